"""CPU oracle of the MoE block forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import
this module. The product path (the CUDA library and its binding) never does.

Two independent fp64 formulations of the same block:

* **O-loop** (``moe_forward``): the C file ``moe_oracle.c`` walks token by token and slot by
  slot: router logits, softmax, top-K, weights, one SwiGLU expert per selected slot,
  identity-expert fold, shared expert. OpenMP over tokens.
* **O-dense** (``moe_forward_dense``): numpy, written separately: every expert runs on every
  token as a dense fp64 matmul and the routing is applied as a [N, E] weight mask. It never
  permutes or gathers, so it also cross-checks the sort/unpermute reading.

Plus the stable expert sort (``sort_by_expert``) that defines the permutation outputs, and
the E4M3 / E2M1 helpers. NVFP4 experts: the C file decodes each E2M1 nibble from its bit
fields, the dense form from a table of the format's eight magnitudes. Citations are to the pages of MoE dispatch code the block is taken from
(see ``moe_oracle.c``'s header).

Parity pins live in ``tests/test_oracle_pins.py``. Parity unpinned: full-size outputs
beyond the agreement of the two formulations and the invariants checked there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_moe.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (fp64, no FP contraction, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp",
                               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Config(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("router_width", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("shared_inter", ctypes.c_int32), ("scoring", ctypes.c_int32),
                ("norm_topk_prob", ctypes.c_int32), ("routed_scaling_factor", ctypes.c_double),
                ("weight_dtype", ctypes.c_int32), ("rms_norm_eps", ctypes.c_double)]


_WEIGHTS = ("router_w", "router_logit_bias", "correction_bias", "w_gate", "w_up", "w_down",
            "s_gate", "s_up", "s_down", "sh_gate", "sh_up", "sh_down", "sh_gate_vec",
            "pre_expert_norm_w", "sf_gate", "sf_up", "sf_down", "scale2_gate", "scale2_up",
            "scale2_down")


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _WEIGHTS]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.orc_moe_forward.restype = ctypes.c_int
            lib.orc_moe_forward.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_Weights)] \
                + [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 9 + [ctypes.c_int]
            lib.orc_e2m1_decode.restype = ctypes.c_double
            lib.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_decode.restype = ctypes.c_double
            lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_e4m3_encode.argtypes = [ctypes.c_double]
            lib.orc_e4m3_encode_array.restype = None
            lib.orc_e4m3_encode_array.argtypes = [ctypes.c_void_p, ctypes.c_long, ctypes.c_void_p]
            lib.orc_quant_1x128.restype = None
            lib.orc_quant_1x128.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_void_p]
            _lib = lib
    return _lib


def _host(t: Optional[torch.Tensor], keep: list):
    """Contiguous CPU copy of ``t`` (kept alive in ``keep``) and its address; bf16 is passed
    as its raw 16-bit pattern."""
    if t is None:
        return None
    t = t.detach().to("cpu").contiguous()
    keep.append(t)
    return t.data_ptr()


def _cfg(shape) -> _Config:
    return _Config(shape.num_tokens, shape.hidden, shape.num_experts, shape.router_width,
                   shape.top_k, shape.inter, shape.shared_inter, shape.scoring,
                   int(shape.norm_topk_prob), float(shape.routed_scaling_factor),
                   shape.weight_dtype, float(shape.rms_norm_eps))


def moe_forward(inp, tokens=None, forced_idx=None, routing_only: bool = False):
    """O-loop forward of the tokens in ``tokens`` (all if None).

    Returns a dict of numpy arrays: ``out`` [n, H] fp64, ``idx`` [n, K] int32, ``w`` [n, K]
    fp64, ``zsum`` [n], ``gap`` [n] (selection-score gap between the K-th and (K+1)-th
    choice), ``gamma`` [n] (shared-expert blend weight), ``sel`` [n, R] (selection score of
    every router column)."""
    lib = _load()
    s = inp.shape
    keep: list = []
    wts = _Weights(*[_host(getattr(inp, n), keep) for n in _WEIGHTS])
    x = _host(inp.x, keep)
    if tokens is None:
        tok = None
        n = s.num_tokens
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        n = len(tok)
    fi = None
    if forced_idx is not None:
        fi = np.ascontiguousarray(np.asarray(forced_idx, dtype=np.int32).reshape(s.num_tokens, s.top_k))
    out = np.zeros((n, s.hidden), dtype=np.float64)
    idx = np.zeros((n, s.top_k), dtype=np.int32)
    w = np.zeros((n, s.top_k), dtype=np.float64)
    zsum = np.zeros(n, dtype=np.float64)
    gap = np.zeros(n, dtype=np.float64)
    gamma = np.zeros(n, dtype=np.float64)
    sel = np.zeros((n, s.router_width), dtype=np.float64)

    def ptr(a):
        return None if a is None else a.ctypes.data

    cfg = _cfg(s)
    rc = lib.orc_moe_forward(ctypes.byref(cfg), ctypes.byref(wts), x, n, ptr(tok), ptr(fi),
                             ptr(out), ptr(idx), ptr(w), ptr(zsum), ptr(gap), ptr(gamma),
                             ptr(sel), int(routing_only))
    if rc != 0:
        raise ValueError("oracle rejected the configuration or token list")
    return {"out": out, "idx": idx, "w": w, "zsum": zsum, "gap": gap, "gamma": gamma,
            "sel": sel}


def e2m1_decode(nibble: int) -> float:
    """The C oracle's decode of one 4-bit E2M1 code."""
    return _load().orc_e2m1_decode(nibble)


def e4m3_decode(code: int) -> float:
    return _load().orc_e4m3_decode(code)


def e4m3_encode(v: float) -> int:
    return _load().orc_e4m3_encode(v)


def e4m3_encode_array(v) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
    codes = np.zeros(v.size, dtype=np.uint8)
    _load().orc_e4m3_encode_array(v.ctypes.data, v.size, codes.ctypes.data)
    return codes.reshape(v.shape)


def quant_1x128(v: np.ndarray):
    """Per-1x128 E4M3 quantisation of fp32 values (decided in fp32). Returns (codes, scales,
    dequantised fp64)."""
    lib = _load()
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    n = v.size
    codes = np.zeros(n, dtype=np.uint8)
    scales = np.zeros(n // 128, dtype=np.float32)
    deq = np.zeros(n, dtype=np.float64)
    lib.orc_quant_1x128(v.ctypes.data, n, codes.ctypes.data, scales.ctypes.data, deq.ctypes.data)
    return codes, scales, deq


# ------------------------------------------------------------------ stable expert sort

def sort_by_expert(idx: np.ndarray, num_experts: int):
    """Counting sort of the (token, slot) pairs by expert id, stable in the flat pair index
    t*K + k ("sort the (row, slot) pairs by expert", forward_prefill.rs, `moe_sort_by_expert`).
    Pairs routed to identity experts (id >= E) take no row.

    Returns ``offsets`` [E+1] (exclusive prefix sum of per-expert counts), ``sorted_pairs``
    [Z] (flat pair index at each sorted row) and ``pair_to_row`` [N*K] (the sorted row of each
    pair, 0xFFFFFFFF for identity-expert pairs)."""
    flat = np.asarray(idx, dtype=np.int64).reshape(-1)
    counts = [0] * num_experts
    for e in flat:
        if e < num_experts:
            counts[e] += 1
    offsets = [0] * (num_experts + 1)
    for e in range(num_experts):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = list(offsets[:-1])
    sorted_pairs = [0] * offsets[-1]
    pair_to_row = [0xFFFFFFFF] * len(flat)
    for pair, e in enumerate(flat):
        if e < num_experts:
            row = fill[e]
            fill[e] += 1
            sorted_pairs[row] = pair
            pair_to_row[pair] = row
    return (np.array(offsets, dtype=np.uint32), np.array(sorted_pairs, dtype=np.uint32),
            np.array(pair_to_row, dtype=np.uint32))


# ------------------------------------------------------------------ O-dense (numpy)

def _f64(t: Optional[torch.Tensor]):
    return None if t is None else t.detach().to("cpu").to(torch.float64).numpy()


def _e4m3_table() -> np.ndarray:
    """All 256 E4M3 code values, from the format's definition (independently of the C file)."""
    tab = np.zeros(256, dtype=np.float64)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            v = np.nan
        elif e == 0:
            v = (m / 8.0) * 2.0 ** -6
        else:
            v = (1.0 + m / 8.0) * 2.0 ** (e - 7)
        tab[c] = -v if s else v
    return tab


def _dequant_blocks(codes: torch.Tensor, scales: torch.Tensor) -> np.ndarray:
    tab = _e4m3_table()
    q = tab[codes.detach().cpu().numpy()]
    s = scales.detach().cpu().numpy().astype(np.float64)
    s = np.repeat(np.repeat(s, 128, axis=-2), 128, axis=-1)
    return q * s


def _quant_rows_np(a: np.ndarray) -> np.ndarray:
    """Per-1x128 quantisation of the rows of ``a`` in fp32, nearest-even to E4M3 by table
    search (numpy restatement, independent of the C file)."""
    tab = _e4m3_table()
    pos = tab[:127]                          # non-negative finite codes 0..126
    a32 = a.astype(np.float32)
    n, m = a32.shape
    g = a32.reshape(n, m // 128, 128)
    amax = np.abs(g).max(axis=-1)
    s = np.where(amax > 0, (amax / np.float32(448.0)).astype(np.float32), np.float32(1.0))
    q = (g / s[..., None]).astype(np.float32).astype(np.float64)
    mag = np.minimum(np.abs(q), 448.0)
    # nearest code; on an exact tie the even code
    d = np.abs(mag[..., None] - pos)
    best = np.argmin(d, axis=-1)
    dmin = np.take_along_axis(d, best[..., None], -1)[..., 0]
    up = np.minimum(best + 1, 126)
    tie = (np.abs(mag - pos[up]) == dmin) & (up != best) & (best % 2 == 1)
    best = np.where(tie, up, best)
    deq = np.sign(q) * pos[best] * s[..., None].astype(np.float64)
    return deq.reshape(n, m)


# E2M1 magnitudes of codes 0..7 as the OCP MX format lists them; bit 3 is the sign.
_E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _dequant_nvfp4(packed: torch.Tensor, sf: torch.Tensor, scale2: torch.Tensor) -> np.ndarray:
    """[E, rows, cols/2] packed E2M1 codes (element 2j in the low nibble), [E, rows, cols/16]
    E4M3 scale codes, fp32 [E] -> fp64 [E, rows, cols]."""
    p = packed.detach().cpu().numpy()
    codes = np.stack([p & 15, p >> 4], axis=-1).reshape(*p.shape[:-1], p.shape[-1] * 2)
    mag = np.asarray(_E2M1_MAGNITUDES)[codes & 7]
    val = np.where(codes >= 8, -mag, mag)
    scal = _e4m3_table()[sf.detach().cpu().numpy().astype(np.int64)]       # [E, rows, cols/16]
    val = val * np.repeat(scal, 16, axis=-1)
    return val * scale2.detach().cpu().double().numpy()[:, None, None]


def moe_forward_dense(inp, forced_idx=None):
    """O-dense: every expert on every token (fp64 matmuls), masked by the routing.
    Returns dict with ``out`` [N,H], ``idx`` [N,K], ``w`` [N,K]."""
    s = inp.shape
    N, E, R, K = s.num_tokens, s.num_experts, s.router_width, s.top_k
    x = _f64(inp.x)
    L = x @ _f64(inp.router_w).T
    if inp.router_logit_bias is not None:
        L = L + _f64(inp.router_logit_bias)[None, :]
    if s.scoring == 2:                     # sigmoid arm: each column scored on its own
        p = 0.5 * (1.0 + np.tanh(0.5 * L))   # = 1 / (1 + e^-L), written differently
    else:
        L = L - L.max(axis=1, keepdims=True)
        p = np.exp(L)
        p = p / p.sum(axis=1, keepdims=True)
    sel = p.copy()
    if s.scoring in (1, 2) and inp.correction_bias is not None:
        sel = sel + _f64(inp.correction_bias)[None, :]
    # K best by (score desc, index asc): lexsort with the index as the secondary key
    order = np.lexsort((np.broadcast_to(np.arange(R), sel.shape), -sel), axis=1)
    idx = order[:, :K] if forced_idx is None else np.asarray(forced_idx).reshape(N, K)
    w = np.take_along_axis(p, idx, axis=1)
    if s.norm_topk_prob:
        w = w / w.sum(axis=1, keepdims=True)
    w = w * s.routed_scaling_factor
    # dense [N, R] routing weight matrix
    M = np.zeros((N, R))
    for k in range(K):
        M[np.arange(N), idx[:, k]] += w[:, k]
    xr = x                                  # routed experts' input
    if inp.pre_expert_norm_w is not None:   # RMSNorm, stored as bf16 like the pages' buffer
        rms = np.sqrt(np.mean(x * x, axis=1, keepdims=True) + s.rms_norm_eps)
        xr = x / rms * _f64(inp.pre_expert_norm_w)[None, :]
        xr = torch.from_numpy(xr).to(torch.float32).to(torch.bfloat16).double().numpy()
    if s.weight_dtype == 1:
        Wg = _dequant_blocks(inp.w_gate, inp.s_gate)
        Wu = _dequant_blocks(inp.w_up, inp.s_up)
        Wd = _dequant_blocks(inp.w_down, inp.s_down)
        xe = _quant_rows_np(xr)
    elif s.weight_dtype == 2:
        Wg = _dequant_nvfp4(inp.w_gate, inp.sf_gate, inp.scale2_gate)
        Wu = _dequant_nvfp4(inp.w_up, inp.sf_up, inp.scale2_up)
        Wd = _dequant_nvfp4(inp.w_down, inp.sf_down, inp.scale2_down)
        xe = xr
    else:
        Wg, Wu, Wd = _f64(inp.w_gate), _f64(inp.w_up), _f64(inp.w_down)
        xe = xr
    out = np.zeros_like(x)
    for e in range(E):
        if not M[:, e].any():
            continue
        g = xe @ Wg[e].T
        u = xe @ Wu[e].T
        h = g / (1.0 + np.exp(-g)) * u
        if s.weight_dtype == 1:
            h = _quant_rows_np(h)
        out += M[:, e:e + 1] * (h @ Wd[e].T)
    out += M[:, E:].sum(axis=1, keepdims=True) * x
    if s.shared_inter > 0:
        g = x @ _f64(inp.sh_gate).T
        u = x @ _f64(inp.sh_up).T
        sh = (g / (1.0 + np.exp(-g)) * u) @ _f64(inp.sh_down).T
        gamma = np.ones((N, 1))
        if inp.sh_gate_vec is not None:
            gamma = 1.0 / (1.0 + np.exp(-(x @ _f64(inp.sh_gate_vec))))[:, None]
        out += gamma * sh
    return {"out": out, "idx": idx.astype(np.int32), "w": w}
