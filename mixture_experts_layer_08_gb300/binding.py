"""ctypes binding of the C ABI in ``include/moe.h``.

Argument marshalling only: every step of the forward runs in the CUDA library. Importing
this module loads ``_build/libmoe_gb300.so`` and fails loudly if it has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import inputs as _inputs

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE_TOO_SMALL = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_TIMEOUT = 5

PATH_AUTO, PATH_DECODE, PATH_GROUPED = 0, 1, 2


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        detail = ""
        if status == MOE_ERR_CUDA:
            detail = " -- " + _lib.moe_last_error_detail().decode()
        super().__init__(f"{what}: {moe_status_string(status)} (status {status}){detail}")
        self.status = status


class moe_config_t(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("router_width", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("shared_inter", ctypes.c_int32), ("scoring", ctypes.c_int32),
                ("norm_topk_prob", ctypes.c_int32), ("routed_scaling_factor", ctypes.c_float),
                ("weight_dtype", ctypes.c_int32), ("deterministic", ctypes.c_int32),
                ("path", ctypes.c_int32), ("pre_expert_norm", ctypes.c_int32),
                ("rms_norm_eps", ctypes.c_float)]


_WEIGHT_FIELDS = ("router_w", "router_logit_bias", "correction_bias", "w_gate", "w_up", "w_down",
                  "s_gate", "s_up", "s_down", "sh_gate", "sh_up", "sh_down", "sh_gate_vec",
                  "pre_expert_norm_w", "sf_gate", "sf_up", "sf_down", "scale2_gate",
                  "scale2_up", "scale2_down")


class moe_weights_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _WEIGHT_FIELDS]


if not os.path.exists(_LIB_PATH):
    raise ImportError(f"CUDA library not built: {_LIB_PATH} is missing "
                      "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
_lib = ctypes.CDLL(_LIB_PATH)
_vp = ctypes.c_void_p
_lib.moe_workspace_size.restype = ctypes.c_int
_lib.moe_workspace_size.argtypes = [ctypes.POINTER(moe_config_t), ctypes.POINTER(ctypes.c_size_t)]
_lib.moe_forward.restype = ctypes.c_int
_lib.moe_forward.argtypes = [ctypes.POINTER(moe_config_t), ctypes.POINTER(moe_weights_t), _vp, _vp,
                             _vp, ctypes.c_size_t, _vp, _vp, _vp, _vp]
_lib.moe_forward_profiled.restype = ctypes.c_int
_lib.moe_forward_profiled.argtypes = [ctypes.POINTER(moe_config_t), ctypes.POINTER(moe_weights_t),
                                      _vp, _vp, _vp, ctypes.c_size_t, _vp,
                                      ctypes.POINTER(ctypes.c_void_p)]
_lib.moe_route.restype = ctypes.c_int
_lib.moe_route.argtypes = [ctypes.POINTER(moe_config_t), ctypes.POINTER(moe_weights_t), _vp, _vp,
                           ctypes.c_size_t, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
_lib.moe_read_device_status.restype = ctypes.c_int
_lib.moe_read_device_status.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_int32)]
_lib.moe_selftest_bounded_wait.restype = ctypes.c_int
_lib.moe_selftest_bounded_wait.argtypes = [_vp, ctypes.c_longlong, _vp]
_lib.moe_last_error_detail.restype = ctypes.c_char_p
_lib.moe_last_error_detail.argtypes = []
_lib.moe_status_string.restype = ctypes.c_char_p
_lib.moe_status_string.argtypes = [ctypes.c_int]

LIB_PATH = _LIB_PATH
lib = _lib


def moe_status_string(status: int) -> str:
    return _lib.moe_status_string(status).decode()


def make_config(shape: "_inputs.MoeShape", deterministic: bool = True,
                path: int = PATH_AUTO) -> moe_config_t:
    return moe_config_t(shape.num_tokens, shape.hidden, shape.num_experts, shape.router_width,
                        shape.top_k, shape.inter, shape.shared_inter, shape.scoring,
                        int(shape.norm_topk_prob), float(shape.routed_scaling_factor),
                        shape.weight_dtype, int(deterministic), path,
                        int(shape.pre_expert_norm), float(shape.rms_norm_eps))


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return t.data_ptr()


def make_weights(inp: "_inputs.MoeInputs") -> moe_weights_t:
    return moe_weights_t(*[_ptr(getattr(inp, n)) for n in _WEIGHT_FIELDS])


def moe_workspace_size(cfg: moe_config_t) -> int:
    n = ctypes.c_size_t(0)
    st = _lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n))
    if st != MOE_OK:
        raise MoeError(st, "moe_workspace_size")
    return n.value


def alloc_workspace(cfg: moe_config_t, device="cuda") -> torch.Tensor:
    return torch.empty(max(moe_workspace_size(cfg), 256), dtype=torch.uint8, device=device)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def moe_forward(cfg: moe_config_t, weights: moe_weights_t, x: torch.Tensor, out: torch.Tensor,
                workspace: torch.Tensor, stream=None, topk_idx_out=None, topk_w_out=None,
                forced_idx=None, check: bool = True) -> int:
    st = _lib.moe_forward(ctypes.byref(cfg), ctypes.byref(weights), _ptr(x), _ptr(out),
                          _ptr(workspace), workspace.numel(), _stream(stream), _ptr(topk_idx_out),
                          _ptr(topk_w_out), _ptr(forced_idx))
    if check and st != MOE_OK:
        raise MoeError(st, "moe_forward")
    return st


STAGES = ("route", "shared", "gate_up", "down", "combine")


def moe_forward_profiled(cfg: moe_config_t, weights: moe_weights_t, x: torch.Tensor,
                         out: torch.Tensor, workspace: torch.Tensor, events, stream=None) -> int:
    """``events``: 2 * len(STAGES) torch.cuda.Event objects (start/end per stage, None to
    skip), recorded on ``stream`` around each stage."""
    arr = (ctypes.c_void_p * (2 * len(STAGES)))(
        *[None if e is None else e.cuda_event for e in events])
    st = _lib.moe_forward_profiled(ctypes.byref(cfg), ctypes.byref(weights), _ptr(x), _ptr(out),
                                   _ptr(workspace), workspace.numel(), _stream(stream), arr)
    if st != MOE_OK:
        raise MoeError(st, "moe_forward_profiled")
    return st


def moe_route(cfg: moe_config_t, weights: moe_weights_t, x: torch.Tensor,
              workspace: torch.Tensor, stream=None, idx_out=None, w_out=None, zsum_out=None,
              offsets_out=None, sorted_pairs_out=None, pair_to_row_out=None,
              check: bool = True) -> int:
    st = _lib.moe_route(ctypes.byref(cfg), ctypes.byref(weights), _ptr(x), _ptr(workspace),
                        workspace.numel(), _stream(stream), _ptr(idx_out), _ptr(w_out),
                        _ptr(zsum_out), _ptr(offsets_out), _ptr(sorted_pairs_out),
                        _ptr(pair_to_row_out))
    if check and st != MOE_OK:
        raise MoeError(st, "moe_route")
    return st


def moe_read_device_status(workspace: torch.Tensor, stream=None) -> int:
    v = ctypes.c_int32(-1)
    st = _lib.moe_read_device_status(_ptr(workspace), _stream(stream), ctypes.byref(v))
    if st != MOE_OK:
        raise MoeError(st, "moe_read_device_status")
    return v.value


def moe_selftest_bounded_wait(workspace: torch.Tensor, limit_cycles: int, stream=None) -> int:
    st = _lib.moe_selftest_bounded_wait(_ptr(workspace), int(limit_cycles), _stream(stream))
    if st != MOE_OK:
        raise MoeError(st, "moe_selftest_bounded_wait")
    return st


class MoeBlock:
    """Convenience holder: config + device weights + workspace, one forward per call."""

    def __init__(self, inp: "_inputs.MoeInputs", deterministic: bool = True,
                 path: int = PATH_AUTO):
        self.inputs = inp
        self.cfg = make_config(inp.shape, deterministic, path)
        self.weights = make_weights(inp)
        self.workspace = alloc_workspace(self.cfg, inp.x.device)

    def __call__(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None,
                 topk_idx_out=None, topk_w_out=None, forced_idx=None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(x)
        moe_forward(self.cfg, self.weights, x, out, self.workspace, stream, topk_idx_out,
                    topk_w_out, forced_idx)
        return out
