"""Seeded synthetic MoE workloads.

This module only draws random tensors: it holds none of the MoE block's arithmetic, so
both the CUDA path and the CPU oracle may take their inputs from it.

Generation recipe (one ``torch.Generator`` per tensor, seeded ``seed * 1000 + tensor_id``,
in the fixed order x, Wr, Wg, Wu, Wd, Sg, Su, Sd, g, bias):

* activations ``x ~ N(0, 1)``, all weight matrices ``~ N(0, 0.02)``, drawn in fp32 and
  rounded to bf16;
* skewed prefill: a per-expert additive router-logit offset ``-s * ln(rank_e)`` with
  ``rank`` a seeded permutation of ``1..E`` and ``s = 1.1`` (Zipf), shifted to mean 0;
* zero-computation experts: a selection-only correction bias ``~ N(0, 0.1)`` (fp32);
* FP8 experts: weights are handed to the layer already quantised to E4M3 with one fp32
  scale per 128x128 block (``scale = amax / 448``, 1 where the block is all zero); the
  rounding to E4M3 is done by ``torch``'s own cast, so neither the kernels nor the oracle
  supply it.
* NVFP4 experts: the packed representation is drawn directly (no quantiser): each 4-bit
  E2M1 code has a uniform sign bit and a magnitude index 0..7 from the fixed categorical
  distribution ``NVFP4_MAG_PROBS``; every 16 consecutive elements along the contraction
  share one E4M3 scale code drawn uniformly from 0x30..0x3F (the E4M3 values in [0.5, 2));
  each expert matrix has one fp32 ``scale2 = 0.007 * (1 + 0.1 * N(0, 1))``, which puts the
  weights near the ``N(0, 0.02)`` magnitude of the bf16 experts. Codes are packed two per
  byte, element ``2j`` in the low nibble and ``2j + 1`` in the high nibble.

Weight layout is ``[out_features, in_features]`` (K-contiguous): gate/up ``[E, I, H]``,
down ``[E, H, I]``, shared gate/up ``[S, H]``, shared down ``[H, S]``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

SCORING_SOFTMAX = 0
SCORING_SOFTMAX_BIAS = 1
SCORING_SIGMOID_BIAS = 2

WDTYPE_BF16 = 0
WDTYPE_FP8_E4M3_B128 = 1
WDTYPE_NVFP4 = 2

# probabilities of the E2M1 magnitude indices 0..7 of the drawn NVFP4 codes
NVFP4_MAG_PROBS = (0.10, 0.16, 0.18, 0.16, 0.14, 0.14, 0.08, 0.04)

_TENSOR_IDS = {"x": 0, "router_w": 1, "w_gate": 2, "w_up": 3, "w_down": 4,
               "sh_gate": 5, "sh_up": 6, "sh_down": 7, "sh_gate_vec": 8, "bias": 9,
               "norm_w": 10, "sf_gate": 11, "sf_up": 12, "sf_down": 13, "scale2": 14}


@dataclasses.dataclass(frozen=True)
class MoeShape:
    """Sizes and routing options of one MoE block forward."""
    name: str
    num_tokens: int            # N
    hidden: int                # H
    num_experts: int           # E (SwiGLU experts)
    router_width: int          # R >= E; ids E..R-1 are identity (zero-computation) experts
    top_k: int                 # K
    inter: int                 # I
    shared_inter: int = 0      # S (0: no shared expert)
    shared_gated: bool = False  # sigmoid(x . g) blend weight for the shared expert
    scoring: int = SCORING_SOFTMAX
    norm_topk_prob: bool = True
    routed_scaling_factor: float = 1.0
    weight_dtype: int = WDTYPE_BF16
    zipf_s: float = 0.0        # >0: skewed per-expert router-logit offsets
    correction_bias_std: float = 0.0  # >0 with the *_BIAS scorings
    pre_expert_norm: bool = False     # RMSNorm of the routed experts' input (weight ~ 1 + N(0, 0.1))
    rms_norm_eps: float = 1e-6
    seed: int = 0

    def with_(self, **kw) -> "MoeShape":
        return dataclasses.replace(self, **kw)

    @property
    def te(self) -> int:
        return self.num_tokens * self.top_k


# The five workloads the layer is measured and checked on.
TINY = MoeShape("tiny_bf16_n16", 16, 256, 8, 8, 2, 128, shared_inter=256)
DECODE = MoeShape("decode_bf16_n4", 4, 2048, 128, 128, 8, 768, shared_inter=512,
                  shared_gated=True)
PREFILL = MoeShape("prefill_zipf_bf16_n4096", 4096, 2048, 128, 128, 8, 768,
                   shared_inter=512, zipf_s=1.1)
ZERO_EXPERT = MoeShape("zero_expert_bf16_n1024", 1024, 2048, 256, 384, 8, 1024,
                       scoring=SCORING_SOFTMAX_BIAS, correction_bias_std=0.1)
FP8_PREFILL = MoeShape("fp8_prefill_n8192", 8192, 4096, 128, 128, 8, 1536,
                       weight_dtype=WDTYPE_FP8_E4M3_B128)

# The decode workload with a pre-expert RMSNorm of the routed experts' input, and with E4M3
# routed experts (128x128 block scales; the shared expert stays bf16).
DECODE_PRENORM = DECODE.with_(name="decode_prenorm_bf16_n4", pre_expert_norm=True)
DECODE_FP8 = DECODE.with_(name="decode_fp8_n4", weight_dtype=WDTYPE_FP8_E4M3_B128)
# NVFP4 routed experts (E2M1 + E4M3 scale per 16 + fp32 scale per expert matrix) on the
# decode and prefill shapes
DECODE_NVFP4 = DECODE.with_(name="decode_nvfp4_n4", weight_dtype=WDTYPE_NVFP4)
PREFILL_NVFP4 = PREFILL.with_(name="prefill_nvfp4_n4096", weight_dtype=WDTYPE_NVFP4)

WORKLOADS = {s.name: s for s in (TINY, DECODE, PREFILL, ZERO_EXPERT, FP8_PREFILL, DECODE_PRENORM,
                                 DECODE_FP8, DECODE_NVFP4, PREFILL_NVFP4)}


def _gen(shape: MoeShape, key: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(shape.seed * 1000 + _TENSOR_IDS[key])
    return g


def _randn(shape: MoeShape, key: str, size, std: float, device) -> torch.Tensor:
    t = torch.randn(*size, generator=_gen(shape, key, device), device=device,
                    dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def quantize_weight_e4m3_b128(w: torch.Tensor):
    """Quantise ``[..., rows, cols]`` fp32 weights to E4M3 with one fp32 scale per 128x128
    block. Returns (codes as uint8 view of float8_e4m3fn, scales ``[..., rows/128, cols/128]``).
    Uses torch's float8 cast for the rounding (input preparation, not part of the layer)."""
    *lead, rows, cols = w.shape
    assert rows % 128 == 0 and cols % 128 == 0
    blk = w.reshape(*lead, rows // 128, 128, cols // 128, 128)
    amax = blk.abs().amax(dim=(-3, -1))                       # [..., rows/128, cols/128]
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (blk / scale[..., :, None, :, None]).clamp_(-448.0, 448.0)
    q8 = q.reshape(*lead, rows, cols).to(torch.float8_e4m3fn)
    return q8.view(torch.uint8), scale.to(torch.float32).contiguous()


def draw_nvfp4(shape: "MoeShape", key: str, size, device):
    """Draw a packed NVFP4 matrix ``[E, rows, cols]`` (see the module docstring): returns
    (codes uint8 ``[E, rows, cols/2]``, E4M3 scale codes uint8 ``[E, rows, cols/16]``)."""
    E, rows, cols = size
    assert cols % 16 == 0
    g = _gen(shape, key, device)
    cum = torch.tensor(NVFP4_MAG_PROBS, dtype=torch.float64).cumsum(0)[:-1]
    cum = cum.to(device=device, dtype=torch.float32)
    packed = torch.empty(E, rows, cols // 2, dtype=torch.uint8, device=device)
    for e in range(E):   # one expert at a time keeps the temporaries small
        u = torch.rand(rows, cols, generator=g, device=device)
        neg = u >= 0.5
        mag = torch.bucketize((u - 0.5 * neg.float()) * 2.0, cum, right=True)
        code = (mag | (neg.to(torch.int64) << 3)).to(torch.uint8)
        packed[e] = code[:, 0::2] | (code[:, 1::2] << 4)
    sf = torch.randint(0x30, 0x40, (E, rows, cols // 16), generator=_gen(shape, "sf_" + key[2:],
                       device), device=device, dtype=torch.int64).to(torch.uint8)
    return packed, sf


@dataclasses.dataclass
class MoeInputs:
    """All tensors of one forward. bf16 tensors are torch.bfloat16; FP8 weights are uint8
    E4M3 codes with fp32 block scales."""
    shape: MoeShape
    x: torch.Tensor
    router_w: torch.Tensor
    w_gate: torch.Tensor
    w_up: torch.Tensor
    w_down: torch.Tensor
    s_gate: Optional[torch.Tensor] = None
    s_up: Optional[torch.Tensor] = None
    s_down: Optional[torch.Tensor] = None
    sf_gate: Optional[torch.Tensor] = None     # NVFP4: E4M3 scale codes per 16 elements
    sf_up: Optional[torch.Tensor] = None
    sf_down: Optional[torch.Tensor] = None
    scale2_gate: Optional[torch.Tensor] = None  # NVFP4: fp32 [E] per expert matrix
    scale2_up: Optional[torch.Tensor] = None
    scale2_down: Optional[torch.Tensor] = None
    sh_gate: Optional[torch.Tensor] = None
    sh_up: Optional[torch.Tensor] = None
    sh_down: Optional[torch.Tensor] = None
    sh_gate_vec: Optional[torch.Tensor] = None
    router_logit_bias: Optional[torch.Tensor] = None
    correction_bias: Optional[torch.Tensor] = None
    pre_expert_norm_w: Optional[torch.Tensor] = None

    def tensors(self):
        return {k: v for k, v in dataclasses.asdict(self).items()
                if isinstance(v, torch.Tensor)}

    def to(self, device) -> "MoeInputs":
        kw = {k: (v.to(device) if isinstance(v, torch.Tensor) else v)
              for k, v in self.__dict__.items()}
        return MoeInputs(**kw)


def make_inputs(shape: MoeShape, device="cpu", x_only_tokens: Optional[int] = None) -> MoeInputs:
    """Draw every tensor of ``shape`` on ``device`` (a CPU or CUDA generator; the two give
    different but equally seeded values)."""
    N, H, E, R, I, S = (shape.num_tokens, shape.hidden, shape.num_experts,
                        shape.router_width, shape.inter, shape.shared_inter)
    bf = torch.bfloat16
    x = _randn(shape, "x", (N, H), 1.0, device).to(bf)
    router_w = _randn(shape, "router_w", (R, H), 0.02, device).to(bf)
    out = {}
    for key, size in (("w_gate", (E, I, H)), ("w_up", (E, I, H)), ("w_down", (E, H, I))):
        if shape.weight_dtype == WDTYPE_NVFP4:
            out[key], out["sf_" + key[2:]] = draw_nvfp4(shape, key, size, device)
            continue
        w = _randn(shape, key, size, 0.02, device)
        if shape.weight_dtype == WDTYPE_FP8_E4M3_B128:
            q, s = quantize_weight_e4m3_b128(w)
            out[key] = q
            out["s_" + key[2:]] = s
        else:
            out[key] = w.to(bf)
        del w
    if shape.weight_dtype == WDTYPE_NVFP4:
        s2 = 0.007 * (1.0 + 0.1 * _randn(shape, "scale2", (3, E), 1.0, device))
        out["scale2_gate"], out["scale2_up"], out["scale2_down"] = (s2[0].contiguous(),
                                                                    s2[1].contiguous(),
                                                                    s2[2].contiguous())
    sh = {}
    if S > 0:
        sh["sh_gate"] = _randn(shape, "sh_gate", (S, H), 0.02, device).to(bf)
        sh["sh_up"] = _randn(shape, "sh_up", (S, H), 0.02, device).to(bf)
        sh["sh_down"] = _randn(shape, "sh_down", (H, S), 0.02, device).to(bf)
        if shape.shared_gated:
            sh["sh_gate_vec"] = _randn(shape, "sh_gate_vec", (H,), 0.02, device).to(bf)
    rlb = None
    cb = None
    if shape.zipf_s > 0:
        perm = torch.randperm(E, generator=_gen(shape, "bias", "cpu"))
        rank = (perm + 1).to(torch.float64)
        b = -shape.zipf_s * torch.log(rank)
        b = b - b.mean()
        rlb = torch.zeros(R, dtype=torch.float64)
        rlb[:E] = b
        rlb = rlb.to(torch.float32).to(device)
    if shape.correction_bias_std > 0:
        cb = _randn(shape, "bias", (R,), shape.correction_bias_std, device)
    nw = None
    if shape.pre_expert_norm:
        nw = (1.0 + _randn(shape, "norm_w", (H,), 0.1, device)).to(bf)
    return MoeInputs(shape=shape, x=x, router_w=router_w, **out, **sh,
                     router_logit_bias=rlb, correction_bias=cb, pre_expert_norm_w=nw)


def l2_flush_bytes() -> int:
    """Bytes written between timed iterations so no input stays in the 126.5 MiB L2."""
    return 512 * 1024 * 1024


def zipf_expected_share(E: int, s: float) -> list:
    """Expected routing share per rank under a pure Zipf(s) prior (for reporting only)."""
    z = [r ** (-s) for r in range(1, E + 1)]
    tot = math.fsum(z)
    return [v / tot for v in z]
