"""CUDA path vs the CPU oracle, through the C ABI (GPU only).

Bars (element by element):
  * routing: top-K index sets exact on every token whose K-th and (K+1)-th selection scores
    differ by more than 1e-3; weights within 1e-5 relative; sort outputs bit-exact;
  * bf16 experts: |out - ref| <= 2e-2 + 2e-2 |ref| per element, and -- because expert outputs
    here are ~0.1 in magnitude, where that absolute term alone would hide real errors -- a
    relative L2 error <= 1e-2 over the whole output.
The output reference is the oracle run with the GPU's own index set (`forced_idx`), so
near-tie tokens whose selection legitimately differs are still checked.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_08_gb300 import inputs as I
from oracle import oracle as O

pytestmark = pytest.mark.gpu

TIE_GAP = 1e-3
ATOL, RTOL, REL_L2 = 2e-2, 2e-2, 1e-2


@pytest.fixture(scope="module")
def B():
    from mixture_experts_layer_08_gb300 import build as _b
    _b.build()
    from mixture_experts_layer_08_gb300 import binding
    assert torch.cuda.is_available()
    return binding


# ------------------------------------------------------------------ workloads

# Reduced copies of the five workloads: several tiles and ragged per-expert tails, small
# enough for the full oracle.
SMALL = {
    "tiny": I.TINY,
    "decode": I.DECODE,
    "prefill_zipf_small": I.PREFILL.with_(name="prefill_zipf_small", num_tokens=300, hidden=512,
                                          num_experts=16, router_width=16, top_k=4, inter=256,
                                          shared_inter=256),
    "zero_expert_small": I.ZERO_EXPERT.with_(name="zero_expert_small", num_tokens=200,
                                             hidden=512, num_experts=32, router_width=48,
                                             top_k=8, inter=256),
    "wide_small": I.PREFILL.with_(name="wide_small", num_tokens=1000, hidden=1024,
                                  num_experts=8, router_width=8, top_k=2, inter=384,
                                  shared_inter=128, zipf_s=0.0, shared_gated=True),
    # decode-sized batches on both chains: identity experts and a router wider than 256 columns
    # (the fused decode kernel's arg-max-rounds top-K), 128-row weight tiles (H, I, S not
    # multiples of 256), a full 16-token batch
    "zero_expert_decode": I.ZERO_EXPERT.with_(name="zero_expert_decode", num_tokens=9,
                                              hidden=512, num_experts=256, router_width=384,
                                              top_k=8, inter=256),
    "odd_tiles_decode": I.DECODE.with_(name="odd_tiles_decode", num_tokens=16, hidden=384,
                                       num_experts=24, router_width=24, top_k=3, inter=384,
                                       shared_inter=128),
    # sigmoid + correction-bias scoring: 32 routed pairs (the decode kernel's split routing),
    # a router wider than 256 columns (arg-max rounds), and a grouped-chain batch
    "sigmoid_bias_decode": I.DECODE.with_(name="sigmoid_bias_decode", hidden=512,
                                          num_experts=64, router_width=64, inter=256,
                                          shared_inter=256, scoring=I.SCORING_SIGMOID_BIAS,
                                          correction_bias_std=0.05, routed_scaling_factor=2.5),
    "sigmoid_wide_decode": I.DECODE.with_(name="sigmoid_wide_decode", num_tokens=3, hidden=256,
                                          num_experts=320, router_width=320, top_k=4,
                                          inter=128, shared_inter=0, shared_gated=False,
                                          scoring=I.SCORING_SIGMOID_BIAS,
                                          correction_bias_std=0.05, norm_topk_prob=False),
    # pre-expert RMSNorm of the routed experts' input (router and shared expert read raw x)
    "prenorm_decode": I.DECODE.with_(name="prenorm_decode", hidden=512, num_experts=64,
                                     router_width=64, inter=256, shared_inter=256,
                                     pre_expert_norm=True),
    "prenorm_grouped": I.PREFILL.with_(name="prenorm_grouped", num_tokens=300, hidden=512,
                                       num_experts=16, router_width=16, top_k=4, inter=256,
                                       shared_inter=256, shared_gated=True,
                                       pre_expert_norm=True),
    # the fused tensor-core router (N > 64, R a multiple of 32): a ragged last token tile,
    # R > 256 (two MMAs per K step) with identity experts and the correction bias
    "fused_router_wide": I.ZERO_EXPERT.with_(name="fused_router_wide", num_tokens=300,
                                             hidden=1024, num_experts=256, router_width=384,
                                             top_k=8, inter=128),
    "fused_router_narrow": I.PREFILL.with_(name="fused_router_narrow", num_tokens=333,
                                           hidden=768, num_experts=64, router_width=64,
                                           top_k=6, inter=256, shared_inter=128,
                                           shared_gated=True),
    # K > 8: the fused router's K rounds of arg-max instead of its sorting networks
    "fused_router_k12": I.PREFILL.with_(name="fused_router_k12", num_tokens=130, hidden=512,
                                        num_experts=64, router_width=64, top_k=12, inter=128,
                                        shared_inter=0, zipf_s=0.0),
    "sigmoid_bias_small": I.PREFILL.with_(name="sigmoid_bias_small", num_tokens=200,
                                          hidden=512, num_experts=32, router_width=32,
                                          top_k=6, inter=256, shared_inter=0, zipf_s=0.0,
                                          scoring=I.SCORING_SIGMOID_BIAS,
                                          correction_bias_std=0.05, norm_topk_prob=False,
                                          routed_scaling_factor=1.5),
}


def run_gpu(B, inp, path=0, deterministic=True, forced=None):
    dev = inp.to("cuda")
    cfg = B.make_config(inp.shape, deterministic, path)
    w = B.make_weights(dev)
    ws = B.alloc_workspace(cfg)
    N, K = inp.shape.num_tokens, inp.shape.top_k
    out = torch.empty_like(dev.x)
    idx = torch.empty(N, K, dtype=torch.int32, device="cuda")
    wt = torch.empty(N, K, dtype=torch.float32, device="cuda")
    f = None if forced is None else torch.as_tensor(forced, dtype=torch.int32, device="cuda")
    B.moe_forward(cfg, w, dev.x, out, ws, None, idx, wt, f)
    torch.cuda.synchronize()
    assert B.moe_read_device_status(ws) == B.MOE_OK
    return out.float().cpu().numpy(), idx.cpu().numpy(), wt.cpu().numpy()


def check_routing(gpu_idx, ref, eps=1e-5):
    """Index sets equal the oracle's on every token whose K-th/(K+1)-th selection-score gap
    exceeds 1e-3; on every token, the GPU's set is a valid top-K of the oracle's fp64 scores
    (each chosen score >= each unchosen score - eps, eps >> the fp32-vs-fp64 score error).
    Returns the number of near-tie tokens."""
    far = ref["gap"] > TIE_GAP
    np.testing.assert_array_equal(gpu_idx[far], ref["idx"][far])
    sel = ref["sel"]
    n, R = sel.shape
    chosen = np.zeros((n, R), dtype=bool)
    np.put_along_axis(chosen, gpu_idx.astype(np.int64), True, axis=1)
    assert (chosen.sum(axis=1) == gpu_idx.shape[1]).all(), "repeated expert id in a token"
    lo = np.where(chosen, sel, np.inf).min(axis=1)
    hi = np.where(chosen, -np.inf, sel).max(axis=1)
    bad = lo < hi - eps
    assert not bad.any(), f"{bad.sum()} tokens with an invalid top-K selection"
    return int((~far).sum())


def check_out(got, ref, atol=ATOL, rtol=RTOL, rel_l2=REL_L2):
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), f"{bad.sum()} elements out of tolerance, max err {err.max():.3e}"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= rel_l2, f"relative L2 error {rel:.3e}"
    return rel


# ------------------------------------------------------------------ routing

@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("path", [1, 2], ids=["decode", "grouped"])
def test_route_matches_oracle(B, name, path):
    shape = SMALL[name]
    if path == 1 and shape.num_tokens > 16:
        pytest.skip("decode chain is for <= 16 tokens")
    inp = I.make_inputs(shape)
    dev = inp.to("cuda")
    cfg = B.make_config(shape, True, path)
    ws = B.alloc_workspace(cfg)
    N, K, E = shape.num_tokens, shape.top_k, shape.num_experts
    idx = torch.empty(N, K, dtype=torch.int32, device="cuda")
    wt = torch.empty(N, K, dtype=torch.float32, device="cuda")
    zs = torch.empty(N, dtype=torch.float32, device="cuda")
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    spairs = torch.empty(N * K, dtype=torch.int32, device="cuda")
    p2r = torch.empty(N * K, dtype=torch.int32, device="cuda")
    B.moe_route(cfg, B.make_weights(dev), dev.x, ws, None, idx, wt, zs, offs, spairs, p2r)
    torch.cuda.synchronize()
    ref = O.moe_forward(inp, routing_only=True)
    gi = idx.cpu().numpy()
    check_routing(gi, ref)
    far = ref["gap"] > TIE_GAP
    np.testing.assert_allclose(wt.cpu().numpy()[far], ref["w"][far], rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(zs.cpu().numpy()[far], ref["zsum"][far], rtol=1e-5, atol=1e-7)
    # the sort is integer work: bit-exact against the oracle's stable sort of the GPU's ids
    o_off, o_pairs, o_p2r = O.sort_by_expert(gi, E)
    np.testing.assert_array_equal(offs.cpu().numpy().view(np.uint32), o_off)
    Z = int(o_off[-1])
    np.testing.assert_array_equal(spairs.cpu().numpy().view(np.uint32)[:Z], o_pairs)
    np.testing.assert_array_equal(p2r.cpu().numpy().view(np.uint32), o_p2r)


@pytest.mark.parametrize("name", ["fused_router_wide", "fused_router_narrow",
                                  "fused_router_k12", "sigmoid_bias_small"])
def test_fused_router_is_repeatable(B, name):
    """The tensor-core router with the top-K fused (N > 64, R a multiple of 32) splits each
    token tile's contraction over a cluster of CTAs and combines the partial sums through
    distributed shared memory in a fixed order: 12 launches give bit-identical ids, weights
    and zsum, each a valid routing against the oracle."""
    shape = SMALL[name]
    inp = I.make_inputs(shape)
    dev = inp.to("cuda")
    cfg = B.make_config(shape, True, 2)
    ws = B.alloc_workspace(cfg)
    w = B.make_weights(dev)
    N, K, E = shape.num_tokens, shape.top_k, shape.num_experts
    ref = O.moe_forward(inp, routing_only=True)
    far = ref["gap"] > TIE_GAP
    first = None
    for _ in range(12):
        idx = torch.empty(N, K, dtype=torch.int32, device="cuda")
        wt = torch.empty(N, K, dtype=torch.float32, device="cuda")
        zs = torch.empty(N, dtype=torch.float32, device="cuda")
        offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
        spairs = torch.empty(N * K, dtype=torch.int32, device="cuda")
        p2r = torch.empty(N * K, dtype=torch.int32, device="cuda")
        B.moe_route(cfg, w, dev.x, ws, None, idx, wt, zs, offs, spairs, p2r)
        torch.cuda.synchronize()
        got = (idx.cpu().numpy(), wt.cpu().numpy(), zs.cpu().numpy())
        check_routing(got[0], ref)
        np.testing.assert_allclose(got[1][far], ref["w"][far], rtol=1e-5, atol=1e-7)
        if first is None:
            first = got
        else:
            for a, b in zip(first, got):
                np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))


# ------------------------------------------------------------------ whole forward

@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("path", [0, 1, 2], ids=["auto", "decode", "grouped"])
def test_forward_matches_oracle(B, name, path):
    shape = SMALL[name]
    if path == 1 and shape.num_tokens > 16:
        pytest.skip("decode chain is for <= 16 tokens")
    inp = I.make_inputs(shape)
    got, gidx, gw = run_gpu(B, inp, path)
    ref_sel = O.moe_forward(inp, routing_only=True)
    check_routing(gidx, ref_sel)
    ref = O.moe_forward(inp, forced_idx=gidx)
    np.testing.assert_allclose(gw, ref["w"], rtol=1e-5, atol=1e-7)
    check_out(got, ref["out"])


def _assert_identity_exact(got, x, w):
    """Token by token: out[t] == bf16(z * x[t]) bit for bit, for one fp32 z -- the kernel's own
    sum of the token's K identity-expert weights, which may add them in another order than
    numpy: z is searched within 8 fp32 ulps of numpy's sum."""
    xf = x.float()
    for t in range(got.shape[0]):
        z0 = np.float32(w[t].astype(np.float32).sum())
        cands = [z0]
        up = dn = z0
        for _ in range(8):
            up, dn = np.nextafter(up, np.float32(np.inf)), np.nextafter(dn, np.float32(-np.inf))
            cands += [up, dn]
        ok = False
        for z in cands:
            want = (torch.tensor(z, dtype=torch.float32) * xf[t]).to(torch.bfloat16).float().numpy()
            if np.array_equal(got[t], want):
                ok = True
                break
        assert ok, f"token {t}: out != bf16(zsum * x) for every zsum near {z0}"


@pytest.mark.parametrize("path", [1, 2], ids=["decode", "grouped"])
@pytest.mark.parametrize("name", ["zero_expert_small", "zero_expert_decode", "zero_split_decode",
                                  "fused_router_wide"])
def test_forced_identity_experts_are_exact(B, name, path):
    """Every slot on an identity expert, no shared expert: out == bf16(zsum * x) bitwise, on
    both chains (the decode kernel adds the identity experts in its combine phase, the grouped
    chain in the combine kernel). zero_split_decode has at most 32 pairs and a router of at most
    256 columns (the decode kernel's split routing); zero_expert_decode a 384-wide router;
    fused_router_wide the tensor-core router with the top-K fused (forced ids)."""
    shape = (SMALL[name] if name in SMALL else
             SMALL["zero_expert_small"].with_(name=name, num_tokens=4, num_experts=64,
                                              router_width=96))
    if path == 1 and shape.num_tokens > 16:
        pytest.skip("decode chain is for <= 16 tokens")
    inp = I.make_inputs(shape)
    N, K, E, R = shape.num_tokens, shape.top_k, shape.num_experts, shape.router_width
    rng = np.random.default_rng(3)
    forced = np.stack([rng.choice(np.arange(E, R), K, replace=False) for _ in range(N)])
    got, gidx, gw = run_gpu(B, inp, path, forced=forced)
    assert (gidx == forced).all()
    _assert_identity_exact(got, inp.x, gw)


def test_decode_and_grouped_chains_agree(B):
    for n in (4, 16):
        inp = I.make_inputs(I.DECODE.with_(num_tokens=n))
        a, ia, _ = run_gpu(B, inp, 1)
        b, ib, _ = run_gpu(B, inp, 2)
        np.testing.assert_array_equal(ia, ib)
        check_out(a, b.astype(np.float64), rel_l2=1e-2)


@pytest.mark.parametrize("path", [1, 2], ids=["decode", "grouped"])
def test_forward_replays_from_a_cuda_graph(B, path):
    """A forward captured once into a CUDA graph replays to the stream-launched result, bit for
    bit (deterministic mode), on both chains."""
    shape = I.DECODE.with_(num_tokens=8) if path == 1 else SMALL["prefill_zipf_small"]
    dev = I.make_inputs(shape).to("cuda")
    cfg = B.make_config(shape, True, path)
    w = B.make_weights(dev)
    ws = B.alloc_workspace(cfg)
    ref = torch.empty_like(dev.x)
    B.moe_forward(cfg, w, dev.x, ref, ws)
    out = torch.zeros_like(dev.x)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):     # first call outside the capture (sets kernel attributes)
        B.moe_forward(cfg, w, dev.x, out, ws, side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        B.moe_forward(cfg, w, dev.x, out, ws, torch.cuda.current_stream())
    for _ in range(2):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)


@pytest.mark.parametrize("path", [1, 2], ids=["decode", "grouped"])
def test_deterministic_mode_is_bitwise_stable(B, path):
    inp = I.make_inputs(I.DECODE.with_(num_tokens=12) if path == 1 else SMALL["prefill_zipf_small"])
    first = run_gpu(B, inp, path)[0]
    for _ in range(4):
        assert np.array_equal(run_gpu(B, inp, path)[0], first)


def test_atomic_decode_accumulation_matches_oracle(B):
    inp = I.make_inputs(I.DECODE)
    got, gidx, _ = run_gpu(B, inp, 1, deterministic=False)
    ref = O.moe_forward(inp, forced_idx=gidx)
    check_out(got, ref["out"])


def test_output_guard_bands_untouched(B):
    inp = I.make_inputs(SMALL["prefill_zipf_small"])
    dev = inp.to("cuda")
    cfg = B.make_config(inp.shape, True, 2)
    ws = B.alloc_workspace(cfg)
    N, H = inp.shape.num_tokens, inp.shape.hidden
    buf = torch.full((N * H + 2 * 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[4096:4096 + N * H].view(N, H)
    B.moe_forward(cfg, B.make_weights(dev), dev.x, out, ws)
    torch.cuda.synchronize()
    assert (buf[:4096] == 7.0).all() and (buf[-4096:] == 7.0).all()


# ------------------------------------------------------------------ full-size workloads

def _sample_tokens(n, k=12, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, n - 1], rng.choice(n, min(k, n), replace=False)]))


# the prefill workload's grouped chain with the sigmoid + correction-bias scoring (scaled,
# not renormalised), and with the pre-expert RMSNorm of the routed experts' input
PREFILL_SIGMOID = I.PREFILL.with_(name="prefill_sigmoid_bias", scoring=I.SCORING_SIGMOID_BIAS,
                                  correction_bias_std=0.05, norm_topk_prob=False,
                                  routed_scaling_factor=2.5)
PREFILL_PRENORM = I.PREFILL.with_(name="prefill_prenorm", pre_expert_norm=True)


@pytest.mark.parametrize("shape", [I.DECODE, I.PREFILL, I.ZERO_EXPERT, I.DECODE_PRENORM,
                                   PREFILL_SIGMOID, PREFILL_PRENORM],
                         ids=lambda s: s.name)
def test_full_size_sampled_tokens(B, shape):
    """The bench's launch configuration at full size; the oracle recomputes sampled tokens
    one by one, and the routing of every token is checked."""
    inp = I.make_inputs(shape, device="cuda")
    got, gidx, gw = run_gpu(B, inp, 0)
    ref_sel = O.moe_forward(inp, routing_only=True)
    check_routing(gidx, ref_sel)
    toks = _sample_tokens(shape.num_tokens)
    ref = O.moe_forward(inp, tokens=toks, forced_idx=gidx)
    np.testing.assert_allclose(gw[toks], ref["w"], rtol=1e-5, atol=1e-7)
    check_out(got[toks], ref["out"])


# ------------------------------------------------------------------ FP8 experts

FP8_ATOL, FP8_RTOL, FP8_REL_L2 = 5e-2, 5e-2, 2e-2

FP8_SMALL = I.FP8_PREFILL.with_(name="fp8_small", num_tokens=300, hidden=512, num_experts=8,
                                router_width=8, top_k=2, inter=256)


@pytest.mark.parametrize("shape", [FP8_SMALL,
                                   FP8_SMALL.with_(name="fp8_small_k4", num_tokens=77,
                                                   num_experts=16, router_width=16, top_k=4,
                                                   inter=384, hidden=768),
                                   FP8_SMALL.with_(name="fp8_small_prenorm",
                                                   pre_expert_norm=True),
                                   # decode-sized: 4 tokens, top-8 of 32, a gated bf16 shared
                                   # expert beside the E4M3 routed experts
                                   FP8_SMALL.with_(name="fp8_decode_n4", num_tokens=4,
                                                   num_experts=32, router_width=32, top_k=8,
                                                   shared_inter=256, shared_gated=True)],
                         ids=lambda s: s.name)
def test_fp8_forward_matches_oracle(B, shape):
    inp = I.make_inputs(shape)
    got, gidx, gw = run_gpu(B, inp, 0)
    check_routing(gidx, O.moe_forward(inp, routing_only=True))
    ref = O.moe_forward(inp, forced_idx=gidx)
    check_out(got, ref["out"], FP8_ATOL, FP8_RTOL, FP8_REL_L2)


# decode-sized FP8 batches, on the decode kernel (E4M3 items, per-item scale promotion) and on
# the grouped chain: 32 routed pairs with a gated shared expert; 64 pairs over 128-row gate/up
# tiles (I = 384); a pre-expert norm (the kernel quantises xn)
FP8_DECODE = [FP8_SMALL.with_(name="fp8_decode_n4", num_tokens=4, num_experts=32, router_width=32,
                              top_k=8, shared_inter=256, shared_gated=True),
              FP8_SMALL.with_(name="fp8_decode_n16_k4", num_tokens=16, num_experts=16,
                              router_width=16, top_k=4, inter=384, hidden=768, shared_inter=128),
              FP8_SMALL.with_(name="fp8_decode_prenorm", num_tokens=3, num_experts=16,
                              router_width=16, top_k=2, pre_expert_norm=True)]


@pytest.mark.parametrize("path", [1, 2], ids=["decode", "grouped"])
@pytest.mark.parametrize("shape", FP8_DECODE, ids=lambda s: s.name)
def test_fp8_decode_matches_oracle(B, shape, path):
    inp = I.make_inputs(shape)
    got, gidx, gw = run_gpu(B, inp, path)
    check_routing(gidx, O.moe_forward(inp, routing_only=True))
    ref = O.moe_forward(inp, forced_idx=gidx)
    check_out(got, ref["out"], FP8_ATOL, FP8_RTOL, FP8_REL_L2)


def test_fp8_decode_kernel_modes(B):
    """E4M3 experts on the decode kernel: the deterministic mode repeats bit for bit, the
    FP32-atomic accumulation matches the oracle."""
    inp = I.make_inputs(FP8_DECODE[0])
    first = run_gpu(B, inp, 1)[0]
    for _ in range(3):
        assert np.array_equal(run_gpu(B, inp, 1)[0], first)
    got, gidx, _ = run_gpu(B, inp, 1, deterministic=False)
    check_out(got, O.moe_forward(inp, forced_idx=gidx)["out"], FP8_ATOL, FP8_RTOL, FP8_REL_L2)


@pytest.mark.parametrize("shape", [I.FP8_PREFILL, I.DECODE_FP8], ids=lambda s: s.name)
def test_fp8_full_size_sampled_tokens(B, shape):
    inp = I.make_inputs(shape, device="cuda")
    got, gidx, gw = run_gpu(B, inp, 0)
    check_routing(gidx, O.moe_forward(inp, routing_only=True))
    toks = _sample_tokens(shape.num_tokens, k=10)
    ref = O.moe_forward(inp, tokens=toks, forced_idx=gidx)
    check_out(got[toks], ref["out"], FP8_ATOL, FP8_RTOL, FP8_REL_L2)


# ------------------------------------------------------------------ NVFP4 experts

# The weights are dequantised exactly to bf16 and the activations stay bf16 (w4a16): the same
# arithmetic as the bf16 experts, so the same bars.
NV_SMALL = I.PREFILL.with_(name="nvfp4_small", num_tokens=300, hidden=512, num_experts=16,
                           router_width=16, top_k=4, inter=256, shared_inter=256,
                           shared_gated=True, weight_dtype=I.WDTYPE_NVFP4)
NV_SHAPES = [
    NV_SMALL,
    # decode-sized: 4 tokens, top-8 of 32
    NV_SMALL.with_(name="nvfp4_decode_n4", num_tokens=4, num_experts=32, router_width=32,
                   top_k=8),
    # 6 gate/up n-tiles, 12 down contraction stages (3 scale boxes), no shared expert
    NV_SMALL.with_(name="nvfp4_wide", num_tokens=130, hidden=1024, inter=768, num_experts=8,
                   router_width=8, top_k=2, shared_inter=0, zipf_s=0.0),
    # sigmoid + correction bias, pre-expert RMSNorm of the routed experts' input
    NV_SMALL.with_(name="nvfp4_sigmoid_prenorm", num_tokens=200, hidden=768, inter=512,
                   num_experts=32, router_width=32, top_k=6, shared_inter=0, zipf_s=0.0,
                   scoring=I.SCORING_SIGMOID_BIAS, correction_bias_std=0.05,
                   pre_expert_norm=True, norm_topk_prob=False, routed_scaling_factor=1.5),
]


@pytest.mark.parametrize("path", [0, 1, 2], ids=["auto", "decode", "grouped"])
@pytest.mark.parametrize("shape", NV_SHAPES + [
    # decode-sized on the decode kernel: 16 tokens, top-4, an ungated shared expert
    NV_SMALL.with_(name="nvfp4_decode_n16", num_tokens=16, num_experts=16, router_width=16,
                   top_k=4, shared_gated=False)], ids=lambda s: s.name)
def test_nvfp4_forward_matches_oracle(B, shape, path):
    if path == 1 and shape.num_tokens > 16:
        pytest.skip("decode chain is for <= 16 tokens")
    inp = I.make_inputs(shape)
    got, gidx, gw = run_gpu(B, inp, path)
    check_routing(gidx, O.moe_forward(inp, routing_only=True))
    ref = O.moe_forward(inp, forced_idx=gidx)
    check_out(got, ref["out"])
    # deterministic mode repeats bit for bit
    assert np.array_equal(run_gpu(B, inp, path)[0], got)


def test_nvfp4_decode_kernel_atomic_mode(B):
    """NVFP4 experts on the decode kernel with the FP32-atomic down accumulation."""
    inp = I.make_inputs(NV_SHAPES[1])
    got, gidx, _ = run_gpu(B, inp, 1, deterministic=False)
    check_out(got, O.moe_forward(inp, forced_idx=gidx)["out"])


def test_nvfp4_rejected_where_unsupported(B):
    """NVFP4 needs hidden and inter multiples of 256."""
    ok = NV_SMALL.with_(num_tokens=4)
    for path in (1, 2):
        assert B.moe_workspace_size(B.make_config(ok, True, path)) > 0
    with pytest.raises(B.MoeError):
        B.moe_workspace_size(B.make_config(NV_SMALL.with_(inter=384), True, 0))


@pytest.mark.parametrize("shape", [I.DECODE_NVFP4, I.PREFILL_NVFP4], ids=lambda s: s.name)
def test_nvfp4_full_size(B, shape):
    inp = I.make_inputs(shape, device="cuda")
    got, gidx, gw = run_gpu(B, inp, 0)
    check_routing(gidx, O.moe_forward(inp, routing_only=True))
    toks = _sample_tokens(shape.num_tokens, k=10) if shape.num_tokens > 16 else \
        list(range(shape.num_tokens))
    ref = O.moe_forward(inp, tokens=toks, forced_idx=gidx)
    np.testing.assert_allclose(gw[toks], ref["w"], rtol=1e-5, atol=1e-7)
    check_out(got[toks], ref["out"])


# ------------------------------------------------------------------ failure detection

def test_bounded_wait_reports_timeout_and_context_survives(B):
    """A device wait on a barrier nothing completes gives up after its limit and reports
    MOE_ERR_DEVICE_TIMEOUT; the next forward on the same context still matches the oracle."""
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    B.moe_selftest_bounded_wait(ws, 20_000_000)       # ~10 ms
    assert B.moe_read_device_status(ws) == B.MOE_ERR_DEVICE_TIMEOUT
    inp = I.make_inputs(I.TINY)
    got, gidx, _ = run_gpu(B, inp, 2)
    check_out(got, O.moe_forward(inp, forced_idx=gidx)["out"])
