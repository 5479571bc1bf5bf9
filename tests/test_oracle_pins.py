"""Pins of the CPU oracle against things other than itself: hand-worked closed forms, brute
force, library routines (torch softmax / silu / matmul / float8 cast), exact identities and a
second independent formulation. CPU only."""
import itertools
import math
import os

import numpy as np
import pytest
import torch

from mixture_experts_layer_08_gb300 import inputs as I
from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.txt")


# ------------------------------------------------------------------ helpers

def _rows(text, dtype=float):
    return [[dtype(v) for v in r.split()] for r in text.split(";")]


def load_worked_examples():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "case":
            cur = {"name": rest}
            cases.append(cur)
        else:
            cur[key] = rest
    return cases


def _closed_form(expr):
    env = {"exp": math.exp, "silu": lambda z: z / (1 + math.exp(-z)),
           "sigmoid": lambda z: 1 / (1 + math.exp(-z))}
    return eval(expr, {"__builtins__": {}}, env)  # fixture-only arithmetic expressions


def inputs_from_case(c):
    kv = dict(p.split("=") for p in c["shape"].split())
    shape = I.MoeShape(c["name"], int(kv["N"]), int(kv["H"]), int(kv["E"]), int(kv["R"]),
                       int(kv["K"]), int(kv["I"]), shared_inter=int(kv["S"]),
                       scoring=int(kv["scoring"]), norm_topk_prob=bool(int(kv["norm"])),
                       routed_scaling_factor=float(kv["scale"]),
                       pre_expert_norm="pre_expert_norm_w" in c,
                       rms_norm_eps=float(kv.get("eps", 1e-6)))
    bf = torch.bfloat16
    N, H, E, R, Ii, S = (shape.num_tokens, shape.hidden, shape.num_experts, shape.router_width,
                         shape.inter, shape.shared_inter)

    def mat(key, rows, cols):
        t = torch.tensor(_rows(c[key]), dtype=torch.float32).reshape(rows, cols)
        assert torch.equal(t.to(bf).float(), t), "fixture values must be exact in bf16"
        return t.to(bf)

    kw = dict(x=mat("x", N, H), router_w=mat("router_w", R, H),
              w_gate=mat("w_gate", E * Ii, H).reshape(E, Ii, H),
              w_up=mat("w_up", E * Ii, H).reshape(E, Ii, H),
              w_down=mat("w_down", E * H, Ii).reshape(E, H, Ii))
    if "correction_bias" in c:
        kw["correction_bias"] = torch.tensor(_rows(c["correction_bias"])[0], dtype=torch.float32)
    if "pre_expert_norm_w" in c:
        kw["pre_expert_norm_w"] = mat("pre_expert_norm_w", 1, H).reshape(H)
    if S:
        kw["sh_gate"] = mat("sh_gate", S, H)
        kw["sh_up"] = mat("sh_up", S, H)
        kw["sh_down"] = mat("sh_down", H, S)
        if "sh_gate_vec" in c:
            kw["sh_gate_vec"] = mat("sh_gate_vec", 1, H).reshape(H)
    return I.MoeInputs(shape=shape, **kw)


def small(shape: I.MoeShape, **kw) -> I.MoeShape:
    return shape.with_(**kw)


def torch_probs(inp):
    """Router probabilities through torch (library matmul + softmax, fp64)."""
    L = inp.x.double() @ inp.router_w.double().T
    if inp.router_logit_bias is not None:
        L = L + inp.router_logit_bias.double()
    return torch.softmax(L, dim=1).numpy()


# ------------------------------------------------------------------ worked examples

@pytest.mark.parametrize("case", load_worked_examples(), ids=lambda c: c["name"])
def test_worked_examples_closed_form(case):
    inp = inputs_from_case(case)
    K = inp.shape.top_k
    want_out = np.array([_closed_form(e) for r in case["expect_out"].split(";")
                         for e in [r]]).reshape(inp.shape.num_tokens, inp.shape.hidden)
    want_idx = np.array(_rows(case["expect_idx"], int)).reshape(-1, K)
    want_w = np.array([[_closed_form(v) for v in r.split()] for r in case["expect_w"].split(";")])
    want_z = np.array([_closed_form(v) for v in case["expect_zsum"].split(";")])
    for impl in (O.moe_forward, O.moe_forward_dense):
        r = impl(inp)
        np.testing.assert_array_equal(r["idx"], want_idx)
        np.testing.assert_allclose(r["w"], want_w, rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(r["out"], want_out, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(O.moe_forward(inp)["zsum"], want_z, rtol=1e-14, atol=1e-15)


# ------------------------------------------------------------------ routing

def test_topk_brute_force_tiny():
    """C1-sized router (R=8, K=2): the chosen set is the unique subset whose every member
    ranks before every non-member under (score desc, index asc); order is that ranking."""
    inp = I.make_inputs(I.TINY)
    r = O.moe_forward(inp, routing_only=True)
    p = torch_probs(inp)
    R, K = inp.shape.router_width, inp.shape.top_k
    for t in range(inp.shape.num_tokens):
        def before(a, b):
            return p[t, a] > p[t, b] or (p[t, a] == p[t, b] and a < b)
        winners = [S for S in itertools.combinations(range(R), K)
                   if all(before(a, b) for a in S for b in range(R) if b not in S)]
        assert len(winners) == 1
        assert sorted(r["idx"][t]) == sorted(winners[0])
        got = list(r["idx"][t])
        assert all(before(got[i], got[i + 1]) for i in range(K - 1))
        srt = np.sort(p[t])[::-1]
        assert r["gap"][t] == pytest.approx(srt[K - 1] - srt[K], abs=1e-12)


def test_all_equal_logits_tie_break():
    shape = small(I.TINY, router_width=16, num_experts=16, top_k=4)
    inp = I.make_inputs(shape)
    inp.router_w = torch.zeros_like(inp.router_w)
    for impl in (O.moe_forward, O.moe_forward_dense):
        r = impl(inp)
        assert (r["idx"] == np.arange(4)[None, :]).all()
        np.testing.assert_allclose(r["w"], 0.25, rtol=0, atol=1e-15)


def test_renormalised_weights_sum_to_one():
    shape = small(I.ZERO_EXPERT, num_tokens=64, hidden=256, num_experts=32, router_width=48,
                  inter=128)
    r = O.moe_forward(I.make_inputs(shape), routing_only=True)
    np.testing.assert_allclose(r["w"].sum(axis=1), 1.0, rtol=0, atol=1e-12)


def test_all_columns_selected_gives_softmax():
    """R == K with renormalisation: every column is chosen and w equals softmax(L)."""
    shape = small(I.TINY, router_width=8, num_experts=8, top_k=8)
    inp = I.make_inputs(shape)
    r = O.moe_forward(inp, routing_only=True)
    p = torch_probs(inp)
    np.testing.assert_allclose(r["w"], np.take_along_axis(p, r["idx"], 1), rtol=1e-13)
    assert np.isinf(r["gap"]).all()


def test_no_renorm_scaling():
    shape = small(I.TINY, norm_topk_prob=False, routed_scaling_factor=2.5)
    inp = I.make_inputs(shape)
    r = O.moe_forward(inp, routing_only=True)
    p = torch_probs(inp)
    np.testing.assert_allclose(r["w"], 2.5 * np.take_along_axis(p, r["idx"], 1), rtol=1e-13)


def test_correction_bias_selects_but_does_not_weight():
    """A +1 bias on ids {5, 9, 2} forces them to be chosen; their weights are the unbiased
    probabilities renormalised, ordered by probability."""
    shape = small(I.ZERO_EXPERT, num_tokens=8, hidden=256, num_experts=12, router_width=12,
                  top_k=3, inter=128)
    inp = I.make_inputs(shape)
    cb = torch.zeros(12)
    cb[[5, 9, 2]] = 1.0
    inp.correction_bias = cb
    p = torch_probs(inp)
    for impl in (O.moe_forward, O.moe_forward_dense):
        r = impl(inp)
        for t in range(8):
            assert set(r["idx"][t]) == {5, 9, 2}
            want = p[t, r["idx"][t]] / p[t, [5, 9, 2]].sum()
            np.testing.assert_allclose(r["w"][t], want, rtol=1e-13)
            assert list(r["idx"][t]) == sorted([5, 9, 2], key=lambda e: (-p[t, e], e))


def test_selection_scores_are_probabilities_plus_bias():
    shape = small(I.ZERO_EXPERT, num_tokens=16, hidden=256, num_experts=16, router_width=24,
                  inter=128)
    inp = I.make_inputs(shape)
    r = O.moe_forward(inp, routing_only=True)
    want = torch_probs(inp) + inp.correction_bias.double().numpy()[None, :]
    np.testing.assert_allclose(r["sel"], want, rtol=1e-12, atol=1e-15)


def test_sigmoid_topk_brute_force_with_bias():
    """Sigmoid + bias arm: the chosen set is the unique K-subset ranking before every other
    column under (sigmoid(L) + bias desc, index asc), sigmoid taken from torch; the selection
    scores are those; the weights are the chosen unbiased scores, renormalised."""
    shape = small(I.TINY, num_tokens=12, router_width=8, num_experts=8, top_k=3,
                  scoring=I.SCORING_SIGMOID_BIAS, correction_bias_std=0.05,
                  routed_scaling_factor=1.5)
    inp = I.make_inputs(shape)
    L = inp.x.double() @ inp.router_w.double().T
    s = torch.sigmoid(L).numpy()
    sel = s + inp.correction_bias.double().numpy()[None, :]
    R, K = 8, 3
    for impl in (O.moe_forward, O.moe_forward_dense):
        r = impl(inp)
        for t in range(shape.num_tokens):
            def before(a, b):
                return sel[t, a] > sel[t, b] or (sel[t, a] == sel[t, b] and a < b)
            winners = [S for S in itertools.combinations(range(R), K)
                       if all(before(a, b) for a in S for b in range(R) if b not in S)]
            assert len(winners) == 1 and sorted(r["idx"][t]) == sorted(winners[0])
            got = list(r["idx"][t])
            assert all(before(got[i], got[i + 1]) for i in range(K - 1))
            np.testing.assert_allclose(r["w"][t].sum(), 1.5, rtol=1e-13)
            np.testing.assert_allclose(r["w"][t] / r["w"][t].sum(),
                                       s[t, got] / s[t, got].sum(), rtol=1e-12)
    np.testing.assert_allclose(O.moe_forward(inp, routing_only=True)["sel"], sel, rtol=1e-12,
                               atol=1e-15)


def test_sigmoid_without_bias_selects_by_logits():
    """Sigmoid is increasing, so with a zero bias the K chosen columns are the K largest
    logits (numpy argsort of the library matmul), the same set softmax scoring picks."""
    shape = small(I.TINY, num_tokens=32, router_width=16, num_experts=16, top_k=4,
                  scoring=I.SCORING_SIGMOID_BIAS)
    inp = I.make_inputs(shape)
    inp.correction_bias = torch.zeros(16)
    L = (inp.x.double() @ inp.router_w.double().T).numpy()
    order = np.lexsort((np.broadcast_to(np.arange(16), L.shape), -L), axis=1)[:, :4]
    r = O.moe_forward(inp, routing_only=True)
    np.testing.assert_array_equal(r["idx"], order)
    soft = O.moe_forward(I.make_inputs(shape.with_(scoring=I.SCORING_SOFTMAX)),
                         routing_only=True)
    np.testing.assert_array_equal(np.sort(soft["idx"], 1), np.sort(r["idx"], 1))


def test_gap_matches_sorted_scores_with_bias():
    shape = small(I.ZERO_EXPERT, num_tokens=32, hidden=256, num_experts=16, router_width=24,
                  inter=128)
    inp = I.make_inputs(shape)
    r = O.moe_forward(inp, routing_only=True)
    sel = torch_probs(inp) + inp.correction_bias.double().numpy()[None, :]
    srt = -np.sort(-sel, axis=1)
    K = shape.top_k
    np.testing.assert_allclose(r["gap"], srt[:, K - 1] - srt[:, K], rtol=1e-10, atol=1e-15)


# ------------------------------------------------------------------ experts

def test_single_expert_equals_dense_swiglu():
    """E = R = K = 1 with renormalisation: w = 1, the block is one dense SwiGLU FFN."""
    shape = small(I.TINY, num_experts=1, router_width=1, top_k=1, shared_inter=0)
    inp = I.make_inputs(shape)
    x = inp.x.double()
    g = x @ inp.w_gate[0].double().T
    u = x @ inp.w_up[0].double().T
    want = (torch.nn.functional.silu(g) * u) @ inp.w_down[0].double().T
    for impl in (O.moe_forward, O.moe_forward_dense):
        np.testing.assert_allclose(impl(inp)["out"], want.numpy(), rtol=1e-11, atol=1e-14)


def test_shared_expert_equals_dense_swiglu_and_gate():
    """Zero routed weights isolate the shared expert: out = gamma * SwiGLU_shared(x), with
    gamma = 1 without a gate vector, 1/2 with a zero gate vector, sigmoid(x.g) otherwise."""
    shape = small(I.DECODE, num_tokens=5, hidden=256, num_experts=4, router_width=4, top_k=2,
                  inter=128, shared_inter=256)
    inp = I.make_inputs(shape)
    for k in ("w_gate", "w_up", "w_down"):
        setattr(inp, k, torch.zeros_like(getattr(inp, k)))
    x = inp.x.double()
    sh = (torch.nn.functional.silu(x @ inp.sh_gate.double().T) * (x @ inp.sh_up.double().T)) \
        @ inp.sh_down.double().T
    gamma = torch.sigmoid(x @ inp.sh_gate_vec.double())
    r = O.moe_forward(inp)
    np.testing.assert_allclose(r["out"], (gamma[:, None] * sh).numpy(), rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(r["gamma"], gamma.numpy(), rtol=1e-13)
    inp.sh_gate_vec = torch.zeros_like(inp.sh_gate_vec)
    r0 = O.moe_forward(inp)
    assert (r0["gamma"] == 0.5).all()
    np.testing.assert_allclose(r0["out"], 0.5 * sh.numpy(), rtol=1e-11, atol=1e-14)
    inp.sh_gate_vec = None
    r1 = O.moe_forward(inp)
    assert (r1["gamma"] == 1.0).all()
    np.testing.assert_allclose(r1["out"], sh.numpy(), rtol=1e-11, atol=1e-14)


def test_identity_experts_exact():
    """A bias that forces every choice onto identity experts (ids >= E) and no shared expert:
    out == zero_accum * x exactly; with renormalisation zero_accum == 1 so out == x."""
    shape = small(I.ZERO_EXPERT, num_tokens=16, hidden=256, num_experts=8, router_width=16,
                  top_k=4, inter=128, norm_topk_prob=False)
    inp = I.make_inputs(shape)
    cb = torch.zeros(16)
    cb[8:] = 1.0
    inp.correction_bias = cb
    x = inp.x.double().numpy()
    for impl in (O.moe_forward,):
        r = impl(inp)
        assert (r["idx"] >= 8).all()
        p = torch_probs(inp)
        np.testing.assert_allclose(r["zsum"], np.take_along_axis(p, r["idx"], 1).sum(1),
                                   rtol=1e-13)
        assert np.array_equal(r["out"], r["zsum"][:, None] * x)
    inp2 = I.make_inputs(shape.with_(norm_topk_prob=True))
    inp2.correction_bias = cb
    r2 = O.moe_forward(inp2)
    np.testing.assert_allclose(r2["zsum"], 1.0, rtol=0, atol=4e-16)
    assert np.array_equal(r2["out"], r2["zsum"][:, None] * x)
    np.testing.assert_allclose(O.moe_forward_dense(inp2)["out"], x, rtol=4e-16, atol=0)


def test_mixed_identity_and_zero_weight_experts():
    """With all routed expert matrices zero, the output is exactly zero_accum * x even when
    the routing mixes real and identity experts."""
    shape = small(I.ZERO_EXPERT, num_tokens=32, hidden=256, num_experts=8, router_width=16,
                  top_k=4, inter=128)
    inp = I.make_inputs(shape)
    inp.correction_bias = torch.zeros(16)
    for k in ("w_gate", "w_up", "w_down"):
        setattr(inp, k, torch.zeros_like(getattr(inp, k)))
    r = O.moe_forward(inp)
    assert ((r["idx"] >= 8).any(axis=1) & (r["idx"] < 8).any(axis=1)).any()
    assert np.array_equal(r["out"], r["zsum"][:, None] * inp.x.double().numpy())


@pytest.mark.parametrize("base", [I.TINY, I.DECODE, I.ZERO_EXPERT, I.PREFILL,
                                  I.DECODE.with_(name="decode_prenorm", pre_expert_norm=True),
                                  I.PREFILL.with_(name="sigmoid_prenorm", pre_expert_norm=True,
                                                  scoring=I.SCORING_SIGMOID_BIAS,
                                                  correction_bias_std=0.05, zipf_s=0.0)],
                         ids=lambda s: s.name)
def test_loop_and_dense_formulations_agree(base):
    shape = base.with_(num_tokens=min(base.num_tokens, 24), hidden=256,
                       num_experts=min(base.num_experts, 16),
                       router_width=min(base.num_experts, 16) + (base.router_width - base.num_experts) // 16,
                       inter=128, shared_inter=min(base.shared_inter, 128))
    inp = I.make_inputs(shape)
    a, b = O.moe_forward(inp), O.moe_forward_dense(inp)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    np.testing.assert_allclose(a["w"], b["w"], rtol=1e-13)
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-10, atol=1e-14)


def test_forced_routing_overrides_selection():
    inp = I.make_inputs(I.TINY)
    forced = np.tile(np.array([[3, 1]], dtype=np.int32), (16, 1))
    a = O.moe_forward(inp, forced_idx=forced)
    b = O.moe_forward_dense(inp, forced_idx=forced)
    assert (a["idx"] == forced).all()
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-10, atol=1e-14)


# ------------------------------------------------------------------ sort / permute

def test_sort_by_expert_matches_stable_argsort_and_roundtrips():
    rng = np.random.default_rng(0)
    N, K, E, R = 37, 3, 6, 9
    idx = np.stack([rng.choice(R, K, replace=False) for _ in range(N)])
    off, pairs, p2r = O.sort_by_expert(idx, E)
    flat = idx.reshape(-1)
    real = np.nonzero(flat < E)[0]
    order = real[np.argsort(flat[real], kind="stable")]
    assert np.array_equal(pairs, order)
    assert off[0] == 0 and off[-1] == len(real) and (np.diff(off.astype(np.int64)) >= 0).all()
    for e in range(E):
        assert (flat[pairs[off[e]:off[e + 1]]] == e).all()
    # permute then unpermute with unit weights is the identity on the routed pairs
    payload = rng.standard_normal(N * K)
    permuted = payload[pairs]
    back = np.full(N * K, np.nan)
    back[real] = permuted[p2r[real]]
    assert np.array_equal(back[real], payload[real])
    assert (p2r[flat >= E] == 0xFFFFFFFF).all()


# ------------------------------------------------------------------ E4M3

def test_e4m3_decode_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([O.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all() and nan.sum() == 2
    assert np.array_equal(ours[~nan], ref[~nan])
    assert O.e4m3_decode(0x7E) == 448.0 and O.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_sweep_matches_torch_cast():
    rng = np.random.default_rng(1)
    mag = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 1_000_000))
    v = mag * rng.choice([-1.0, 1.0], mag.size)
    # exact midpoints between neighbouring codes exercise ties-to-even
    pos = np.array([O.e4m3_decode(c) for c in range(127)])
    mids = (pos[:-1] + pos[1:]) / 2
    v = np.concatenate([v, mids, -mids, [0.0, -0.0, 448.0, -448.0, 2.0 ** -10]]).astype(np.float32)
    ours = O.e4m3_encode_array(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encode_saturates():
    for v, c in ((500.0, 0x7E), (1e9, 0x7E), (-1e9, 0xFE), (464.0, 0x7E), (449.0, 0x7E)):
        assert O.e4m3_encode(v) == c


def test_quant_1x128_rules():
    v = np.zeros(384, dtype=np.float32)
    v[:128] = np.linspace(-448, 448, 128, dtype=np.float32)   # amax 448 -> scale 1
    v[256:] = np.float32(3.0) * np.linspace(-1, 1, 128, dtype=np.float32)
    codes, scales, deq = O.quant_1x128(v)
    assert scales[0] == 1.0 and scales[1] == 1.0 and scales[2] == np.float32(3.0) / np.float32(448.0)
    ref0 = torch.from_numpy(v[:128]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes[:128], ref0)
    assert (codes[128:256] == 0).all() and (deq[128:256] == 0).all()
    q2 = (v[256:] / scales[2]).astype(np.float32)
    ref2 = torch.from_numpy(q2).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(deq[256:], ref2 * np.float64(scales[2]))
    # the numpy restatement used by the dense formulation agrees code for code
    dn = O._quant_rows_np(v.reshape(1, -1).astype(np.float64))
    np.testing.assert_array_equal(dn.reshape(-1), deq)


def test_fp8_formulations_agree_and_stay_near_unquantised():
    shape = I.FP8_PREFILL.with_(num_tokens=12, hidden=256, num_experts=6, router_width=6,
                                top_k=2, inter=256)
    inp = I.make_inputs(shape)
    a, b = O.moe_forward(inp), O.moe_forward_dense(inp)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    rel = np.linalg.norm(a["out"] - b["out"]) / np.linalg.norm(b["out"])
    assert rel < 1e-6
    # same weights dequantised, activations not quantised: close but not equal
    deq = {}
    for k, sk in (("w_gate", "s_gate"), ("w_up", "s_up"), ("w_down", "s_down")):
        deq[k] = torch.from_numpy(O._dequant_blocks(getattr(inp, k), getattr(inp, sk)))
    ref_inp = I.MoeInputs(shape=shape.with_(weight_dtype=I.WDTYPE_BF16), x=inp.x,
                          router_w=inp.router_w, **deq)
    c = O.moe_forward_dense(ref_inp, forced_idx=a["idx"])
    rel_q = np.linalg.norm(a["out"] - c["out"]) / np.linalg.norm(c["out"])
    assert 1e-4 < rel_q < 0.08


# ------------------------------------------------------------------ NVFP4 experts

E2M1_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_ocp_mx.txt")


def test_e2m1_decode_all_codes_match_the_ocp_table():
    rows = [l.split() for l in open(E2M1_GOLDEN) if l.strip() and not l.startswith("#")]
    assert len(rows) == 16
    for code, val in rows:
        got = O.e2m1_decode(int(code))
        assert got == float(val) and math.copysign(1.0, got) == math.copysign(1.0, float(val))


def _nvfp4_inputs(shape, placements, sf_codes, scale2):
    """NVFP4 weights that are zero except for hand-placed codes. `placements` maps a matrix
    name to [(row, col, code)]; `sf_codes` to {(row, group): E4M3 code} (others 0x38 = 1.0);
    `scale2` to its fp32 value. Returns the inputs and the dense fp64 matrices they encode,
    built from the placements by hand (value table, scale table, product)."""
    base = I.make_inputs(shape.with_(weight_dtype=I.WDTYPE_BF16))
    E, H, Ii = shape.num_experts, shape.hidden, shape.inter
    e2m1 = {2: 1.0, 5: 3.0, 7: 6.0, 9: -0.5, 12: -2.0}
    e4m3 = {0x38: 1.0, 0x40: 2.0, 0x30: 0.5, 0x3C: 1.5}
    kw, dense = {}, {}
    for name, (rows, cols) in (("gate", (Ii, H)), ("up", (Ii, H)), ("down", (H, Ii))):
        packed = torch.zeros(E, rows, cols // 2, dtype=torch.uint8)
        sf = torch.full((E, rows, cols // 16), 0x38, dtype=torch.uint8)
        d = torch.zeros(E, rows, cols, dtype=torch.float64)
        for (r, g), code in sf_codes.get(name, {}).items():
            sf[0, r, g] = code
        for r, c, code in placements.get(name, []):
            byte = int(packed[0, r, c // 2])
            byte |= code << 4 if c % 2 else code
            packed[0, r, c // 2] = byte
            d[0, r, c] = e2m1[code] * e4m3[int(sf[0, r, c // 16])] * scale2[name]
        kw["w_" + name], kw["sf_" + name] = packed, sf
        kw["scale2_" + name] = torch.full((E,), scale2[name], dtype=torch.float32)
        dense[name] = d
    inp = I.MoeInputs(shape=shape, x=base.x, router_w=base.router_w, **kw)
    return inp, dense


def test_nvfp4_packing_scales_and_scale2_against_dense_swiglu():
    """E = R = K = 1: the block is one dense SwiGLU FFN whose weights are the hand-placed
    values: the nibble order (odd columns in the high nibble), the 16-wide scale groups and
    the per-matrix scale2 are checked against torch's matmul + silu."""
    shape = I.TINY.with_(num_experts=1, router_width=1, top_k=1, shared_inter=0, hidden=64,
                         inter=32, weight_dtype=I.WDTYPE_NVFP4)
    placements = {
        "gate": [(0, 5, 2), (0, 21, 7), (3, 0, 9), (3, 63, 12), (31, 16, 5)],
        "up": [(0, 4, 5), (0, 21, 2), (3, 1, 7), (3, 62, 9), (31, 17, 12)],
        "down": [(0, 0, 2), (7, 3, 5), (7, 31, 9), (63, 16, 7), (40, 15, 12)],
    }
    sf_codes = {"gate": {(0, 1): 0x40, (3, 3): 0x30}, "up": {(0, 1): 0x3C},
                "down": {(7, 1): 0x40, (63, 1): 0x30}}
    scale2 = {"gate": 0.25, "up": 0.5, "down": 0.125}
    inp, d = _nvfp4_inputs(shape, placements, sf_codes, scale2)
    x = inp.x.double()
    g = x @ d["gate"][0].T
    u = x @ d["up"][0].T
    want = (torch.nn.functional.silu(g) * u) @ d["down"][0].T
    assert (want != 0).sum() > 3
    for impl in (O.moe_forward, O.moe_forward_dense):
        np.testing.assert_allclose(impl(inp)["out"], want.numpy(), rtol=1e-12, atol=1e-15)


def test_nvfp4_formulations_agree():
    shape = I.PREFILL.with_(name="nvfp4_pin", num_tokens=24, hidden=256, num_experts=6,
                            router_width=6, top_k=2, inter=128, shared_inter=64,
                            weight_dtype=I.WDTYPE_NVFP4)
    inp = I.make_inputs(shape)
    a, b = O.moe_forward(inp), O.moe_forward_dense(inp)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-10, atol=1e-15)
