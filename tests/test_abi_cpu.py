"""The C-ABI library loads, exports every entry point its header declares, and refuses bad
arguments on the host (no GPU needed: every call here returns before touching CUDA)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from mixture_experts_layer_08_gb300 import build as _b
    _b.build()
    from mixture_experts_layer_08_gb300 import binding
    return binding


def header_symbols():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    syms = header_symbols()
    for s in ("moe_forward", "moe_workspace_size", "moe_route", "moe_status_string",
              "moe_read_device_status"):
        assert s in syms


def test_library_exports_every_header_symbol(B):
    lib = ctypes.CDLL(B.LIB_PATH)
    for s in header_symbols():
        assert hasattr(lib, s), f"{s} declared in include/moe.h but not exported"


def test_status_strings(B):
    assert B.moe_status_string(0) == "ok"
    for s in range(1, 6):
        assert B.moe_status_string(s) != "unknown status"
    assert B.moe_status_string(99) == "unknown status"


def _cfg(B, **kw):
    from mixture_experts_layer_08_gb300 import inputs as I
    return B.make_config(I.TINY.with_(**kw))


@pytest.mark.parametrize("kw,status", [
    (dict(num_tokens=-1), 1),
    (dict(hidden=0), 1),
    (dict(top_k=9), 1),                       # K > R
    (dict(router_width=4), 1),                # R < E
    (dict(hidden=200), 2),                    # not a multiple of 128
    (dict(inter=96), 2),
    (dict(shared_inter=100), 2),
    (dict(router_width=12), 2),               # identity experts need softmax + bias scoring
    (dict(router_width=12, scoring=2), 2),    # ... not the sigmoid + bias scoring
    (dict(scoring=3), 1),                     # no such scoring
    (dict(top_k=33, router_width=64, num_experts=64), 2),
    (dict(router_width=2048, num_experts=2048, scoring=1), 2),
])
def test_workspace_size_refusals(B, kw, status):
    n = ctypes.c_size_t(0)
    assert B.lib.moe_workspace_size(ctypes.byref(_cfg(B, **kw)), ctypes.byref(n)) == status


def test_decode_path_limits(B):
    n = ctypes.c_size_t(0)
    cfg = _cfg(B, num_tokens=17)
    cfg.path = B.PATH_DECODE
    assert B.lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == B.MOE_ERR_UNSUPPORTED
    cfg.path = B.PATH_GROUPED
    assert B.lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == B.MOE_OK
    cfg.path = 7
    assert B.lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == B.MOE_ERR_INVALID_ARG


def test_workspace_grows_with_tokens(B):
    sizes = [B.moe_workspace_size(_cfg(B, num_tokens=n)) for n in (1, 16, 17, 300, 5000)]
    assert sizes[1] >= sizes[0] and sizes[3] > sizes[2] and sizes[4] > sizes[3]
    assert all(s % 256 == 0 for s in sizes)


def test_forward_refuses_before_touching_the_gpu(B):
    cfg = _cfg(B)
    w = B.moe_weights_t()
    # missing weights
    st = B.lib.moe_forward(ctypes.byref(cfg), ctypes.byref(w), None, None, None, 0, None, None,
                           None, None)
    assert st == B.MOE_ERR_INVALID_ARG
    # a workspace that is too small (fake, never dereferenced: the size check comes first)
    fake = 1 << 20
    for n in B.moe_weights_t._fields_:
        setattr(w, n[0], fake)
    w.router_logit_bias = None
    w.correction_bias = None
    w.s_gate = w.s_up = w.s_down = None
    w.sh_gate_vec = None
    st = B.lib.moe_forward(ctypes.byref(cfg), ctypes.byref(w), fake, fake, fake, 256, None, None,
                           None, None)
    assert st == B.MOE_ERR_WORKSPACE_TOO_SMALL
    # misaligned workspace
    st = B.lib.moe_forward(ctypes.byref(cfg), ctypes.byref(w), fake, fake, fake + 16, 1 << 30,
                           None, None, None, None)
    assert st == B.MOE_ERR_INVALID_ARG
    # bias scoring without a bias vector
    cfg2 = _cfg(B, scoring=1)
    st = B.lib.moe_forward(ctypes.byref(cfg2), ctypes.byref(w), fake, fake, fake, 1 << 30, None,
                           None, None, None)
    assert st == B.MOE_ERR_INVALID_ARG
    # a pre-expert norm without its weight vector
    w.pre_expert_norm_w = None
    cfg3 = _cfg(B, pre_expert_norm=True)
    st = B.lib.moe_forward(ctypes.byref(cfg3), ctypes.byref(w), fake, fake, fake, 1 << 30, None,
                           None, None, None)
    assert st == B.MOE_ERR_INVALID_ARG


def test_pre_expert_norm_config(B):
    n = ctypes.c_size_t(0)
    plain = B.moe_workspace_size(_cfg(B))
    normed = B.moe_workspace_size(_cfg(B, pre_expert_norm=True))
    assert normed >= plain + 16 * 256 * 2          # room for the [N, H] normed copy
    for eps in (-1.0, float("inf"), float("nan")):
        cfg = _cfg(B, pre_expert_norm=True, rms_norm_eps=eps)
        assert B.lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == \
            B.MOE_ERR_INVALID_ARG
    cfg = _cfg(B, pre_expert_norm=False, rms_norm_eps=-1.0)   # ignored without the norm
    assert B.lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == B.MOE_OK


def test_zero_tokens_is_a_no_op(B):
    cfg = _cfg(B, num_tokens=0)
    w = B.moe_weights_t()
    fake = 1 << 20
    for n in B.moe_weights_t._fields_:
        setattr(w, n[0], fake)
    w.router_logit_bias = w.correction_bias = w.s_gate = w.s_up = w.s_down = None
    w.sh_gate_vec = None
    assert B.lib.moe_forward(ctypes.byref(cfg), ctypes.byref(w), None, None, None, 0, None, None,
                             None, None) == B.MOE_OK


def test_selftest_refuses_bad_arguments(B):
    assert B.lib.moe_selftest_bounded_wait(None, 1000, None) == B.MOE_ERR_INVALID_ARG
    assert B.lib.moe_selftest_bounded_wait(1 << 20, 0, None) == B.MOE_ERR_INVALID_ARG
    assert B.lib.moe_selftest_bounded_wait((1 << 20) + 8, 1000, None) == B.MOE_ERR_INVALID_ARG
    assert B.lib.moe_selftest_bounded_wait(1 << 20, 10 ** 12, None) == B.MOE_ERR_INVALID_ARG
