"""moe_forward_decode_noalloc: the decode chain for callers that cannot allocate device
memory (a plugin inside another runtime that owns all allocations, or a latency-critical
loop where cudaMalloc's device-wide synchronisation is not acceptable). It runs on a fixed
4 MiB device array owned by the library instead of a caller workspace.

Checked against the workspace entry point (moe_forward) on two calls in a row, with the
output tolerance the other parity tests use. Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_08_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from mixture_experts_layer_08_gb300 import build as _b
    _b.build()
    from mixture_experts_layer_08_gb300 import binding
    fn = binding.lib.moe_forward_decode_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(binding.moe_config_t), ctypes.POINTER(binding.moe_weights_t),
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return binding


def _noalloc(B, cfg, w, x, out):
    return B.lib.moe_forward_decode_noalloc(ctypes.byref(cfg), ctypes.byref(w), x.data_ptr(),
                                            out.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("shape", [I.DECODE, I.TINY, I.DECODE.with_(num_tokens=16)],
                         ids=["decode_n4", "tiny_n16", "decode_n16"])
def test_noalloc_matches_workspace_entry_point(B, shape):
    """Deterministic mode: both entry points run the same kernel on the same inputs, so the
    outputs must agree bit for bit on both calls (a scratch region the second call reused
    without clearing would show here); the tolerance check is the one the parity tests use.
    Then one call in the atomic-accumulation mode, whose FP32 accumulator the kernel clears in
    the shared array itself, against moe_forward in the same mode within that tolerance."""
    inp = I.make_inputs(shape, device="cuda")
    w = B.make_weights(inp)
    for det in (True, False):
        cfg = B.make_config(shape, det, B.PATH_DECODE)
        ref = torch.empty_like(inp.x)
        B.moe_forward(cfg, w, inp.x, ref, B.alloc_workspace(cfg))
        torch.cuda.synchronize()
        r = ref.float().cpu().numpy()
        for _ in range(2 if det else 1):
            out = torch.full_like(inp.x, float("nan"))
            assert _noalloc(B, cfg, w, inp.x, out) == B.MOE_OK
            torch.cuda.synchronize()
            got = out.float().cpu().numpy()
            err = np.abs(got - r)
            assert (err <= 2e-2 + 2e-2 * np.abs(r)).all(), f"max err {err.max()}"
            assert np.linalg.norm(got - r) <= 1e-2 * np.linalg.norm(r)
            if det:
                assert torch.equal(out, ref)


def test_noalloc_rejects_what_it_cannot_hold(B):
    inp = I.make_inputs(I.TINY, device="cuda")
    w = B.make_weights(inp)
    out = torch.empty_like(inp.x)
    too_many = B.make_config(I.TINY.with_(num_tokens=17))
    assert _noalloc(B, too_many, w, inp.x, out) == B.MOE_ERR_UNSUPPORTED
    grouped = B.make_config(I.TINY, True, B.PATH_GROUPED)
    assert _noalloc(B, grouped, w, inp.x, out) == B.MOE_ERR_UNSUPPORTED
    # a decode config whose scratch exceeds the 4 MiB array (never launched: refused first)
    big = B.make_config(I.DECODE.with_(num_tokens=16, top_k=32, hidden=8192, inter=1024))
    assert B.moe_workspace_size(big) > (4 << 20)
    assert _noalloc(B, big, w, inp.x, out) == B.MOE_ERR_WORKSPACE_TOO_SMALL


def test_noalloc_status_word_reads_ok_after_a_call(B):
    """moe_noalloc_read_device_status reads the status word of the no-alloc array: MOE_OK
    after a forward whose device waits all completed."""
    fn = B.lib.moe_noalloc_read_device_status
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
    inp = I.make_inputs(I.TINY, device="cuda")
    w = B.make_weights(inp)
    cfg = B.make_config(I.TINY, True, B.PATH_DECODE)
    out = torch.empty_like(inp.x)
    assert _noalloc(B, cfg, w, inp.x, out) == B.MOE_OK
    st = ctypes.c_int32(-1)
    assert fn(torch.cuda.current_stream().cuda_stream, ctypes.byref(st)) == B.MOE_OK
    assert st.value == B.MOE_OK
