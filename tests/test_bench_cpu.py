"""Host logic of the benchmark (no GPU): the launch count it claims per forward and the rule
that a recorded DRAM-traffic figure is reported only while the measured kernel's sources are
unchanged."""
import importlib.util
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test",
                                                  os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


@pytest.fixture(scope="module")
def B():
    from mixture_experts_layer_08_gb300 import build as _b
    _b.build()
    from mixture_experts_layer_08_gb300 import binding
    return binding


def test_traffic_reported_only_while_sources_match(tmp_path, monkeypatch):
    b = _bench()
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_text("kernel, first version")
    entry = {"kernel": "k", "workload": "w", "sources": ["k.cu"],
             "dram_bytes_per_launch": 123, "sources_sha256": b.sources_sha256(["k.cu"])}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"entries": [entry]}))
    assert b.measured_traffic("k", "w") == 123
    assert b.measured_traffic("k", "another workload") is None
    assert b.measured_traffic("another kernel", "w") is None
    src.write_text("kernel, edited")
    assert b.measured_traffic("k", "w") is None
    src.unlink()
    assert b.measured_traffic("k", "w") is None


def test_committed_traffic_records_are_well_formed():
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for e in rec["entries"]:
        assert e["dram_bytes_per_launch"] == e["dram_read_bytes"] + e["dram_write_bytes"]
        assert len(e["sources_sha256"]) == 64 and e["command"].startswith("ncu ")
        assert "--clock-control none" in e["command"]
        for p in e["sources"]:
            assert os.path.exists(os.path.join(ROOT, p)), p


def test_launches_per_forward(B):
    from mixture_experts_layer_08_gb300 import inputs as I
    b = _bench()
    n = lambda shape, path=B.PATH_AUTO: b.kernels_per_step(B, B.make_config(shape, True, path))
    assert n(I.DECODE) == 1                      # one cooperative kernel
    assert n(I.TINY) == 8                        # 1.6 MB of weights: the grouped chain
    assert n(I.TINY, B.PATH_DECODE) == 1
    assert n(I.DECODE_PRENORM) == 1              # the norm runs in its phase 0
    assert n(I.PREFILL) == 7                     # fused router, 3 sort, 2 GEMMs, combine
    assert n(I.PREFILL.with_(pre_expert_norm=True)) == 8
    assert n(I.PREFILL.with_(num_experts=144, router_width=144)) == 8   # 144 % 32: not fused
    assert n(I.ZERO_EXPERT) == 7                 # a 384-wide router, fused
    assert n(I.DECODE, B.PATH_GROUPED) == 8      # 4 tokens: router + top-K
    assert n(I.FP8_PREFILL) == 8                 # + the token-row quantiser, no shared expert
    assert n(I.FP8_PREFILL.with_(shared_inter=512)) == 10
    assert n(I.DECODE_FP8) == 1                  # E4M3 experts through the decode kernel too
    assert n(I.DECODE_FP8, B.PATH_GROUPED) == 11
    assert n(I.DECODE_NVFP4) == 1                # NVFP4 experts through the decode kernel
    assert n(I.DECODE_NVFP4, B.PATH_GROUPED) == 10   # grouped: shared expert apart
    assert n(I.PREFILL_NVFP4) == 9
