"""MoE block forward benchmark: tokens/s and roofline fraction on one GB300.

Headline: the decode workload (N=4 tokens, H=2048, 128 experts of inter 768, top-8, sigmoid-
gated shared expert of inter 512), HBM-bound. The prefill workload (N=4096, Zipf-skewed
routing) is measured in the same run and reported under "prefill" (tensor-bound).

A step is one moe_forward over one batch with inputs resident in HBM; L2 is flushed before every
timed step, outside the timed region: a 512 MiB write, then a 512 MiB read, so that L2 holds no
line of the workload and no dirty line (a write-only flush leaves ~126 MB of dirty lines whose
write-back lands inside the next timed step; that variant is reported too, as "l2_write_only"). Times come from CUDA events on the
launching stream. `--impl reference` times the CPU oracle instead (the only baseline there
is). Multi-GPU runs are independent replicas (the block does not shard): value = all ranks'
tokens / the slowest rank's time.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_layer_08_gb300 import inputs as I  # noqa: E402

METRIC = "MoE-layer tokens/s (prefill N=4096, decode N=4) and % tensor/HBM roofline"
# The FP8 prefill workload cut to 2048 tokens and 32 experts (same H, I, K, block scales): the
# grouped FP8 GEMMs see the same tiles, and a profiler capture holds under 2 GB of device memory.
FP8_PREFILL_SMALL = I.FP8_PREFILL.with_(name="fp8_prefill_n2048_e32", num_tokens=2048,
                                        num_experts=32, router_width=32)
FLUSH_BYTES = 512 << 20


class L2Flush:
    """Evicts the workload from L2 between timed steps: a write of FLUSH_BYTES, then (unless
    `dirty`) a read of as many bytes, which leaves L2 clean."""

    def __init__(self, device, dirty=False):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.acc = torch.empty((), dtype=torch.float32, device=device)
        self.dirty = dirty

    def __call__(self):
        self.w.zero_()
        if not self.dirty:
            torch.sum(self.r, dim=0, out=self.acc)


def workload_config(shape):
    """The workload keys of the JSON line's config, the same on both arms."""
    return {"workload": shape.name, "N": shape.num_tokens, "H": shape.hidden,
            "E": shape.num_experts, "R": shape.router_width, "K": shape.top_k,
            "I": shape.inter, "S": shape.shared_inter, "parallelism": "replicas"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "src": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev: int):
        self.dev = dev
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def routing_stats(inp, idx):
    s = inp.shape
    flat = idx.reshape(-1)
    real = flat[flat < s.num_experts]
    counts = np.bincount(real, minlength=s.num_experts)
    return {"Z": int(real.size), "distinct": int((counts > 0).sum()), "counts": counts}


def algorithmic(inp, rs):
    """Work the method must do (routed rows Z, not tile-padded; touched experts read once)."""
    s = inp.shape
    H, I_, S, R = s.hidden, s.inter, s.shared_inter, s.router_width
    # bytes per expert weight: bf16 2, E4M3 1 (block scales negligible), NVFP4 half a byte
    # of code plus one E4M3 scale per 16
    wb = {I.WDTYPE_FP8_E4M3_B128: 1.0, I.WDTYPE_NVFP4: 0.5 + 1.0 / 16}.get(s.weight_dtype, 2.0)
    own_shared = s.weight_dtype != I.WDTYPE_BF16   # shared expert in launches of its own
    expert_bytes = 3 * I_ * H * wb
    bytes_ = (rs["distinct"] * expert_bytes + 3 * S * H * 2 + R * H * 2
              + 2 * s.num_tokens * H * 2 + (H * 2 if s.shared_gated else 0))
    flops_routed = 6.0 * rs["Z"] * H * I_
    flops = flops_routed + 6.0 * s.num_tokens * H * S + 2.0 * s.num_tokens * H * R
    # with bf16 experts the gate/up and down launches also run the shared expert's projections
    gate_up_flops = 4.0 * rs["Z"] * H * I_ + (0.0 if own_shared else 4.0 * s.num_tokens * H * S)
    down_flops = 2.0 * rs["Z"] * I_ * H + (0.0 if own_shared else 2.0 * s.num_tokens * S * H)
    gate_up_bytes = rs["distinct"] * 2 * I_ * H * wb + (0 if own_shared else 2 * S * H * 2)
    # the decode chain's one kernel reads every touched expert, the shared expert, the router
    # and x, and writes out: all of the step's algorithmic bytes
    ffn_bytes = bytes_
    return {"bytes": bytes_, "flops": flops, "gate_up_flops": gate_up_flops, "down_flops": down_flops,
            "gate_up_bytes": gate_up_bytes, "ffn_bytes": ffn_bytes, "expert_bytes": expert_bytes}


def sources_sha256(paths):
    """SHA-256 over the bytes of the given repository files, in order."""
    import hashlib
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(kernel, workload):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from the committed ncu
    summary (profiles/traffic.json), or None when none was taken or the kernel's sources have
    changed since (the summary records the SHA-256 of the source files it measured)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    for e in rec.get("entries", []):
        if e.get("kernel") != kernel or e.get("workload") != workload:
            continue
        try:
            sha = sources_sha256(e["sources"])
        except (OSError, KeyError):
            return None
        return e["dram_bytes_per_launch"] if sha == e.get("sources_sha256") else None
    return None


def fused_router(cfg, num_sms):
    """Whether the grouped chain routes with the fused tensor-core router (one launch: router
    GEMM, scoring and top-K) -- the library's own rule: more than 64 tokens, a router width
    that is a multiple of 32 up to 384 (of 128 above 256), the contraction split over a
    cluster of at least 2 CTAs, and the shared memory it needs."""
    N, H, R = cfg.num_tokens, cfg.hidden, cfg.router_width
    if N <= 64 or R < 32 or R > 384 or R % 32 or H % 64 or (R > 256 and R % 128):
        return False
    mt, nkb, ks = (N + 127) // 128, H // 64, 1
    while ks < 8 and mt * ks * 2 <= num_sms and nkb % (ks * 2) == 0:
        ks *= 2
    stage = 16384 + R * 128
    nst = min(8, (192 * 1024) // stage, nkb // ks)
    ld = R + 4
    if nst < 1 or (128 - 128 // ks) * ld < 32 * 2 * R:
        return False
    region = (max(nst * stage, 128 * ld * 4) + 7) & ~7
    return region + 1024 + 18 * 8 <= 227 * 1024


def kernels_per_step(B, cfg, num_sms=152):
    """Kernels of this library one forward launches (memsets are not kernels)."""
    per_weight = {0: 2.0, 1: 1.0}.get(cfg.weight_dtype, 0.5625)
    touched = (min(cfg.num_experts, cfg.num_tokens * cfg.top_k) * 3.0 * cfg.inter * cfg.hidden
               * per_weight + 3.0 * cfg.shared_inter * cfg.hidden * 2.0)
    decode = cfg.path == B.PATH_DECODE or (
        cfg.path == B.PATH_AUTO and cfg.num_tokens <= 16 and cfg.inter <= 1024
        and cfg.shared_inter <= 1024 and (cfg.weight_dtype == 0 or cfg.hidden % 256 == 0)
        and touched >= 8.0 * (1 << 20))
    if decode:   # router, top-K, sort, projections, combine (and any pre-expert norm): one kernel
        return 1
    # routing: the fused router (1) or router + top-K (2); then 3 sort, gate/up GEMM, down GEMM,
    # combine; FP8 experts add the token-row quantiser; FP8 and NVFP4 experts run the bf16
    # shared expert in two launches of their own; a pre-expert norm adds its row kernel
    n = (1 if fused_router(cfg, num_sms) else 2) + 6 + (1 if cfg.pre_expert_norm else 0)
    if cfg.weight_dtype == 1:
        n += 1
    if cfg.weight_dtype in (1, 2) and cfg.shared_inter:
        n += 2
    return n


def replicas_value(ms_local, tokens_per_replica, device="cpu"):
    """Independent replicas, one per rank: the job's time is the slowest rank's and its
    throughput every rank's tokens over that time. Returns (ms, tokens/s)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    ms = ms_local
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * tokens_per_replica / (ms / 1000.0)


def barrier():
    if int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist
        dist.barrier()


def time_ours(B, shape, steps, warmup, dev, peaks, with_e2e=True):
    torch.cuda.set_device(dev)
    inp = I.make_inputs(shape, device=f"cuda:{dev}")
    blk = B.MoeBlock(inp)
    N, K = shape.num_tokens, shape.top_k
    idx = torch.empty(N, K, dtype=torch.int32, device=f"cuda:{dev}")
    out = torch.empty_like(inp.x)
    blk(inp.x, out=out, topk_idx_out=idx)
    torch.cuda.synchronize()
    rs = routing_stats(inp, idx.cpu().numpy())
    alg = algorithmic(inp, rs)
    flush = L2Flush(f"cuda:{dev}")
    stream = torch.cuda.current_stream()
    nst = len(B.STAGES)

    def one(events):
        B.moe_forward_profiled(blk.cfg, blk.weights, inp.x, out, blk.workspace, events, stream)

    for _ in range(warmup):
        flush()
        one([None] * (2 * nst))
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    # the timed steps: one event pair around each forward (events between the stages would add
    # their own cost to the step)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for e in ev0 + ev1:     # torch creates the CUDA event on first record
        e.record()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        t_wall0 = time.time()
        for i in range(steps):
            flush()
            ev0[i].record()
            B.moe_forward(blk.cfg, blk.weights, inp.x, out, blk.workspace, stream)
            ev1[i].record()
        torch.cuda.synchronize()
        t_wall = time.time() - t_wall0
    step_ms = [ev0[i].elapsed_time(ev1[i]) for i in range(steps)]
    ms = statistics.mean(step_ms)
    # the same loop after a write-only flush (dirty L2)
    dirty = L2Flush(f"cuda:{dev}", dirty=True)
    for i in range(steps):
        dirty()
        ev0[i].record()
        B.moe_forward(blk.cfg, blk.weights, inp.x, out, blk.workspace, stream)
        ev1[i].record()
    torch.cuda.synchronize()
    ms_dirty = statistics.mean([ev0[i].elapsed_time(ev1[i]) for i in range(steps)])
    del dirty
    # the same loop in the non-deterministic mode (routed down rows FP32-atomic-added into one
    # accumulator per token), where the chain supports it
    ms_atomic = None
    if with_e2e:
        blk_a = B.MoeBlock(inp, deterministic=False)
        for _ in range(warmup):
            flush()
            B.moe_forward(blk_a.cfg, blk_a.weights, inp.x, out, blk_a.workspace, stream)
        for i in range(steps):
            flush()
            ev0[i].record()
            B.moe_forward(blk_a.cfg, blk_a.weights, inp.x, out, blk_a.workspace, stream)
            ev1[i].record()
        torch.cuda.synchronize()
        ms_atomic = statistics.mean([ev0[i].elapsed_time(ev1[i]) for i in range(steps)])
        del blk_a
    # the stage breakdown: the same steps again, with the caller's events around every stage
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nst)] for _ in range(steps)]
    for row in ev:
        for e in row:
            e.record()
    torch.cuda.synchronize()
    for i in range(steps):
        flush()
        one(ev[i])
    torch.cuda.synchronize()
    stage_ms = {n: [] for n in B.STAGES}
    for i in range(steps):
        e = ev[i]
        for s, n in enumerate(B.STAGES):
            stage_ms[n].append(e[2 * s].elapsed_time(e[2 * s + 1]))
    res = {"inp": inp, "rs": rs, "alg": alg, "ms": ms, "ms_dirty": ms_dirty, "ms_atomic": ms_atomic, "stage_ms": {k: statistics.mean(v)
                                                                     for k, v in stage_ms.items()},
           "clocks": clk.summary(), "wall_s": t_wall,
           "launches_per_step": kernels_per_step(
               B, blk.cfg, torch.cuda.get_device_properties(0).multi_processor_count)}
    if with_e2e:
        res["graph"] = time_graph(B, blk, inp, out, flush, steps, warmup)
        hx = torch.empty(inp.x.shape, dtype=inp.x.dtype, pin_memory=True)
        hx.copy_(inp.x.cpu())
        ho = torch.empty(inp.x.shape, dtype=inp.x.dtype, pin_memory=True)
        dx = torch.empty_like(inp.x)
        e2e = []
        for i in range(warmup + steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            dx.copy_(hx, non_blocking=True)
            B.moe_forward(blk.cfg, blk.weights, dx, out, blk.workspace, stream)
            ho.copy_(out, non_blocking=True)
            b.record()
            torch.cuda.synchronize()
            if i >= warmup:
                e2e.append(a.elapsed_time(b))
        res["e2e_ms"] = statistics.mean(e2e)
        res["io_bytes"] = hx.numel() * hx.element_size()
    return res


def time_graph(B, blk, inp, out, flush, steps, warmup):
    """The same forward captured once in a CUDA graph and replayed (L2 flushed before each
    replay, outside the graph). Returns ms per replay, or the reason capture failed."""
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            B.moe_forward(blk.cfg, blk.weights, inp.x, out, blk.workspace, side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            B.moe_forward(blk.cfg, blk.weights, inp.x, out, blk.workspace,
                          torch.cuda.current_stream())
        times = []
        for i in range(warmup + steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            if i >= warmup:
                times.append(a.elapsed_time(b))
        return {"ms_per_step": statistics.mean(times)}
    except Exception as exc:   # reported, not fatal: the stream-launched number stands
        return {"error": f"{type(exc).__name__}: {exc}"[:300]}


def host_cpu():
    """Host cores this process may run on and the CPU model (lscpu, else /proc/cpuinfo)."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for l in out.splitlines():
            if l.strip().startswith("Model name:"):
                model = l.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            for l in open("/proc/cpuinfo"):
                if l.lower().startswith("model name"):
                    model = l.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return {"host_cores": cores, "cpu_model": model or "unknown"}


def _omp_threads(n):
    """Sets the OpenMP thread count of this (the calling) thread's next parallel regions; the
    oracle's library shares the process's libgomp."""
    try:
        import ctypes
        ctypes.CDLL("libgomp.so.1").omp_set_num_threads(int(n))
        return True
    except OSError:
        return False


def _time_oracle(host, tokens, budget_s, max_reps=50):
    from oracle import oracle as O
    O.moe_forward(host, tokens=tokens[:1])   # build + warm-up, untimed
    done, reps, t0 = 0, 0, time.time()
    while True:
        O.moe_forward(host, tokens=tokens)
        done += len(tokens)
        reps += 1
        if time.time() - t0 > budget_s or reps >= max_reps:
            break
    dt = time.time() - t0
    return done / dt, reps, dt


def cpu_oracle_tokens_per_s(inp, budget_s=12.0, max_tokens=None, extra=True):
    """Times the oracle (as it stands) on the host cores on a bounded sample of tokens: the
    given workload with every host core (OpenMP over tokens: a batch of n tokens keeps at
    most n threads busy), and, when `extra`, the tiny and decode workloads on one thread and
    a 64-token sample of the prefill workload on every core."""
    hc = host_cpu()
    n = inp.shape.num_tokens
    tokens = np.arange(n if max_tokens is None else min(n, max_tokens))
    host = inp.to("cpu")
    _omp_threads(hc["host_cores"])
    v, reps, dt = _time_oracle(host, tokens, budget_s)
    res = {"value": v, "unit": "tokens/s", "cores": min(hc["host_cores"], len(tokens)),
           "kind": "oracle", **hc,
           "sample": f"{reps} x {len(tokens)} tokens of the {inp.shape.name} workload "
                     f"(fp64 C oracle, OpenMP over tokens), {dt:.1f} s"}
    if extra:
        per = {}
        if _omp_threads(1):
            for shp, src in ((I.TINY, None), (I.DECODE, host if inp.shape == I.DECODE else None)):
                h = src if src is not None else I.make_inputs(shp)
                t = np.arange(shp.num_tokens)
                tv, treps, tdt = _time_oracle(h, t, 3.0)
                per[shp.name + "_1thread"] = {"value": tv, "unit": "tokens/s", "cores": 1,
                                              "sample": f"{treps} x {len(t)} tokens, {tdt:.1f} s"}
            _omp_threads(hc["host_cores"])
        pre = I.make_inputs(I.PREFILL)
        t = np.linspace(0, I.PREFILL.num_tokens - 1, 64).astype(np.int64)
        pv, preps, pdt = _time_oracle(pre, t, 3.0)
        per[I.PREFILL.name + "_sampled"] = {
            "value": pv, "unit": "tokens/s", "cores": min(hc["host_cores"], len(t)),
            "sample": f"{preps} x 64 evenly spaced tokens of {I.PREFILL.num_tokens}, {pdt:.1f} s"}
        del pre
        res["per_workload"] = per
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the zero-expert, FP8 and tiny workloads")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--profile-only", choices=["decode", "prefill", "fp8", "zero_expert",
                                               "fp8_small", "tiny", "decode_fp8",
                                               "decode_nvfp4", "prefill_nvfp4"],
                    help="run one workload's timing loop only (for ncu captures); prints a "
                         "reduced line")
    args = ap.parse_args()
    warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    shape = I.DECODE
    peaks = load_peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        inp = I.make_inputs(shape)
        times = []
        from oracle import oracle as O
        O.moe_forward(inp, tokens=[0])
        for _ in range(warmup):
            O.moe_forward(inp)
        for _ in range(args.steps):
            t0 = time.time()
            O.moe_forward(inp)
            times.append(time.time() - t0)
        ms = 1000 * statistics.mean(times)
        v = shape.num_tokens / (ms / 1000)
        hc = host_cpu()
        threads = int(os.environ.get("OMP_NUM_THREADS", hc["host_cores"]))
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": workload_config(shape),
                "cpu_baseline": {"value": v, "unit": "tokens/s",
                                 "cores": min(threads, shape.num_tokens), "kind": "oracle",
                                 **hc,
                                 "sample": f"each step: the whole {shape.num_tokens}-token batch"},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    dev = local
    torch.cuda.set_device(dev)
    try:
        from mixture_experts_layer_08_gb300 import binding as B
    except ImportError:
        from mixture_experts_layer_08_gb300 import build as _b
        _b.build()
        from mixture_experts_layer_08_gb300 import binding as B

    if args.profile_only:
        shp = {"decode": I.DECODE, "prefill": I.PREFILL, "fp8": I.FP8_PREFILL,
               "zero_expert": I.ZERO_EXPERT, "fp8_small": FP8_PREFILL_SMALL, "tiny": I.TINY,
               "decode_fp8": I.DECODE_FP8, "decode_nvfp4": I.DECODE_NVFP4,
               "prefill_nvfp4": I.PREFILL_NVFP4}[args.profile_only]
        r = time_ours(B, shp, args.steps, warmup, dev, peaks, with_e2e=False)
        print(json.dumps({"profile_only": shp.name, "ms_per_step": r["ms"], "clocks": r["clocks"],
                          "tokens_per_s": shp.num_tokens / (r["ms"] / 1000.0),
                          "stage_us": {k: 1000 * v for k, v in r["stage_ms"].items()},
                          "Z": r["rs"]["Z"], "distinct_experts": r["rs"]["distinct"]}))
        return

    r = time_ours(B, shape, args.steps, warmup, dev, peaks)
    ms, value = replicas_value(r["ms"], shape.num_tokens, f"cuda:{dev}")
    alg = r["alg"]
    # the decode chain's kernel (timed as the gate/up stage): router, top-K, sort, projections
    # and combine; algorithmic bytes = every touched expert's weights once, the shared expert,
    # the router, x and out
    gu_ms = r["stage_ms"]["gate_up"]
    gu_ach = alg["ffn_bytes"] / (gu_ms / 1000.0) / 1e9
    traffic = measured_traffic("decode_forward_kernel", shape.name)
    step_ach = alg["bytes"] / (ms / 1000.0) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(shape),
        "notes": {"l2": "flushed before every timed step (512 MiB write, then 512 MiB read; "
                        "untimed)",
                  "distinct_experts": r["rs"]["distinct"]},
        "roofline": {"bound": "hbm", "kernel": "decode_forward_kernel",
                     "achieved": gu_ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gu_ach / peaks["hbm_gbs"], "traffic": traffic,
                     "peak_src": peaks["src"],
                     "step_achieved_gbs": step_ach, "step_frac": step_ach / peaks["hbm_gbs"],
                     "algorithmic_bytes_per_launch": alg["ffn_bytes"],
                     "algorithmic_bytes_per_step": alg["bytes"]},
        "l2_write_only": {"ms_per_step": r["ms_dirty"],
                          "value": world * shape.num_tokens / (r["ms_dirty"] / 1000.0),
                          "unit": "tokens/s"},
        "atomic_accumulation": {"ms_per_step": r["ms_atomic"],
                                "value": world * shape.num_tokens / (r["ms_atomic"] / 1000.0),
                                "unit": "tokens/s",
                                "note": "deterministic=0: down rows FP32-atomic-added per token"},
        "stage_us": {k: 1000 * v for k, v in r["stage_ms"].items()},
        "gpu_launches": r["launches_per_step"] * 3 * args.steps,
        "clocks": r["clocks"],
        "e2e": {"value": world * shape.num_tokens / (r["e2e_ms"] / 1000.0), "unit": "tokens/s",
                "h2d_bytes_per_step": r["io_bytes"], "d2h_bytes_per_step": r["io_bytes"]},
        "graph_replay": (dict(r["graph"], value=world * shape.num_tokens /
                              (r["graph"]["ms_per_step"] / 1000.0), unit="tokens/s")
                         if "ms_per_step" in r["graph"] else r["graph"]),
    }
    if not args.no_prefill:
        p = time_ours(B, I.PREFILL, max(3, args.steps // 2), warmup, dev, peaks, with_e2e=False)
        pa = p["alg"]
        gu = p["stage_ms"]["gate_up"]
        gu_tf = pa["gate_up_flops"] / (gu / 1000.0) / 1e12
        p_traffic = measured_traffic("gemm_bf16_kernel<256,SwiGLU>", I.PREFILL.name)
        line["prefill"] = {
            "workload": I.PREFILL.name, "value": I.PREFILL.num_tokens / (p["ms"] / 1000.0),
            "unit": "tokens/s", "ms_per_step": p["ms"],
            "stage_us": {k: 1000 * v for k, v in p["stage_ms"].items()},
            "roofline": {"bound": "tensor", "kernel": "gemm_bf16_kernel<256,SwiGLU>",
                         "achieved": gu_tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": gu_tf / peaks["bf16_tflops"], "traffic": p_traffic,
                         # the same launch against the HBM roofline: measured DRAM bytes
                         # (ncu, one launch) over its CUDA-event time
                         "hbm_frac": (p_traffic / (gu / 1000.0) / 1e9 / peaks["hbm_gbs"]
                                      if p_traffic else None),
                         "down_kernel": "gemm_bf16_kernel<256,bf16>",
                         "down_tflops": pa["down_flops"] / (p["stage_ms"]["down"] / 1000.0) / 1e12,
                         "down_frac": pa["down_flops"] / (p["stage_ms"]["down"] / 1000.0) / 1e12
                         / peaks["bf16_tflops"],
                         "down_traffic": measured_traffic("gemm_bf16_kernel<256,bf16>",
                                                          I.PREFILL.name),
                         "step_tflops": pa["flops"] / (p["ms"] / 1000.0) / 1e12,
                         "step_frac": pa["flops"] / (p["ms"] / 1000.0) / 1e12 / peaks["bf16_tflops"]},
            "Z": p["rs"]["Z"], "max_expert_rows": int(p["rs"]["counts"].max()),
            "min_expert_rows": int(p["rs"]["counts"].min()),
            "clocks": p["clocks"]}
        line["gpu_launches"] += p["launches_per_step"] * max(3, args.steps // 2)
    if not args.no_extra:
        extra = {}
        for shp in (I.ZERO_EXPERT, I.FP8_PREFILL, I.TINY, I.DECODE_PRENORM, I.DECODE_FP8,
                    I.DECODE_NVFP4, I.PREFILL_NVFP4):
            x = time_ours(B, shp, max(3, args.steps // 2), warmup, dev, peaks, with_e2e=False)
            xa = x["alg"]
            fp8 = shp.weight_dtype == I.WDTYPE_FP8_E4M3_B128
            nv = shp.weight_dtype == I.WDTYPE_NVFP4   # dequantised to bf16: the bf16 MMA
            tpeak = peaks["bf16_tflops"] * (2.0 if fp8 else 1.0)
            gu = x["stage_ms"]["gate_up"]
            extra[shp.name] = {
                "value": shp.num_tokens / (x["ms"] / 1000.0), "unit": "tokens/s",
                "ms_per_step": x["ms"],
                "stage_us": {k: 1000 * v for k, v in x["stage_ms"].items()},
                "gate_up_tflops": xa["gate_up_flops"] / (gu / 1000.0) / 1e12,
                "gate_up_tensor_frac": xa["gate_up_flops"] / (gu / 1000.0) / 1e12 / tpeak,
                "gate_up_hbm_frac": xa["gate_up_bytes"] / (gu / 1000.0) / 1e9 / peaks["hbm_gbs"],
                "tensor_peak_tflops": tpeak,
                "tensor_peak_src": "2 x measured bf16 (nominal fp8:bf16 ratio)" if fp8 else "measured bf16",
                "down_tflops": xa["down_flops"] / (x["stage_ms"]["down"] / 1000.0) / 1e12
                if x["stage_ms"]["down"] > 0.01 else None,
                "down_tensor_frac": xa["down_flops"] / (x["stage_ms"]["down"] / 1000.0) / 1e12 / tpeak
                if x["stage_ms"]["down"] > 0.01 else None,
                "gate_up_traffic": measured_traffic(
                    "gemm_fp8_kernel<0>" if fp8 else "gemm_nvfp4_kernel<256,SwiGLU>" if nv
                    else "gemm_bf16_kernel<256,SwiGLU>", shp.name),
                "down_traffic": measured_traffic(
                    "gemm_fp8_kernel<1>" if fp8 else "gemm_nvfp4_kernel<256,bf16>" if nv
                    else "gemm_bf16_kernel<256,bf16>", shp.name),
                "step_hbm_frac": xa["bytes"] / (x["ms"] / 1000.0) / 1e9 / peaks["hbm_gbs"],
                "step_tensor_frac": xa["flops"] / (x["ms"] / 1000.0) / 1e12 / tpeak,
                "Z": x["rs"]["Z"], "distinct_experts": x["rs"]["distinct"]}
            line["gpu_launches"] += x["launches_per_step"] * max(3, args.steps // 2)
            del x
            torch.cuda.empty_cache()
        line["other_workloads"] = extra
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_oracle_tokens_per_s(r["inp"])
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
