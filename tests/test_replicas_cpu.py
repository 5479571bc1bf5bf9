"""The N-GPU benchmark path (independent replicas, no data-path collective) on CPU ranks:
two gloo processes, each with its own step time; the job's time must be the slower rank's and
its throughput both ranks' tokens over that time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier()
        ms, value = bench.replicas_value(1.0 + rank, 4)   # rank r: (1 + r) ms per 4 tokens
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, value in got:
        assert ms == pytest.approx(2.0)                    # the slower rank
        assert value == pytest.approx(2 * 4 / 0.002)       # both ranks' tokens


def test_single_process_is_its_own_job(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "1")
    import bench
    ms, value = bench.replicas_value(0.5, 4)
    assert ms == 0.5 and value == pytest.approx(8000.0)
