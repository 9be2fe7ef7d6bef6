"""Multi-rank host logic of bench.py on the CPU: two gloo ranks (the GPU run
uses one process per GPU over NCCL with the same helpers).  Each rank times a
different step; both must report the slowest rank's time, and the whole-job
throughput counts every rank's tokens over that time."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, local_ms, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(local_ms[rank], dist, "cpu")
        q.put((rank, ms, bench.job_throughput(8192, world, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    local_ms = [0.625, 0.700]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, local_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [0.700, 0.700]
    assert res[0][2] == pytest.approx(2 * 8192 / 0.700e-3)


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, None, "cpu") == 1.5
    assert bench.job_throughput(8192, 1, 0.5) == pytest.approx(8192 / 0.5e-3)
