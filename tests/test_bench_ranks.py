"""Multi-process (gloo, world size 2, CPU) check of the benchmark's cross-rank
timing: the job's step time is the slowest replica's, and the job's throughput
counts every replica's units over that time (weak scaling)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, per_rank_ms, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms_max = bench.max_over_ranks(per_rank_ms[rank], world, "cpu")
        out[rank] = (ms_max, bench.job_rate(1000.0, world, ms_max))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_world2():
    world = 2
    per_rank_ms = [1.5, 2.5]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), per_rank_ms, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms_max, rate = res[rank]
        assert ms_max == 2.5
        assert rate == pytest.approx(world * 1000.0 / 2.5e-3)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)
