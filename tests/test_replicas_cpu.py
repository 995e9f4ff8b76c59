"""The replicated bench's aggregation on CPU (gloo, world size 2, 127.0.0.1): every rank
gets the slowest rank's time, and the whole-job throughput counts every rank's units
against that time.  No data-path collective exists; this is the only cross-rank step."""
from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        got = bench.max_over_ranks_of(times[rank], world, "cpu")
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world, port = 2, _free_port()
    times = [3.5, 7.25]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, times, out), nprocs=world, join=True)
        assert out[0] == out[1] == 7.25


def test_job_throughput_counts_every_replica():
    import bench
    # two replicas, 100 units each per step, 10 steps, slowest rank 2 ms in all
    assert bench.job_throughput(100, 10, 2.0, 2) == pytest.approx(2 * 100 * 10 / 2e-3)
    assert bench.job_throughput(100, 10, 2.0, 1) == pytest.approx(100 * 10 / 2e-3)
    assert bench.max_over_ranks_of(1.5, 1, "cpu") == 1.5
