"""Replica timing of bench.py on CPU: two gloo ranks, each with its own time;
the job's time is the slowest rank's and the rate counts every rank's units."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = 10.0 * (rank + 1)          # rank 1 is the slow one
        ms_max = bench.max_over_ranks(ms, "cpu", world)
        out[rank] = (ms_max, bench.whole_job_rate(1000.0, world, ms_max))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_rate_with_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms_max, rate = res[r]
        assert ms_max == pytest.approx(20.0)
        assert rate == pytest.approx(2 * 1000.0 / 0.020)


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(7.5, "cpu", 1) == 7.5
    assert bench.whole_job_rate(500.0, 1, 250.0) == pytest.approx(2000.0)
