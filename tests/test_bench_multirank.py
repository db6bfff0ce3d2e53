"""The multi-rank path of bench.py on CPU: two gloo ranks (replicas) each time
their own step; both must report the slowest rank's time, and the whole-job
value counts the work of every rank in that time (weak scaling)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        ms = bench.max_over_ranks(times[rank], w, "cpu")
        out[rank] = (ms, bench.job_value(1e12, w, ms))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    world, times = 2, [3.0, 5.0]
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True)
    for rank in range(world):
        ms, value = out[rank]
        assert ms == max(times)
        # 1e12 units per rank, both ranks, in 5 ms -> 400 (units / 1e12 per second)
        assert value == pytest.approx(2 * 1e12 / 5e-3 / 1e12)


def test_single_rank_is_unchanged():
    assert bench.max_over_ranks(4.0, 1, "cpu") == 4.0
    assert bench.job_value(2e12, 1, 4.0) == pytest.approx(500.0)
