"""bench.py's multi-rank aggregation on CPU: two gloo ranks with different timed-region
lengths both see the slowest one, and the whole-job throughput counts every rank's work."""
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


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.slowest_rank_ms(times[rank], world, torch.device("cpu"))
        out[rank] = (ms, bench.job_tflops(1e12, 3, world, ms))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(10.0, 25.0), (40.0, 5.0)])
def test_two_ranks_take_the_slowest(times):
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), list(times), out), nprocs=world, join=True)
    slow = max(times)
    for r in range(world):
        ms, tf = out[r]
        assert ms == slow
        assert tf == pytest.approx(1e12 * 3 * world / (slow / 1e3) / 1e12)


def test_single_rank_is_unchanged():
    assert bench.slowest_rank_ms(12.5, 1, None) == 12.5
    assert bench.job_tflops(2e12, 2, 1, 1000.0) == pytest.approx(4.0)
