"""The N>1 host logic of bench.py on CPU: two gloo ranks (127.0.0.1), each with its
own timing, agree on the slowest rank's time, and the whole-job throughput counts the
work of every rank over that time.  The path has no data-path collective (replicas
only), so this timing reduction and the barrier are the only cross-rank steps."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = 30.0 + 5.0 * rank  # this rank's own step time
        slow = bench.max_over_ranks(dist, ms, "cpu")
        flops = 42.0e12  # one rank's work per step
        out[rank] = (slow, bench.job_tflops(world, flops, slow))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    slowest = 30.0 + 5.0 * (world - 1)
    for r in range(world):
        ms, tflops = out[r]
        assert ms == slowest
        assert tflops == pytest.approx(world * 42.0e12 / (slowest * 1e-3) / 1e12)


def test_single_process_needs_no_collective():
    assert bench.max_over_ranks(None, 12.5, "cpu") == 12.5
    assert bench.job_tflops(1, 42.0e12, 32.5) == pytest.approx(42.0e12 / 32.5e-3 / 1e12)
