"""The N-GPU bench path on CPU: two gloo ranks run independent replicas; the
job time is the slowest rank's and the rate counts every rank's rows."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], world, "cpu")
        out[rank] = (ms, bench.job_rate(64, 10, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_time():
    world = 2
    times = [3.0, 5.0]  # ms for 10 steps of 64 rows on each rank
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), times, out), nprocs=world,
                       join=True, start_method="spawn")
    for r in range(world):
        ms, rate = out[r]
        assert ms == 5.0
        assert rate == pytest.approx(64 * 10 * 2 / 5e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1, "cpu") == 2.5
    assert bench.job_rate(8, 4, 1, 2.0) == pytest.approx(8 * 4 / 2e-3)
