"""The benchmark's multi-process timing logic on CPU: two gloo ranks.

bench.py runs one replica of the workload per GPU (weak scaling, no collective
on the data path); the job's time per step is the slowest rank's and its
throughput counts every rank's tokens.  Here two CPU processes with different
local times check that aggregation through torch.distributed (gloo, world
size 2), without a GPU.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(local_ms[rank], dist)
        out[rank] = ms
        out[world + rank] = bench.job_tokens_per_s(world, 131072, ms)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world, port = 2, _free_port()
    local_ms = [2.5, 3.75]
    out = torch.zeros(2 * world, dtype=torch.float64).share_memory_()
    mp.spawn(_rank_main, args=(world, port, local_ms, out), nprocs=world, join=True)
    # every rank sees the slowest rank's time ...
    assert out[0].item() == pytest.approx(3.75) and out[1].item() == pytest.approx(3.75)
    # ... and the throughput counts both ranks' tokens over that time
    expect = 2 * 131072 / 3.75e-3
    assert out[2].item() == pytest.approx(expect) and out[3].item() == pytest.approx(expect)


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.job_tokens_per_s(1, 1000, 2.0) == pytest.approx(5e5)
