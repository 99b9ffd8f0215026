"""The benchmark's multi-rank logic on CPU (gloo, world size 2): every rank
runs an independent replica, the time is the maximum over ranks, the value is
the sum of all ranks' work, and the reference arm prints from rank 0 only."""
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


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 10.0 + 5.0 * rank                 # rank 1 is the slowest replica
    ms_max = bench.max_over_ranks(local_ms)
    value = bench.whole_job_tflops(world, 2e12, ms_max)
    # a decision every rank must share (the end-to-end leg's memory check):
    # one rank without room makes all of them skip
    agreed = bench.min_over_ranks(1.0 if rank == 0 else 0.0)

    class Args:
        config, steps, warmup = "smoke", 1, 3
    ref = bench.run_reference(Args(), rank)
    out[rank] = (ms_max, value, ref is None, agreed)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_gloo():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        ms_max, value, ref_none, agreed = out[rank]
        assert ms_max == 15.0
        assert agreed == 0.0
        assert value == pytest.approx(2 * 2e12 / 15e-3 / 1e12)
        assert ref_none == (rank != 0)


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.min_over_ranks(2.5) == 2.5
    assert bench.whole_job_tflops(1, 1e12, 1000.0) == pytest.approx(1.0)
