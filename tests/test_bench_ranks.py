"""The multi-replica host logic of bench.py on CPU: two gloo ranks, each with
its own timings; both see the maximum, and the whole-job rate counts every
replica's rows over the slowest step."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 3.0 - rank]          # rank 0: (1, 3), rank 1: (2, 2)
        got = bench.max_over_ranks(mine, dist, "cpu")
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_with_two_gloo_ranks():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == [2.0, 3.0] and out[1] == [2.0, 3.0]
    import sys
    sys.path.insert(0, ROOT)
    import bench
    rows = int(bench.ragged_layout()[1][-1])
    assert rows == 2256568
    assert bench.job_rate_gbs(rows, world, 2.0) == pytest.approx(2 * rows * 584 / 2e-3 / 1e9)
    assert bench.job_rate_gbs(rows, world, 2.0, 296) == pytest.approx(2 * rows * 296 / 2e-3 / 1e9)
    assert bench.job_rate_gbs(rows, 1, 2.0) * 2 == pytest.approx(bench.job_rate_gbs(rows, 2, 2.0))


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the reference arm's other ranks exit without work."""
    import argparse
    import sys
    sys.path.insert(0, ROOT)
    import bench
    args = argparse.Namespace(steps=1, warmup=0)
    assert bench.run_reference(args, rank=1, world=2) is None
