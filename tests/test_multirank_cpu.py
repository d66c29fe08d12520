"""The multi-GPU bench path runs one replica of the block per rank and
reduces only its timings across ranks. Checked here with two gloo ranks on
the CPU: the reduction returns every rank the element-wise maximum, and the
whole-job value divides the slowest rank's step time by the replica count."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    vals = [10.0 + rank, 5.0 - rank, 1.0 * rank]
    red = bench.max_over_ranks(vals)
    out[rank] = red
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    mgr = mp.get_context("spawn").Manager()  # no fork of a multi-threaded process
    out = mgr.dict()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        assert out[r] == [11.0, 5.0, 1.0]


def test_single_rank_is_identity_and_job_value():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.job_value(80.0, 1) == 80.0
    assert bench.job_value(80.0, 4) == 20.0
