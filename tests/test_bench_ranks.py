"""The multi-rank host logic of bench.py on CPU: two gloo ranks (replicas, weak scaling)
reduce their step times with MAX and report the whole job's tokens/s from the slowest rank."""
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + 0.25 * rank, 2.0 - 0.5 * rank]          # step ms, e2e ms of this rank
        ms, e2e = bench.max_over_ranks(mine, world, "cpu")
        dist.barrier()
        out[rank] = (ms, e2e, bench.whole_job_rate(world, 2048, ms))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_rank():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        ms, e2e, rate = out[r]
        assert ms == pytest.approx(1.25) and e2e == pytest.approx(2.0)   # max over ranks
        assert rate == pytest.approx(2 * 2048 / 1.25e-3)                  # whole job, weak scaling


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1, "cpu") == [3.0, 4.0]
    assert bench.whole_job_rate(1, 2048, 2.0) == pytest.approx(1.024e6)
