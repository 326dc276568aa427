"""The bench's multi-rank bookkeeping on CPU with gloo, world size 2: each
rank is an independent replica, the step time is the maximum over ranks and
the reported value is the whole job's units over that time."""

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, rank, world)
        ms = 2.0 + rank                       # rank 1 is the slower replica
        ms_max = bench.reduce_max(ms)
        value = bench.aggregate(1e9, world, ms_max)
        bench.barrier()
        out[rank] = (ms_max, value)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for r in range(world):
        ms_max, value = res[r]
        assert ms_max == 3.0                  # the slowest rank's time, on every rank
        assert value == pytest.approx(2 * 1e9 / 3e-3)


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(1.5) == 1.5
    assert bench.aggregate(10, 1, 1000.0) == 10.0
