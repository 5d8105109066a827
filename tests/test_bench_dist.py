"""bench.py's multi-rank bookkeeping on CPU: two gloo ranks, max time, summed work."""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        ms, units = bench.aggregate_over_ranks(10.0 + 5.0 * rank, 100.0 * (rank + 1), world)
        out[rank] = (ms, units)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_takes_max_time_and_sums_work():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1] == (15.0, 300.0)


def test_single_rank_is_identity():
    assert bench.aggregate_over_ranks(3.5, 7.0, 1) == (3.5, 7.0)
    assert bench.dist_env()[1] >= 1
