"""Replica aggregation of bench.py over two gloo ranks on CPU (no GPU): the
reported time is the slowest rank's, the work is every rank's."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier()
        ms, units = bench.reduce_max_sum(1.5 + rank, 100.0 * (rank + 1))
        bench.barrier()
        out[rank] = (ms, units)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_sum_work():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == (2.5, 300.0) and res[1] == (2.5, 300.0)


def test_single_process_passthrough():
    import bench
    assert not (dist.is_available() and dist.is_initialized())
    assert bench.reduce_max_sum(3.0, 7.0) == (3.0, 7.0)
