"""The bench's N-rank host logic on CPU: two gloo ranks (no GPU).

The path does not shard beyond independent replicas (every batch row is independent),
so `bench.py --gpus N` runs N replicas: the only cross-rank steps are the barrier around
the timed region and the max over ranks of the measured time. Those run here as two
processes over gloo on 127.0.0.1.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    ws, r, local = bench.dist_setup()
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(ws)
    t = bench.max_over_ranks(10.0 + 5.0 * rank, ws)   # each rank's own time
    out[rank] = t
    bench.barrier(ws)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_ranks_barrier_and_max_time():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, join=True, start_method="spawn")
    assert dict(out) == {0: 15.0, 1: 15.0}   # every rank reports the slowest rank's time


def test_single_rank_needs_no_process_group():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    ws, rank, local = bench.dist_setup()
    assert (ws, rank) == (1, 0)
    assert bench.max_over_ranks(3.5, ws) == 3.5
    bench.barrier(ws)   # no-op
