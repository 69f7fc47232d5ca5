"""The N>1 path of bench.py on CPU: two gloo ranks exercise the replica
plumbing (rendezvous on 127.0.0.1, barrier, max-over-ranks timing, the
whole-job value as all ranks' bytes over the slowest rank's time).  The path
has no data exchange, so nothing else crosses ranks."""
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


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # each replica reports its own elapsed time; the job takes the slowest
        elapsed = 10.0 + 5.0 * rank
        slowest = bench.max_over_ranks(elapsed, world)
        bytes_per_rank = 1000
        value = bytes_per_rank * world / slowest
        results[rank] = (slowest, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        got = dict(results)
    assert got[0] == got[1] == (15.0, 2000 / 15.0)
