"""The benchmark's multi-rank host logic on CPU with the gloo backend
(world size 2): every rank's time reduces to the slowest rank's, and the
whole-job value of replicated ranks is world x per-rank work / that time.

The attention path has no exchange step (every (batch, kv head) unit is
independent), so N GPUs run N replicas; only this timing aggregation spans
ranks, and it runs the same on gloo as on NCCL.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        mine = 10.0 + 5.0 * rank  # rank 1 is the slow one
        slow = bench.max_over_ranks(mine, torch.device("cpu"))
        results[rank] = (w, r, local, slow, bench.replica_throughput(1e12, slow * 1e-3, w))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        got = dict(results)
    for rank in range(world):
        w, r, local, slow, value = got[rank]
        assert (w, r, local) == (world, rank, rank)
        assert slow == 15.0                      # max over ranks, seen by every rank
        assert value == pytest.approx(2 * 1e12 / 15e-3)


def test_single_process_is_its_own_maximum():
    import torch
    import bench
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
    assert bench.replica_throughput(6.0, 2.0, 1) == 3.0
