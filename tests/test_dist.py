"""The multi-rank timing path of bench.py on CPU: two gloo ranks agree on the
slowest rank's time and on the whole-job rate (replicas, no data exchange)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    bench.barrier(w)
    mine = 0.5 + rank                              # rank 1 is the slow one
    slowest = bench.max_over_ranks(mine, w)
    rate = bench.aggregate(per_rank_units=10.0, world=w, seconds_max=slowest)
    out[rank] = (slowest, rate)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == (1.5, 20.0 / 1.5)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.aggregate(10.0, 1, 2.0) == 5.0
