"""The multi-process harness of bench.py on CPU (gloo, world size 2): each
rank runs an independent replica; the timing is the slowest rank's and the
rate counts every rank's rows."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = 0.5 + rank          # rank 1 is the slow one
    slowest = bench.max_over_ranks(local)
    out[rank] = (slowest, bench.replica_rate(1000, world, slowest), bench.dist_env())
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas():
    import torch.multiprocessing as mp
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
    for r in (0, 1):
        slowest, rate, env = out[r]
        assert slowest == pytest.approx(1.5)
        assert rate == pytest.approx(2 * 1000 / 1.5)
        assert env == (2, r, r)


def test_single_process_uses_local_time():
    import bench
    assert bench.max_over_ranks(0.25) == 0.25
    assert bench.replica_rate(131072, 1, 0.5) == 262144
