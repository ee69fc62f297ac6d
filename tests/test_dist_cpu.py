"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

On the GPU pool every run uses one GPU; the N > 1 bench path runs independent
replicas (no collective in the data path).  This checks its host side: the
barrier, the max-over-ranks timing, per-rank seeds and the aggregate value.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench._barrier(world)
        t = bench._max_over_ranks(1.5 + rank, world)          # rank 1 is the slow one
        seeds = [None] * world
        dist.all_gather_object(seeds, bench.rank_seed(rank))
        v = bench.aggregate_value(1000, 10, world, t)
        q.put((rank, t, seeds, v))
    finally:
        dist.destroy_process_group()


def test_two_rank_host_logic():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, seeds, v in res:
        assert t == 2.5                                    # max over ranks, on every rank
        assert len(set(seeds)) == 2                        # independent weights per rank
        assert v == pytest.approx(1000 * 10 * 2 / 2.5 / 1e9)
