"""The benchmark's multi-rank host logic (per-rank seeds, max-over-ranks timing, summed work) on
two gloo ranks on CPU."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, l = bench.dist_env()
        t = bench.max_over_ranks(10.0 + rank)
        s = bench.sum_over_ranks(100.0 * (rank + 1))
        seed = bench.rank_seed(1002, rank)
        seeds = [None] * world
        dist.all_gather_object(seeds, seed)
        bench.barrier()
        q.put((rank, r, w, l, t, s, seeds))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
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
    for rank, r, w, l, t, s, seeds in res:
        assert (r, w, l) == (rank, 2, rank)
        assert t == 11.0          # max over ranks
        assert s == 300.0         # work summed over ranks
        assert len(set(seeds)) == 2  # independent batches per rank
