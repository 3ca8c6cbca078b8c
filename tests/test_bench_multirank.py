"""bench.py's multi-rank plumbing on the CPU: two gloo ranks, barrier and the
max-over-ranks time (the job time is the slowest rank's).  No GPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    # Rank r "took" 10 + 5 r milliseconds: every rank must see the maximum.
    got = bench.max_over_ranks(10.0 + 5.0 * r, w)
    out[rank] = got
    bench.barrier(w)
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
