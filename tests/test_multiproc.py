"""Multi-rank plumbing of bench.py on CPU (gloo, world size 2): the barrier
and the max-over-ranks reduction of the timed region, and the per-rank
batches of a weak-scaling run (same shape, different draws).  The scan itself
needs no collective: heads and sequences are independent."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from bayesian_scan_gb300 import workloads
    d = bench.Dist(use_gpu=False)
    try:
        d.barrier()
        m = d.max(float(10 + rank))
        w = workloads.get("small")
        w_rank = w if rank == 0 else type(w)(**{**w.__dict__, "seed": w.seed + 7919 * rank})
        x = workloads.make(w_rank, with_mobius=False)
        q.put((rank, d.world, m, float(x["q"].sum())))
    finally:
        d.close()


def test_two_ranks_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    assert [r[1] for r in res] == [2, 2]
    assert [r[2] for r in res] == [11.0, 11.0]          # max over ranks seen by both
    assert res[0][3] != res[1][3]                          # each rank draws its own batch
