"""Replica aggregation of bench.py across ranks (gloo, world size 2, CPU only).

The decode path does not shard across GPUs (every virtual rank runs on one
GPU); `bench.py --gpus N` runs N independent replicas and reports the max of
the ranks' times with a barrier around the timed region.  These tests run the
same helpers in two gloo processes on the host.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        bench.barrier(w)
        # rank-dependent times: the max over ranks must come back on every rank
        got = bench.reduce_max([1.0 + r, 10.0 - r, 0.5 * r], w)
        bench.barrier(w)
        out[r] = (r, w, local, got)
    finally:
        dist.destroy_process_group()


def test_replica_max_over_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert sorted(res) == [0, 1]
    for r in range(world):
        rank, w, local, got = res[r]
        assert (rank, w, local) == (r, world, r)
        assert got == [2.0, 10.0, 0.5]


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max([3.0, 1.0], 1) == [3.0, 1.0]
    bench.barrier(1)  # no-op without a process group
