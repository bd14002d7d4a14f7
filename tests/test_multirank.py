"""The benchmark's multi-rank host logic on CPU: two gloo ranks, no GPU.

bench.py runs one replica of the workload per GPU (weak scaling, no collective on the data path);
its only cross-rank steps are the barriers around the timed region and the max-over-ranks of the
elapsed time.  This runs those helpers in two processes with the gloo backend.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r = bench.init_dist("gloo")
    assert (w, r) == (world, rank)
    bench.barrier(world)
    elapsed = 1.0 + rank  # rank 1 is the slow one
    m = bench.max_over_ranks(elapsed, world)
    seed = bench.rank_seed(0, rank)
    wl = bench.make_workload("decode", seed) if rank < 2 else None
    value = bench.aggregate_throughput(256, 10, world, m)
    results[rank] = (m, seed, float(wl.q[0, 0]), value)
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks_report_slowest_time_and_distinct_replicas():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=300)
            assert p.exitcode == 0
        res = dict(results)
    assert res[0][0] == res[1][0] == 2.0          # max over ranks
    assert res[0][1] != res[1][1]                 # each rank draws its own replica
    assert res[0][2] != res[1][2]
    assert res[0][3] == pytest.approx(256 * 10 * 2 / 2.0)
