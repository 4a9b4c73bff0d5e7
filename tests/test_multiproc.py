"""The benchmark's multi-process path on CPU: two gloo ranks, the barrier and
the max/sum reductions the JSON line is computed from (no GPU)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    dist = bench.init_dist(ws, "gloo")
    bench.barrier(dist)
    # each rank "timed" a different duration and processed the same work
    mx = bench.max_over_ranks(dist, 10.0 + rank)
    sm = bench.sum_over_ranks(dist, 1.5)
    out.put((rank, mx, sm))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_json_line():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    # every rank sees the slowest rank's time and the whole job's work
    assert [r[1] for r in res] == [11.0, 11.0]
    assert [r[2] for r in res] == [3.0, 3.0]


def test_single_process_needs_no_process_group():
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 2.5) == 2.5
    assert bench.sum_over_ranks(None, 2.5) == 2.5
