"""The benchmark's multi-rank path on CPU: two gloo ranks.

With N replicas (one per GPU under torchrun) the reported value is every
rank's bytes over the slowest rank's time, and the ranks meet at a barrier
on both sides of the timed region.  This runs that aggregation with two
processes on the gloo backend (no GPU), giving the ranks different local
times, and checks both ranks see the same maximum and the same value.
"""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        bench.barrier(w)
        local_ms = 10.0 * (rank + 1)            # rank 1 is the slow one
        value, max_ms = bench.aggregate(1e9, 5, local_ms, w)
        bench.barrier(w)
        q.put((r, w, local, value, max_ms))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_all_bytes_over_the_slowest_time():
    pytest.importorskip("torch")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(2))
    # 2 ranks x 1e9 B x 5 steps over the slower rank's 20 ms = 500 GB/s
    for r, (rank, world, local, value, max_ms) in enumerate(got):
        assert (rank, world, local) == (r, 2, r)
        assert max_ms == pytest.approx(20.0)
        assert value == pytest.approx(500.0)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    value, max_ms = bench.aggregate(2e9, 4, 8.0, 1)
    assert max_ms == 8.0 and value == pytest.approx(1000.0)
