"""The multi-process path of bench.py (one process per GPU), on CPU with gloo.

The data path has no collective: every rank solves its own problem (weak
scaling).  What the ranks share is bookkeeping -- a barrier and the maximum of
the per-rank times -- and the job throughput computed from it.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    w, r, lr = bench.rank_info()
    assert (w, r, lr) == (world, rank, rank)
    bench.init_ranks(w)
    bench.barrier(w)
    local_ms = 10.0 * (rank + 1)  # rank 1 is the slowest
    total = bench.max_over_ranks(local_ms, w)
    value, ms_per_step = bench.job_throughput(total, steps=4, macs=1024**3, world=w)
    out.put((rank, total, value, ms_per_step))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_rank_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(world))
    for rank, total, value, ms_per_step in got:
        assert total == 20.0  # the maximum over ranks, on every rank
        assert ms_per_step == 5.0
        assert value == pytest.approx(2 * 4 * 2.0 * 1024**3 / 20e-3 / 1e12)


def test_single_rank_needs_no_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    value, ms = bench.job_throughput(2.0, steps=2, macs=10**12, world=1)
    assert ms == 1.0 and value == pytest.approx(2000.0)  # 2 * 2e12 operations in 2 ms
