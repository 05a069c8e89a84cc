"""bench.py's multi-rank timing on CPU: two gloo ranks (no GPU).  Each rank
reports its own step time; the job uses the slowest rank's and counts every
rank's bytes (one independent replica per GPU)."""
from __future__ import annotations

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 100.0 + 25.0 * rank                      # rank 1 is the slower one
    worst = bench.max_over_ranks(ms)
    dist.barrier()
    out.put((rank, worst, bench.whole_job_gbs(10**12, 4, worst, world)))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [125.0, 125.0]
    # 2 ranks x 1e12 B x 4 steps in 0.125 s
    assert got[0][2] == pytest.approx(2 * 4 * 1e12 / 0.125 / 1e9)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_gbs(10**9, 10, 1000.0, 1) == pytest.approx(10.0)
