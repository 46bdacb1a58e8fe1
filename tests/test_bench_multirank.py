"""bench.py's multi-rank aggregation on CPU: two gloo ranks (no GPU).

Under torchrun every rank runs its own replica (no collective in the data
path); the reported rate is all ranks' tokens over the slowest rank's time.
Each rank reports a different time here: both must get the maximum, and the
whole-job rate must use it.
"""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, times, out):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.slowest(times[rank], dist)
        out[rank] = (t, bench.job_rate(16 * 20, world, t))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(0.75, 2.5), (3.0, 1.25)])
def test_two_ranks_agree_on_the_slowest_time(times):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, times, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        got = dict(out)
    top = max(times)
    for r in range(2):
        assert got[r][0] == top
        assert got[r][1] == pytest.approx(16 * 20 * 2 / top)


def test_one_rank_keeps_its_own_time():
    import bench
    assert bench.slowest(1.5, None) == 1.5
    assert bench.job_rate(50, 1, 0.1) == pytest.approx(500.0)
