"""The bench's multi-rank host logic on two gloo ranks (CPU, no GPU).

The path shards with no exchange (replicas only), so the only cross-rank step
is the timing reduction: every rank must report the slowest rank's times, and
the whole-job value is world x step bytes over that time.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        mine = [1.0 + rank, 10.0 - rank, 0.5 * (rank + 1), 3.0]
        q.put((rank, bench.max_over_ranks(mine, torch.device("cpu"))))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        assert got[r] == [2.0, 10.0, 1.0, 3.0]


def test_whole_job_value_scales_with_world():
    import bench
    one = bench.whole_job_gbs(1, 331_350_016, 0.2)
    assert one == pytest.approx(331_350_016 / 0.2e-3 / 1e9)
    assert bench.whole_job_gbs(4, 331_350_016, 0.2) == pytest.approx(4 * one)
