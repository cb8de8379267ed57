"""Host logic of bench.py's multi-rank mode, on two gloo ranks on the CPU.

Sequences are independent, so under torchrun every rank decodes its own replica and nothing
is exchanged on the data path; the only cross-rank steps are the barrier around the timed
region, the slowest rank's time (max over ranks) and the whole-job total.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    try:
        r, ws = bench.dist_setup(world)
        assert (r, ws) == (rank, world)
        assert dist.get_backend() == "gloo"
        bench.barrier(ws)
        secs = 0.5 + rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(secs, ws)
        total = bench.whole_job(1000, ws, slowest)
        q.put((rank, slowest, total))
        dist.destroy_process_group()
    except Exception as e:  # report instead of hanging the parent
        q.put((rank, "error", repr(e)))


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    try:
        for _ in range(world):
            rank, a, b = q.get(timeout=120)
            got[rank] = (a, b)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    for rank in range(world):
        assert got[rank][0] != "error", got[rank][1]
        slowest, total = got[rank]
        assert slowest == pytest.approx(1.5)
        assert total == pytest.approx(2 * 1000 / 1.5)  # units of all ranks / slowest rank's time


def test_single_process_needs_no_process_group():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    assert bench.dist_setup(1) == (0, 1)
    assert bench.max_over_ranks(0.25, 1) == 0.25
    assert bench.whole_job(10, 1, 2.0) == 5.0
