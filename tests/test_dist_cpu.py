"""The bench's multi-rank path on the CPU: two gloo ranks exercise the barrier, the
max-over-ranks timing and the whole-job aggregation (each rank runs its own batch)."""

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        my_ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
        slowest = bench.max_over_ranks(my_ms, world)
        rate = bench.whole_job_rate(1000.0, 4, slowest, world)
        results[rank] = (slowest, rate)
        bench.barrier(world)
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        got = dict(results)
    for r in range(world):
        slowest, rate = got[r]
        assert slowest == 15.0
        # 2 ranks x 1000 units x 4 steps in 15 ms
        assert rate == pytest.approx(2 * 1000 * 4 / 0.015)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(10.0, 2, 1000.0, 1) == pytest.approx(20.0)
