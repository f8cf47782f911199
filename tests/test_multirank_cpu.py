"""The benchmark's multi-rank path on CPU: two gloo ranks, no GPU.

Layers and weight tiles are independent, so each rank runs its own copy of the per-GPU work and
the only collectives are barriers and the max-over-ranks of the timings (weak scaling).
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        mine = [10.0 + rank, 20.0 - rank, 30.0 + 2 * rank]  # per-rank step times (ms)
        dist.barrier()
        got = bench.max_over_ranks(mine, world)
        q.put((rank, got, bench.job_throughput(1e12, world, got[0])))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_aggregate_weakly():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict((r, (got, tp)) for r, got, tp in (q.get(timeout=10) for _ in range(2)))
    for r in (0, 1):
        got, tp = res[r]
        assert got == [11.0, 20.0, 32.0]
        # 2 ranks x 1 TFLOP each in 11 ms
        assert tp == pytest.approx(2 * 1e12 / 11e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.job_throughput(2e12, 1, 1000.0) == pytest.approx(2.0)
