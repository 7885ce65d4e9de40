"""The multi-rank logic of bench.py on CPU: two gloo ranks, as torchrun would launch them.

Each rank is an independent replica of the step; the step time is the slowest
rank's and the reported value aggregates all replicas (weak scaling).
"""
import os

import pytest

torch = pytest.importorskip("torch")


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 100.0 + 25.0 * rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, dist, "cpu")
        out.put((rank, slowest, bench.whole_job_tflops(world, 2.0e12, slowest)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    import socket

    import torch.multiprocessing as mp

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, tflops in res:
        assert slowest == 125.0
        assert abs(tflops - 2 * 2.0e12 / 0.125 / 1e12) < 1e-9


def test_single_process_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tflops(1, 1e12, 1000.0) == 1.0
