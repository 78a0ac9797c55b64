"""The benchmark's multi-rank logic on two gloo ranks (CPU, no GPU).

Multi-GPU runs are independent replicas of the workload (weak scaling, no
collective on the data path); the only cross-rank steps are the barrier and
the max-over-ranks of the measured times, checked here.
"""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5 * rank])
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert results[r] == [2.0, 10.0, 0.5]


def test_max_over_ranks_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]


def test_whole_job_throughput_is_weak_scaling():
    import bench
    one = bench.whole_job_gbs(1, 33_423_360, 0.1)
    assert one == pytest.approx(334.2336)
    assert bench.whole_job_gbs(4, 33_423_360, 0.1) == pytest.approx(4 * one)
