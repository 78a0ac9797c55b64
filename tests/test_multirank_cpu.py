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


def test_reference_arm_prints_once_from_rank_zero():
    """bench.py --impl reference launched as two ranks: rank 0 times the oracle
    and prints one JSON line (impl reference, the oracle's own cpu_baseline and
    e2e keys); rank 1 exits 0 without output."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    outs = []
    for rank in (0, 1):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
        r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                            "--warmup", "3", "--ref-budget", "0.5"], capture_output=True, text=True, env=env,
                           cwd=root, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append([line for line in r.stdout.splitlines() if line.strip()])
    assert outs[1] == []
    assert len(outs[0]) == 1
    line = json.loads(outs[0][0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
