"""The bench's multi-replica bookkeeping on two CPU ranks (gloo).

The attention path does not shard: several GPUs run independent replicas and
the bench reports the tokens of all replicas over the slowest rank's time.
These tests run that host logic in two processes without a GPU.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                            rank=rank, world_size=world)
    try:
        # rank r spent (r + 1) * 10 ms over its timed steps
        mine = 10.0 * (rank + 1)
        total = bench.max_over_ranks(mine)
        rate = bench.whole_job_rate(8192, world, 30, total)
        q.put((rank, total, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, total, rate in got:
        assert total == 20.0                       # the slowest rank's time
        assert rate == pytest.approx(8192 * 2 * 30 / 0.020)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(100, 1, 10, 1000.0) == pytest.approx(1000.0)


def test_reference_arm_only_on_rank_zero():
    # a non-zero rank of the reference arm exits at once without output
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl",
                          "reference", "--steps", "1", "--warmup", "3"],
                         capture_output=True, text=True, env=env, timeout=120)
    assert out.returncode == 0
    assert out.stdout.strip() == ""
