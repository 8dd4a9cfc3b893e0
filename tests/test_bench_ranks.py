"""Multi-process host logic of bench.py on CPU (gloo, two ranks): the job's
time is the slowest rank's, the value counts every rank's work, and the
reference arm's non-zero ranks exit without work."""
from __future__ import annotations

import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 10 + 3r ms for the step and 4 - r ms per e2e step
        got = bench.ranks_max_ms([10.0 + 3 * rank, 4.0 - rank])
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time_gloo_two_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: [13.0, 4.0], 1: [13.0, 4.0]}


def test_job_throughput_counts_all_ranks():
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 3 steps x 1e12 MACs in 1.5 s -> 4 TMAC/s
    assert bench.job_tmacs(1e12, 3, 2, 1500.0) == pytest.approx(4.0)
    assert bench.ranks_max_ms([2.5, 1.0]) == [2.5, 1.0]   # one process: unchanged


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
