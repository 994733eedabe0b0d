"""The multi-replica bench path on CPU: two gloo ranks (one process each, as
torchrun starts them) agree on the slowest rank's time and on the whole-job
rate built from it; the reference arm leaves every rank but 0 idle."""

import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, _ = bench.dist_env()
    bench.init_distributed(w)
    try:
        bench.barrier()
        local_ms = 100.0 + 50.0 * r          # rank 1 is the slow one
        value, t = bench.job_rate(32, 10, w, local_ms)
        q.put((r, value, t))
    finally:
        bench._dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, value, t in got:
        assert t == 150.0                                   # max over ranks
        assert value == pytest.approx(32 * 10 * 2 / 0.150)  # both ranks' units over that time


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._dist is None
    value, t = bench.job_rate(4, 5, 1, 20.0)
    assert t == 20.0 and value == pytest.approx(4 * 5 / 0.020)


def test_reference_arm_runs_on_rank_0_only():
    import subprocess
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
