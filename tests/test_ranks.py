"""Host-side logic of bench.py's multi-rank run (replicas, weak scaling), on CPU with gloo.

Each rank times its own replica; the job's time is the slowest rank's and the job's rate
counts the bytes of every rank. No GPU is involved."""
import os
import socket
import subprocess
import sys

import pytest
import torch
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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.0 + 0.5 * rank, torch.device("cpu"))
        q.put((rank, ms, bench.job_rate_gbs(10**9, ms, world)))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(30)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    for _, ms, rate in res:
        assert ms == 1.5                       # the slower rank's time on every rank
        assert rate == pytest.approx(2 * 10**9 / 1.5e-3 / 1e9)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_rate_gbs(47_394_816, 0.01, 1) == pytest.approx(4739.4816)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
