"""The benchmark's multi-rank logic on CPU (gloo, world size 2): the step
time is the maximum over ranks, the value counts every rank's replica, and
under torchrun the reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [3.0, 7.5][rank]
    got = bench.max_over_ranks(ms, dist, "cpu")
    q.put((rank, got, bench.whole_job_value(1000, world, got)))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [7.5, 7.5]                 # both ranks see the slowest
    assert res[0][2] == pytest.approx(1000 * 2 / 7.5e-3)      # tokens of both replicas / max time


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(4.25, None, "cpu") == 4.25
    assert bench.whole_job_value(16384, 1, 9.0) == pytest.approx(16384 / 9e-3)


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
