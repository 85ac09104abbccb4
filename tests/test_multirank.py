"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the
replicas' time is the maximum over ranks, the value counts every rank's work,
and only rank 0 of the reference arm prints."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        mine = [0.25, 0.5][rank]
        worst = bench.max_over_ranks(mine, dist, torch.device("cpu"))
        results[rank] = (worst, bench.whole_job_tflops(world, 1e12, 10, worst))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = free_port()
    mp.start_processes(_worker, args=(2, port, results), nprocs=2, start_method="spawn", join=True)
    assert results[0] == results[1] == (0.5, 2 * 1e12 * 10 / 0.5 / 1e12)


def test_single_rank_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, None, None) == 3.0
    assert bench.whole_job_tflops(1, 2e12, 5, 2.0) == 5.0


@pytest.mark.timeout(300)
def test_reference_arm_two_ranks_only_rank0_prints():
    env = dict(os.environ, PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0", "--workload", "gemm_256_f16_f32"]
    res = subprocess.run(cmd, capture_output=True, text=True, env=env, cwd=ROOT, timeout=280)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["n_gpus"] == 2
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
