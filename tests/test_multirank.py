"""The N > 1 path on CPU with gloo, world size 2.

The product has no exchange step, so several GPUs run independent replicas:
the only cross-rank logic is the barrier and the max-over-ranks timing in
bench.py, and rank 0 alone printing the JSON line.  Both are exercised here
with two gloo ranks on the CPU."""
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports a step time of 10*(r+1) ms and a kernel time of 5 - r ms
        got = bench.max_over_ranks([10.0 * (rank + 1), 5.0 - rank], torch.device("cpu"))
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1] == [20.0, 5.0]


def test_job_tflops_aggregates_ranks():
    sys.path.insert(0, ROOT)
    import bench

    one = bench.job_tflops(2 * 8192 ** 3, 1, 4.0)
    assert abs(bench.job_tflops(2 * 8192 ** 3, 2, 4.0) - 2 * one) < 1e-9


def test_reference_arm_under_torchrun_world2():
    """Rank 0 prints exactly one JSON line; rank 1 exits 0 without output."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "sq256_uniform", "--steps", "2",
           "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "TFLOP/s" and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["config"]["workload"] == "sq256_uniform"
