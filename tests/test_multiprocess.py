"""The replicas path on CPU: with torchrun (N > 1) every rank runs its own
replica, the job's time is the slowest rank's (max over ranks, gloo) and
`value` counts every rank's tokens; the reference arm runs on rank 0 alone
and prints the only line."""

from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(10.0 * (rank + 1), dist)
        v = bench.job_value(world, 128, 50, t)
        with open(os.path.join(out_dir, "r%d.json" % rank), "w") as f:
            json.dump({"max": t, "value": v}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_with_gloo(tmp_path):
    world = 2
    mp.spawn(_rank, args=(world, free_port(), str(tmp_path)), nprocs=world, join=True)
    got = [json.load(open(tmp_path / ("r%d.json" % r))) for r in range(world)]
    for g in got:
        assert g["max"] == 20.0                     # the slower rank's time
        assert g["value"] == 2 * 128 * 50 / 0.020   # both ranks' tokens over it
    assert bench.max_over_ranks(3.5, None) == 3.5


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1",
           "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
           "--master-port", str(free_port()), "bench.py", "--impl", "reference",
           "--workload", "tiny_prefill", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, OMP_NUM_THREADS="1"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
