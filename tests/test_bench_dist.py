"""The benchmark's multi-process path on CPU (no GPU): two gloo ranks.

bench.py runs one process per GPU under torchrun: each rank solves its own
problem of the same shape (weak scaling, no collective on the data path),
the timings are reduced to their maximum over ranks, and rank 0 alone
prints.  These tests run that host-side logic with world_size 2 on gloo."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synthetic

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 10.0 - rank, 5.0 * (rank + 1)]
        got = bench.max_over_ranks(mine, torch.device("cpu"), world)
        w = bench.rank_problem(synthetic.WORKLOADS["t128_h4_kv2"], rank)
        q, _, _ = synthetic.make_inputs(w)
        out[rank] = (got, w.seed, float(np.abs(q.astype(np.float32)).sum()))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_independent_problems_gloo():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, free_port(), out), nprocs=world, join=True)
    want = [2.0, 10.0, 10.0]          # element-wise max of the two ranks' timings
    assert out[0][0] == want and out[1][0] == want
    assert out[0][1] != out[1][1]     # each rank its own seed ...
    assert out[0][2] != out[1][2]     # ... hence its own inputs


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}", "bench.py",
           "--impl", "reference", "--steps", "1", "--warmup", "3",
           "--workload", "t128_h4_kv2", "--reference-budget-s", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    for key in ("metric", "unit", "steps", "warmup", "ms_per_step", "higher_is_better",
                "cpu_baseline", "e2e", "config"):
        assert key in rec
