#!/usr/bin/env python
"""Causal GQA attention forward benchmark on GB300.

Metric: causal attention forward TFLOP/s, counting 4 * T^2 * 64 * heads / 2
FLOPs per pass, on the headline workload (T = 8192, 32 query heads over 8 K/V
heads, head width 64, binary16 inputs from the seeded generator), and its
fraction of the GB300's dense fp16 tensor peak.

One step = one forward pass (one kernel launch) over the whole workload.
Inputs are resident in HBM; the 129 MB L2 is flushed (a 512 MiB write)
between timed steps because the workload's inputs (85 MB) would otherwise stay
in it.  Each launch is timed with CUDA events on the launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores
  python bench.py --pass backward ...    # the backward pass instead (see below)
  python bench.py --all-configs          # one line per workload: timing + full parity
  python bench.py --all-configs --pass backward   # the same for the backward call

The --all-configs mode (one GPU) prints one JSON line per workload of the
benchmark list: the kernel's time (CUDA events; the three small workloads as
20 event pairs around 200 back-to-back launches each, the two large ones as
launches with L2 flushed between them), causal TFLOP/s and fraction of the
peaks, max |dO| and max |dLSE| of one launch against the fp64 oracle on every
element, the oracle's wall time, its thread count, the host's hardware thread
count and CPU model.  It is a record of every configuration, not the contract
line.

The materialised mode (--pass materialised) times one attn_fwd_materialised
call per step: the same forward through a binary32 scores plane and a
binary16 probability plane (three launches), reported in the same causal
TFLOP/s and against the HBM roofline, since it moves the planes through memory.

The producer mode (--pass producer) times one attn_qkv_rope call per step:
the fused QKV product of the workload's tokens (width = heads * 64, the
model's width) with a QKV matrix of heads + 2 kv_heads heads, rotary
embedding and value transpose in its epilogue; it counts
2 * T * width * (heads + 2 kv_heads) * 64 FLOPs against the tensor roofline.

The backward mode times one attn_bwd call per step (the query launch and the
key launch) on the same workload, with O and LSE from one forward pass made
before timing and dO from the seeded generator; it counts the five products
of the backward, 10 * T^2 * 64 * heads / 2 FLOPs per pass.

For N > 1 (torchrun), every rank runs its own independent problem of the same
shape (weak scaling, no collective on the data path); the barrier and the
max-over-ranks timing use torch.distributed.
"""
from __future__ import annotations

import argparse
import csv
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic  # noqa: E402

METRIC = "causal attn fwd TFLOP/s and % of GB300 dense fp16 tensor peak, T=8192"
METRIC_BWD = "causal attn bwd TFLOP/s (five products) and % of GB300 dense fp16 tensor peak"
METRIC_MAT = "materialised causal attn fwd TFLOP/s (scores + probability planes), HBM roofline"
METRIC_QKV = "fused QKV producer (product + rotary + V transpose) TFLOP/s and % of fp16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
# NVIDIA's nominal dense (no 2:4 sparsity) fp16/bf16 tensor rate of one GB300
DATASHEET_FP16_TFLOPS = 2250.0
FLUSH_BYTES = 512 << 20
KERNEL_SOURCE = os.path.join(ROOT, "transformer_causal_gqa_gb300", "csrc", "attn_fwd.cu")
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "attn_fwd_kernel_t8192_h32_kv8.md")
BWD_SOURCE = os.path.join(ROOT, "transformer_causal_gqa_gb300", "csrc", "attn_bwd.cu")
BWD_TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "attn_bwd_t8192_h32_kv8.md")
QKV_SOURCE = os.path.join(ROOT, "transformer_causal_gqa_gb300", "csrc", "attn_qkv.cu")
QKV_TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "qkv_kernel_t8192_w2048_h32_kv8.md")
MAT_SOURCE = os.path.join(ROOT, "transformer_causal_gqa_gb300", "csrc", "attn_materialised.cu")
MAT_TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "attn_materialised_t8192_and_t2048.md")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default=synthetic.HEADLINE,
                    choices=list(synthetic.WORKLOADS) + list(synthetic.PROFILE_SHAPES))
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reference-budget-s", type=float, default=120.0,
                    help="CPU seconds the reference arm spends over warm-up and timed steps")
    ap.add_argument("--all-configs", action="store_true",
                    help="one line per workload: kernel time and full-oracle parity")
    ap.add_argument("--pass", dest="which",
                    choices=["forward", "backward", "materialised", "producer"], default="forward")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def rank_problem(base, rank):
    """The workload each rank runs: the same shape, its own seed (an independent problem)."""
    return dataclasses.replace(base, seed=base.seed + 7919 * rank)


def max_over_ranks(values, device, world):
    """Element-wise maximum of per-rank timings over all ranks (the slowest rank sets the
    step time); the values themselves when world == 1."""
    import torch
    import torch.distributed as dist
    vals = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(vals, op=dist.ReduceOp.MAX)
    return [float(x) for x in vals.tolist()]


def workload_config(w, l2_note):
    return {"workload": w.name, "T": w.T, "heads": w.heads, "kv_heads": w.kv_heads,
            "head_dim": 64, "group": w.group, "causal_flops_per_step": w.causal_flops,
            "inputs": "seeded synthetic binary16 (Philox), c = fl32(0.125/ln 2)",
            "l2": l2_note}


def sampled_flops(rows):
    """FLOPs the metric credits a sample of query rows: 4 * 64 per causal (row, key) pair."""
    return float(256.0 * (np.asarray(rows, dtype=np.float64) + 1.0).sum())


def oracle_sample(w, inputs, n_rows, seed):
    import oracle
    q, k, vT = inputs
    rng = np.random.default_rng(seed)
    hs = rng.integers(0, w.heads, n_rows)
    rs = rng.integers(0, w.T, n_rows)
    t0 = time.perf_counter()
    oracle.attn_fwd_rows(q, k, vT, w.T, w.heads, w.kv_heads, synthetic.scale_c(), hs, rs)
    return time.perf_counter() - t0, sampled_flops(rs)


def calibrate_rows(w, inputs, target_s):
    """Rows of the workload the oracle covers in about target_s seconds."""
    n = 64
    while True:
        dt, _ = oracle_sample(w, inputs, n, seed=1)
        if dt > 0.5 or n >= 1 << 22:
            break
        n *= 4
    return max(8, int(n * target_s / max(dt, 1e-6)))


def cpu_baseline(w, inputs, target_s=15.0):
    """The oracle on the host cores, on about target_s seconds of the workload's rows,
    or on every row once if that fits."""
    import oracle
    q, k, vT = inputs
    n = calibrate_rows(w, inputs, target_s)
    if n >= w.heads * w.T:
        t0 = time.perf_counter()
        oracle.attn_fwd(q, k, vT, w.T, w.heads, w.kv_heads, synthetic.scale_c())
        dt = time.perf_counter() - t0
        fl = w.causal_flops   # the metric's count for the whole workload
        sample = f"every row of {w.name} once (fp64 two-pass oracle, {dt:.1f} s)"
    else:
        dt, fl = oracle_sample(w, inputs, n, seed=2)
        sample = (f"{n} query rows of {w.name} drawn uniformly over heads and rows "
                  f"(fp64 two-pass oracle, {dt:.1f} s); FLOPs credited 256 per causal "
                  f"(row, key) pair as in the metric")
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": oracle.max_threads(),
            "kind": "oracle", "sample": sample}


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        with open(self.path) as f:
            for rec in csv.reader(f):
                if len(rec) >= 9:
                    rows.append([x.strip() for x in rec])
        os.unlink(self.path)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm, smax, pw = [], [], []
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                pw.append(float(r[3]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def gpu_uuid():
    import torch
    try:
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ----------------------------------------------------------------------------- roofline
def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["bf16_tflops"]), "measured (cuBLAS bf16 burst; fp16 dense rate = bf16)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback (1.9 PFLOP/s bf16; fp16 dense rate = bf16)"


def kernel_traffic(summary=TRAFFIC_SUMMARY, source=KERNEL_SOURCE, key="traffic_bytes_per_launch"):
    """DRAM bytes per launch (or per call) from a committed ncu summary, if it was
    taken on the current kernel source; else None."""
    try:
        text = open(summary).read()
    except OSError:
        return None
    m_b = re.search(key + r":\s*([0-9.eE+]+)", text)
    m_h = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    if not (m_b and m_h):
        return None
    cur = hashlib.sha256(open(source, "rb").read()).hexdigest()
    return float(m_b.group(1)) if cur == m_h.group(1) else None


# ----------------------------------------------------------------------------- GPU arm
def run_gb300(args):
    import torch
    import torch.distributed as dist

    import transformer_causal_gqa_gb300 as tcg
    from transformer_causal_gqa_gb300 import build as tcg_build

    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or world == 1:
        tcg_build.build()
    if world > 1:
        dist.barrier()
    tcg.load_library()

    base = synthetic.lookup(args.workload)
    w = rank_problem(base, rank)
    inputs = synthetic.make_inputs(w)
    c = synthetic.scale_c()
    q, k, vT = (torch.from_numpy(x).to(dev) for x in inputs)
    o = torch.empty((w.T, w.heads * 64), dtype=torch.float16, device=dev)
    lse = torch.empty((w.heads, w.T), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        tcg.attn_fwd(q, k, vT, o, lse, w.T, w.heads, w.kv_heads, c, stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    if tcg.last_device_status(stream) != tcg.ATTN_OK:
        raise RuntimeError("device status after warm-up is not OK")

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(gpu_uuid())
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()               # evict the previous step's inputs from L2
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    if tcg.last_device_status(stream) != tcg.ATTN_OK:
        raise RuntimeError("device status after the timed steps is not OK")
    per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    dev_s = sum(per_launch_ms) / 1e3

    # end to end through the host-buffer entry point: H2D inputs, kernel, D2H outputs
    qh, kh, vh = (torch.from_numpy(x).pin_memory() for x in inputs)
    oh = torch.empty((w.T, w.heads * 64), dtype=torch.float16).pin_memory()
    lh = torch.empty((w.heads, w.T), dtype=torch.float32).pin_memory()
    ws = torch.empty(tcg.attn_fwd_workspace_bytes(w.T, w.heads, w.kv_heads),
                     dtype=torch.uint8, device=dev)

    def e2e_step():
        tcg.attn_fwd_host(qh, kh, vh, oh, lh, w.T, w.heads, w.kv_heads, c, ws, stream)

    for _ in range(3):
        e2e_step()
    E = max(1, args.e2e_steps)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = time.perf_counter()
    for _ in range(E):
        e2e_step()
        stream.synchronize()        # the result is on the host before the next step
    e2e_s = time.perf_counter() - e0
    h2d = sum(x.numel() * x.element_size() for x in (qh, kh, vh))
    d2h = oh.numel() * oh.element_size() + lh.numel() * lh.element_size()

    dev_s, e2e_s, wall = max_over_ranks([dev_s, e2e_s, wall], dev, world)

    if rank == 0:
        flops = w.causal_flops
        value = world * K * flops / dev_s / 1e12
        avg_launch_s = statistics.fmean(per_launch_ms) / 1e3
        achieved = flops / avg_launch_s / 1e12
        peak, peak_note = measured_peak()
        traffic = kernel_traffic()
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": dev_s / K * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16", "data": "synthetic",
            "config": dict(workload_config(w, "flushed between timed steps (512 MiB write); "
                                              "each launch timed by CUDA events"),
                           parallelism=f"independent problem per GPU x{world}"),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": peak_note,
                         "datasheet": {"peak": DATASHEET_FP16_TFLOPS,
                                       "frac": achieved / DATASHEET_FP16_TFLOPS,
                                       "source": "NVIDIA GB300 nominal dense fp16/bf16 rate"},
                         "ncu_tensor_pipe_active_pct": kernel_traffic(
                             key="tensor_pipe_active_pct"),
                         "kernel": "attn_fwd_kernel",
                         "launch_ms": {"mean": avg_launch_s * 1e3,
                                       "median": statistics.median(per_launch_ms),
                                       "min": min(per_launch_ms)}},
            "e2e": {"value": world * E * flops / e2e_s / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "path": "attn_fwd_host: pinned host buffers; four K/V-head chunks, copies in "
                            "and out on two library streams overlapping the kernel on the "
                            "caller's stream; synchronised each step"},
            "gpu_launches": K,
            "clocks": clocks,
            "wall_s_timed_region": wall,
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(base, inputs)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, metric=METRIC):
    import oracle
    rank, _, world = dist_env()
    if rank != 0:
        return
    w = synthetic.lookup(args.workload)
    inputs = synthetic.make_inputs(w)
    K, W = max(1, args.steps), max(3, args.warmup)
    budget_s = args.reference_budget_s
    rows = calibrate_rows(w, inputs, budget_s / (K + W))
    for i in range(W):
        oracle_sample(w, inputs, rows, seed=100 + i)
    tot_s = tot_fl = 0.0
    for i in range(K):
        dt, fl = oracle_sample(w, inputs, rows, seed=1000 + i)
        tot_s += dt
        tot_fl += fl
    value = tot_fl / tot_s / 1e12
    sample = (f"each step: {rows} query rows of {w.name} drawn uniformly over heads and rows; "
              f"FLOPs credited 256 per causal (row, key) pair as in the metric")
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": tot_s / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(workload_config(w, "not applicable (host CPU)"),
                       parallelism="host cores of rank 0"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- backward pass
def bwd_flops(w):
    """Five causal-half products of 2 * T^2/2 * 64 FLOPs per head each."""
    return 2.5 * w.causal_flops


def oracle_bwd_sample(w, inputs, o, lse, dO, n_rows, seed):
    """Times the oracle on n_rows query rows (dQ) and n_rows // group key rows
    (dK, dV); credits 384 FLOPs per causal (row, key) pair of a query row and
    256 per (query, key) pair of a key row, the five products' split."""
    import oracle
    q, k, vT = inputs
    rng = np.random.default_rng(seed)
    qh = rng.integers(0, w.heads, n_rows)
    qi = rng.integers(0, w.T, n_rows)
    nk = max(1, n_rows // w.group)
    kg = rng.integers(0, w.kv_heads, nk)
    kj = rng.integers(0, w.T, nk)
    t0 = time.perf_counter()
    oracle.attn_bwd_rows(q, k, vT, o, lse, dO, w.T, w.heads, w.kv_heads, synthetic.scale_c(),
                         0.125, qh, qi, kg, kj)
    dt = time.perf_counter() - t0
    fl = 384.0 * (qi + 1.0).sum() + 256.0 * w.group * (w.T - kj).astype(np.float64).sum()
    return dt, float(fl)


def bwd_oracle_inputs(w, inputs):
    """The forward's O and LSE from the oracle (fp64, as the reference arm has no GPU)."""
    import oracle
    q, k, vT = inputs
    return oracle.attn_fwd(q, k, vT, w.T, w.heads, w.kv_heads, synthetic.scale_c())


def bwd_calibrate(w, inputs, o, lse, dO, target_s):
    n = 4
    while True:
        dt, _ = oracle_bwd_sample(w, inputs, o, lse, dO, n, seed=1)
        if dt > 0.5 or n >= 1 << 20:
            break
        n *= 4
    return max(1, int(n * target_s / max(dt, 1e-6)))


def run_gb300_backward(args):
    import torch
    import torch.distributed as dist

    import transformer_causal_gqa_gb300 as tcg
    from transformer_causal_gqa_gb300 import build as tcg_build

    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or world == 1:
        tcg_build.build()
    if world > 1:
        dist.barrier()
    tcg.load_library()

    base = synthetic.lookup(args.workload)
    w = rank_problem(base, rank)
    inputs = synthetic.make_inputs(w)
    dO_np = synthetic.make_output_grad(w)
    c, s_nat = synthetic.scale_c(), 0.125
    T, H, G = w.T, w.heads, w.kv_heads
    q, k, vT = (torch.from_numpy(x).to(dev) for x in inputs)
    dO = torch.from_numpy(dO_np).to(dev)
    o = torch.empty((T, H * 64), dtype=torch.float16, device=dev)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    dq = torch.empty((H, T, 64), dtype=torch.float32, device=dev)
    dk = torch.empty((G, T, 64), dtype=torch.float32, device=dev)
    dvT = torch.empty((G, 64, T), dtype=torch.float32, device=dev)
    ws = torch.empty(tcg.attn_bwd_workspace_bytes(T, H, G), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    tcg.attn_fwd(q, k, vT, o, lse, T, H, G, c, stream)

    def step():
        tcg.attn_bwd(q, k, vT, o, lse, dO, dq, dk, dvT, T, H, G, c, s_nat, ws, stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    if tcg.bwd_last_device_status(stream) != tcg.ATTN_OK:
        raise RuntimeError("backward device status after warm-up is not OK")
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(gpu_uuid())
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    if tcg.bwd_last_device_status(stream) != tcg.ATTN_OK:
        raise RuntimeError("backward device status after the timed steps is not OK")
    per_call_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    dev_s = sum(per_call_ms) / 1e3

    # end to end through the public API: pinned host inputs copied in, the call,
    # the three gradients copied back, synchronised every step
    host_in = [x.cpu().pin_memory() for x in (q, k, vT, o, lse, dO)]
    host_out = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (dq, dk, dvT)]
    dev_in = [torch.empty_like(x) for x in (q, k, vT, o, lse, dO)]

    def e2e_step():
        for d, h in zip(dev_in, host_in):
            d.copy_(h, non_blocking=True)
        tcg.attn_bwd(*dev_in, dq, dk, dvT, T, H, G, c, s_nat, ws, stream)
        for h, d in zip(host_out, (dq, dk, dvT)):
            h.copy_(d, non_blocking=True)

    for _ in range(3):
        e2e_step()
        stream.synchronize()
    E = max(1, args.e2e_steps)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = time.perf_counter()
    for _ in range(E):
        e2e_step()
        stream.synchronize()
    e2e_s = time.perf_counter() - e0
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = sum(x.numel() * x.element_size() for x in host_out)

    dev_s, e2e_s, wall = max_over_ranks([dev_s, e2e_s, wall], dev, world)
    if rank == 0:
        flops = bwd_flops(w)
        avg_s = statistics.fmean(per_call_ms) / 1e3
        achieved = flops / avg_s / 1e12
        peak, peak_note = measured_peak()
        line = {
            "metric": METRIC_BWD, "value": world * K * flops / dev_s / 1e12, "unit": UNIT,
            "n_gpus": world, "steps": K, "warmup": max(3, args.warmup),
            "ms_per_step": dev_s / K * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": dict(workload_config(w, "flushed between timed steps (512 MiB write); "
                                              "each call timed by CUDA events"),
                           **{"pass": "backward"}, flops_per_step=flops,
                           parallelism=f"independent problem per GPU x{world}"),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak,
                         "traffic": kernel_traffic(BWD_TRAFFIC_SUMMARY, BWD_SOURCE,
                                                   "traffic_bytes_per_call"),
                         "peak_source": peak_note,
                         "datasheet": {"peak": DATASHEET_FP16_TFLOPS,
                                       "frac": achieved / DATASHEET_FP16_TFLOPS,
                                       "source": "NVIDIA GB300 nominal dense fp16/bf16 rate"},
                         "kernel": "attn_bwd call (query_kernel then key_kernel)",
                         "launch_ms": {"mean": avg_s * 1e3,
                                       "median": statistics.median(per_call_ms),
                                       "min": min(per_call_ms)}},
            "e2e": {"value": world * E * flops / e2e_s / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "path": "attn_bwd binding: pinned host inputs copied in, the call, "
                            "gradients copied out, one stream, synchronised each step"},
            "gpu_launches": 2 * K,
            "clocks": clocks,
            "wall_s_timed_region": wall,
        }
        if world == 1 and not args.no_cpu_baseline:
            o_h = o.cpu().numpy()
            l_h = lse.cpu().numpy()
            n = bwd_calibrate(base, inputs, o_h, l_h, dO_np, 15.0)
            dt, fl = oracle_bwd_sample(base, inputs, o_h, l_h, dO_np, n, seed=2)
            import oracle
            line["cpu_baseline"] = {
                "value": fl / dt / 1e12, "unit": UNIT, "cores": oracle.max_threads(),
                "kind": "oracle",
                "sample": f"{n} query rows (dQ) and {max(1, n // w.group)} key rows (dK, dV) "
                          f"of {w.name} drawn uniformly (fp64 oracle, {dt:.1f} s); FLOPs "
                          f"credited 384 per causal pair of a query row, 256 per pair of a "
                          f"key row"}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference_backward(args):
    import oracle
    rank, _, world = dist_env()
    if rank != 0:
        return
    w = synthetic.lookup(args.workload)
    inputs = synthetic.make_inputs(w)
    dO = synthetic.make_output_grad(w)
    o, lse = bwd_oracle_inputs(w, inputs)
    K, W = max(1, args.steps), max(3, args.warmup)
    n = bwd_calibrate(w, inputs, o, lse, dO, args.reference_budget_s / (K + W))
    for i in range(W):
        oracle_bwd_sample(w, inputs, o, lse, dO, n, seed=100 + i)
    tot_s = tot_fl = 0.0
    for i in range(K):
        dt, fl = oracle_bwd_sample(w, inputs, o, lse, dO, n, seed=1000 + i)
        tot_s += dt
        tot_fl += fl
    value = tot_fl / tot_s / 1e12
    sample = (f"each step: {n} query rows (dQ) and {max(1, n // w.group)} key rows (dK, dV) of "
              f"{w.name}; FLOPs credited 384 per causal pair of a query row, 256 per pair of a "
              f"key row")
    print(json.dumps({
        "impl": "reference", "metric": METRIC_BWD, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": tot_s / K * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": dict(workload_config(w, "not applicable (host CPU)"), **{"pass": "backward"},
                       parallelism="host cores of rank 0"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ----------------------------------------------------------------------------- materialised path
def measured_hbm():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (STREAM-style copy)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback (6.8 TB/s)"


def materialised_bytes(w):
    """Algorithmic DRAM bytes of one attn_fwd_materialised call: the scores plane's
    causal tiles written once and their causal elements read once, the probability
    plane written up to each row's diagonal-tile end and its causal tiles read once,
    plus Q, K, V^T read and O, LSE written once."""
    T, H, G = w.T, w.heads, w.kv_heads
    nt = (T + 127) // 128
    tile_elems = 0
    for qt in range(nt):
        rows = min(128, T - 128 * qt)
        for kt in range(qt + 1):
            tile_elems += rows * min(128, T - 128 * kt)
    causal = T * (T + 1) // 2
    p_written = sum(min(T, (i // 128 + 1) * 128) for i in range(T))
    io = 2 * H * T * 64 + 2 * 2 * G * T * 64 + 2 * T * H * 64 + 4 * H * T
    return H * (4 * tile_elems + 4 * causal + 2 * p_written + 2 * tile_elems) + io


def run_gb300_materialised(args):
    import torch
    import torch.distributed as dist

    import transformer_causal_gqa_gb300 as tcg
    from transformer_causal_gqa_gb300 import build as tcg_build

    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or world == 1:
        tcg_build.build()
    if world > 1:
        dist.barrier()
    tcg.load_library()
    base = synthetic.lookup(args.workload)
    w = rank_problem(base, rank)
    inputs = synthetic.make_inputs(w)
    c = synthetic.scale_c()
    T, H, G = w.T, w.heads, w.kv_heads
    q, k, vT = (torch.from_numpy(x).to(dev) for x in inputs)
    o = torch.empty((T, H * 64), dtype=torch.float16, device=dev)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    ws = torch.empty(tcg.attn_materialised_workspace_bytes(T, H, G), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        tcg.attn_fwd_materialised(q, k, vT, o, lse, T, H, G, c, ws, stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    if tcg.materialised_last_device_status(stream) != tcg.ATTN_OK:
        raise RuntimeError("materialised device status after warm-up is not OK")
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(gpu_uuid())
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    if tcg.materialised_last_device_status(stream) != tcg.ATTN_OK:
        raise RuntimeError("materialised device status after the timed steps is not OK")
    per_call_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    dev_s = sum(per_call_ms) / 1e3

    qh, kh, vh = (torch.from_numpy(x).pin_memory() for x in inputs)
    oh = torch.empty((T, H * 64), dtype=torch.float16).pin_memory()
    lh = torch.empty((H, T), dtype=torch.float32).pin_memory()
    qd, kd, vd = torch.empty_like(q), torch.empty_like(k), torch.empty_like(vT)

    def e2e_step():
        qd.copy_(qh, non_blocking=True)
        kd.copy_(kh, non_blocking=True)
        vd.copy_(vh, non_blocking=True)
        tcg.attn_fwd_materialised(qd, kd, vd, o, lse, T, H, G, c, ws, stream)
        oh.copy_(o, non_blocking=True)
        lh.copy_(lse, non_blocking=True)

    for _ in range(3):
        e2e_step()
        stream.synchronize()
    E = max(1, args.e2e_steps)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = time.perf_counter()
    for _ in range(E):
        e2e_step()
        stream.synchronize()
    e2e_s = time.perf_counter() - e0
    h2d = sum(x.numel() * x.element_size() for x in (qh, kh, vh))
    d2h = oh.numel() * oh.element_size() + lh.numel() * lh.element_size()

    dev_s, e2e_s, wall = max_over_ranks([dev_s, e2e_s, wall], dev, world)
    if rank == 0:
        flops = w.causal_flops
        avg_s = statistics.fmean(per_call_ms) / 1e3
        nbytes = materialised_bytes(w)
        peak, peak_note = measured_hbm()
        achieved = nbytes / avg_s / 1e9
        line = {
            "metric": METRIC_MAT, "value": world * K * flops / dev_s / 1e12, "unit": UNIT,
            "n_gpus": world, "steps": K, "warmup": max(3, args.warmup),
            "ms_per_step": dev_s / K * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": dict(workload_config(w, "flushed between timed steps (512 MiB write); "
                                              "each call timed by CUDA events"),
                           **{"pass": "materialised"}, algorithmic_bytes_per_step=nbytes,
                           workspace_bytes=ws.numel(),
                           parallelism=f"independent problem per GPU x{world}"),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak,
                         # counted on 4 query heads over 1 K/V head at T = 8192 and scaled
                         # by the head count (independent per-head planes, each beyond L2)
                         "traffic": (kernel_traffic(MAT_TRAFFIC_SUMMARY, MAT_SOURCE,
                                                    "traffic_bytes_per_call")
                                     if args.workload == synthetic.HEADLINE else None),
                         "peak_source": peak_note,
                         "kernel": "attn_fwd_materialised call (scores, softmax, pv kernels)",
                         "launch_ms": {"mean": avg_s * 1e3,
                                       "median": statistics.median(per_call_ms),
                                       "min": min(per_call_ms)}},
            "e2e": {"value": world * E * flops / e2e_s / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "path": "attn_fwd_materialised binding: pinned host inputs copied in, the "
                            "call, O and LSE copied out, synchronised each step"},
            "gpu_launches": 3 * K,
            "clocks": clocks,
            "wall_s_timed_region": wall,
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(base, inputs)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- QKV producer
def producer_shape(w):
    width = w.heads * 64
    n_out = (w.heads + 2 * w.kv_heads) * 64
    return width, n_out, 2.0 * w.T * width * n_out


def oracle_producer_sample(w, x, wt, c, s, n_tok):
    """The oracle producer on the first n_tok tokens (every token costs the same)."""
    import oracle
    width, n_out, _ = producer_shape(w)
    t0 = time.perf_counter()
    oracle.qkv_rope(x[:n_tok], wt, c[:n_tok], s[:n_tok], n_tok, width, w.heads, w.kv_heads)
    return time.perf_counter() - t0, 2.0 * n_tok * width * n_out


def producer_calibrate(w, x, wt, c, s, target_s):
    n = 8
    while True:
        dt, _ = oracle_producer_sample(w, x, wt, c, s, n)
        if dt > 0.5 or n >= w.T:
            break
        n = min(w.T, n * 4)
    return max(1, min(w.T, int(n * target_s / max(dt, 1e-6))))


def run_gb300_producer(args):
    import torch
    import torch.distributed as dist

    import transformer_causal_gqa_gb300 as tcg
    from transformer_causal_gqa_gb300 import build as tcg_build

    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or world == 1:
        tcg_build.build()
    if world > 1:
        dist.barrier()
    tcg.load_library()
    base = synthetic.lookup(args.workload)
    w = rank_problem(base, rank)
    T, H, G = w.T, w.heads, w.kv_heads
    width, n_out, flops = producer_shape(w)
    host = synthetic.make_producer_inputs(T, width, H, G, w.seed)
    xd, wd, cd, sd = (torch.from_numpy(a).to(dev) for a in host)
    q = torch.empty((H, T, 64), dtype=torch.float16, device=dev)
    k = torch.empty((G, T, 64), dtype=torch.float16, device=dev)
    vT = torch.empty((G, 64, T), dtype=torch.float16, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        tcg.attn_qkv_rope(xd, wd, cd, sd, q, k, vT, T, width, H, G, stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    if tcg.qkv_last_device_status(stream) != tcg.ATTN_OK:
        raise RuntimeError("producer device status after warm-up is not OK")
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(gpu_uuid())
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    if tcg.qkv_last_device_status(stream) != tcg.ATTN_OK:
        raise RuntimeError("producer device status after the timed steps is not OK")
    per_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    dev_s = sum(per_ms) / 1e3

    hin = [torch.from_numpy(a).pin_memory() for a in host]
    hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (q, k, vT)]
    din = [torch.empty_like(t) for t in (xd, wd, cd, sd)]

    def e2e_step():
        for d, h in zip(din, hin):
            d.copy_(h, non_blocking=True)
        tcg.attn_qkv_rope(*din, q, k, vT, T, width, H, G, stream)
        for h, d in zip(hout, (q, k, vT)):
            h.copy_(d, non_blocking=True)

    for _ in range(3):
        e2e_step()
        stream.synchronize()
    E = max(1, args.e2e_steps)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = time.perf_counter()
    for _ in range(E):
        e2e_step()
        stream.synchronize()
    e2e_s = time.perf_counter() - e0
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in hout)

    dev_s, e2e_s, wall = max_over_ranks([dev_s, e2e_s, wall], dev, world)
    if rank == 0:
        avg_s = statistics.fmean(per_ms) / 1e3
        peak, peak_note = measured_peak()
        achieved = flops / avg_s / 1e12
        cfg = dict(workload_config(w, "flushed between timed steps (512 MiB write); each launch "
                                      "timed by CUDA events"),
                   **{"pass": "producer"}, width=width, outputs=n_out, flops_per_step=flops,
                   inputs_producer="X ~ N(0,1), W ~ N(0,1/width) binary16 (Philox); rotary "
                                   "tables cos/sin(t * 10000^(-p/32)) binary32",
                   parallelism=f"independent problem per GPU x{world}")
        cfg.pop("causal_flops_per_step", None)
        line = {
            "metric": METRIC_QKV, "value": world * K * flops / dev_s / 1e12, "unit": UNIT,
            "n_gpus": world, "steps": K, "warmup": max(3, args.warmup),
            "ms_per_step": dev_s / K * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic", "config": cfg,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak,
                         "traffic": kernel_traffic(QKV_TRAFFIC_SUMMARY, QKV_SOURCE),
                         "peak_source": peak_note, "kernel": "qkv_kernel",
                         "datasheet": {"peak": DATASHEET_FP16_TFLOPS,
                                       "frac": achieved / DATASHEET_FP16_TFLOPS,
                                       "source": "NVIDIA GB300 nominal dense fp16/bf16 rate"},
                         "launch_ms": {"mean": avg_s * 1e3, "median": statistics.median(per_ms),
                                       "min": min(per_ms)}},
            "e2e": {"value": world * E * flops / e2e_s / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "path": "attn_qkv_rope binding: pinned host inputs copied in, the call, "
                            "Q, K, V^T copied out, synchronised each step"},
            "gpu_launches": K,
            "clocks": clocks,
            "wall_s_timed_region": wall,
        }
        if world == 1 and not args.no_cpu_baseline:
            import oracle
            n = producer_calibrate(base, *host, 15.0)
            dt, fl = oracle_producer_sample(base, *host, n)
            line["cpu_baseline"] = {
                "value": fl / dt / 1e12, "unit": UNIT, "cores": oracle.max_threads(),
                "kind": "oracle",
                "sample": f"the first {n} of {T} tokens (every token costs the same; fp64 "
                          f"oracle, {dt:.1f} s)"}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference_producer(args):
    import oracle
    rank, _, world = dist_env()
    if rank != 0:
        return
    w = synthetic.lookup(args.workload)
    width, n_out, _ = producer_shape(w)
    host = synthetic.make_producer_inputs(w.T, width, w.heads, w.kv_heads, w.seed)
    K, W = max(1, args.steps), max(3, args.warmup)
    n = producer_calibrate(w, *host, args.reference_budget_s / (K + W))
    for _ in range(W):
        oracle_producer_sample(w, *host, n)
    tot_s = tot_fl = 0.0
    for _ in range(K):
        dt, fl = oracle_producer_sample(w, *host, n)
        tot_s += dt
        tot_fl += fl
    value = tot_fl / tot_s / 1e12
    cfg = dict(workload_config(w, "not applicable (host CPU)"), **{"pass": "producer"},
               width=width, outputs=n_out, parallelism="host cores of rank 0")
    cfg.pop("causal_flops_per_step", None)
    print(json.dumps({
        "impl": "reference", "metric": METRIC_QKV, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": tot_s / K * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": f"each step: the first {n} tokens"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)

# ----------------------------------------------------------------------------- every workload
def cpu_model():
    """The host CPU's model name, from /proc/cpuinfo or lscpu."""
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return "unknown"


def run_all_configs(args):
    import torch

    import oracle
    import transformer_causal_gqa_gb300 as tcg
    from transformer_causal_gqa_gb300 import build as tcg_build

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    tcg_build.build()
    tcg.load_library()
    c = synthetic.scale_c()
    peak, peak_note = measured_peak()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    host = {"cpu_model": cpu_model(), "hardware_concurrency": os.cpu_count(),
            "oracle_threads": oracle.max_threads()}
    for w in synthetic.WORKLOADS.values():
        inputs = synthetic.make_inputs(w)
        q, k, vT = (torch.from_numpy(x).to(dev) for x in inputs)
        o = torch.full((w.T, w.heads * 64), float("nan"), dtype=torch.float16, device=dev)
        lse = torch.full((w.heads, w.T), float("nan"), dtype=torch.float32, device=dev)

        def step():
            tcg.attn_fwd(q, k, vT, o, lse, w.T, w.heads, w.kv_heads, c, stream)

        step()
        if tcg.last_device_status(stream) != tcg.ATTN_OK:
            raise RuntimeError(f"{w.name}: device status after the parity launch is not OK")
        o_gpu = o.cpu().numpy().astype(np.float64)
        l_gpu = lse.cpu().numpy().astype(np.float64)
        for _ in range(max(3, args.warmup)):
            step()
        small = w.T <= 2048
        per_pair = 200 if small else 1
        pairs = 20 if small else max(20, min(args.steps, 200))
        sampler = ClockSampler(gpu_uuid())
        sampler.start()
        times = []
        torch.cuda.synchronize()
        for _ in range(pairs):
            if not small:
                flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(per_pair):
                step()
            b.record(stream)
            times.append((a, b))
        torch.cuda.synchronize()
        clocks = sampler.stop()
        if tcg.last_device_status(stream) != tcg.ATTN_OK:
            raise RuntimeError(f"{w.name}: device status after timing is not OK")
        ms = [a.elapsed_time(b) / per_pair for a, b in times]
        t0 = time.perf_counter()
        o_ref, l_ref = oracle.attn_fwd(*inputs, w.T, w.heads, w.kv_heads, c)
        oracle_s = time.perf_counter() - t0
        d_o = float(np.abs(o_gpu - o_ref).max())
        d_l = float(np.abs(l_gpu - l_ref).max())
        med = statistics.median(ms)
        tflops = w.causal_flops / (med / 1e3) / 1e12
        print(json.dumps({
            "mode": "all-configs", "workload": w.name, "T": w.T, "heads": w.heads,
            "kv_heads": w.kv_heads, "gpu_ms_median": med, "gpu_ms_mean": statistics.fmean(ms),
            "gpu_ms_min": min(ms), "event_pairs": pairs, "launches_per_event_pair": per_pair,
            "l2": ("warm: back-to-back launches inside each event pair" if small else
                   "flushed before each launch (512 MiB write)"),
            "tflops": tflops, "frac_of_measured_peak": tflops / peak, "peak": peak,
            "peak_source": peak_note, "frac_of_datasheet_fp16": tflops / DATASHEET_FP16_TFLOPS,
            "max_abs_dO": d_o, "max_abs_dLSE": d_l, "tol_dO": 4e-3, "tol_dLSE": 1e-3,
            "parity": "pass" if (d_o <= 4e-3 and d_l <= 1e-3) else "FAIL",
            "oracle_s": oracle_s, "oracle_rows": "every row", **host,
            "oracle_gflops": w.causal_flops / oracle_s / 1e9, "clocks": clocks,
        }), flush=True)
        del q, k, vT, o, lse, o_ref, l_ref, o_gpu, l_gpu
        torch.cuda.empty_cache()


def run_all_configs_backward(args):
    """One line per workload for the backward call: its time (CUDA events), TFLOP/s over
    the five products, and its agreement with the fp64 oracle: every element of the three
    small workloads, 256 query rows and 128 key rows of the two large ones."""
    import torch

    import oracle
    import transformer_causal_gqa_gb300 as tcg
    from transformer_causal_gqa_gb300 import build as tcg_build

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    tcg_build.build()
    tcg.load_library()
    c, s_nat = synthetic.scale_c(), 0.125
    peak, peak_note = measured_peak()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    host = {"cpu_model": cpu_model(), "hardware_concurrency": os.cpu_count(),
            "oracle_threads": oracle.max_threads()}

    def agreement(got, ref):
        got = np.asarray(got, dtype=np.float64)
        return {"rel_frobenius": float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)),
                "max_err_over_max_ref": float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))}

    for w in synthetic.WORKLOADS.values():
        T, H, G = w.T, w.heads, w.kv_heads
        inputs = synthetic.make_inputs(w)
        dO_np = synthetic.make_output_grad(w)
        q, k, vT = (torch.from_numpy(x).to(dev) for x in inputs)
        dO = torch.from_numpy(dO_np).to(dev)
        o, lse = tcg.attention(q, k, vT, c)
        dq = torch.empty((H, T, 64), dtype=torch.float32, device=dev)
        dk = torch.empty((G, T, 64), dtype=torch.float32, device=dev)
        dvT = torch.empty((G, 64, T), dtype=torch.float32, device=dev)
        ws = torch.empty(tcg.attn_bwd_workspace_bytes(T, H, G), dtype=torch.uint8, device=dev)

        def step():
            tcg.attn_bwd(q, k, vT, o, lse, dO, dq, dk, dvT, T, H, G, c, s_nat, ws, stream)

        step()
        if tcg.bwd_last_device_status(stream) != tcg.ATTN_OK:
            raise RuntimeError(f"{w.name}: backward device status is not OK")
        got = (dq.cpu().numpy(), dk.cpu().numpy(), dvT.cpu().numpy())
        o_h, l_h = o.cpu().numpy(), lse.cpu().numpy()
        for _ in range(max(3, args.warmup)):
            step()
        small = T <= 2048
        per_pair = 50 if small else 1
        pairs = 20 if small else 50
        sampler = ClockSampler(gpu_uuid())
        sampler.start()
        times = []
        torch.cuda.synchronize()
        for _ in range(pairs):
            if not small:
                flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(per_pair):
                step()
            b.record(stream)
            times.append((a, b))
        torch.cuda.synchronize()
        clocks = sampler.stop()
        if tcg.bwd_last_device_status(stream) != tcg.ATTN_OK:
            raise RuntimeError(f"{w.name}: backward device status after timing is not OK")
        ms = [a.elapsed_time(b) / per_pair for a, b in times]
        t0 = time.perf_counter()
        if small:
            rq, rk, rv, _ = oracle.attn_bwd(*inputs, o_h, l_h, dO_np, T, H, G, c, s_nat)
            rows = "every element"
            parity = {"dQ": agreement(got[0], rq), "dK": agreement(got[1], rk),
                      "dV^T": agreement(got[2], rv)}
        else:
            rng = np.random.default_rng(w.seed)
            qh, qi = rng.integers(0, H, 256), rng.integers(0, T, 256)
            kg, kj = rng.integers(0, G, 128), rng.integers(0, T, 128)
            rq, rk, rv = oracle.attn_bwd_rows(*inputs, o_h, l_h, dO_np, T, H, G, c, s_nat,
                                              qh, qi, kg, kj)
            rows = "256 query rows (dQ) and 128 key rows (dK, dV) drawn uniformly"
            parity = {"dQ": agreement(got[0][qh, qi], rq), "dK": agreement(got[1][kg, kj], rk),
                      "dV^T": agreement(got[2][kg, :, kj], rv)}
        oracle_s = time.perf_counter() - t0
        med = statistics.median(ms)
        flops = bwd_flops(w)
        tflops = flops / (med / 1e3) / 1e12
        print(json.dumps({
            "mode": "all-configs", "pass": "backward", "workload": w.name, "T": T, "heads": H,
            "kv_heads": G, "gpu_ms_median": med, "gpu_ms_mean": statistics.fmean(ms),
            "gpu_ms_min": min(ms), "event_pairs": pairs, "launches_per_event_pair": per_pair,
            "l2": ("warm: back-to-back calls inside each event pair" if small else
                   "flushed before each call (512 MiB write)"),
            "flops_five_products": flops, "tflops": tflops, "frac_of_measured_peak": tflops / peak,
            "peak": peak, "peak_source": peak_note,
            "frac_of_datasheet_fp16": tflops / DATASHEET_FP16_TFLOPS,
            "oracle_rows": rows, "parity": parity, "oracle_s": oracle_s, **host, "clocks": clocks,
        }), flush=True)
        del q, k, vT, dO, o, lse, dq, dk, dvT, ws, got
        torch.cuda.empty_cache()


def main():
    args = parse_args()
    if args.all_configs:
        if args.impl == "reference":
            raise SystemExit("--all-configs times the GPU kernel; the oracle is timed inside it")
        if args.which == "backward":
            run_all_configs_backward(args)
        elif args.which == "forward":
            run_all_configs(args)
        else:
            raise SystemExit("--all-configs covers --pass forward and --pass backward")
        return
    if args.which == "producer":
        (run_reference_producer if args.impl == "reference" else run_gb300_producer)(args)
    elif args.which == "materialised":
        if args.impl == "reference":
            run_reference(args, metric=METRIC_MAT)
        else:
            run_gb300_materialised(args)
    elif args.which == "backward":
        (run_reference_backward if args.impl == "reference" else run_gb300_backward)(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gb300(args)


if __name__ == "__main__":
    main()
