"""Seeded synthetic inputs for the causal grouped-query attention forward and
backward passes.

This module is shared by the CUDA path's tests and benchmark and by the oracle
tests.  It draws random numbers and lays them out; it holds none of the
attention arithmetic.

Recipe (identical for both sides, which then read the same binary16 buffers):
  * a counter-based generator, numpy's Philox (Salmon et al., "Parallel random
    numbers: as easy as 1, 2, 3", SC'11), keyed by the workload's seed;
  * draws in this order: Q [heads][T][64], K [kv_heads][T][64], V [kv_heads][T][64],
    each as float32 (standard normal, or uniform on [-1, 1) where stated);
  * the workload's power-of-two scale factors applied in float32 (exact);
  * rounded to binary16 with round-to-nearest-even (numpy's cast);
  * V transposed per K/V head to V^T [kv_heads][64][T].
For the backward pass the output gradient dO [T][heads*64] (O's token-major
layout) is drawn from its own Philox stream, keyed by the seed plus
0x9E3779B9, as standard-normal float32 rounded to binary16.  For the fused
QKV producer, X and W come from a stream keyed by the seed plus 0x51ED2700,
and the rotary tables are the nearest binary32 values of cos and sin of
t * 10000^(-p/32).
The scale constant c is the binary32 value nearest 0.125 / ln 2 (the head
width 64 gives the score scale 1/sqrt(64) = 0.125).
"""
from __future__ import annotations

import dataclasses

import numpy as np

HEAD_DIM = 64


def scale_c() -> float:
    """c = the binary32 nearest 0.125 / ln 2, returned as a Python float."""
    return float(np.float32(0.125 / np.log(2.0)))


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    heads: int
    kv_heads: int
    seed: int
    qk_scale: float = 1.0            # Q and K multiplied by this (peaked softmax)
    k_outlier_every: int = 0         # key rows j with (j+1) % every == 0 ...
    k_outlier_scale: float = 1.0     # ... multiplied by this
    v_uniform: bool = False          # V ~ U(-1, 1) instead of N(0, 1)

    @property
    def group(self) -> int:
        return self.heads // self.kv_heads

    @property
    def causal_flops(self) -> float:
        """4 * T^2 * 64 * heads / 2: the metric's FLOP count."""
        return 4.0 * self.T * self.T * HEAD_DIM * self.heads / 2.0

    @property
    def io_bytes(self) -> int:
        """Q + K + V^T read once, O + LSE written once."""
        T, H, G = self.T, self.heads, self.kv_heads
        return 2 * H * T * HEAD_DIM + 2 * 2 * G * T * HEAD_DIM + 2 * T * H * HEAD_DIM + 4 * H * T


# The five workloads of the headline benchmark, smallest first.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("t128_h4_kv2", 128, 4, 2, seed=0x5EED0000),
        Workload("t1024_h12_kv12_mha", 1024, 12, 12, seed=0x5EED0001),
        Workload("t2048_h16_kv4_peaked", 2048, 16, 4, seed=0x5EED0002, qk_scale=4.0),
        Workload("t8192_h32_kv8", 8192, 32, 8, seed=0x5EED0003),
        Workload("t16384_h64_kv8_outliers", 16384, 64, 8, seed=0x5EED0004,
                 k_outlier_every=97, k_outlier_scale=16.0, v_uniform=True),
    ]
}
HEADLINE = "t8192_h32_kv8"

# Shapes for profiler captures only, not benchmark workloads: the headline length with
# fewer heads, so that a capture holds a few GB of device memory while the rows of the
# materialised planes are as long as the headline's.
PROFILE_SHAPES = {
    w.name: w
    for w in [
        Workload("t8192_h4_kv1_profile", 8192, 4, 1, seed=0x5EED0005),
    ]
}


def lookup(name: str) -> Workload:
    """A benchmark workload or a profiling shape, by name."""
    if name in WORKLOADS:
        return WORKLOADS[name]
    return PROFILE_SHAPES[name]


def custom(T: int, heads: int, kv_heads: int, seed: int, **kw) -> Workload:
    return Workload(f"t{T}_h{heads}_kv{kv_heads}_s{seed}", T, heads, kv_heads, seed, **kw)


def make_inputs(w: Workload):
    """Returns (q [H][T][64], k [G][T][64], vT [G][64][T]) as binary16 numpy arrays."""
    rng = np.random.Generator(np.random.Philox(w.seed))
    T, H, G = w.T, w.heads, w.kv_heads
    q = rng.standard_normal((H, T, HEAD_DIM), dtype=np.float32)
    k = rng.standard_normal((G, T, HEAD_DIM), dtype=np.float32)
    if w.v_uniform:
        v = rng.uniform(-1.0, 1.0, size=(G, T, HEAD_DIM)).astype(np.float32)
    else:
        v = rng.standard_normal((G, T, HEAD_DIM), dtype=np.float32)
    if w.qk_scale != 1.0:
        q *= np.float32(w.qk_scale)
        k *= np.float32(w.qk_scale)
    if w.k_outlier_every:
        rows = np.arange(T)
        sel = (rows + 1) % w.k_outlier_every == 0
        k[:, sel, :] *= np.float32(w.k_outlier_scale)
    q16 = q.astype(np.float16)
    k16 = k.astype(np.float16)
    vT16 = np.ascontiguousarray(v.astype(np.float16).transpose(0, 2, 1))
    return q16, k16, vT16


GRAD_SEED_OFFSET = 0x9E3779B9


def make_output_grad(w: Workload):
    """Returns dO [T][H*64] as a binary16 numpy array (the backward's input)."""
    rng = np.random.Generator(np.random.Philox(w.seed + GRAD_SEED_OFFSET))
    g = rng.standard_normal((w.T, w.heads * HEAD_DIM), dtype=np.float32)
    return g.astype(np.float16)


ROPE_BASE = 10000.0
PRODUCER_SEED_OFFSET = 0x51ED2700


def rotary_tables(T: int):
    """cos and sin tables [T][32] as binary32: column p holds position t times
    theta_p = 10000^(-p/32), evaluated in float64 and rounded once (the table is an
    input of the producer, made here as the nearest binary32 values)."""
    p = np.arange(HEAD_DIM // 2, dtype=np.float64)
    theta = ROPE_BASE ** (-p / (HEAD_DIM // 2))
    ang = np.arange(T, dtype=np.float64)[:, None] * theta[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def make_producer_inputs(T: int, width: int, heads: int, kv_heads: int, seed: int):
    """Inputs of the fused QKV producer from their own Philox stream: X [T][width]
    ~ N(0, 1) and W [(heads + 2 kv_heads) * 64][width] ~ N(0, 1/width), both
    rounded to binary16, and the rotary tables."""
    rng = np.random.Generator(np.random.Philox(seed + PRODUCER_SEED_OFFSET))
    x = rng.standard_normal((T, width), dtype=np.float32)
    n_out = (heads + 2 * kv_heads) * HEAD_DIM
    w = rng.standard_normal((n_out, width), dtype=np.float32) * np.float32(1.0 / np.sqrt(width))
    cos_t, sin_t = rotary_tables(T)
    return x.astype(np.float16), w.astype(np.float16), cos_t, sin_t
