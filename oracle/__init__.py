"""fp64 CPU oracle for the causal grouped-query attention forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this package.  The
product path (``transformer_causal_gqa_gb300``) never imports it and has no
CPU fallback.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64); this module only
compiles it with gcc (once, into ``oracle/_build/``) and marshals numpy arrays
through ctypes.  What it computes follows the page
"Realization/Nvidia/SM86/StreamingAttentionSM86.alpha", header comment:
softmax(Q K^T scale) V per query head in base-2 units, t = S c, weights
2^(t - m), output O / l and log-sum-exp m + log2 l.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
HEAD_DIM = 64

_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile attn_oracle.c into a shared library (OpenMP if gcc supports it)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    fresh = os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src)
    if fresh and not force:
        return out
    tmp = out + f".{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, src, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def open_library(path: str):
    """ctypes handle on a compiled oracle library, with its signatures declared."""
    lib = ctypes.CDLL(path)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_attn_fwd.argtypes = [u16p, u16p, u16p, i64, i64, i64, ctypes.c_float,
                                    f64p, f64p, ctypes.c_int]
    lib.oracle_attn_fwd.restype = ctypes.c_int
    lib.oracle_attn_fwd_rows.argtypes = [u16p, u16p, u16p, i64, i64, i64, ctypes.c_float,
                                         i64p, i64p, i64, f64p, f64p, ctypes.c_int]
    lib.oracle_attn_fwd_rows.restype = ctypes.c_int
    f = ctypes.c_float
    lib.oracle_attn_bwd.argtypes = [u16p, u16p, u16p, f64p, f64p, u16p, i64, i64, i64, f, f,
                                    f64p, f64p, f64p, f64p, ctypes.c_int]
    lib.oracle_attn_bwd.restype = ctypes.c_int
    lib.oracle_attn_bwd_rows.argtypes = [u16p, u16p, u16p, f64p, f64p, u16p, i64, i64, i64, f, f,
                                         i64p, i64p, i64, i64p, i64p, i64, f64p, f64p, f64p,
                                         ctypes.c_int]
    lib.oracle_attn_bwd_rows.restype = ctypes.c_int
    f32p = ctypes.POINTER(ctypes.c_float)
    lib.oracle_qkv_rope.argtypes = [u16p, u16p, f32p, f32p, i64, i64, i64, i64, f64p, f64p, f64p,
                                    ctypes.c_int]
    lib.oracle_qkv_rope.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = open_library(build())
    return _lib


def _bits(a: np.ndarray, shape: tuple) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.float16:
        raise TypeError("oracle inputs are binary16 arrays")
    if a.shape != shape:
        raise ValueError(f"expected shape {shape}, got {a.shape}")
    return a.view(np.uint16)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def half_to_double(bits: int) -> float:
    """Exact value of one binary16 bit pattern, decoded by the oracle's own routine."""
    return float(_load().oracle_half_to_double(int(bits) & 0xFFFF))


def max_threads() -> int:
    """Threads the oracle uses when ``threads`` is not given."""
    return int(_load().oracle_max_threads())


def attn_fwd(q: np.ndarray, k: np.ndarray, vT: np.ndarray, T: int, heads: int,
             kv_heads: int, c: float, threads: int = 0, lib=None):
    """Every row.  Returns (O float64 [T][heads*64], LSE float64 [heads][T])."""
    lib = lib or _load()
    qb = _bits(q, (heads, T, HEAD_DIM))
    kb = _bits(k, (kv_heads, T, HEAD_DIM))
    vb = _bits(vT, (kv_heads, HEAD_DIM, T))
    o = np.empty((T, heads * HEAD_DIM), dtype=np.float64)
    lse = np.empty((heads, T), dtype=np.float64)
    rc = lib.oracle_attn_fwd(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                             _ptr(vb, ctypes.c_uint16), T, heads, kv_heads,
                             ctypes.c_float(c), _ptr(o, ctypes.c_double),
                             _ptr(lse, ctypes.c_double), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the shape")
    return o, lse


def attn_fwd_rows(q: np.ndarray, k: np.ndarray, vT: np.ndarray, T: int, heads: int,
                  kv_heads: int, c: float, heads_idx, rows_idx, threads: int = 0,
                  lib=None):
    """Selected (head, row) pairs.  Returns (O float64 [n][64], LSE float64 [n])."""
    lib = lib or _load()
    qb = _bits(q, (heads, T, HEAD_DIM))
    kb = _bits(k, (kv_heads, T, HEAD_DIM))
    vb = _bits(vT, (kv_heads, HEAD_DIM, T))
    hi = np.ascontiguousarray(heads_idx, dtype=np.int64)
    ri = np.ascontiguousarray(rows_idx, dtype=np.int64)
    if hi.shape != ri.shape or hi.ndim != 1:
        raise ValueError("heads_idx and rows_idx must be 1-D and equal length")
    n = hi.shape[0]
    o = np.empty((n, HEAD_DIM), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = lib.oracle_attn_fwd_rows(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                  _ptr(vb, ctypes.c_uint16), T, heads, kv_heads,
                                  ctypes.c_float(c), _ptr(hi, ctypes.c_int64),
                                  _ptr(ri, ctypes.c_int64), n, _ptr(o, ctypes.c_double),
                                  _ptr(lse, ctypes.c_double), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the shape or an index")
    return o, lse


def _f64(a, shape):
    a = np.ascontiguousarray(a, dtype=np.float64)
    if a.shape != shape:
        raise ValueError(f"expected shape {shape}, got {a.shape}")
    return a


def attn_bwd(q, k, vT, o, lse, dO, T: int, heads: int, kv_heads: int, c: float, s: float,
             threads: int = 0, lib=None):
    """Backward pass.  o, lse: the forward's output and base-2 log-sum-exp (any float
    dtype; taken as given); dO: binary16 [T][heads*64].  Returns (dQ [heads][T][64],
    dK [kv_heads][T][64], dV^T [kv_heads][64][T], D [heads][T]), all float64."""
    lib = lib or _load()
    qb = _bits(q, (heads, T, HEAD_DIM))
    kb = _bits(k, (kv_heads, T, HEAD_DIM))
    vb = _bits(vT, (kv_heads, HEAD_DIM, T))
    gb = _bits(dO, (T, heads * HEAD_DIM))
    od = _f64(o, (T, heads * HEAD_DIM))
    ld = _f64(lse, (heads, T))
    dq = np.empty((heads, T, HEAD_DIM))
    dk = np.empty((kv_heads, T, HEAD_DIM))
    dvT = np.empty((kv_heads, HEAD_DIM, T))
    D = np.empty((heads, T))
    rc = lib.oracle_attn_bwd(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                             _ptr(vb, ctypes.c_uint16), _ptr(od, ctypes.c_double),
                             _ptr(ld, ctypes.c_double), _ptr(gb, ctypes.c_uint16), T, heads,
                             kv_heads, ctypes.c_float(c), ctypes.c_float(s),
                             _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double),
                             _ptr(dvT, ctypes.c_double), _ptr(D, ctypes.c_double), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the shape")
    return dq, dk, dvT, D


def attn_bwd_rows(q, k, vT, o, lse, dO, T: int, heads: int, kv_heads: int, c: float, s: float,
                  q_heads, q_rows, kv_heads_idx, kv_rows, threads: int = 0, lib=None):
    """Sampled rows of the backward: dQ at (q_heads[r], q_rows[r]) and dK, dV at
    (kv_heads_idx[r], kv_rows[r]).  Returns (dQ [n_q][64], dK [n_kv][64], dV [n_kv][64])."""
    lib = lib or _load()
    qb = _bits(q, (heads, T, HEAD_DIM))
    kb = _bits(k, (kv_heads, T, HEAD_DIM))
    vb = _bits(vT, (kv_heads, HEAD_DIM, T))
    gb = _bits(dO, (T, heads * HEAD_DIM))
    od = _f64(o, (T, heads * HEAD_DIM))
    ld = _f64(lse, (heads, T))
    qh = np.ascontiguousarray(q_heads, dtype=np.int64)
    qi = np.ascontiguousarray(q_rows, dtype=np.int64)
    kg = np.ascontiguousarray(kv_heads_idx, dtype=np.int64)
    kj = np.ascontiguousarray(kv_rows, dtype=np.int64)
    if qh.shape != qi.shape or kg.shape != kj.shape:
        raise ValueError("index arrays must pair up")
    dq = np.empty((qh.shape[0], HEAD_DIM))
    dk = np.empty((kg.shape[0], HEAD_DIM))
    dv = np.empty((kg.shape[0], HEAD_DIM))
    rc = lib.oracle_attn_bwd_rows(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                  _ptr(vb, ctypes.c_uint16), _ptr(od, ctypes.c_double),
                                  _ptr(ld, ctypes.c_double), _ptr(gb, ctypes.c_uint16), T, heads,
                                  kv_heads, ctypes.c_float(c), ctypes.c_float(s),
                                  _ptr(qh, ctypes.c_int64), _ptr(qi, ctypes.c_int64), qh.shape[0],
                                  _ptr(kg, ctypes.c_int64), _ptr(kj, ctypes.c_int64), kg.shape[0],
                                  _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double),
                                  _ptr(dv, ctypes.c_double), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the shape or an index")
    return dq, dk, dv


def qkv_rope(x, w, cos_tab, sin_tab, T: int, width: int, heads: int, kv_heads: int,
             threads: int = 0, lib=None):
    """The fused QKV producer.  x: binary16 [T][width]; w: binary16
    [(heads + 2 kv_heads) * 64][width] (parts Q, K, V); cos_tab, sin_tab: binary32
    [T][32].  Returns (q [heads][T][64], k [kv_heads][T][64], vT [kv_heads][64][T]),
    float64, unrounded."""
    lib = lib or _load()
    n_out = (heads + 2 * kv_heads) * HEAD_DIM
    xb = _bits(x, (T, width))
    wb = _bits(w, (n_out, width))
    ct = np.ascontiguousarray(cos_tab, dtype=np.float32)
    st = np.ascontiguousarray(sin_tab, dtype=np.float32)
    if ct.shape != (T, HEAD_DIM // 2) or st.shape != (T, HEAD_DIM // 2):
        raise ValueError("rotary tables must be [T][32] float32")
    q = np.empty((heads, T, HEAD_DIM))
    k = np.empty((kv_heads, T, HEAD_DIM))
    vT = np.empty((kv_heads, HEAD_DIM, T))
    rc = lib.oracle_qkv_rope(_ptr(xb, ctypes.c_uint16), _ptr(wb, ctypes.c_uint16),
                             _ptr(ct, ctypes.c_float), _ptr(st, ctypes.c_float), T, width, heads,
                             kv_heads, _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                             _ptr(vT, ctypes.c_double), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the shape")
    return q, k, vT
