"""Pins for the fp64 oracle of the fused QKV producer (no GPU).

The product is pinned to numpy's float64 matrix product of the exact binary16
values (with the rotation switched off: cos = 1, sin = 0), the rotation to a
hand-worked example (a unit input in one pair comes out as (cos, sin)), and
both together to invariants of a rotation: pair norms are kept, and the
rotated query-key dot product depends only on the positions' difference.  A
planted-mistake test checks that these pins catch plausible errors."""
import os
import shutil

import numpy as np
import pytest

import oracle
import synthetic


def identity_tables(T):
    return np.ones((T, 32), np.float32), np.zeros((T, 32), np.float32)


def layout_reference(x, w, heads, kv_heads):
    """numpy float64 product, cut into the outputs' layouts (no rotation)."""
    y = x.astype(np.float64) @ w.astype(np.float64).T          # [T][n_out]
    T = x.shape[0]
    q = y[:, :heads * 64].reshape(T, heads, 64).transpose(1, 0, 2)
    k = y[:, heads * 64:(heads + kv_heads) * 64].reshape(T, kv_heads, 64).transpose(1, 0, 2)
    v = y[:, (heads + kv_heads) * 64:].reshape(T, kv_heads, 64).transpose(1, 2, 0)
    return q, k, v


@pytest.mark.parametrize("T,width,H,G", [(5, 64, 1, 1), (17, 128, 4, 2), (9, 192, 2, 2)])
def test_product_and_layouts_match_numpy(T, width, H, G):
    x, w, _, _ = synthetic.make_producer_inputs(T, width, H, G, seed=T + width)
    c, s = identity_tables(T)
    q, k, vT = oracle.qkv_rope(x, w, c, s, T, width, H, G)
    rq, rk, rv = layout_reference(x, w, H, G)
    np.testing.assert_allclose(q, rq, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(k, rk, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(vT, rv, rtol=1e-12, atol=1e-12)


def test_rotation_worked_example():
    # one head of width 64: W routes input element i to output i of every part
    # (the identity), X a unit vector in pair p: the rotated query pair p is
    # (cos, sin) for (1, 0) and (-sin, cos) for (0, 1), the other pairs stay zero,
    # V is not rotated
    T, width = 3, 64
    w = np.zeros((3 * 64, 64), np.float16)
    for part in range(3):
        w[part * 64:(part + 1) * 64] = np.eye(64, dtype=np.float16)
    cos_t = np.array([[np.float32(0.25 * (p + 1) / 32)] * 1 for p in range(32)], np.float32).T.repeat(T, 0)
    sin_t = np.array([[np.float32(-0.5 + p / 64)] for p in range(32)], np.float32).T.repeat(T, 0)
    for p in (0, 7, 31):
        for second in (False, True):
            x = np.zeros((T, width), np.float16)
            x[:, 2 * p + second] = 1.0
            q, k, vT = oracle.qkv_rope(x, w, cos_t, sin_t, T, width, 1, 1)
            for t in range(T):
                want = np.zeros(64)
                c, s = np.float64(cos_t[t, p]), np.float64(sin_t[t, p])
                # (1, 0) -> (cos, sin); (0, 1) -> (-sin, cos)
                want[2 * p], want[2 * p + 1] = (-s, c) if second else (c, s)
                assert np.array_equal(q[0, t], want)
                assert np.array_equal(k[0, t], want)
            assert np.array_equal(vT[0, :, :], x.astype(np.float64).T)   # V: the input, transposed


def test_rotation_keeps_pair_norms():
    T, width, H, G = 11, 128, 2, 1
    x, w, c, s = synthetic.make_producer_inputs(T, width, H, G, seed=3)
    q, k, _ = oracle.qkv_rope(x, w, c, s, T, width, H, G)
    q0, k0, _ = oracle.qkv_rope(x, w, *identity_tables(T), T, width, H, G)
    for a, b in ((q, q0), (k, k0)):
        na = a[..., 0::2] ** 2 + a[..., 1::2] ** 2
        nb = b[..., 0::2] ** 2 + b[..., 1::2] ** 2
        np.testing.assert_allclose(na, nb, rtol=1e-6, atol=1e-9)   # tables are binary32


def test_relative_position_property():
    # the same input at every position: the rotated query-key dot product depends
    # only on the positions' difference (cos/sin of the same angles, binary32 tables)
    T, width = 24, 64
    rng = np.random.default_rng(9)
    row = rng.standard_normal(width).astype(np.float16)
    x = np.tile(row, (T, 1))
    w = (rng.standard_normal((3 * 64, width)) / 8).astype(np.float16)
    c, s = synthetic.rotary_tables(T)
    q, k, _ = oracle.qkv_rope(x, w, c, s, T, width, 1, 1)
    dots = q[0] @ k[0].T                                    # [m][n]
    for d in range(-5, 6):
        vals = np.array([dots[m, m - d] for m in range(max(0, d), min(T, T + d))])
        assert np.abs(vals - vals[0]).max() <= 1e-4 * np.abs(dots).max()


MUTANTS = {
    "sin_sign": ("dst[2 * p] = a * c - b * s;", "dst[2 * p] = a * c + b * s;"),
    "cos_sin_swapped": ("const double c = (double)cos_tab[t * (HEAD_DIM / 2) + p];",
                        "const double c = (double)sin_tab[t * (HEAD_DIM / 2) + p];"),
    "half_split_pairs": ("const double a = src[2 * p], b = src[2 * p + 1];",
                         "const double a = src[p], b = src[p + HEAD_DIM / 2];"),
    "value_part_offset": ("const double *src = y + (heads + kv_heads + g) * HEAD_DIM;",
                          "const double *src = y + (heads + g) * HEAD_DIM;"),
    "value_not_transposed": ("vT[(g * HEAD_DIM + e) * T + t] = src[e];",
                             "vT[(g * T + t) * HEAD_DIM + e] = src[e];"),
}


def _pins_pass(lib):
    T, width, H, G = 7, 128, 4, 2
    x, w, c, s = synthetic.make_producer_inputs(T, width, H, G, seed=11)
    ci, si = identity_tables(T)
    q, k, vT = oracle.qkv_rope(x, w, ci, si, T, width, H, G, lib=lib)
    rq, rk, rv = layout_reference(x, w, H, G)
    if not (np.allclose(q, rq) and np.allclose(k, rk) and np.allclose(vT, rv)):
        return False
    # the worked example
    w1 = np.zeros((3 * 64, 64), np.float16)
    for part in range(3):
        w1[part * 64:(part + 1) * 64] = np.eye(64, dtype=np.float16)
    x1 = np.zeros((2, 64), np.float16)
    x1[:, 6] = 1.0
    c1 = np.full((2, 32), 0.6, np.float32)
    s1 = np.full((2, 32), 0.8, np.float32)
    q1, _, _ = oracle.qkv_rope(x1, w1, c1, s1, 2, 64, 1, 1, lib=lib)
    want = np.zeros(64)
    want[6], want[7] = np.float32(0.6), np.float32(0.8)
    x2 = np.zeros((2, 64), np.float16)
    x2[:, 7] = 1.0                                  # the pair's second element: (-sin, cos)
    q2, _, _ = oracle.qkv_rope(x2, w1, c1, s1, 2, 64, 1, 1, lib=lib)
    want2 = np.zeros(64)
    want2[6], want2[7] = -np.float32(0.8), np.float32(0.6)
    return bool(np.array_equal(q1[0, 0], want) and np.array_equal(q2[0, 0], want2))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_pins_catch_planted_mistakes(tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()
    good = tmp_path / "good.c"
    good.write_text(src)
    assert _pins_pass(oracle.open_library(oracle.build(src=str(good), out=str(tmp_path / "good.so"))))
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, name
        path = tmp_path / f"{name}.c"
        path.write_text(src.replace(old, new))
        lib = oracle.open_library(oracle.build(src=str(path), out=str(tmp_path / f"{name}.so")))
        assert not _pins_pass(lib), f"planted mistake '{name}' was not caught"
