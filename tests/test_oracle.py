"""Pins for the fp64 CPU oracle (no GPU).

Each test ties the oracle to something other than itself: hand-derived worked
examples (tests/golden/), a library routine (torch's scaled-dot-product
attention and logsumexp in float64), closed forms and invariants of the
definition, and an exhaustive check of its binary16 decoder.  The last test
plants mistakes in a copy of the oracle's C source and checks that these pins
catch every one.
"""
import math
import os
import re
import shutil

import numpy as np
import pytest
import torch

import oracle
import synthetic
from tests._golden import load_case, load_constants

LN2 = math.log(2.0)


def rand_inputs(T, H, G, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((H, T, 64)) * scale).astype(np.float16)
    k = (rng.standard_normal((G, T, 64)) * scale).astype(np.float16)
    vT = rng.standard_normal((G, 64, T)).astype(np.float16)
    return q, k, vT


def sdpa_reference(q, k, vT, H, G, c):
    """torch's causal scaled-dot-product attention in float64 with the natural
    scale c * ln 2 (2^(S c) = e^(S c ln 2)); K/V expanded to every query head of
    its group (query head h reads K/V head h // (H/G)).  Also the base-2
    log-sum-exp from torch.logsumexp over the materialised natural-unit scores."""
    g = H // G
    Q = torch.from_numpy(q.astype(np.float64))
    K = torch.from_numpy(k.astype(np.float64)).repeat_interleave(g, dim=0)
    V = torch.from_numpy(vT.astype(np.float64)).transpose(1, 2).repeat_interleave(g, dim=0)
    s = float(np.float64(np.float32(c))) * LN2
    O = torch.nn.functional.scaled_dot_product_attention(
        Q.unsqueeze(0), K.unsqueeze(0), V.unsqueeze(0), is_causal=True, scale=s)[0]
    T = q.shape[1]
    S = (Q @ K.transpose(1, 2)) * s
    mask = torch.triu(torch.ones(T, T, dtype=torch.bool), diagonal=1)
    S = S.masked_fill(mask, float("-inf"))
    lse = torch.logsumexp(S, dim=-1) / LN2
    # O as [T][H*64]
    return O.permute(1, 0, 2).reshape(T, H * 64).numpy(), lse.numpy()


# ---------------------------------------------------------------- decoder
def test_half_decoder_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # the sign of zero survives
    assert math.copysign(1.0, oracle.half_to_double(0x8000)) == -1.0


# ---------------------------------------------------------------- worked examples
@pytest.mark.parametrize("name", ["base2_ladder.txt", "gqa_grouping.txt"])
def test_golden_worked_example(name):
    case = load_case(name)
    T, H, G = case["T"], case["heads"], case["kv_heads"]
    o, lse = oracle.attn_fwd(case["q"], case["k"], case["vT"], T, H, G, case["c"])
    for (h, i, e), frac in case["o"].items():
        assert o[i, h * 64 + e] == pytest.approx(float(frac), rel=1e-14, abs=1e-15), (h, i, e)
    for (h, i), frac in case["lse"].items():
        assert lse[h, i] == pytest.approx(math.log2(frac), rel=1e-14, abs=1e-15), (h, i)


def test_scale_constant():
    k = load_constants()
    # 1/sqrt(64) as binary32
    assert int(np.float32(1.0 / math.sqrt(64.0)).view(np.uint32)) == k["score_scale_bits"]
    # the pages' construction: bits(binary32 log2 e) - 3 * 2^23
    assert int(np.float32(math.log2(math.e)).view(np.uint32)) == k["log2e_bits"]
    assert k["log2e_bits"] - 3 * 2 ** 23 == k["c_bits"]
    # the workload generator's c is that value: nearest binary32 to 0.125/ln 2
    assert int(np.float32(synthetic.scale_c()).view(np.uint32)) == k["c_bits"]


# ---------------------------------------------------------------- library routine
@pytest.mark.parametrize("T", [1, 2, 5, 64, 128, 192, 200])
@pytest.mark.parametrize("H,G", [(1, 1), (2, 1), (4, 2), (8, 2)])
def test_matches_torch_sdpa(T, H, G):
    c = synthetic.scale_c()
    q, k, vT = rand_inputs(T, H, G, seed=1000 * T + 10 * H + G)
    o, lse = oracle.attn_fwd(q, k, vT, T, H, G, c)
    o_ref, lse_ref = sdpa_reference(q, k, vT, H, G, c)
    np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


def test_matches_torch_sdpa_peaked():
    # large scores: the running maximum matters, weights span many binades
    c = synthetic.scale_c()
    q, k, vT = rand_inputs(160, 4, 1, seed=7, scale=4.0)
    o, lse = oracle.attn_fwd(q, k, vT, 160, 4, 1, c)
    o_ref, lse_ref = sdpa_reference(q, k, vT, 4, 1, c)
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-11)


# ---------------------------------------------------------------- closed forms
def test_first_row_is_first_value_row():
    c = synthetic.scale_c()
    T, H, G = 96, 4, 2
    q, k, vT = rand_inputs(T, H, G, seed=3)
    o, lse = oracle.attn_fwd(q, k, vT, T, H, G, c)
    for h in range(H):
        g = h // (H // G)
        # one key: weight 1, sum 1, output = V row 0 exactly
        assert np.array_equal(o[0, h * 64:(h + 1) * 64], vT[g, :, 0].astype(np.float64))
        s = math.fsum(float(a) * float(b) for a, b in zip(q[h, 0], k[g, 0]))
        assert lse[h, 0] == pytest.approx(float(np.float32(c)) * s, rel=1e-14, abs=1e-14)


def test_second_row_two_key_closed_form():
    c = synthetic.scale_c()
    q, k, vT = rand_inputs(64, 1, 1, seed=4)
    o, lse = oracle.attn_fwd(q, k, vT, 64, 1, 1, c)
    cd = float(np.float32(c))
    t0 = cd * math.fsum(float(a) * float(b) for a, b in zip(q[0, 1], k[0, 0]))
    t1 = cd * math.fsum(float(a) * float(b) for a, b in zip(q[0, 1], k[0, 1]))
    # two keys: O = sigma v0 + (1 - sigma) v1 with sigma = 1 / (1 + 2^(t1 - t0))
    sigma = 1.0 / (1.0 + 2.0 ** (t1 - t0))
    want = sigma * vT[0, :, 0].astype(np.float64) + (1 - sigma) * vT[0, :, 1].astype(np.float64)
    np.testing.assert_allclose(o[1], want, rtol=1e-13, atol=1e-14)
    assert lse[0, 1] == pytest.approx(max(t0, t1) + math.log2(1 + 2.0 ** (-abs(t1 - t0))),
                                      rel=1e-14)


# ---------------------------------------------------------------- invariants
def test_constant_value_rows_give_that_row():
    c = synthetic.scale_c()
    T, H, G = 130, 4, 2
    q, k, _ = rand_inputs(T, H, G, seed=5, scale=3.0)
    u = np.random.default_rng(6).standard_normal(64).astype(np.float16)
    vT = np.ascontiguousarray(np.broadcast_to(u[None, :, None], (G, 64, T)))
    o, _ = oracle.attn_fwd(q, k, vT, T, H, G, c)
    want = np.tile(u.astype(np.float64), H)
    np.testing.assert_allclose(o, np.broadcast_to(want, o.shape), rtol=1e-13, atol=1e-14)


def test_weights_sum_to_one_and_respect_causality():
    # V row j = e_j for j < 64: the output row is the weight vector itself
    c = synthetic.scale_c()
    T = 64
    q, k, _ = rand_inputs(T, 2, 1, seed=8, scale=2.0)
    vT = np.zeros((1, 64, T), np.float16)
    vT[0, np.arange(64), np.arange(64)] = 1.0
    o, lse = oracle.attn_fwd(q, k, vT, T, 2, 1, c)
    for h in range(2):
        P = o[:, h * 64:(h + 1) * 64]
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert np.all(P[np.triu_indices(T, 1)] == 0.0)      # no weight on later keys
        assert np.all(np.diag(P) > 0.0)                      # the diagonal key is kept
        # LSE = log2 sum_j 2^t_ij, so 2^(t_ij - LSE_i) is the weight
        S = q[h].astype(np.float64) @ k[0].astype(np.float64).T * float(np.float32(c))
        W = np.exp2(S - lse[h][:, None])
        np.testing.assert_allclose(np.tril(W), P, rtol=1e-12, atol=1e-15)


def test_gqa_equals_expanded_mha():
    c = synthetic.scale_c()
    T, H, G = 100, 8, 2
    q, k, vT = rand_inputs(T, H, G, seed=9)
    o, lse = oracle.attn_fwd(q, k, vT, T, H, G, c)
    ke = np.repeat(k, H // G, axis=0)
    ve = np.repeat(vT, H // G, axis=0)
    o2, lse2 = oracle.attn_fwd(q, ke, ve, T, H, H, c)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_scale_equivalence():
    # (2Q, c) and (Q, 2c) give the same scores exactly
    c = synthetic.scale_c()
    T, H, G = 70, 2, 2
    q, k, vT = rand_inputs(T, H, G, seed=10)
    o1, l1 = oracle.attn_fwd((q.astype(np.float32) * 2).astype(np.float16), k, vT, T, H, G, c)
    o2, l2 = oracle.attn_fwd(q, k, vT, T, H, G, 2 * c)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_later_keys_do_not_change_earlier_rows():
    c = synthetic.scale_c()
    T, H, G = 120, 4, 1
    q, k, vT = rand_inputs(T, H, G, seed=11)
    o1, l1 = oracle.attn_fwd(q, k, vT, T, H, G, c)
    cut = 57
    k2, v2 = k.copy(), vT.copy()
    k2[:, cut + 1:, :] = np.float16(9.0)
    v2[:, :, cut + 1:] = np.float16(-5.0)
    o2, l2 = oracle.attn_fwd(q, k2, v2, T, H, G, c)
    assert np.array_equal(o1[:cut + 1], o2[:cut + 1])
    assert np.array_equal(l1[:, :cut + 1], l2[:, :cut + 1])
    assert not np.array_equal(o1[cut + 1:], o2[cut + 1:])


def test_rows_entry_matches_full_and_thread_count():
    c = synthetic.scale_c()
    T, H, G = 150, 4, 2
    q, k, vT = rand_inputs(T, H, G, seed=12)
    o, lse = oracle.attn_fwd(q, k, vT, T, H, G, c, threads=1)
    o4, lse4 = oracle.attn_fwd(q, k, vT, T, H, G, c, threads=4)
    assert np.array_equal(o, o4) and np.array_equal(lse, lse4)
    hs = np.array([0, 3, 1, 2, 3])
    rs = np.array([0, 149, 77, 1, 64])
    ro, rl = oracle.attn_fwd_rows(q, k, vT, T, H, G, c, hs, rs)
    for n, (h, i) in enumerate(zip(hs, rs)):
        assert np.array_equal(ro[n], o[i, h * 64:(h + 1) * 64])
        assert rl[n] == lse[h, i]


def test_rejects_bad_shapes():
    q, k, vT = rand_inputs(8, 3, 2, seed=0)
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, k, vT, 8, 3, 2, 0.18)          # 3 heads over 2 K/V heads
    q, k, vT = rand_inputs(8, 2, 1, seed=0)
    with pytest.raises(ValueError):
        oracle.attn_fwd_rows(q, k, vT, 8, 2, 1, 0.18, [0], [8])  # row out of range


# ---------------------------------------------------------------- pins catch planted mistakes
MUTANTS = {
    "natural_exp": ("t[j] = exp2(t[j] - m);", "t[j] = exp(t[j] - m);"),
    "natural_log": ("*lse = m + log2(l);", "*lse = m + log(l);"),
    "no_diagonal": ("for (int64_t j = 0; j <= i; ++j) {\n        const uint16_t *kj = k + (g * T + j) * HEAD_DIM;\n        double s = 0.0;",
                    "for (int64_t j = 0; j < i; ++j) {\n        const uint16_t *kj = k + (g * T + j) * HEAD_DIM;\n        double s = 0.0;"),
    "interleaved_groups": ("const int64_t g = h / group;", "const int64_t g = h % kv_heads;"),
    "v_not_transposed": ("acc += t[j] * g_half[ve[j]];",
                         "acc += t[j] * g_half[vT[(g * T + j) * HEAD_DIM + e]];"),
    "scale_dropped": ("t[j] = c * s;", "t[j] = s;"),
    "unnormalised": ("o_row[e] = acc / l;", "o_row[e] = acc;"),
    "max_not_subtracted_in_lse": ("*lse = m + log2(l);", "*lse = log2(l);"),
}


def _pins_pass(lib):
    """The worked examples and the library comparison, against one oracle build."""
    try:
        for name in ["base2_ladder.txt", "gqa_grouping.txt"]:
            case = load_case(name)
            o, lse = oracle.attn_fwd(case["q"], case["k"], case["vT"], case["T"],
                                     case["heads"], case["kv_heads"], case["c"], lib=lib)
            for (h, i, e), frac in case["o"].items():
                if not math.isclose(o[i, h * 64 + e], float(frac), rel_tol=1e-12, abs_tol=1e-14):
                    return False
            for (h, i), frac in case["lse"].items():
                if not math.isclose(lse[h, i], math.log2(frac), rel_tol=1e-12, abs_tol=1e-14):
                    return False
        c = synthetic.scale_c()
        q, k, vT = rand_inputs(80, 4, 2, seed=99)
        o, lse = oracle.attn_fwd(q, k, vT, 80, 4, 2, c, lib=lib)
        o_ref, lse_ref = sdpa_reference(q, k, vT, 4, 2, c)
        return bool(np.allclose(o, o_ref, rtol=1e-10, atol=1e-11)
                    and np.allclose(lse, lse_ref, rtol=1e-10, atol=1e-11))
    except ValueError:
        return False


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_pins_catch_planted_mistakes(tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()
    # the unmodified source passes
    good = oracle.build(src=_write(tmp_path, "good.c", src), out=str(tmp_path / "good.so"))
    assert _pins_pass(oracle.open_library(good))
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, name
        path = _write(tmp_path, f"{name}.c", src.replace(old, new))
        lib = oracle.open_library(oracle.build(src=path, out=str(tmp_path / f"{name}.so")))
        assert not _pins_pass(lib), f"planted mistake '{name}' was not caught"


def _write(d, name, text):
    p = d / name
    p.write_text(text)
    return str(p)
