"""Pins for the fp64 backward oracle (no GPU).

The backward follows the page's statement: P = 2^(S c - L), dP = dO V^T,
D = rowsum(dO * O), dS = P (dP - D), dQ = s dS K, dK = s dS^T Q, dV = P^T dO,
dK and dV summed over each K/V head's group.  It is pinned against torch's
float64 autograd through scaled-dot-product attention (a library routine), a
closed form for one key, the identity D = rowsum(P * dP) at the exact forward,
causality, and agreement of its sampled-rows entry with the full one.  The
last test plants mistakes in a copy of the C source and checks the pins catch
each one.
"""
import math
import os
import shutil

import numpy as np
import pytest
import torch

import oracle
import synthetic

LN2 = math.log(2.0)


def rand_case(T, H, G, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((H, T, 64)) * scale).astype(np.float16)
    k = (rng.standard_normal((G, T, 64)) * scale).astype(np.float16)
    vT = rng.standard_normal((G, 64, T)).astype(np.float16)
    dO = rng.standard_normal((T, H * 64)).astype(np.float16)
    return q, k, vT, dO


def autograd_reference(q, k, vT, dO, H, G, c):
    """torch float64 causal SDPA with the natural scale c ln 2 (2^(S c) = e^(S c ln 2)),
    K/V expanded over each group (query head h reads K/V head h // (H/G)); gradients by
    autograd.  Returns (dQ [H][T][64], dK [G][T][64], dV^T [G][64][T]) and the scale."""
    g = H // G
    T = q.shape[1]
    s_nat = float(np.float64(np.float32(c))) * LN2
    Q = torch.from_numpy(q.astype(np.float64)).requires_grad_(True)
    K = torch.from_numpy(k.astype(np.float64)).requires_grad_(True)
    V = torch.from_numpy(vT.astype(np.float64)).transpose(1, 2).contiguous().requires_grad_(True)
    O = torch.nn.functional.scaled_dot_product_attention(
        Q.unsqueeze(0), K.repeat_interleave(g, 0).unsqueeze(0),
        V.repeat_interleave(g, 0).unsqueeze(0), is_causal=True, scale=s_nat)[0]
    G_ = torch.from_numpy(dO.astype(np.float64)).reshape(T, H, 64).permute(1, 0, 2)
    O.backward(G_)
    return (Q.grad.numpy(), K.grad.numpy(), V.grad.numpy().transpose(0, 2, 1), s_nat)


def exact_forward(q, k, vT, T, H, G, c):
    return oracle.attn_fwd(q, k, vT, T, H, G, c)


@pytest.mark.parametrize("T", [1, 3, 64, 130])
@pytest.mark.parametrize("H,G", [(1, 1), (4, 2), (4, 1)])
def test_matches_torch_autograd(T, H, G):
    c = synthetic.scale_c()
    q, k, vT, dO = rand_case(T, H, G, seed=100 * T + 10 * H + G)
    o, lse = exact_forward(q, k, vT, T, H, G, c)
    dq_ref, dk_ref, dvT_ref, s_nat = autograd_reference(q, k, vT, dO, H, G, c)
    dq, dk, dvT, _ = oracle.attn_bwd(q, k, vT, o, lse, dO, T, H, G, c, s_nat)
    np.testing.assert_allclose(dq, dq_ref, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(dk, dk_ref, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(dvT, dvT_ref, rtol=1e-9, atol=1e-11)


def test_single_key_closed_form():
    # one key: P = 1, O = V_0, so D = dO . V_0 = dP and dS = 0: dQ = dK = 0, dV = sum of dO
    c = synthetic.scale_c()
    q, k, vT, dO = rand_case(1, 4, 2, seed=3)
    o, lse = exact_forward(q, k, vT, 1, 4, 2, c)
    dq, dk, dvT, D = oracle.attn_bwd(q, k, vT, o, lse, dO, 1, 4, 2, c, 0.125)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    g = dO.astype(np.float64).reshape(1, 4, 64)
    want = np.stack([g[0, 0] + g[0, 1], g[0, 2] + g[0, 3]])     # per K/V head, over its group
    np.testing.assert_allclose(dvT[:, :, 0], want, rtol=1e-14, atol=1e-14)


def test_row_term_identity_at_exact_forward():
    # D = rowsum(dO * O) equals rowsum(P * dP) when O and L are the exact forward's
    c = synthetic.scale_c()
    T, H, G = 96, 2, 1
    q, k, vT, dO = rand_case(T, H, G, seed=4)
    o, lse = exact_forward(q, k, vT, T, H, G, c)
    _, _, _, D = oracle.attn_bwd(q, k, vT, o, lse, dO, T, H, G, c, 0.125)
    for h in range(H):
        S = q[h].astype(np.float64) @ k[0].astype(np.float64).T
        P = np.tril(np.exp2(S * float(np.float32(c)) - lse[h][:, None]))
        dP = dO.astype(np.float64)[:, h * 64:(h + 1) * 64] @ vT[0].astype(np.float64)
        np.testing.assert_allclose(D[h], (P * dP).sum(1), rtol=1e-11, atol=1e-12)


def test_earlier_queries_do_not_change_later_key_gradients():
    c = synthetic.scale_c()
    T, H, G = 80, 2, 1
    q, k, vT, dO = rand_case(T, H, G, seed=5)
    o, lse = exact_forward(q, k, vT, T, H, G, c)
    _, dk1, dv1, _ = oracle.attn_bwd(q, k, vT, o, lse, dO, T, H, G, c, 0.125)
    cut = 33          # query rows < cut changed: key rows >= cut only see queries >= cut
    q2, dO2, o2, lse2 = q.copy(), dO.copy(), o.copy(), lse.copy()
    q2[:, :cut] = np.float16(0.7)
    dO2[:cut] = np.float16(-2.0)
    o2[:cut] = 0.3
    lse2[:, :cut] = 5.0
    _, dk2, dv2, _ = oracle.attn_bwd(q2, k, vT, o2, lse2, dO2, T, H, G, c, 0.125)
    assert np.array_equal(dk1[:, cut:], dk2[:, cut:])
    assert np.array_equal(dv1[:, :, cut:], dv2[:, :, cut:])
    assert not np.array_equal(dk1[:, :cut], dk2[:, :cut])


def test_rows_entry_matches_full():
    c = synthetic.scale_c()
    T, H, G = 70, 4, 2
    q, k, vT, dO = rand_case(T, H, G, seed=6)
    o, lse = exact_forward(q, k, vT, T, H, G, c)
    dq, dk, dvT, _ = oracle.attn_bwd(q, k, vT, o, lse, dO, T, H, G, c, 0.125)
    qh, qi = np.array([0, 3, 2, 1]), np.array([0, 69, 33, 64])
    kg, kj = np.array([0, 1, 1]), np.array([69, 0, 40])
    rq, rk, rv = oracle.attn_bwd_rows(q, k, vT, o, lse, dO, T, H, G, c, 0.125, qh, qi, kg, kj)
    for n, (h, i) in enumerate(zip(qh, qi)):
        assert np.array_equal(rq[n], dq[h, i])
    for n, (g, j) in enumerate(zip(kg, kj)):
        assert np.array_equal(rk[n], dk[g, j])
        assert np.array_equal(rv[n], dvT[g, :, j])


MUTANTS = {
    "natural_exp": ("const double p = exp2(c * dot64_hq(kj, qd) - lse[h * T + i]);",
                    "const double p = exp(c * dot64_hq(kj, qd) - lse[h * T + i]);"),
    "row_term_sign": ("const double ds = p * (dp - D[h * T + i]);\n        for (int e = 0; e < HEAD_DIM; ++e)\n            acc",
                      "const double ds = p * (dp + D[h * T + i]);\n        for (int e = 0; e < HEAD_DIM; ++e)\n            acc"),
    "dq_scale_dropped": ("out[e] = s * acc[e];", "out[e] = acc[e];"),
    "dv_uses_ds": ("dv[e] += p * g_half[gi[e]];", "dv[e] += ds * g_half[gi[e]];"),
    "dk_uses_k": ("dk[e] += ds * g_half[qi[e]];", "dk[e] += ds * kd[e];"),
    "key_range_strict": ("for (int64_t i = j; i < T; ++i) {", "for (int64_t i = j + 1; i < T; ++i) {"),
}


def _bwd_pins_pass(lib):
    c = synthetic.scale_c()
    for T, H, G in [(1, 2, 1), (40, 4, 2)]:
        q, k, vT, dO = rand_case(T, H, G, seed=77 + T)
        o, lse = oracle.attn_fwd(q, k, vT, T, H, G, c)
        dq_ref, dk_ref, dvT_ref, s_nat = autograd_reference(q, k, vT, dO, H, G, c)
        dq, dk, dvT, _ = oracle.attn_bwd(q, k, vT, o, lse, dO, T, H, G, c, s_nat, lib=lib)
        ok = (np.allclose(dq, dq_ref, rtol=1e-6, atol=1e-9) and np.allclose(dk, dk_ref, rtol=1e-6, atol=1e-9)
              and np.allclose(dvT, dvT_ref, rtol=1e-9, atol=1e-11))
        if not ok:
            return False
    return True


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_backward_pins_catch_planted_mistakes(tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()
    good = tmp_path / "good.c"
    good.write_text(src)
    assert _bwd_pins_pass(oracle.open_library(oracle.build(src=str(good), out=str(tmp_path / "good.so"))))
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, name
        path = tmp_path / f"{name}.c"
        path.write_text(src.replace(old, new))
        lib = oracle.open_library(oracle.build(src=str(path), out=str(tmp_path / f"{name}.so")))
        assert not _bwd_pins_pass(lib), f"planted mistake '{name}' was not caught"
