"""Edge cases of the forward and backward passes at the admission limits, and
degenerate scales.

Admission (the page's predicate for the forward program): heads <= 65535 and
heads * 64 * T * 4 <= 2^32 - 1.  Two launches sit on those limits:
  * 65535 query heads over 257 K/V heads (groups of 255), T = 128;
  * 4 query heads over one K/V head at T = 4194240, the largest multiple of 64
    with 4 * 64 * T * 4 <= 2^32 - 1 (2.1 GB each for Q and O, 9.0e15 FLOP).
Both are compared with the fp64 oracle on sampled (head, row) pairs it
computes one by one, and checked at every element on the device (finite; each
output row a convex combination of V rows, so |O| <= max |V|).

Degenerate scales: c tiny (every weight 2^(t - m) is 1 to binary32 precision,
so O is the mean of the visible V rows), c denormal (the fused t = S c rounds
to zero), and c large (scores 30+ base-2 units apart: nearly one-hot rows).
These are compared on every element.

Tolerances as everywhere: max |dO| <= 4e-3, max |dLSE| <= 1e-3 (base 2) for the
forward; the per-element bound of tests/test_attn_bwd_gpu.py for the backward (below).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import transformer_causal_gqa_gb300 as tcg
from transformer_causal_gqa_gb300 import build as tcg_build

pytestmark = pytest.mark.gpu

TOL_O = 4e-3
TOL_LSE = 1e-3


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tcg_build.build()
    return tcg.load_library()


def _sampled_check(w, n_random, seed):
    q, k, vT = synthetic.make_inputs(w)
    c = synthetic.scale_c()
    T, H, G = w.T, w.heads, w.kv_heads
    assert H * 64 * T * 4 <= 2 ** 32 - 1
    dev = torch.device("cuda:0")
    qd, kd, vd = (torch.from_numpy(x).to(dev) for x in (q, k, vT))
    o = torch.full((T, H * 64), float("nan"), dtype=torch.float16, device=dev)
    lse = torch.full((H, T), float("nan"), dtype=torch.float32, device=dev)
    tcg.attn_fwd(qd, kd, vd, o, lse, T, H, G, c)
    assert tcg.last_device_status() == tcg.ATTN_OK
    # every element, on the device
    assert bool(torch.isfinite(o).all().item()) and bool(torch.isfinite(lse).all().item())
    vmax = float(vd.abs().max().item())
    assert float(o.abs().max().item()) <= vmax * (1 + 1e-3)
    # sampled rows against the oracle: the first, the last and tile-boundary rows, random ones
    rng = np.random.default_rng(seed)
    fixed_rows = [0, 1, 63, 64, 127, T - 1] + ([128, 255, 256, T // 2, T - 128] if T > 256 else [])
    rows = np.concatenate([np.array(fixed_rows), rng.integers(0, T, n_random)])
    heads = np.concatenate([np.array([0, H - 1] * ((len(fixed_rows) + 1) // 2))[:len(fixed_rows)],
                            rng.integers(0, H, n_random)])
    o_ref, l_ref = oracle.attn_fwd_rows(q, k, vT, T, H, G, c, heads, rows)
    got_o = torch.stack([o[int(r), int(h) * 64:(int(h) + 1) * 64] for h, r in zip(heads, rows)])
    got_o = got_o.double().cpu().numpy()
    got_l = lse[torch.as_tensor(heads, device=dev), torch.as_tensor(rows, device=dev)]
    got_l = got_l.double().cpu().numpy()
    d_o = float(np.abs(got_o - o_ref).max())
    d_l = float(np.abs(got_l - l_ref).max())
    assert d_o <= TOL_O, f"max |dO| = {d_o}"
    assert d_l <= TOL_LSE, f"max |dLSE| = {d_l}"
    return d_o, d_l


def test_most_heads_admitted():
    # 65535 units of one row block: many more units than SMs, the largest head index
    _sampled_check(synthetic.custom(128, 65535, 257, seed=65535), n_random=1500, seed=11)


def test_longest_sequence_admitted():
    # the largest T the predicate admits for four query heads: one CTA's units hold up to
    # 32768 key tiles, and every index of Q, K, V^T, O and LSE is past 2^31 bytes
    T = (2 ** 32 - 1) // (4 * 64 * 4) // 64 * 64
    assert T == 4194240
    _sampled_check(synthetic.custom(T, 4, 1, seed=4242), n_random=64, seed=12)


@pytest.mark.parametrize("c", [1e-6, 1e-40, 32.0])
def test_degenerate_scales(c):
    w = synthetic.custom(1088, 8, 2, seed=909)
    q, k, vT = synthetic.make_inputs(w)
    c32 = float(np.float32(c))
    assert c32 > 0.0
    dev = torch.device("cuda:0")
    qd, kd, vd = (torch.from_numpy(x).to(dev) for x in (q, k, vT))
    o = torch.full((w.T, w.heads * 64), float("nan"), dtype=torch.float16, device=dev)
    lse = torch.full((w.heads, w.T), float("nan"), dtype=torch.float32, device=dev)
    tcg.attn_fwd(qd, kd, vd, o, lse, w.T, w.heads, w.kv_heads, c32)
    assert tcg.last_device_status() == tcg.ATTN_OK
    o_ref, l_ref = oracle.attn_fwd(q, k, vT, w.T, w.heads, w.kv_heads, c32)
    got_o = o.double().cpu().numpy()
    got_l = lse.double().cpu().numpy()
    assert np.isfinite(got_o).all() and np.isfinite(got_l).all()
    assert np.abs(got_o - o_ref).max() <= TOL_O
    assert np.abs(got_l - l_ref).max() <= TOL_LSE


# ---------------------------------------------------------------------------- backward
# The backward pass at the same kind of limits, on sampled rows.  The bound is that of
# tests/test_attn_bwd_gpu.py made rigorous for long rows: a binary16 operand (P or dS)
# carries a relative rounding error of at most u = 2^-11 while it is normal, but below
# 2^-14 it is subnormal and its rounding error is absolute, at most 2^-25.  At T = 2^20
# the normalised weights P ~ 1/T are deep in that range.  So each element satisfies
#     |dGPU - oracle| <= 8 (u A + 2^-25 F) + 2^-16 max A,
# A the sum of its terms' magnitudes and F the sum of the other factor's magnitudes
# (s sum |K| for dQ, s sum |Q| for dK, sum |dO| for dV).  The relative Frobenius
# criterion of the other backward tests assumes normal operands and is not applied to
# the long sequence.  A and F are formed from binary32 copies of the inputs, one sampled
# row at a time, and inflated by 1e-3 for their own binary32 rounding.  The long case
# uses T = 2^20: the oracle's host wrapper holds O in float64 (2 GB here), which at the
# predicate's largest T would take 8.6 GB of host memory.

S_NAT = 0.125
U16 = 2.0 ** -11
SUB16 = 2.0 ** -25      # half the spacing of binary16 subnormals


def _bwd_rows_magnitudes(q, k, vT, o, lse, dO, H, G, c, qh, qi, kg, kj, s=S_NAT):
    """(A, F) for dQ at (qh, qi) and for dK, dV at (kg, kj)."""
    grp = H // G
    T = q.shape[1]
    qf = q.astype(np.float32)
    kf = k.astype(np.float32)
    vf = vT.astype(np.float32)
    of = o.astype(np.float32).reshape(T, H, 64)
    gf = dO.astype(np.float32).reshape(T, H, 64)
    L = lse.astype(np.float32)
    a_dq, f_dq = np.zeros((len(qi), 64)), np.zeros((len(qi), 64))
    for r, (h, i) in enumerate(zip(qh, qi)):
        g = h // grp
        P = np.exp2(np.minimum((kf[g][:i + 1] @ qf[h][i]) * c - L[h, i], 60.0))
        dP = gf[i, h] @ vf[g][:, :i + 1]
        D = float(gf[i, h] @ of[i, h])
        a_dq[r] = s * (np.abs(P * (dP - D)) @ np.abs(kf[g][:i + 1]))
        f_dq[r] = s * np.abs(kf[g][:i + 1]).sum(axis=0)
    a_dk, f_dk = np.zeros((len(kj), 64)), np.zeros((len(kj), 64))
    a_dv, f_dv = np.zeros((len(kj), 64)), np.zeros((len(kj), 64))
    for r, (g, j) in enumerate(zip(kg, kj)):
        for h in range(g * grp, (g + 1) * grp):
            P = np.exp2(np.minimum((qf[h][j:] @ kf[g][j]) * c - L[h, j:], 60.0))
            dP = gf[j:, h] @ vf[g][:, j]
            D = np.einsum("te,te->t", gf[j:, h], of[j:, h])
            a_dk[r] += s * (np.abs(P * (dP - D)) @ np.abs(qf[h][j:]))
            f_dk[r] += s * np.abs(qf[h][j:]).sum(axis=0)
            a_dv[r] += P @ np.abs(gf[j:, h])
            f_dv[r] += np.abs(gf[j:, h]).sum(axis=0)
    z = 1 + 1e-3
    return (a_dq * z, f_dq * z), (a_dk * z, f_dk * z), (a_dv * z, f_dv * z)


def _bound_check(name, got, ref, mag, frobenius=True):
    a, f = mag
    assert np.isfinite(got).all(), name
    err = np.abs(got - ref)
    bound = 8.0 * (U16 * a + SUB16 * f) + 2.0 ** -16 * float(a.max())
    ratio = float((err / bound).max())
    print(f"{name}: max |error| / bound {ratio:.3f}")
    assert ratio <= 1.0, (name, float(err.max()), ratio)
    if frobenius:
        rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
        assert rel <= 1e-3, (name, rel)


def _bwd_sampled_check(w, n_q, n_k, seed, frobenius=True):
    q, k, vT = synthetic.make_inputs(w)
    dO = synthetic.make_output_grad(w)
    c = synthetic.scale_c()
    T, H, G = w.T, w.heads, w.kv_heads
    dev = torch.device("cuda:0")
    qd, kd, vd, gd = (torch.from_numpy(x).to(dev) for x in (q, k, vT, dO))
    o, lse = tcg.attention(qd, kd, vd, c)
    assert tcg.last_device_status() == tcg.ATTN_OK
    dq, dk, dvT = tcg.attention_backward(qd, kd, vd, o, lse, gd, c, S_NAT)
    assert tcg.bwd_last_device_status() == tcg.ATTN_OK
    for x in (dq, dk, dvT):
        assert bool(torch.isfinite(x).all().item())
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 63, T - 1] + ([127, 128, T // 2, T - 129] if T > 256 else [])
    qi = np.concatenate([np.array(fixed), rng.integers(0, T, n_q)]).astype(np.int64)
    qh = np.concatenate([np.arange(len(fixed)) * (H - 1) % H, rng.integers(0, H, n_q)]).astype(np.int64)
    kj = np.concatenate([np.array(fixed), rng.integers(0, T, n_k)]).astype(np.int64)
    kg = np.concatenate([np.arange(len(fixed)) * (G - 1) % G, rng.integers(0, G, n_k)]).astype(np.int64)
    o_h, l_h = o.cpu().numpy(), lse.cpu().numpy()
    rq, rk, rv = oracle.attn_bwd_rows(q, k, vT, o_h, l_h, dO, T, H, G, c, S_NAT, qh, qi, kg, kj)
    a_dq, a_dk, a_dv = _bwd_rows_magnitudes(q, k, vT, o_h, l_h, dO, H, G, c, qh, qi, kg, kj)
    qh_d, qi_d = torch.as_tensor(qh, device=dev), torch.as_tensor(qi, device=dev)
    kg_d, kj_d = torch.as_tensor(kg, device=dev), torch.as_tensor(kj, device=dev)
    _bound_check("dQ rows", dq[qh_d, qi_d].double().cpu().numpy(), rq, a_dq, frobenius)
    _bound_check("dK rows", dk[kg_d, kj_d].double().cpu().numpy(), rk, a_dk, frobenius)
    _bound_check("dV rows", dvT[kg_d, :, kj_d].double().cpu().numpy(), rv, a_dv, frobenius)


def test_backward_most_heads_admitted():
    # 65535 query units of one tile; 257 key units, each walking a group of 255 heads
    _bwd_sampled_check(synthetic.custom(64, 65535, 257, seed=6553), n_q=200, n_k=40, seed=21)


def test_backward_long_sequence():
    # P ~ 1/T: binary16 subnormals, so only the rigorous per-element bound applies
    _bwd_sampled_check(synthetic.custom(1 << 20, 4, 1, seed=2020), n_q=12, n_k=6, seed=22,
                       frobenius=False)


@pytest.mark.parametrize("c", [1e-6, 32.0])
def test_backward_degenerate_scales(c):
    from tests.test_attn_bwd_gpu import check, term_magnitudes
    w = synthetic.custom(640, 8, 2, seed=919)
    q, k, vT = synthetic.make_inputs(w)
    dO = synthetic.make_output_grad(w)
    c32 = float(np.float32(c))
    dev = torch.device("cuda:0")
    qd, kd, vd, gd = (torch.from_numpy(x).to(dev) for x in (q, k, vT, dO))
    o, lse = tcg.attention(qd, kd, vd, c32)
    dq, dk, dvT = tcg.attention_backward(qd, kd, vd, o, lse, gd, c32, S_NAT)
    assert tcg.bwd_last_device_status() == tcg.ATTN_OK
    o_h, l_h = o.cpu().numpy(), lse.cpu().numpy()
    rq, rk, rv, _ = oracle.attn_bwd(q, k, vT, o_h, l_h, dO, w.T, 8, 2, c32, S_NAT)
    a_dq, a_dk, a_dv = term_magnitudes(q, k, vT, o_h, l_h, dO, w.T, 8, 2, c32)
    check("dQ", dq.double().cpu().numpy(), rq, a_dq)
    check("dK", dk.double().cpu().numpy(), rk, a_dk)
    check("dV^T", dvT.double().cpu().numpy(), rv, a_dv)
