"""GPU parity of the backward pass: the CUDA path through the C ABI against the
fp64 CPU oracle, on the same seeded binary16 inputs and on the forward's own
O and LSE (the GPU forward's, handed to both sides).

Tolerance (derived from the arithmetic, as the method states none for the
backward).  P and dS are rounded to binary16 before their products, unit
roundoff u = 2^-11; every other step is binary32 (u32 = 2^-24).  Each gradient
element is a sum of products of such rounded operands:
    dQ[i,e]  = s sum_j  dS[i,j] K[j,e]
    dK[j,e]  = s sum_(h,i) dS[i,j] Q[i,e]      (i over the group's query heads)
    dV[j,e]  =   sum_(h,i) P[i,j] dO[i,e]
so its rounding error is at most u * A with A the sum of the terms' magnitudes
(s sum_j |dS[i,j]| |K[j,e]| and so on), plus binary32 effects (the binary32
sums over up to 16384 terms, the binary32 exp2 and row terms) that stay below
u * A by orders of magnitude.  The tests therefore ask, element by element,
    |GPU - oracle| <= 8 u A + 2^-16 max A,
where the floor covers elements whose terms cancel exactly in the oracle (the
first query row, where dS is zero) but only to binary32 rounding on the GPU.
The magnitudes A are formed here in float64 from the same inputs, O and LSE.
Per output tensor the tests also ask ||GPU - oracle||_F <= 1e-3 ||oracle||_F
(about 2u).  Small and ragged shapes are compared on every element; the two
largest workloads, in the launch configuration the benchmark times, on 512
query rows and 256 key rows the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import transformer_causal_gqa_gb300 as tcg
from transformer_causal_gqa_gb300 import build as tcg_build

pytestmark = pytest.mark.gpu

TOL_FRO = 1e-3
U16 = 2.0 ** -11       # binary16 unit roundoff
S_NAT = 0.125          # natural score scale for head width 64


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tcg_build.build()
    return tcg.load_library()


def run_gpu(q, k, vT, dO, T, H, G, c, s=S_NAT, ws_fill=None):
    """Forward then backward on cuda:0; returns host copies (o fp16, lse f32,
    dq, dk, dvT f32)."""
    dev = torch.device("cuda:0")
    qd, kd, vd, gd = (torch.from_numpy(x).to(dev) for x in (q, k, vT, dO))
    o = torch.empty((T, H * 64), dtype=torch.float16, device=dev)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    tcg.attn_fwd(qd, kd, vd, o, lse, T, H, G, c)
    assert tcg.last_device_status() == tcg.ATTN_OK
    dq = torch.full((H, T, 64), float("nan"), dtype=torch.float32, device=dev)
    dk = torch.full((G, T, 64), float("nan"), dtype=torch.float32, device=dev)
    dvT = torch.full((G, 64, T), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(tcg.attn_bwd_workspace_bytes(T, H, G), dtype=torch.uint8, device=dev)
    if ws_fill is not None:
        ws.fill_(ws_fill)
    tcg.attn_bwd(qd, kd, vd, o, lse, gd, dq, dk, dvT, T, H, G, c, s, ws)
    assert tcg.bwd_last_device_status() == tcg.ATTN_OK
    return (o.cpu().numpy(), lse.cpu().numpy(), dq.cpu().numpy().astype(np.float64),
            dk.cpu().numpy().astype(np.float64), dvT.cpu().numpy().astype(np.float64))


def check(name, got, ref, mag):
    """got, ref: the gradient elements; mag: the sum of their terms' magnitudes."""
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    err = got - ref
    fro = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30))
    assert fro <= TOL_FRO, f"{name}: relative Frobenius error {fro:.3e}"
    bound = 8.0 * U16 * mag + 2.0 ** -16 * float(mag.max())
    ratio = np.abs(err) / bound
    worst = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
    print(f"{name}: rel. Frobenius {fro:.2e}, max |error| / bound {float(ratio.max()):.3f}, "
          f"max |error| / (u A) {float((np.abs(err) / (U16 * np.maximum(mag, 1e-30))).max()):.3f}")
    assert float(ratio.max()) <= 1.0, (
        f"{name}: |error| {abs(float(err[worst])):.3e} exceeds its bound {float(bound[worst]):.3e} "
        f"at {worst} (ref {float(ref[worst]):.3e}, term magnitude {float(mag[worst]):.3e})")
    return fro, float(ratio.max())


def _head_views(q, k, vT, o, dO, H, G):
    f = lambda a: a.astype(np.float64)
    T = q.shape[1]
    o3 = f(o).reshape(T, H, 64)
    g3 = f(dO).reshape(T, H, 64)
    D = (o3 * g3).sum(axis=2)                        # [T][H]: the row terms
    return f(q), f(k), f(vT), g3, D


def term_magnitudes(q, k, vT, o, lse, dO, T, H, G, c, s=S_NAT):
    """Every element's sum of term magnitudes (dQ [H][T][64], dK [G][T][64],
    dV^T [G][64][T]), float64."""
    qf, kf, vf, g3, D = _head_views(q, k, vT, o, dO, H, G)
    grp = H // G
    tri = np.tril(np.ones((T, T), dtype=bool))
    a_dq = np.zeros((H, T, 64))
    a_dk = np.zeros((G, T, 64))
    a_dv = np.zeros((G, T, 64))
    for h in range(H):
        g = h // grp
        t = (qf[h] @ kf[g].T) * c - lse[h].astype(np.float64)[:, None]
        P = np.where(tri, np.exp2(np.minimum(t, 60.0)), 0.0)
        dP = g3[:, h, :] @ vf[g]
        dS = np.abs(P * (dP - D[:, h][:, None]))
        a_dq[h] = s * (dS @ np.abs(kf[g]))
        a_dk[g] += s * (dS.T @ np.abs(qf[h]))
        a_dv[g] += P.T @ np.abs(g3[:, h, :])
    return a_dq, a_dk, np.ascontiguousarray(a_dv.transpose(0, 2, 1))


def term_magnitudes_rows(q, k, vT, o, lse, dO, T, H, G, c, qh, qi, kg, kj, s=S_NAT):
    """The same for sampled rows: dQ at (qh[r], qi[r]); dK and dV at (kg[r], kj[r])."""
    qf, kf, vf, g3, D = _head_views(q, k, vT, o, dO, H, G)
    grp = H // G
    L = lse.astype(np.float64)
    a_dq = np.zeros((len(qi), 64))
    for r, (h, i) in enumerate(zip(qh, qi)):
        g = h // grp
        t = (kf[g][:i + 1] @ qf[h][i]) * c - L[h, i]
        P = np.exp2(np.minimum(t, 60.0))
        dP = vf[g][:, :i + 1].T @ g3[i, h, :]
        a_dq[r] = s * (np.abs(P * (dP - D[i, h])) @ np.abs(kf[g][:i + 1]))
    a_dk = np.zeros((len(kj), 64))
    a_dv = np.zeros((len(kj), 64))
    for r, (g, j) in enumerate(zip(kg, kj)):
        for h in range(g * grp, (g + 1) * grp):
            t = (qf[h][j:] @ kf[g][j]) * c - L[h, j:]
            P = np.exp2(np.minimum(t, 60.0))
            dP = g3[j:, h, :] @ vf[g][:, j]
            a_dk[r] += s * (np.abs(P * (dP - D[j:, h])) @ np.abs(qf[h][j:]))
            a_dv[r] += P @ np.abs(g3[j:, h, :])
    return a_dq, a_dk, a_dv


def compare_full(w):
    q, k, vT = synthetic.make_inputs(w)
    dO = synthetic.make_output_grad(w)
    c = synthetic.scale_c()
    T, H, G = w.T, w.heads, w.kv_heads
    o, lse, dq, dk, dvT = run_gpu(q, k, vT, dO, T, H, G, c)
    dq_ref, dk_ref, dvT_ref, _ = oracle.attn_bwd(q, k, vT, o, lse, dO, T, H, G, c, S_NAT)
    a_dq, a_dk, a_dv = term_magnitudes(q, k, vT, o, lse, dO, T, H, G, c)
    return [check("dQ", dq, dq_ref, a_dq), check("dK", dk, dk_ref, a_dk),
            check("dV^T", dvT, dvT_ref, a_dv)]


@pytest.mark.parametrize("name", ["t128_h4_kv2", "t1024_h12_kv12_mha", "t2048_h16_kv4_peaked"])
def test_workload_every_element(name):
    compare_full(synthetic.WORKLOADS[name])


# ragged tails (T mod 128 = 64), one tile, several; groups 1, 2, 4, 8, and odd ones
# (6 over 3; 5 over 1, whose short problems share each key unit's steps five ways)
@pytest.mark.parametrize("T", [64, 128, 192, 320, 1088])
@pytest.mark.parametrize("H,G", [(1, 1), (4, 2), (8, 2), (8, 1), (6, 3), (5, 1)])
def test_shapes_every_element(T, H, G):
    compare_full(synthetic.custom(T, H, G, seed=T * 100 + H * 10 + G + 7))


def test_outlier_keys_small():
    compare_full(synthetic.custom(1152, 16, 2, seed=91, k_outlier_every=97,
                                  k_outlier_scale=16.0, v_uniform=True))


def test_more_units_than_sms():
    # 160 heads x 4 query tiles = 640 query units, 20 x 4 = 80 key units of 32 steps each
    compare_full(synthetic.custom(512, 160, 20, seed=92))


def test_workspace_contents_do_not_matter():
    w = synthetic.custom(384, 8, 2, seed=93)
    q, k, vT = synthetic.make_inputs(w)
    dO = synthetic.make_output_grad(w)
    c = synthetic.scale_c()
    a = run_gpu(q, k, vT, dO, w.T, 8, 2, c, ws_fill=0)
    b = run_gpu(q, k, vT, dO, w.T, 8, 2, c, ws_fill=0xFF)      # NaN binary16 / binary32 patterns
    for x, y in zip(a[2:], b[2:]):
        assert np.array_equal(x, y)


def test_deterministic():
    w = synthetic.custom(1024, 16, 4, seed=94)
    q, k, vT = synthetic.make_inputs(w)
    dO = synthetic.make_output_grad(w)
    c = synthetic.scale_c()
    a = run_gpu(q, k, vT, dO, w.T, 16, 4, c)
    b = run_gpu(q, k, vT, dO, w.T, 16, 4, c)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def sampled_rows(T, n, rng):
    fixed = [0, 1, 63, 64, 127, 128, T // 2, T - 129, T - 128, T - 65, T - 64, T - 1]
    extra = rng.integers(0, T, size=max(0, n - len(fixed)))
    return np.concatenate([np.array(fixed), extra]).astype(np.int64)


@pytest.mark.parametrize("name", [synthetic.HEADLINE, "t16384_h64_kv8_outliers"])
def test_full_size_sampled_rows(name):
    w = synthetic.WORKLOADS[name]
    q, k, vT = synthetic.make_inputs(w)
    dO = synthetic.make_output_grad(w)
    c = synthetic.scale_c()
    T, H, G = w.T, w.heads, w.kv_heads
    o, lse, dq, dk, dvT = run_gpu(q, k, vT, dO, T, H, G, c)
    rng = np.random.default_rng(5)
    qi = sampled_rows(T, 512, rng)
    qh = rng.integers(0, H, size=qi.shape[0])
    kj = sampled_rows(T, 256, rng)
    kg = rng.integers(0, G, size=kj.shape[0])
    rq, rk, rv = oracle.attn_bwd_rows(q, k, vT, o, lse, dO, T, H, G, c, S_NAT, qh, qi, kg, kj)
    a_dq, a_dk, a_dv = term_magnitudes_rows(q, k, vT, o, lse, dO, T, H, G, c, qh, qi, kg, kj)
    check("dQ rows", dq[qh, qi], rq, a_dq)
    check("dK rows", dk[kg, kj], rk, a_dk)
    check("dV rows", dvT[kg, :, kj], rv, a_dv)
    # properties at full size: every element finite; the first query row sees one key,
    # so P = 1 and O = V there, D = dP and dS = 0: dQ of row 0 vanishes up to rounding
    for x in (dq, dk, dvT):
        assert np.isfinite(x).all()
    assert np.abs(dq[:, 0, :]).max() <= 1e-4 * np.abs(dq).max()
