"""GPU parity of the backward pass: the CUDA path through the C ABI against the
fp64 CPU oracle, on the same seeded binary16 inputs and on the forward's own
O and LSE (the GPU forward's, handed to both sides).

Tolerance (derived from the arithmetic, as the method states none for the
backward): P and dS are rounded to binary16 before their products, unit
roundoff u = 2^-11; every other step is binary32 (u = 2^-24).  Each gradient
element is a sum of such rounded products, so its error is at most about
u * sum|terms|, and over a whole tensor the rounding errors (of random sign)
give a relative Frobenius error near u.  The tests ask, per output tensor:
  * ||GPU - oracle||_F <= 1e-3 * ||oracle||_F      (about 2u), and
  * max |GPU - oracle| <= 4e-3 * max |oracle|      (about 8u, elementwise).
Small and ragged shapes are compared on every element; the headline-sized
workload, in the launch configuration the benchmark times, on rows the
oracle computes one by one.
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
TOL_MAX = 4e-3
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


def check(name, got, ref):
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    err = got - ref
    fro = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30))
    mx = float(np.abs(err).max() / max(np.abs(ref).max(), 1e-30))
    assert fro <= TOL_FRO, f"{name}: relative Frobenius error {fro:.3e}"
    assert mx <= TOL_MAX, f"{name}: max error / max |ref| = {mx:.3e}"
    return fro, mx


def compare_full(w):
    q, k, vT = synthetic.make_inputs(w)
    dO = synthetic.make_output_grad(w)
    c = synthetic.scale_c()
    T, H, G = w.T, w.heads, w.kv_heads
    o, lse, dq, dk, dvT = run_gpu(q, k, vT, dO, T, H, G, c)
    dq_ref, dk_ref, dvT_ref, _ = oracle.attn_bwd(q, k, vT, o, lse, dO, T, H, G, c, S_NAT)
    return [check("dQ", dq, dq_ref), check("dK", dk, dk_ref), check("dV^T", dvT, dvT_ref)]


@pytest.mark.parametrize("name", ["t128_h4_kv2", "t1024_h12_kv12_mha", "t2048_h16_kv4_peaked"])
def test_workload_every_element(name):
    compare_full(synthetic.WORKLOADS[name])


# ragged tails (T mod 128 = 64), one tile, several; groups 1, 2, 4, 8
@pytest.mark.parametrize("T", [64, 128, 192, 320, 1088])
@pytest.mark.parametrize("H,G", [(1, 1), (4, 2), (8, 2), (8, 1)])
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
    qi = sampled_rows(T, 48, rng)
    qh = rng.integers(0, H, size=qi.shape[0])
    kj = sampled_rows(T, 24, rng)
    kg = rng.integers(0, G, size=kj.shape[0])
    rq, rk, rv = oracle.attn_bwd_rows(q, k, vT, o, lse, dO, T, H, G, c, S_NAT, qh, qi, kg, kj)
    check("dQ rows", dq[qh, qi], rq)
    check("dK rows", dk[kg, kj], rk)
    check("dV rows", dvT[kg, :, kj], rv)
    # properties at full size: every element finite; the first query row sees one key,
    # so P = 1 and O = V there, D = dP and dS = 0: dQ of row 0 vanishes up to rounding
    for x in (dq, dk, dvT):
        assert np.isfinite(x).all()
    assert np.abs(dq[:, 0, :]).max() <= 1e-4 * np.abs(dq).max()
