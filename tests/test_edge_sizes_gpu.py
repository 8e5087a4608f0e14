"""Edge cases of the forward at the admission limits, and degenerate scales.

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

Tolerances as everywhere: max |dO| <= 4e-3, max |dLSE| <= 1e-3 (base 2).
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
