"""GPU parity of the fused QKV producer against its fp64 oracle.

Tolerance (derived): the product is accumulated in binary32 (relative error
near width * 2^-24 in the worst case, far less in practice) and each output is
rounded once to binary16 (half an ulp, 2^-11 relative).  Elementwise the tests
ask |GPU - oracle| <= 2^-10 |oracle| + 2^-13 max|oracle| over the tensor:
one binary16 ulp plus a floor for outputs near zero, where the binary32
accumulation error of terms of size max|oracle| dominates."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import transformer_causal_gqa_gb300 as tcg
from transformer_causal_gqa_gb300 import build as tcg_build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tcg_build.build()
    return tcg.load_library()


def run(T, width, H, G, seed):
    x, w, c, s = synthetic.make_producer_inputs(T, width, H, G, seed)
    dev = torch.device("cuda:0")
    xd, wd, cd, sd = (torch.from_numpy(a).to(dev) for a in (x, w, c, s))
    q = torch.full((H, T, 64), float("nan"), dtype=torch.float16, device=dev)
    k = torch.full((G, T, 64), float("nan"), dtype=torch.float16, device=dev)
    vT = torch.full((G, 64, T), float("nan"), dtype=torch.float16, device=dev)
    tcg.attn_qkv_rope(xd, wd, cd, sd, q, k, vT, T, width, H, G)
    assert tcg.qkv_last_device_status() == tcg.ATTN_OK
    ref = oracle.qkv_rope(x, w, c, s, T, width, H, G)
    got = (q.cpu().numpy(), k.cpu().numpy(), vT.cpu().numpy())
    for name, g, r in zip(("q", "k", "vT"), got, ref):
        g = g.astype(np.float64)
        assert np.isfinite(g).all(), name
        bound = 2.0 ** -10 * np.abs(r) + 2.0 ** -13 * np.abs(r).max()
        bad = np.abs(g - r) > bound
        assert not bad.any(), f"{name}: {int(bad.sum())} elements out of bound, worst {np.abs(g - r).max():.3e}"
    return got


@pytest.mark.parametrize("T,width,H,G", [
    (64, 64, 1, 1),          # one ragged M tile, one partial N tile (3 heads)
    (128, 128, 4, 2),        # 8 heads: two N tiles
    (192, 256, 8, 2),        # ragged tokens, 12 heads = 3 N tiles
    (320, 512, 4, 4),        # MHA, 12 heads
    (256, 2048, 32, 8),      # the headline's head layout and width
    (1088, 192, 2, 1),       # many M tiles, 4 heads
])
def test_shapes(T, width, H, G):
    run(T, width, H, G, seed=T + width + H)


def test_feeds_the_forward():
    # producer -> streaming forward equals oracle producer -> oracle forward (on the
    # GPU producer's binary16 outputs, so only the forward's tolerance applies)
    T, width, H, G = 384, 256, 8, 2
    q, k, vT = run(T, width, H, G, seed=5)
    c = synthetic.scale_c()
    dev = torch.device("cuda:0")
    o, lse = tcg.attention(*(torch.from_numpy(a).to(dev) for a in (q, k, vT)), c)
    o_ref, lse_ref = oracle.attn_fwd(q, k, vT, T, H, G, c)
    assert np.abs(o.cpu().numpy().astype(np.float64) - o_ref).max() <= 4e-3
    assert np.abs(lse.cpu().numpy().astype(np.float64) - lse_ref).max() <= 1e-3


def test_deterministic():
    a = run(512, 256, 8, 2, seed=9)
    b = run(512, 256, 8, 2, seed=9)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_headline_size_every_element():
    # the benchmark's shape: 8192 tokens, width 2048, 32 query heads over 8 K/V heads
    run(8192, 2048, 32, 8, seed=synthetic.WORKLOADS[synthetic.HEADLINE].seed)
