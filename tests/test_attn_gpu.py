"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Tolerances (written here, from the headline statement of the method's
accuracy): max |dO| <= 4e-3 and max |dLSE| <= 1e-3 (base 2), elementwise, on
the same seeded binary16 inputs.  Every workload of the benchmark list is
compared on every element, the two largest in the launch configuration the
benchmark times (the oracle needs about 5 s and 40 s of 16 host cores for
them); a faster check of those two on sampled rows the oracle computes one by
one, plus properties that hold at any size, runs first.  Small and ragged
shapes are compared on every element.
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


@pytest.fixture
def mode(request):
    """Forces the forward kernel's mode (0 normal, 1 split) for one test."""
    tcg.set_split_mode(request.param)
    yield request.param
    tcg.set_split_mode(-1)


def run_gpu(q, k, vT, T, H, G, c, stream=None):
    dev = torch.device("cuda:0")
    qd, kd, vd = (torch.from_numpy(x).to(dev) for x in (q, k, vT))
    o = torch.full((T, H * 64), float("nan"), dtype=torch.float16, device=dev)
    lse = torch.full((H, T), float("nan"), dtype=torch.float32, device=dev)
    tcg.attn_fwd(qd, kd, vd, o, lse, T, H, G, c, stream)
    assert tcg.last_device_status(stream) == tcg.ATTN_OK
    return o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def compare_full(w):
    q, k, vT = synthetic.make_inputs(w)
    c = synthetic.scale_c()
    o, lse = run_gpu(q, k, vT, w.T, w.heads, w.kv_heads, c)
    o_ref, lse_ref = oracle.attn_fwd(q, k, vT, w.T, w.heads, w.kv_heads, c)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    d_o = float(np.abs(o - o_ref).max())
    d_l = float(np.abs(lse - lse_ref).max())
    assert d_o <= TOL_O, f"max |dO| = {d_o}"
    assert d_l <= TOL_LSE, f"max |dLSE| = {d_l}"
    return d_o, d_l


@pytest.mark.parametrize("name", ["t128_h4_kv2", "t1024_h12_kv12_mha", "t2048_h16_kv4_peaked"])
def test_workload_every_element(name):
    compare_full(synthetic.WORKLOADS[name])


# ragged tails: T mod 256 in {64, 128, 192, 0}; groups 1, 2, 4, 8; both modes of the
# kernel (short problems run split by default: the two subtiles share out a 128-row
# unit's key tiles and merge; the normal mode gives each subtile its own 128 rows)
@pytest.mark.parametrize("mode", [0, 1], indirect=True)
@pytest.mark.parametrize("T", [64, 192, 320, 384, 448, 640, 1088])
@pytest.mark.parametrize("H,G", [(1, 1), (4, 2), (8, 2), (8, 1), (6, 3), (5, 1)])
def test_shapes_every_element(mode, T, H, G):
    compare_full(synthetic.custom(T, H, G, seed=T * 100 + H * 10 + G))


@pytest.mark.parametrize("mode", [0, 1], indirect=True)
@pytest.mark.parametrize("name", ["t128_h4_kv2", "t1024_h12_kv12_mha", "t2048_h16_kv4_peaked"])
def test_small_workloads_both_modes(mode, name):
    compare_full(synthetic.WORKLOADS[name])


def test_outlier_keys_small():
    compare_full(synthetic.custom(1152, 16, 2, seed=77, k_outlier_every=97,
                                  k_outlier_scale=16.0, v_uniform=True))


def test_peaked_many_heads():
    compare_full(synthetic.custom(768, 32, 4, seed=78, qk_scale=4.0))


def test_more_units_than_sms():
    # 160 heads x 2 row blocks = 320 work units: each CTA takes several
    compare_full(synthetic.custom(512, 160, 20, seed=79))


def sample_rows(T, H, n_random, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 63, 64, 127, 128, 129, 255, 256, T // 2, T - 129, T - 128, T - 2, T - 1]
    rows = np.concatenate([np.array(fixed), rng.integers(0, T, n_random)])
    heads = np.concatenate([np.arange(len(fixed)) % H, rng.integers(0, H, n_random)])
    extra_h = np.arange(H)                      # every head, its last row
    return (np.concatenate([heads, extra_h]),
            np.concatenate([rows, np.full(H, T - 1)]))


@pytest.mark.parametrize("name,n_random", [("t8192_h32_kv8", 600), ("t16384_h64_kv8_outliers", 300)])
def test_full_size_sampled_rows(name, n_random):
    w = synthetic.WORKLOADS[name]
    q, k, vT = synthetic.make_inputs(w)
    c = synthetic.scale_c()
    o, lse = run_gpu(q, k, vT, w.T, w.heads, w.kv_heads, c)
    # properties at every element: finite, LSE >= the row's first score's bound
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    vmax = float(np.abs(vT.astype(np.float32)).max())
    assert float(np.abs(o).max()) <= vmax * (1 + 1e-3)   # a convex combination of V rows
    hs, rs = sample_rows(w.T, w.heads, n_random, seed=w.seed)
    o_ref, lse_ref = oracle.attn_fwd_rows(q, k, vT, w.T, w.heads, w.kv_heads, c, hs, rs)
    got_o = np.stack([o[r, h * 64:(h + 1) * 64] for h, r in zip(hs, rs)])
    got_l = lse[hs, rs]
    d_o = float(np.abs(got_o - o_ref).max())
    d_l = float(np.abs(got_l - lse_ref).max())
    assert d_o <= TOL_O, f"max |dO| = {d_o}"
    assert d_l <= TOL_LSE, f"max |dLSE| = {d_l}"


@pytest.mark.parametrize("name", ["t8192_h32_kv8", "t16384_h64_kv8_outliers"])
def test_full_size_every_element(name):
    d_o, d_l = compare_full(synthetic.WORKLOADS[name])
    print(f"{name}: max|dO| = {d_o:.3e}, max|dLSE| = {d_l:.3e}")


def test_deterministic_and_stream():
    w = synthetic.custom(1024, 8, 2, seed=80)
    q, k, vT = synthetic.make_inputs(w)
    c = synthetic.scale_c()
    s = torch.cuda.Stream()
    a = run_gpu(q, k, vT, w.T, w.heads, w.kv_heads, c)
    with torch.cuda.stream(s):
        b = run_gpu(q, k, vT, w.T, w.heads, w.kv_heads, c, stream=s)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# the host entry cuts the problem into up to four K/V-head chunks: one chunk,
# one head per chunk, uneven chunks (6 -> 1, 2, 1, 2; 12 -> 3 each) and MHA
@pytest.mark.parametrize("H,G", [(8, 4), (4, 1), (12, 6), (24, 12), (16, 16)])
def test_host_entry_matches_device_entry(H, G):
    w = synthetic.custom(640, H, G, seed=81 + H)
    q, k, vT = synthetic.make_inputs(w)
    c = synthetic.scale_c()
    o_dev, lse_dev = run_gpu(q, k, vT, w.T, w.heads, w.kv_heads, c)
    qh, kh, vh = (torch.from_numpy(x).pin_memory() for x in (q, k, vT))
    oh = torch.empty((w.T, w.heads * 64), dtype=torch.float16).pin_memory()
    lh = torch.empty((w.heads, w.T), dtype=torch.float32).pin_memory()
    ws = torch.empty(tcg.attn_fwd_workspace_bytes(w.T, w.heads, w.kv_heads),
                     dtype=torch.uint8, device="cuda")
    tcg.attn_fwd_host(qh, kh, vh, oh, lh, w.T, w.heads, w.kv_heads, c, ws)
    torch.cuda.synchronize()
    assert np.array_equal(oh.numpy().astype(np.float64), o_dev)
    assert np.array_equal(lh.numpy().astype(np.float64), lse_dev)


def test_rejections_on_device():
    dev = torch.device("cuda:0")
    q = torch.zeros(4, 128, 64, dtype=torch.float16, device=dev)
    k = torch.zeros(2, 128, 64, dtype=torch.float16, device=dev)
    vT = torch.zeros(2, 64, 128, dtype=torch.float16, device=dev)
    lse = torch.zeros(4, 128, dtype=torch.float32, device=dev)
    # o aliasing q is refused before anything is queued
    with pytest.raises(tcg.AttnError) as e:
        tcg.attn_fwd(q, k, vT, q.view(128, 256), lse, 128, 4, 2, 0.18)
    assert e.value.status == tcg.ATTN_EOVERLAP
    assert tcg.last_device_status() == tcg.ATTN_OK


def test_binding_rejects_bad_cuda_tensors():
    """The binding's checks on CUDA tensors: each bad argument raises its own error
    before the library is called, so the output is left as it was."""
    dev = torch.device("cuda:0")
    T, H, G = 128, 4, 2
    q = torch.zeros(H, T, 64, dtype=torch.float16, device=dev)
    k = torch.zeros(G, T, 64, dtype=torch.float16, device=dev)
    vT = torch.zeros(G, 64, T, dtype=torch.float16, device=dev)
    lse = torch.zeros(H, T, dtype=torch.float32, device=dev)
    sentinel = torch.full((T, H * 64), 7.0, dtype=torch.float16, device=dev)
    o = sentinel.clone()
    cases = [
        ((q.float(), k, vT, o, lse), TypeError),                                # dtype
        ((q, k[:, :64], vT, o, lse), ValueError),                               # shape
        ((q, k, vT.clone(), o, lse), None),                                     # valid: accepted
        ((q, k, torch.zeros(G, T, 64, dtype=torch.float16, device=dev).transpose(1, 2), o, lse),
         ValueError),                                                           # not contiguous
        ((q, k, vT, o, lse.cpu()), ValueError),                                 # not on the device
    ]
    for args, err in cases:
        if err is None:
            tcg.attn_fwd(*args, T, H, G, 0.18)
            torch.cuda.synchronize()
            o.copy_(sentinel)
            continue
        with pytest.raises(err):
            tcg.attn_fwd(*args, T, H, G, 0.18)
        torch.cuda.synchronize()
        assert torch.equal(o, sentinel)
    assert tcg.last_device_status() == tcg.ATTN_OK


def compare_arrays(q, k, vT, T, H, G):
    c = synthetic.scale_c()
    o, lse = run_gpu(q, k, vT, T, H, G, c)
    o_ref, lse_ref = oracle.attn_fwd(q, k, vT, T, H, G, c)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    d_o = float(np.abs(o - o_ref).max())
    d_l = float(np.abs(lse - lse_ref).max())
    assert d_o <= TOL_O, f"max |dO| = {d_o}"
    assert d_l <= TOL_LSE, f"max |dLSE| = {d_l}"


@pytest.mark.parametrize("mode", [0, 1], indirect=True)
@pytest.mark.parametrize("jump", [6.0, 12.0, 14.0, 16.0, 40.0, 120.0, 200.0])
def test_late_score_jump(mode, jump):
    """A key late in the sequence whose score exceeds every earlier one by `jump`
    (base-2 units) for every query row after it.  Each row's weight for that key
    is 2^(jump + d) against its reference maximum, d >= 0 the row's own gap to
    the largest earlier score.  Below the slack of 8 a row keeps its reference
    (weights up to 2^8); above it the reference moves to the tile's maximum and O
    and l are scaled by 2^-jump or less (to zero in binary32 for the largest
    jumps).  Jumps of 14 and 16 put the rows of one warp on both sides of the
    line where a weight against the old reference would pass the largest
    binary16.  Every case must match the exact definition."""
    T, H, G = 1024, 2, 1
    w = synthetic.custom(T, H, G, seed=1234)
    q, k, vT = synthetic.make_inputs(w)
    c = synthetic.scale_c()
    j = 700                                        # key tile 5, row 60 of that tile
    u = np.zeros(64, dtype=np.float64)
    u[0] = 1.0
    q = q.astype(np.float64)
    q[:, :, 0] = 4.0                               # every query row: component 4 along u
    # score of key j for every row: 4 * k0 * scale/ln2 = jump + (largest earlier score)
    base_max = float(np.max(q[:, :, :] @ k[0].astype(np.float64).T * c))
    k = k.astype(np.float64)
    k[0, j, :] = 0.0
    k[0, j, 0] = (jump + base_max) / (4.0 * c)
    q16 = q.astype(np.float16)
    k16 = k.astype(np.float16)
    assert np.isfinite(k16).all()
    compare_arrays(q16, k16, vT, T, H, G)


@pytest.mark.parametrize("mode", [0, 1], indirect=True)
@pytest.mark.parametrize("rise", [1.0, 3.0, 9.0])
def test_tile_wide_rise(mode, rise):
    """Every key of one tile scores `rise` above the largest earlier score, for
    every query row after the tile: 128 equal weights of at least 2^rise, tied at
    the tile's maximum.  With rises 1 and 3 most rows keep their reference (row
    sums of 256 to over 1000 against it), with rise 9 every row moves it.  The
    diagonal tile's mask (query rows inside the tile) is covered too."""
    T, H, G = 1024, 4, 2
    w = synthetic.custom(T, H, G, seed=4321)
    q, k, vT = synthetic.make_inputs(w)
    c = synthetic.scale_c()
    q = q.astype(np.float64)
    q[:, :, 0] = 4.0
    base_max = float(max(np.max(q[h] @ k[h // (H // G)].astype(np.float64).T * c) for h in range(H)))
    k = k.astype(np.float64)
    for g in range(G):
        k[g, 640:768, :] = 0.0                      # key tile 5
        k[g, 640:768, 0] = (rise + base_max) / (4.0 * c)
    q16 = q.astype(np.float16)
    k16 = k.astype(np.float16)
    assert np.isfinite(k16).all()
    compare_arrays(q16, k16, vT, T, H, G)
