"""GPU parity of the materialised forward (scores plane, row softmax, P V): the
same definition as the streaming forward, so it is checked against the same
fp64 oracle with the same tolerances (max |dO| <= 4e-3, max |dLSE| <= 1e-3,
base 2), and against the streaming kernel on the same inputs."""
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


def run_materialised(q, k, vT, T, H, G, c, ws_fill=None):
    dev = torch.device("cuda:0")
    qd, kd, vd = (torch.from_numpy(x).to(dev) for x in (q, k, vT))
    o = torch.full((T, H * 64), float("nan"), dtype=torch.float16, device=dev)
    lse = torch.full((H, T), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(tcg.attn_materialised_workspace_bytes(T, H, G), dtype=torch.uint8, device=dev)
    if ws_fill is not None:
        ws.fill_(ws_fill)
    tcg.attn_fwd_materialised(qd, kd, vd, o, lse, T, H, G, c, ws)
    assert tcg.materialised_last_device_status() == tcg.ATTN_OK
    return o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def compare(w):
    q, k, vT = synthetic.make_inputs(w)
    c = synthetic.scale_c()
    o, lse = run_materialised(q, k, vT, w.T, w.heads, w.kv_heads, c)
    o_ref, lse_ref = oracle.attn_fwd(q, k, vT, w.T, w.heads, w.kv_heads, c)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert np.abs(o - o_ref).max() <= TOL_O
    assert np.abs(lse - lse_ref).max() <= TOL_LSE
    return o, lse


@pytest.mark.parametrize("name", ["t128_h4_kv2", "t1024_h12_kv12_mha", "t2048_h16_kv4_peaked"])
def test_workload_every_element(name):
    compare(synthetic.WORKLOADS[name])


@pytest.mark.parametrize("T", [64, 192, 320, 640])
@pytest.mark.parametrize("H,G", [(1, 1), (4, 2), (8, 1)])
def test_shapes_every_element(T, H, G):
    compare(synthetic.custom(T, H, G, seed=T * 31 + H * 7 + G))


def test_outlier_keys():
    compare(synthetic.custom(1152, 8, 2, seed=95, k_outlier_every=97, k_outlier_scale=16.0,
                             v_uniform=True))


def test_agrees_with_streaming_forward():
    w = synthetic.WORKLOADS["t1024_h12_kv12_mha"]
    q, k, vT = synthetic.make_inputs(w)
    c = synthetic.scale_c()
    o_m, lse_m = run_materialised(q, k, vT, w.T, w.heads, w.kv_heads, c)
    dev = torch.device("cuda:0")
    qd, kd, vd = (torch.from_numpy(x).to(dev) for x in (q, k, vT))
    o_s, lse_s = tcg.attention(qd, kd, vd, c)
    assert np.abs(o_m - o_s.cpu().numpy().astype(np.float64)).max() <= 2 * TOL_O
    assert np.abs(lse_m - lse_s.cpu().numpy().astype(np.float64)).max() <= 2 * TOL_LSE


def test_workspace_contents_do_not_matter():
    w = synthetic.custom(448, 4, 2, seed=96)
    q, k, vT = synthetic.make_inputs(w)
    c = synthetic.scale_c()
    a = run_materialised(q, k, vT, w.T, 4, 2, c, ws_fill=0)
    b = run_materialised(q, k, vT, w.T, 4, 2, c, ws_fill=0xFF)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
