"""Guard bands around every output buffer, checked after each call.

compute-sanitizer cannot be used on these GPUs, so out-of-bounds stores are
looked for directly: each output (and each workspace the library writes) is
carved out of a larger device allocation whose 4 KiB before and after the
buffer hold a sentinel byte.  After the call the sentinel must be intact, on
both sides.  Shapes are chosen where a stray store is likeliest: ragged last
tiles (T mod 128 = 64, T mod 256 = 192), single-tile problems, and more work
units than a wave.  The result inside the buffer is checked too (finite
everywhere, and the forward against the fp64 oracle), so the test also shows
that every element was written.

Entry points covered: attn_fwd, attn_fwd_host (device workspace and the host
outputs), attn_bwd (dQ, dK, dV^T and its row-term workspace),
attn_fwd_materialised (O, LSE and the score/probability planes) and
attn_qkv_rope (Q, K, V^T).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic
import transformer_causal_gqa_gb300 as tcg
from transformer_causal_gqa_gb300 import build as tcg_build

pytestmark = pytest.mark.gpu

PAD = 4096               # bytes of sentinel before and after each buffer
SENTINEL = 0xA5
SHAPES = [(64, 4, 2), (192, 4, 2), (320, 8, 1), (1088, 4, 2)]


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tcg_build.build()
    return tcg.load_library()


class Guarded:
    """A tensor of `shape` and `dtype` inside a byte buffer with PAD sentinel bytes on
    each side.  PAD keeps the tensor's 256-byte alignment."""

    def __init__(self, shape, dtype, device="cuda", fill=float("nan"), pin=False):
        itemsize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = math.prod(shape) * itemsize
        raw = torch.full((2 * PAD + self.nbytes,), SENTINEL, dtype=torch.uint8,
                         device="cpu" if pin else device)
        if pin:
            raw = raw.pin_memory()
        self.raw = raw
        self.t = raw[PAD:PAD + self.nbytes].view(dtype).view(shape)
        if fill is not None:
            self.t.fill_(fill)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        head = self.raw[:PAD]
        tail = self.raw[PAD + self.nbytes:]
        return bool((head == SENTINEL).all().item()) and bool((tail == SENTINEL).all().item())


def _inputs(T, H, G, seed):
    w = synthetic.custom(T, H, G, seed=seed)
    q, k, vT = synthetic.make_inputs(w)
    return w, (q, k, vT)


@pytest.mark.parametrize("T,H,G", SHAPES)
def test_forward_guard_bands(T, H, G):
    w, (q, k, vT) = _inputs(T, H, G, seed=700 + T + H)
    c = synthetic.scale_c()
    qd, kd, vd = (torch.from_numpy(x).cuda() for x in (q, k, vT))
    o = Guarded((T, H * 64), torch.float16)
    lse = Guarded((H, T), torch.float32)
    tcg.attn_fwd(qd, kd, vd, o.t, lse.t, T, H, G, c)
    assert tcg.last_device_status() == tcg.ATTN_OK
    assert o.intact() and lse.intact()
    o_ref, lse_ref = oracle.attn_fwd(q, k, vT, T, H, G, c)
    assert np.abs(o.t.cpu().numpy().astype(np.float64) - o_ref).max() <= 4e-3
    assert np.abs(lse.t.cpu().numpy().astype(np.float64) - lse_ref).max() <= 1e-3


@pytest.mark.parametrize("T,H,G", SHAPES)
def test_host_entry_guard_bands(T, H, G):
    w, (q, k, vT) = _inputs(T, H, G, seed=710 + T + H)
    c = synthetic.scale_c()
    qh, kh, vh = (torch.from_numpy(x).pin_memory() for x in (q, k, vT))
    o = Guarded((T, H * 64), torch.float16, pin=True)
    lse = Guarded((H, T), torch.float32, pin=True)
    ws = Guarded((tcg.attn_fwd_workspace_bytes(T, H, G),), torch.uint8, fill=0)
    tcg.attn_fwd_host(qh, kh, vh, o.t, lse.t, T, H, G, c, ws.t)
    torch.cuda.synchronize()
    assert o.intact() and lse.intact() and ws.intact()
    o_ref, lse_ref = oracle.attn_fwd(q, k, vT, T, H, G, c)
    assert np.abs(o.t.numpy().astype(np.float64) - o_ref).max() <= 4e-3
    assert np.abs(lse.t.numpy().astype(np.float64) - lse_ref).max() <= 1e-3


@pytest.mark.parametrize("T,H,G", SHAPES)
def test_backward_guard_bands(T, H, G):
    w, (q, k, vT) = _inputs(T, H, G, seed=720 + T + H)
    dO = synthetic.make_output_grad(w)
    c = synthetic.scale_c()
    qd, kd, vd, gd = (torch.from_numpy(x).cuda() for x in (q, k, vT, dO))
    o, lse = tcg.attention(qd, kd, vd, c)
    dq = Guarded((H, T, 64), torch.float32)
    dk = Guarded((G, T, 64), torch.float32)
    dvT = Guarded((G, 64, T), torch.float32)
    ws = Guarded((tcg.attn_bwd_workspace_bytes(T, H, G),), torch.uint8, fill=0)
    tcg.attn_bwd(qd, kd, vd, o, lse, gd, dq.t, dk.t, dvT.t, T, H, G, c, 0.125, ws.t)
    assert tcg.bwd_last_device_status() == tcg.ATTN_OK
    for g in (dq, dk, dvT, ws):
        assert g.intact()
    for g in (dq, dk, dvT):
        assert torch.isfinite(g.t).all().item()


@pytest.mark.parametrize("T,H,G", SHAPES)
def test_materialised_guard_bands(T, H, G):
    w, (q, k, vT) = _inputs(T, H, G, seed=730 + T + H)
    c = synthetic.scale_c()
    qd, kd, vd = (torch.from_numpy(x).cuda() for x in (q, k, vT))
    o = Guarded((T, H * 64), torch.float16)
    lse = Guarded((H, T), torch.float32)
    ws = Guarded((tcg.attn_materialised_workspace_bytes(T, H, G),), torch.uint8, fill=0)
    tcg.attn_fwd_materialised(qd, kd, vd, o.t, lse.t, T, H, G, c, ws.t)
    assert tcg.materialised_last_device_status() == tcg.ATTN_OK
    assert o.intact() and lse.intact() and ws.intact()
    o_ref, lse_ref = oracle.attn_fwd(q, k, vT, T, H, G, c)
    assert np.abs(o.t.cpu().numpy().astype(np.float64) - o_ref).max() <= 4e-3
    assert np.abs(lse.t.cpu().numpy().astype(np.float64) - lse_ref).max() <= 1e-3


@pytest.mark.parametrize("T,width,H,G", [(64, 64, 1, 1), (192, 256, 8, 2), (320, 128, 4, 4),
                                         (1088, 192, 2, 1)])
def test_producer_guard_bands(T, width, H, G):
    x, wm, cs, sn = synthetic.make_producer_inputs(T, width, H, G, seed=740 + T)
    xd, wd, cd, sd = (torch.from_numpy(a).cuda() for a in (x, wm, cs, sn))
    q = Guarded((H, T, 64), torch.float16)
    k = Guarded((G, T, 64), torch.float16)
    vT = Guarded((G, 64, T), torch.float16)
    tcg.attn_qkv_rope(xd, wd, cd, sd, q.t, k.t, vT.t, T, width, H, G)
    assert tcg.qkv_last_device_status() == tcg.ATTN_OK
    for g in (q, k, vT):
        assert g.intact()
        assert torch.isfinite(g.t).all().item()
