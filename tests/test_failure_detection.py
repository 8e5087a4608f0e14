"""Failure detection on the GPU without a fault, for every entry point: a wait inside a kernel runs
out (its tile is never loaded), the kernel reports ATTN_ETIMEOUT through the
status word and exits cleanly, and the next launch is correct."""
import time

import numpy as np
import pytest
import torch

import oracle
import synthetic
import transformer_causal_gqa_gb300 as tcg
from transformer_causal_gqa_gb300 import build as tcg_build

pytestmark = pytest.mark.gpu


def test_wait_runs_out_then_recovers():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tcg_build.build()
    lib = tcg.load_library()
    w = synthetic.custom(512, 4, 2, seed=31)
    q, k, vT = synthetic.make_inputs(w)
    c = synthetic.scale_c()
    dev = torch.device("cuda:0")
    qd, kd, vd = (torch.from_numpy(x).to(dev) for x in (q, k, vT))
    o = torch.empty((w.T, w.heads * 64), dtype=torch.float16, device=dev)
    lse = torch.empty((w.heads, w.T), dtype=torch.float32, device=dev)

    assert tcg.last_device_status() == tcg.ATTN_OK
    assert lib.attn_test_inject_stall() == tcg.ATTN_OK
    t0 = time.monotonic()
    tcg.attn_fwd(qd, kd, vd, o, lse, w.T, w.heads, w.kv_heads, c)
    assert tcg.last_device_status() == tcg.ATTN_ETIMEOUT
    assert time.monotonic() - t0 < 10.0         # bounded: a few 1 s waits at most
    assert tcg.last_device_status() == tcg.ATTN_OK  # reading it cleared it

    # the context is usable and the next launch is correct
    tcg.attn_fwd(qd, kd, vd, o, lse, w.T, w.heads, w.kv_heads, c)
    assert tcg.last_device_status() == tcg.ATTN_OK
    o_ref, lse_ref = oracle.attn_fwd(q, k, vT, w.T, w.heads, w.kv_heads, c)
    assert float(np.abs(o.cpu().numpy().astype(np.float64) - o_ref).max()) <= 4e-3
    assert float(np.abs(lse.cpu().numpy().astype(np.float64) - lse_ref).max()) <= 1e-3


def test_backward_wait_runs_out_then_recovers():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tcg_build.build()
    lib = tcg.load_library()
    w = synthetic.custom(512, 8, 2, seed=32)
    q, k, vT = synthetic.make_inputs(w)
    dO = synthetic.make_output_grad(w)
    c = synthetic.scale_c()
    dev = torch.device("cuda:0")
    qd, kd, vd, gd = (torch.from_numpy(x).to(dev) for x in (q, k, vT, dO))
    o, lse = tcg.attention(qd, kd, vd, c)
    assert tcg.last_device_status() == tcg.ATTN_OK
    good = [x.cpu() for x in tcg.attention_backward(qd, kd, vd, o, lse, gd, c, 0.125)]
    assert tcg.bwd_last_device_status() == tcg.ATTN_OK

    assert lib.attn_bwd_test_inject_stall() == tcg.ATTN_OK
    t0 = time.monotonic()
    tcg.attention_backward(qd, kd, vd, o, lse, gd, c, 0.125)
    assert tcg.bwd_last_device_status() == tcg.ATTN_ETIMEOUT
    assert time.monotonic() - t0 < 10.0
    assert tcg.bwd_last_device_status() == tcg.ATTN_OK    # reading it cleared it

    # the context is usable and the next call reproduces the good result bit for bit
    again = [x.cpu() for x in tcg.attention_backward(qd, kd, vd, o, lse, gd, c, 0.125)]
    assert tcg.bwd_last_device_status() == tcg.ATTN_OK
    for a, b in zip(good, again):
        assert torch.equal(a, b)


def test_producer_wait_runs_out_then_recovers():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tcg_build.build()
    lib = tcg.load_library()
    T, width, H, G = 512, 256, 8, 2
    dev = torch.device("cuda:0")
    x, wt, cs, sn = (torch.from_numpy(a).to(dev)
                     for a in synthetic.make_producer_inputs(T, width, H, G, seed=33))
    good = [t.cpu() for t in tcg.qkv_rope(x, wt, cs, sn, H, G)]
    assert tcg.qkv_last_device_status() == tcg.ATTN_OK

    assert lib.attn_qkv_test_inject_stall() == tcg.ATTN_OK
    t0 = time.monotonic()
    tcg.qkv_rope(x, wt, cs, sn, H, G)
    assert tcg.qkv_last_device_status() == tcg.ATTN_ETIMEOUT
    assert time.monotonic() - t0 < 10.0
    assert tcg.qkv_last_device_status() == tcg.ATTN_OK    # reading it cleared it

    # the context is usable and the next call reproduces the good result bit for bit
    again = [t.cpu() for t in tcg.qkv_rope(x, wt, cs, sn, H, G)]
    assert tcg.qkv_last_device_status() == tcg.ATTN_OK
    for a, b in zip(good, again):
        assert torch.equal(a, b)


def test_materialised_wait_runs_out_then_recovers():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tcg_build.build()
    lib = tcg.load_library()
    w = synthetic.custom(512, 4, 2, seed=34)
    q, k, vT = synthetic.make_inputs(w)
    c = synthetic.scale_c()
    dev = torch.device("cuda:0")
    qd, kd, vd = (torch.from_numpy(a).to(dev) for a in (q, k, vT))
    o = torch.empty((w.T, w.heads * 64), dtype=torch.float16, device=dev)
    lse = torch.empty((w.heads, w.T), dtype=torch.float32, device=dev)
    ws = torch.empty(tcg.attn_materialised_workspace_bytes(w.T, w.heads, w.kv_heads),
                     dtype=torch.uint8, device=dev)
    tcg.attn_fwd_materialised(qd, kd, vd, o, lse, w.T, w.heads, w.kv_heads, c, ws)
    good = (o.cpu(), lse.cpu())
    assert tcg.materialised_last_device_status() == tcg.ATTN_OK

    assert lib.attn_materialised_test_inject_stall() == tcg.ATTN_OK
    t0 = time.monotonic()
    tcg.attn_fwd_materialised(qd, kd, vd, o, lse, w.T, w.heads, w.kv_heads, c, ws)
    assert tcg.materialised_last_device_status() == tcg.ATTN_ETIMEOUT
    assert time.monotonic() - t0 < 10.0
    assert tcg.materialised_last_device_status() == tcg.ATTN_OK    # reading it cleared it

    # the context is usable and the next call reproduces the good result bit for bit
    tcg.attn_fwd_materialised(qd, kd, vd, o, lse, w.T, w.heads, w.kv_heads, c, ws)
    assert tcg.materialised_last_device_status() == tcg.ATTN_OK
    assert torch.equal(o.cpu(), good[0]) and torch.equal(lse.cpu(), good[1])
