"""The forward and backward calls inside a CUDA graph.

Both passes are asynchronous, stream-ordered launches with no host
synchronisation after a device's first call, so a caller can capture them into
a CUDA graph (for a decode or training loop that replays a fixed sequence of
launches) and replay it.  Replays must give exactly the results of direct
calls on the same inputs.  The first call on the device is made before the
capture, since it sets up the device's state (a scratch allocation and the
kernels' shared-memory attributes).
"""
import numpy as np
import pytest
import torch

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


def test_forward_and_backward_replayed_from_a_graph():
    w = synthetic.custom(1088, 8, 2, seed=515)
    dev = torch.device("cuda:0")
    q, k, vT = (torch.from_numpy(x).to(dev) for x in synthetic.make_inputs(w))
    dO = torch.from_numpy(synthetic.make_output_grad(w)).to(dev)
    c, s = synthetic.scale_c(), 0.125
    T, H, G = w.T, w.heads, w.kv_heads
    # direct calls (also the first calls on the device: set-up happens here)
    o_ref, l_ref = tcg.attention(q, k, vT, c)
    dq_ref, dk_ref, dv_ref = tcg.attention_backward(q, k, vT, o_ref, l_ref, dO, c, s)
    torch.cuda.synchronize()
    assert tcg.last_device_status() == tcg.ATTN_OK
    assert tcg.bwd_last_device_status() == tcg.ATTN_OK
    # the same sequence captured on a side stream, into preallocated outputs
    o = torch.empty_like(o_ref)
    lse = torch.empty_like(l_ref)
    dq, dk, dv = torch.empty_like(dq_ref), torch.empty_like(dk_ref), torch.empty_like(dv_ref)
    ws = torch.empty(tcg.attn_bwd_workspace_bytes(T, H, G), dtype=torch.uint8, device=dev)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            tcg.attn_fwd(q, k, vT, o, lse, T, H, G, c, side)
            tcg.attn_bwd(q, k, vT, o, lse, dO, dq, dk, dv, T, H, G, c, s, ws, side)
    for _ in range(3):
        for t in (o, lse, dq, dk, dv):
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert tcg.last_device_status() == tcg.ATTN_OK
        assert tcg.bwd_last_device_status() == tcg.ATTN_OK
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
        assert torch.equal(dq, dq_ref) and torch.equal(dk, dk_ref) and torch.equal(dv, dv_ref)
