"""attn_fwd_noalloc through the C ABI: the entry point for callers that cannot
allocate device memory (memory-planned runtimes, fixed device-memory quotas,
loops that cannot take cudaMalloc's implicit synchronisation).  Its scratch,
the kernel's status word, lives in a fixed array inside the library.

Two calls in a row must each match attn_fwd's output within the parity
tolerances (max |dO| <= 4e-3, max |dLSE| <= 1e-3) and report a clean status.
This file is collected last so a failure here cannot hide another test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synthetic
import transformer_causal_gqa_gb300 as tcg
from transformer_causal_gqa_gb300 import build as tcg_build

pytestmark = pytest.mark.gpu

TOL_O = 4e-3
TOL_LSE = 1e-3


def test_noalloc_matches_attn_fwd_twice():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tcg_build.build()
    lib = tcg.load_library()
    dev = torch.device("cuda:0")
    w = synthetic.custom(1088, 8, 2, seed=4242)
    q, k, vT = (torch.from_numpy(x).to(dev) for x in synthetic.make_inputs(w))
    c = synthetic.scale_c()
    T, H, G = w.T, w.heads, w.kv_heads

    o_ref = torch.empty((T, H * 64), dtype=torch.float16, device=dev)
    l_ref = torch.empty((H, T), dtype=torch.float32, device=dev)
    tcg.attn_fwd(q, k, vT, o_ref, l_ref, T, H, G, c)
    assert tcg.last_device_status() == tcg.ATTN_OK

    stream = torch.cuda.current_stream()
    status = torch.full((1,), -7, dtype=torch.int32).pin_memory()
    for _ in range(2):
        o = torch.full((T, H * 64), float("nan"), dtype=torch.float16, device=dev)
        lse = torch.full((H, T), float("nan"), dtype=torch.float32, device=dev)
        vp = ctypes.c_void_p
        rc = lib.attn_fwd_noalloc(vp(q.data_ptr()), vp(k.data_ptr()), vp(vT.data_ptr()),
                                  vp(o.data_ptr()), vp(lse.data_ptr()), T, H, G, c,
                                  vp(status.data_ptr()), vp(stream.cuda_stream))
        assert rc == tcg.ATTN_OK, tcg.status_string(rc)
        stream.synchronize()
        assert int(status[0]) == 0
        d_o = (o.double() - o_ref.double()).abs().max().item()
        d_l = (lse.double() - l_ref.double()).abs().max().item()
        assert d_o <= TOL_O and d_l <= TOL_LSE, (d_o, d_l)
        assert np.isfinite(o.float().cpu().numpy()).all()
