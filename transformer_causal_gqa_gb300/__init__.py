"""GB300 (sm_103a) causal grouped-query attention: the forward pass as a
streaming normalised sum, and its backward pass.

A thin ctypes binding over the C ABI declared in ``include/attn_fwd.h`` and
``include/attn_bwd.h``, ``include/attn_materialised.h`` and ``include/attn_qkv.h``
(``libattn_gb300.so``): it checks tensor dtypes,
devices and contiguity, and passes raw pointers, sizes and the stream handle.
Every step of both passes runs in the library's CUDA kernels; there is no CPU
path.  If the library has not been built, every entry point raises
``RuntimeError``.

Layouts (the page "Realization/Nvidia/SM86/StreamingAttentionSM86.alpha"):
q binary16 [heads][T][64], k binary16 [kv_heads][T][64], vT binary16
[kv_heads][64][T]; forward outputs o binary16 [T][heads*64] and lse binary32
[heads][T] (base-2 log-sum-exp).  Backward: dO binary16 [T][heads*64] (O's
layout); outputs dq binary32 [heads][T][64], dk binary32 [kv_heads][T][64],
dvT binary32 [kv_heads][64][T].
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

HEAD_DIM = 64

ATTN_OK = 0
ATTN_EINVAL = -1
ATTN_EALIGN = -2
ATTN_EOVERLAP = -3
ATTN_ELAUNCH = -4
ATTN_EDEVICE = -5
ATTN_ETIMEOUT = -6

# every symbol the headers under include/ declare
EXPORTED = ("attn_fwd", "attn_fwd_workspace_bytes", "attn_fwd_host",
            "attn_last_device_status", "attn_fwd_noalloc", "attn_test_inject_stall",
            "attn_test_set_split_mode",
            "attn_status_string", "attn_bwd", "attn_bwd_workspace_bytes",
            "attn_bwd_last_device_status", "attn_bwd_test_inject_stall", "attn_fwd_materialised",
            "attn_materialised_workspace_bytes", "attn_materialised_last_device_status",
            "attn_materialised_test_inject_stall",
            "attn_qkv_rope", "attn_qkv_last_device_status", "attn_qkv_test_inject_stall")

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB_PATH


def load_library():
    """Loads libattn_gb300.so (built by ``transformer_causal_gqa_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m transformer_causal_gqa_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, f, vp]
    lib.attn_fwd.restype = i
    lib.attn_fwd_workspace_bytes.argtypes = [i, i, i]
    lib.attn_fwd_workspace_bytes.restype = sz
    lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, f, vp, sz, vp]
    lib.attn_fwd_host.restype = i
    lib.attn_last_device_status.argtypes = [vp]
    lib.attn_last_device_status.restype = i
    lib.attn_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, f, vp, vp]
    lib.attn_fwd_noalloc.restype = i
    lib.attn_test_inject_stall.argtypes = []
    lib.attn_test_inject_stall.restype = i
    lib.attn_test_set_split_mode.argtypes = [i]
    lib.attn_test_set_split_mode.restype = i
    lib.attn_status_string.argtypes = [i]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, f, f, vp, sz, vp]
    lib.attn_bwd.restype = i
    lib.attn_bwd_workspace_bytes.argtypes = [i, i, i]
    lib.attn_bwd_workspace_bytes.restype = sz
    lib.attn_bwd_last_device_status.argtypes = [vp]
    lib.attn_bwd_last_device_status.restype = i
    lib.attn_bwd_test_inject_stall.argtypes = []
    lib.attn_bwd_test_inject_stall.restype = i
    lib.attn_fwd_materialised.argtypes = [vp, vp, vp, vp, vp, i, i, i, f, vp, sz, vp]
    lib.attn_fwd_materialised.restype = i
    lib.attn_materialised_workspace_bytes.argtypes = [i, i, i]
    lib.attn_materialised_workspace_bytes.restype = sz
    lib.attn_materialised_last_device_status.argtypes = [vp]
    lib.attn_materialised_last_device_status.restype = i
    lib.attn_materialised_test_inject_stall.argtypes = []
    lib.attn_materialised_test_inject_stall.restype = i
    lib.attn_qkv_rope.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, vp]
    lib.attn_qkv_rope.restype = i
    lib.attn_qkv_last_device_status.argtypes = [vp]
    lib.attn_qkv_last_device_status.restype = i
    lib.attn_qkv_test_inject_stall.argtypes = []
    lib.attn_qkv_test_inject_stall.restype = i
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def _stream_handle(stream):
    if stream is None:
        import torch
        # torch's current stream as a raw handle, without building a Stream object
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return ctypes.c_void_p(raw(torch.cuda.current_device()))
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(getattr(stream, "cuda_stream", stream))


def _check_tensor(name, t, dtype, shape, device=True):
    # one combined test for the usual case; the separate tests below name the failure
    if (t.dtype is dtype and t.shape == shape and t.is_contiguous()
            and (t.is_cuda if device else t.device.type == "cpu")):
        return
    import torch
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if device and t.device.type != "cuda":
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not device and t.device.type != "cpu":
        raise ValueError(f"{name}: must be a host tensor")
    del torch


def attn_fwd(q, k, vT, o, lse, T: int, heads: int, kv_heads: int, c: float, stream=None) -> None:
    """Forward pass on CUDA tensors, queued on ``stream`` (default: torch's current)."""
    import torch
    _check_tensor("q", q, torch.float16, (heads, T, HEAD_DIM))
    _check_tensor("k", k, torch.float16, (kv_heads, T, HEAD_DIM))
    _check_tensor("vT", vT, torch.float16, (kv_heads, HEAD_DIM, T))
    _check_tensor("o", o, torch.float16, (T, heads * HEAD_DIM))
    _check_tensor("lse", lse, torch.float32, (heads, T))
    rc = load_library().attn_fwd(q.data_ptr(), k.data_ptr(), vT.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), int(T), int(heads), int(kv_heads),
                                 float(c), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")


def attn_fwd_workspace_bytes(T: int, heads: int, kv_heads: int) -> int:
    return int(load_library().attn_fwd_workspace_bytes(int(T), int(heads), int(kv_heads)))


def attn_fwd_host(q, k, vT, o, lse, T: int, heads: int, kv_heads: int, c: float,
                  workspace, stream=None) -> None:
    """Forward pass on host tensors (pinned for asynchronous copies); ``workspace``
    is a CUDA uint8 tensor of at least attn_fwd_workspace_bytes bytes.  Queued on
    ``stream``; synchronise it before reading o and lse."""
    import torch
    _check_tensor("q", q, torch.float16, (heads, T, HEAD_DIM), device=False)
    _check_tensor("k", k, torch.float16, (kv_heads, T, HEAD_DIM), device=False)
    _check_tensor("vT", vT, torch.float16, (kv_heads, HEAD_DIM, T), device=False)
    _check_tensor("o", o, torch.float16, (T, heads * HEAD_DIM), device=False)
    _check_tensor("lse", lse, torch.float32, (heads, T), device=False)
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace: must be a contiguous CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    rc = load_library().attn_fwd_host(q.data_ptr(), k.data_ptr(), vT.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), int(T), int(heads), int(kv_heads),
                                      float(c), workspace.data_ptr(), nbytes,
                                      _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_host")


def attn_fwd_noalloc(q, k, vT, o, lse, T: int, heads: int, kv_heads: int, c: float,
                     status=None, stream=None) -> None:
    """attn_fwd without any device allocation: the kernel's scratch (its status word
    and tile-scheduler counters) lives in a fixed array inside the library.
    ``status``: None, or a 1-element int32 tensor (CUDA, or pinned host memory)
    that receives the word (0 = every kernel wait completed) in stream order.
    Calls that overlap on the GPU share the array."""
    import torch
    _check_tensor("q", q, torch.float16, (heads, T, HEAD_DIM))
    _check_tensor("k", k, torch.float16, (kv_heads, T, HEAD_DIM))
    _check_tensor("vT", vT, torch.float16, (kv_heads, HEAD_DIM, T))
    _check_tensor("o", o, torch.float16, (T, heads * HEAD_DIM))
    _check_tensor("lse", lse, torch.float32, (heads, T))
    if status is not None and (status.dtype != torch.int32 or status.numel() < 1):
        raise TypeError("status: expected an int32 tensor with at least one element")
    rc = load_library().attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), vT.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), int(T), int(heads), int(kv_heads),
                                         float(c), None if status is None else status.data_ptr(),
                                         _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_noalloc")


def set_split_mode(mode: int) -> None:
    """Test hook: -1 lets attn_fwd choose its mode by size, 0 forces the normal mode,
    1 the split mode (short problems' key tiles shared out between the two softmax
    warpgroups of a CTA).  Affects every later forward call in this process."""
    rc = load_library().attn_test_set_split_mode(int(mode))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_test_set_split_mode")


def last_device_status(stream=None) -> int:
    """Synchronises ``stream``; ATTN_OK, or ATTN_ETIMEOUT if a kernel wait gave up."""
    return int(load_library().attn_last_device_status(_stream_handle(stream)))


def attention(q, k, vT, c: float, stream=None):
    """Allocates o and lse with torch and runs attn_fwd; returns (o, lse)."""
    import torch
    heads, T, _ = q.shape
    kv_heads = k.shape[0]
    o = torch.empty((T, heads * HEAD_DIM), dtype=torch.float16, device=q.device)
    lse = torch.empty((heads, T), dtype=torch.float32, device=q.device)
    attn_fwd(q, k, vT, o, lse, T, heads, kv_heads, c, stream)
    return o, lse


def attn_bwd_workspace_bytes(T: int, heads: int, kv_heads: int) -> int:
    return int(load_library().attn_bwd_workspace_bytes(int(T), int(heads), int(kv_heads)))


def attn_bwd(q, k, vT, o, lse, dO, dq, dk, dvT, T: int, heads: int, kv_heads: int, c: float,
             s: float, workspace, stream=None) -> None:
    """Backward pass on CUDA tensors, queued on ``stream`` (default: torch's current).
    o and lse are the forward's outputs for q, k, vT and c; s is the natural score
    scale.  ``workspace`` is a CUDA uint8 tensor of at least attn_bwd_workspace_bytes
    bytes (256-byte aligned, as torch's allocations are)."""
    import torch
    _check_tensor("q", q, torch.float16, (heads, T, HEAD_DIM))
    _check_tensor("k", k, torch.float16, (kv_heads, T, HEAD_DIM))
    _check_tensor("vT", vT, torch.float16, (kv_heads, HEAD_DIM, T))
    _check_tensor("o", o, torch.float16, (T, heads * HEAD_DIM))
    _check_tensor("lse", lse, torch.float32, (heads, T))
    _check_tensor("dO", dO, torch.float16, (T, heads * HEAD_DIM))
    _check_tensor("dq", dq, torch.float32, (heads, T, HEAD_DIM))
    _check_tensor("dk", dk, torch.float32, (kv_heads, T, HEAD_DIM))
    _check_tensor("dvT", dvT, torch.float32, (kv_heads, HEAD_DIM, T))
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace: must be a contiguous CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    rc = load_library().attn_bwd(q.data_ptr(), k.data_ptr(), vT.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), dO.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                 dvT.data_ptr(), int(T), int(heads), int(kv_heads), float(c),
                                 float(s), workspace.data_ptr(), nbytes, _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd")


def bwd_last_device_status(stream=None) -> int:
    """Synchronises ``stream``; ATTN_OK, or ATTN_ETIMEOUT if a backward kernel wait gave up."""
    return int(load_library().attn_bwd_last_device_status(_stream_handle(stream)))


def attention_backward(q, k, vT, o, lse, dO, c: float, s: float, stream=None):
    """Allocates the gradients and the workspace with torch and runs attn_bwd;
    returns (dq, dk, dvT)."""
    import torch
    heads, T, _ = q.shape
    kv_heads = k.shape[0]
    dq = torch.empty((heads, T, HEAD_DIM), dtype=torch.float32, device=q.device)
    dk = torch.empty((kv_heads, T, HEAD_DIM), dtype=torch.float32, device=q.device)
    dvT = torch.empty((kv_heads, HEAD_DIM, T), dtype=torch.float32, device=q.device)
    ws = torch.empty(attn_bwd_workspace_bytes(T, heads, kv_heads), dtype=torch.uint8,
                     device=q.device)
    attn_bwd(q, k, vT, o, lse, dO, dq, dk, dvT, T, heads, kv_heads, c, s, ws, stream)
    return dq, dk, dvT


def attn_materialised_workspace_bytes(T: int, heads: int, kv_heads: int) -> int:
    return int(load_library().attn_materialised_workspace_bytes(int(T), int(heads), int(kv_heads)))


def attn_fwd_materialised(q, k, vT, o, lse, T: int, heads: int, kv_heads: int, c: float,
                          workspace, stream=None) -> None:
    """The forward through materialised scores and probability planes (the design the
    streaming kernel replaces), on CUDA tensors; ``workspace`` is a CUDA uint8 tensor of
    at least attn_materialised_workspace_bytes bytes."""
    import torch
    _check_tensor("q", q, torch.float16, (heads, T, HEAD_DIM))
    _check_tensor("k", k, torch.float16, (kv_heads, T, HEAD_DIM))
    _check_tensor("vT", vT, torch.float16, (kv_heads, HEAD_DIM, T))
    _check_tensor("o", o, torch.float16, (T, heads * HEAD_DIM))
    _check_tensor("lse", lse, torch.float32, (heads, T))
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace: must be a contiguous CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    rc = load_library().attn_fwd_materialised(q.data_ptr(), k.data_ptr(), vT.data_ptr(),
                                              o.data_ptr(), lse.data_ptr(), int(T), int(heads),
                                              int(kv_heads), float(c), workspace.data_ptr(),
                                              nbytes, _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_materialised")


def materialised_last_device_status(stream=None) -> int:
    """Synchronises ``stream``; ATTN_OK, or ATTN_ETIMEOUT if a materialised-path wait gave up."""
    return int(load_library().attn_materialised_last_device_status(_stream_handle(stream)))


def attn_qkv_rope(x, w, cosines, sines, q, k, vT, T: int, width: int, heads: int,
                  kv_heads: int, stream=None) -> None:
    """The fused QKV producer on CUDA tensors: x binary16 [T][width], w binary16
    [(heads + 2 kv_heads) * 64][width], cosines/sines binary32 [T][32]; writes
    q [heads][T][64], k [kv_heads][T][64], vT [kv_heads][64][T] (binary16)."""
    import torch
    n_out = (heads + 2 * kv_heads) * HEAD_DIM
    _check_tensor("x", x, torch.float16, (T, width))
    _check_tensor("w", w, torch.float16, (n_out, width))
    _check_tensor("cosines", cosines, torch.float32, (T, HEAD_DIM // 2))
    _check_tensor("sines", sines, torch.float32, (T, HEAD_DIM // 2))
    _check_tensor("q", q, torch.float16, (heads, T, HEAD_DIM))
    _check_tensor("k", k, torch.float16, (kv_heads, T, HEAD_DIM))
    _check_tensor("vT", vT, torch.float16, (kv_heads, HEAD_DIM, T))
    rc = load_library().attn_qkv_rope(x.data_ptr(), w.data_ptr(), cosines.data_ptr(),
                                      sines.data_ptr(), q.data_ptr(), k.data_ptr(), vT.data_ptr(),
                                      int(T), int(width), int(heads), int(kv_heads),
                                      _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_qkv_rope")


def qkv_last_device_status(stream=None) -> int:
    """Synchronises ``stream``; ATTN_OK, or ATTN_ETIMEOUT if a producer wait gave up."""
    return int(load_library().attn_qkv_last_device_status(_stream_handle(stream)))


def qkv_rope(x, w, cosines, sines, heads: int, kv_heads: int, stream=None):
    """Allocates the outputs with torch and runs attn_qkv_rope; returns (q, k, vT)."""
    import torch
    T, width = x.shape
    q = torch.empty((heads, T, HEAD_DIM), dtype=torch.float16, device=x.device)
    k = torch.empty((kv_heads, T, HEAD_DIM), dtype=torch.float16, device=x.device)
    vT = torch.empty((kv_heads, HEAD_DIM, T), dtype=torch.float16, device=x.device)
    attn_qkv_rope(x, w, cosines, sines, q, k, vT, T, width, heads, kv_heads, stream)
    return q, k, vT
