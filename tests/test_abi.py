"""The C-ABI library on the host (no GPU): it builds, loads, exports every
symbol include/attn_fwd.h declares, and rejects bad arguments before touching
the device."""
import ctypes
import os
import re

import pytest

import transformer_causal_gqa_gb300 as tcg
from transformer_causal_gqa_gb300 import build as tcg_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    tcg_build.build()
    return tcg.load_library()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(attn_\w+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names == set(tcg.EXPORTED)
    for n in names:
        assert getattr(lib, n) is not None


def test_status_strings(lib):
    for code in range(-6, 1):
        assert tcg.status_string(code) != "unknown status"
    assert tcg.status_string(7) == "unknown status"


def call(lib, q=0x1000, k=0x100000, v=0x200000, o=0x300000, l=0x400000, T=128, H=4, G=2, c=0.18):
    vp = ctypes.c_void_p
    return lib.attn_fwd(vp(q), vp(k), vp(v), vp(o), vp(l), T, H, G, c, None)


@pytest.mark.parametrize("T,H,G,c", [
    (0, 4, 2, 0.18), (100, 4, 2, 0.18), (-64, 4, 2, 0.18),   # T > 0, T % 64 == 0
    (128, 0, 1, 0.18), (128, 4, 0, 0.18), (128, 4, 3, 0.18),  # heads % kv_heads == 0
    (128, 65536, 1, 0.18),                                    # heads <= 65535
    (2 ** 24, 1, 1, 0.18),                                     # heads*64*T*4 <= 2^32-1
    (128, 4, 2, 0.0), (128, 4, 2, -1.0), (128, 4, 2, float("inf")), (128, 4, 2, float("nan")),
])
def test_rejects_inadmissible_shapes(lib, T, H, G, c):
    assert call(lib, T=T, H=H, G=G, c=c) == tcg.ATTN_EINVAL


def test_admission_boundary(lib):
    # heads*64*T*4 == 2^32 exactly is one past the limit; 2^32 - 256 * 4 passes the check
    assert call(lib, T=2 ** 24 // 64 * 64 // 1, H=1, G=1) == tcg.ATTN_EINVAL
    big = call(lib, q=0x10000000000, k=0x20000000000, v=0x30000000000, o=0x40000000000,
               l=0x50000000000, T=2 ** 24 - 64, H=1, G=1)
    assert big != tcg.ATTN_EINVAL


def test_rejects_null_pointers(lib):
    assert call(lib, q=0) == tcg.ATTN_EINVAL
    assert call(lib, l=0) == tcg.ATTN_EINVAL


def test_rejects_misaligned_pointers(lib):
    assert call(lib, q=0x1008) == tcg.ATTN_EALIGN
    assert call(lib, o=0x300004) == tcg.ATTN_EALIGN


def test_rejects_overlapping_outputs(lib):
    # q occupies 4*128*64*2 = 65536 bytes from 0x1000
    assert call(lib, o=0x1000 + 65536 - 16) == tcg.ATTN_EOVERLAP
    assert call(lib, l=0x100000 + 16) == tcg.ATTN_EOVERLAP
    assert call(lib, o=0x300000, l=0x300000 + 65536 - 16) == tcg.ATTN_EOVERLAP


def test_no_device_is_reported_not_crashed(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call(lib) == tcg.ATTN_EDEVICE


def test_workspace_bytes(lib):
    T, H, G = 8192, 32, 8
    up = lambda n: (n + 255) // 256 * 256
    want = up(H * T * 128) * 2 + up(G * T * 128) * 2 + up(H * T * 4)
    assert tcg.attn_fwd_workspace_bytes(T, H, G) == want
    assert tcg.attn_fwd_workspace_bytes(100, H, G) == 0


def test_binding_checks_tensors(lib):
    torch = pytest.importorskip("torch")
    q = torch.zeros(4, 128, 64, dtype=torch.float32)
    with pytest.raises(TypeError):
        tcg.attn_fwd(q, q, q, q, q, 128, 4, 2, 0.18)


# ---------------------------------------------------------------------------- backward entry
def bwd_call(lib, T=128, H=4, G=2, c=0.18, s=0.125, ws_bytes=None, **ptr):
    """attn_bwd with fake, well-separated device addresses (no launch happens on a
    rejected call).  Sizes at T=128, H=4, G=2: q/o/dO 64 KiB, k/vT 32 KiB, lse 2 KiB,
    dq 128 KiB, dk/dvT 64 KiB, workspace 2 KiB."""
    base = dict(q=0x100000, k=0x200000, v=0x300000, o=0x400000, l=0x500000, g=0x600000,
                dq=0x700000, dk=0x800000, dv=0x900000, ws=0xA00000)
    base.update(ptr)
    vp = ctypes.c_void_p
    if ws_bytes is None:
        ws_bytes = tcg.attn_bwd_workspace_bytes(T, H, G) if T > 0 and T % 64 == 0 else 1 << 20
    return lib.attn_bwd(vp(base["q"]), vp(base["k"]), vp(base["v"]), vp(base["o"]),
                        vp(base["l"]), vp(base["g"]), vp(base["dq"]), vp(base["dk"]),
                        vp(base["dv"]), T, H, G, c, s, vp(base["ws"]), ws_bytes, None)


@pytest.mark.parametrize("T,H,G,c,s", [
    (0, 4, 2, 0.18, 0.125), (100, 4, 2, 0.18, 0.125), (128, 4, 3, 0.18, 0.125),
    (128, 65536, 1, 0.18, 0.125), (2 ** 24, 1, 1, 0.18, 0.125),
    (128, 4, 2, 0.0, 0.125), (128, 4, 2, 0.18, 0.0), (128, 4, 2, 0.18, float("nan")),
    (128, 4, 2, float("inf"), 0.125), (128, 4, 2, 0.18, -1.0),
])
def test_bwd_rejects_inadmissible_shapes(lib, T, H, G, c, s):
    assert bwd_call(lib, T=T, H=H, G=G, c=c, s=s) == tcg.ATTN_EINVAL


def test_bwd_rejects_null_misaligned_short_workspace(lib):
    assert bwd_call(lib, g=0) == tcg.ATTN_EINVAL
    assert bwd_call(lib, ws=0) == tcg.ATTN_EINVAL
    assert bwd_call(lib, dq=0x700008) == tcg.ATTN_EALIGN
    assert bwd_call(lib, l=0x500004) == tcg.ATTN_EALIGN
    assert bwd_call(lib, ws=0xA00010) == tcg.ATTN_EALIGN          # workspace wants 256 bytes
    assert bwd_call(lib, ws_bytes=tcg.attn_bwd_workspace_bytes(128, 4, 2) - 1) == tcg.ATTN_EINVAL


def test_bwd_rejects_overlaps(lib):
    assert bwd_call(lib, dq=0x100000 + 65536 - 16) == tcg.ATTN_EOVERLAP      # dq over q
    assert bwd_call(lib, dk=0x700000 + 131072 - 16) == tcg.ATTN_EOVERLAP     # dk over dq
    assert bwd_call(lib, ws=0x900000) == tcg.ATTN_EOVERLAP                   # workspace over dvT
    assert bwd_call(lib, dv=0x600000 + 65536) != tcg.ATTN_EOVERLAP           # adjacent is fine


def test_bwd_workspace_bytes(lib):
    # 512 key-launch units (8 K/V heads x 64 tiles): the row terms only
    assert tcg.attn_bwd_workspace_bytes(8192, 32, 8) == 32 * 8192 * 4
    assert tcg.attn_bwd_workspace_bytes(16384, 4, 1) == 4 * 16384 * 4     # 128 units
    # short GQA problems add S partial planes of dK and of dV^T,
    # S = min(group, ceil(256 / units), 8): 4 K/V heads x 16 tiles, groups of 4 -> S = 4
    up = lambda n: (n + 255) // 256 * 256
    plane = 4 * 2048 * 64 * 4
    assert tcg.attn_bwd_workspace_bytes(2048, 16, 4) == up(16 * 2048 * 4) + 2 * up(4 * plane)
    plane = 2 * 1024 * 64 * 4                                          # 2 K/V heads x 8 tiles, groups of 8
    assert tcg.attn_bwd_workspace_bytes(1024, 16, 2) == up(16 * 1024 * 4) + 2 * up(8 * plane)
    assert tcg.attn_bwd_workspace_bytes(1024, 12, 12) == 12 * 1024 * 4  # MHA: no split
    assert tcg.attn_bwd_workspace_bytes(64, 3, 1) == 768        # a 3-step walk: no split
    assert tcg.attn_bwd_workspace_bytes(100, 4, 2) == 0


def test_bwd_binding_checks_tensors(lib):
    torch = pytest.importorskip("torch")
    x = torch.zeros(4, 128, 64, dtype=torch.float16)
    with pytest.raises((TypeError, ValueError)):
        tcg.attn_bwd(x, x, x, x, x, x, x, x, x, 128, 4, 2, 0.18, 0.125, x)


# ---------------------------------------------------------------------------- materialised entry
def mat_call(lib, T=128, H=4, G=2, c=0.18, ws_bytes=None, **ptr):
    """attn_fwd_materialised with fake, well-separated device addresses (no launch
    happens on a rejected call).  At T=128, H=4, G=2: q/o 64 KiB, k/vT 32 KiB, lse 2 KiB,
    workspace 384 KiB."""
    base = dict(q=0x100000, k=0x200000, v=0x300000, o=0x400000, l=0x500000, ws=0x600000)
    base.update(ptr)
    vp = ctypes.c_void_p
    if ws_bytes is None:
        ws_bytes = tcg.attn_materialised_workspace_bytes(T, H, G) or (1 << 20)
    return lib.attn_fwd_materialised(vp(base["q"]), vp(base["k"]), vp(base["v"]), vp(base["o"]),
                                     vp(base["l"]), T, H, G, c, vp(base["ws"]), ws_bytes, None)


@pytest.mark.parametrize("T,H,G,c", [
    (0, 4, 2, 0.18), (100, 4, 2, 0.18), (128, 4, 3, 0.18), (16384 + 64, 1, 1, 0.18),
    (128, 4, 2, 0.0), (128, 4, 2, float("nan")),
])
def test_mat_rejects_inadmissible_shapes(lib, T, H, G, c):
    assert mat_call(lib, T=T, H=H, G=G, c=c) == tcg.ATTN_EINVAL


def test_mat_rejects_bad_pointers_and_workspace(lib):
    assert mat_call(lib, q=0) == tcg.ATTN_EINVAL
    assert mat_call(lib, ws=0x600010) == tcg.ATTN_EALIGN
    assert mat_call(lib, ws_bytes=tcg.attn_materialised_workspace_bytes(128, 4, 2) - 1) == tcg.ATTN_EINVAL
    assert mat_call(lib, o=0x100000 + 65536 - 16) == tcg.ATTN_EOVERLAP      # o over q
    assert mat_call(lib, ws=0x400000) == tcg.ATTN_EOVERLAP                  # workspace over o


def test_mat_workspace_bytes(lib):
    assert tcg.attn_materialised_workspace_bytes(1024, 12, 12) == 12 * 1024 * 1024 * 6
    assert tcg.attn_materialised_workspace_bytes(16384, 1, 1) == 16384 * 16384 * 6
    assert tcg.attn_materialised_workspace_bytes(16384 + 64, 1, 1) == 0


# ---------------------------------------------------------------------------- producer entry
def qkv_call(lib, T=128, width=128, H=4, G=2, **ptr):
    """attn_qkv_rope with fake, well-separated device addresses (no launch happens on a
    rejected call).  At T=128, width=128, H=4, G=2: x 32 KiB, w 64 KiB, tables 16 KiB each,
    q 64 KiB, k and vT 32 KiB."""
    base = dict(x=0x100000, w=0x200000, c=0x300000, s=0x400000, q=0x500000, k=0x600000,
                v=0x700000)
    base.update(ptr)
    vp = ctypes.c_void_p
    return lib.attn_qkv_rope(vp(base["x"]), vp(base["w"]), vp(base["c"]), vp(base["s"]),
                             vp(base["q"]), vp(base["k"]), vp(base["v"]), T, width, H, G, None)


@pytest.mark.parametrize("T,width,H,G", [
    (0, 128, 4, 2), (100, 128, 4, 2), (128, 0, 4, 2), (128, 96, 4, 2), (128, 128, 4, 3),
    (128, 128, 65536, 1), (2 ** 24, 64, 1, 1),
])
def test_qkv_rejects_inadmissible_shapes(lib, T, width, H, G):
    assert qkv_call(lib, T=T, width=width, H=H, G=G) == tcg.ATTN_EINVAL


def test_qkv_rejects_bad_pointers(lib):
    assert qkv_call(lib, w=0) == tcg.ATTN_EINVAL
    assert qkv_call(lib, c=0x300008) == tcg.ATTN_EALIGN
    assert qkv_call(lib, q=0x100000 + 32768 - 16) == tcg.ATTN_EOVERLAP     # q over x
    assert qkv_call(lib, v=0x600000 + 16) == tcg.ATTN_EOVERLAP             # vT over k
