"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/fa4fp4.h declares, sizes its buffers, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from precision_attention_fa4fp4_gb300 import api, build
    build.build()
    return api.load_library()


def declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            txt = open(os.path.join(inc, f)).read()
            names |= set(re.findall(r"FA4FP4_API\s+[\w\s\*]+?\b(\w+)\s*\(", txt))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_qtensor_bytes(lib):
    sb = ctypes.c_size_t(0)
    assert lib.fa4fp4_qtensor_bytes(2, 3, 300, 128, 0, 0, ctypes.byref(sb)) == 2 * 3 * 300 * 64
    assert sb.value == 2 * 3 * 300 * 4
    assert lib.fa4fp4_qtensor_bytes(2, 3, 300, 128, 0, 1, ctypes.byref(sb)) == 2 * 3 * 128 * 384 // 2
    assert sb.value == 2 * 3 * 128 * 384 // 32
    assert lib.fa4fp4_qtensor_bytes(1, 1, 33, 64, 1, 1, ctypes.byref(sb)) == 64 * 128
    assert lib.fa4fp4_qtensor_bytes(1, 1, 33, 96, 0, 0, ctypes.byref(sb)) == 0
    assert lib.fa4fp4_qtensor_bytes(1, 1, 0, 64, 0, 0, None) == 0


def test_argument_errors_before_launch(lib):
    p = ctypes.c_void_p(4096)       # never dereferenced: validation fails first
    odd = ctypes.c_void_p(4097)
    null = None
    INVALID, UNSUP, ALIGN = 1, 2, 3
    assert lib.fa4fp4_quantize(null, 1, 1, 32, 64, 0, 0, p, p, null) == INVALID
    assert lib.fa4fp4_quantize(p, 1, 1, 32, 64, 2, 0, p, p, null) == INVALID
    assert lib.fa4fp4_quantize(p, 1, 1, 32, 96, 0, 0, p, p, null) == UNSUP
    assert lib.fa4fp4_quantize(odd, 1, 1, 32, 64, 0, 0, p, p, null) == ALIGN
    args = [p] * 6
    assert lib.fa4fp4_fwd(*args, 1, 4, 3, 64, 64, 0.0, 0, p, 1, null, null) == UNSUP   # Hq % Hkv
    assert lib.fa4fp4_fwd(*args, 1, 4, 4, 64, 80, 0.0, 0, p, 1, null, null) == UNSUP   # d
    assert lib.fa4fp4_fwd(*args, 1, 4, 4, 0, 64, 0.0, 0, p, 1, null, null) == INVALID  # N
    assert lib.fa4fp4_fwd(*args, 1, 4, 4, 64, 64, 0.0, 0, p, 7, null, null) == INVALID # dtype
    assert lib.fa4fp4_fwd(*([p] * 5 + [odd]), 1, 4, 4, 64, 64, 0.0, 0, p, 1, null, null) == ALIGN
    assert lib.fa4bf16_fwd(null, p, p, 1, 1, 1, 64, 64, 0.0, 0, p, 1, null, null) == INVALID
    assert lib.fa4fp4_quantize_nvfp4(null, 1, 1, 32, 64, p, p, p, null) == INVALID
    assert lib.fa4fp4_quantize_nvfp4(p, 1, 1, 32, 64, p, p, null, null) == INVALID
    assert lib.fa4fp4_quantize_nvfp4(p, 1, 1, 32, 96, p, p, p, null) == UNSUP
    assert lib.fa4fp4_quantize_nvfp4(p, 1, 1, 32, 64, p, p, ctypes.c_void_p(4098), null) == ALIGN
    nv = [p] * 8
    assert lib.fa4fp4_fwd_nvfp4(p, p, null, p, p, p, p, p, 1, 4, 2, 64, 64, 0.0, 0, 0, p, 1, null, null) == INVALID
    assert lib.fa4fp4_fwd_nvfp4(*nv, 1, 4, 2, 64, 64, 0.0, 0, 2, p, 1, null, null) == INVALID   # fp8pv
    assert lib.fa4fp4_fwd_nvfp4(*nv, 1, 4, 3, 64, 64, 0.0, 0, 0, p, 1, null, null) == UNSUP
    assert lib.fa4fp4_fwd_fp8pv(*([p] * 6), 1, 4, 4, 64, 80, 0.0, 0, p, 1, null, null) == UNSUP
    qkv = [p] * 3
    outs = [p] * 6
    assert lib.fa4fp4_quantize_qkv(null, p, p, 1, 4, 2, 64, 64, *outs, null) == INVALID
    assert lib.fa4fp4_quantize_qkv(*qkv, 1, 4, 2, 64, 64, *([p] * 5 + [null]), null) == INVALID
    assert lib.fa4fp4_quantize_qkv(*qkv, 1, 4, 3, 64, 64, *outs, null) == UNSUP      # Hq % Hkv
    assert lib.fa4fp4_quantize_qkv(*qkv, 1, 4, 2, 64, 96, *outs, null) == UNSUP      # d
    assert lib.fa4fp4_quantize_qkv(p, p, odd, 1, 4, 2, 64, 64, *outs, null) == ALIGN
    assert lib.fa4fp4_quantize_qkv(*qkv, 1, 4, 2, 64, 64, *([p] * 4 + [odd, p]), null) == ALIGN
    assert lib.fa4fp4_fwd_qbf16(null, p, p, p, p, 1, 4, 2, 64, 64, 0.0, 0, 0, p, 1, null, null) == INVALID
    assert lib.fa4fp4_fwd_qbf16(p, p, p, p, p, 1, 4, 2, 64, 64, 0.0, 0, 2, p, 1, null, null) == INVALID  # fp8pv
    assert lib.fa4fp4_fwd_qbf16(p, p, p, p, p, 1, 4, 3, 64, 64, 0.0, 0, 0, p, 1, null, null) == UNSUP
    assert lib.fa4fp4_fwd_qbf16(odd, p, p, p, p, 1, 4, 2, 64, 64, 0.0, 0, 0, p, 1, null, null) == ALIGN
    assert lib.fa4fp4_quantize_kv(null, p, 1, 2, 64, 64, p, p, p, p, null) == INVALID
    assert lib.fa4fp4_quantize_kv(p, p, 1, 2, 64, 96, p, p, p, p, null) == UNSUP
    assert lib.fa4fp4_quantize_kv(p, p, 1, 2, 64, 64, p, p, odd, p, null) == ALIGN
    assert lib.fa4fp4_directp_codes(null, 10, 0.0, 1.0, 0, p, null) == INVALID
    assert lib.fa4fp4_directp_codes(p, 10, 0.0, 1.0, 2, p, null) == INVALID
    assert lib.fa4fp4_status_string(5).decode() == "device pipeline wait timed out"


def test_workspace_size(lib):
    """The backward's workspace: the dO row view (codes + scales), the dO
    column view (codes + scales, N padded to 128) and one 16-byte row of
    accumulator offsets per query row, each piece rounded up to 256 bytes."""
    up = lambda x: (x + 255) // 256 * 256
    for B, Hq, Hkv, N, d in ((2, 4, 2, 300, 128), (1, 6, 3, 1, 64), (2, 32, 8, 8192, 128)):
        rows = B * Hq * N
        Np = (N + 127) // 128 * 128
        want = (up(rows * d) + up(rows * d // 32) + up(B * Hq * d * Np) + up(B * Hq * d * Np // 32)
                + up(rows * 16))
        assert lib.fa4fp4_bwd_workspace_bytes(B, Hq, Hkv, N, d) == want
    assert lib.fa4fp4_bwd_workspace_bytes(2, 4, 3, 300, 128) == 0


def test_empty_problems_are_noops(lib):
    """B == 0 or H == 0: shape and options are still checked, then the call
    returns OK without inspecting its (here NULL) pointers or launching."""
    null = None
    OK, INVALID, UNSUP = 0, 1, 2
    n6 = [null] * 6
    for B, H in ((0, 4), (2, 0)):
        Hkv = 2 if H else 0
        assert lib.fa4fp4_quantize(null, B, H, 32, 64, 0, 0, null, null, null) == OK
        assert lib.fa4fp4_quantize(null, B, H, 32, 128, 1, 1, null, null, null) == OK
        assert lib.fa4fp4_quantize_qkv(null, null, null, B, H, Hkv, 64, 128, *n6, null) == OK
        assert lib.fa4fp4_quantize_nvfp4(null, B, H, 32, 64, null, null, null, null) == OK
        assert lib.fa4fp4_fwd(*n6, B, H, Hkv, 300, 128, 0.0, 1, null, 1, null, null) == OK
        assert lib.fa4fp4_fwd_fp8pv(*n6, B, H, Hkv, 300, 64, 0.0, 0, null, 0, null, null) == OK
        assert lib.fa4fp4_fwd_nvfp4(*([null] * 8), B, H, Hkv, 300, 128, 0.0, 1, 1, null, 1, null, null) == OK
        assert lib.fa4bf16_fwd(null, null, null, B, H, Hkv, 300, 128, 0.0, 1, null, 1, null, null) == OK
        assert lib.fa4fp4_fwd_qbf16(*([null] * 5), B, H, Hkv, 300, 128, 0.0, 1, 0, null, 1, null, null) == OK
        assert lib.fa4fp4_quantize_kv(null, null, B, Hkv, 300, 128, null, null, null, null, null) == OK
        assert lib.fa4fp4_bwd(*([null] * 11), 0, null, null, B, H, Hkv, 300, 128, 0.0, 1,
                              null, null, null, null, 0, null) == OK
        assert lib.fa4fp4_bwd_workspace_bytes(B, H, Hkv, 300, 128) == 0
    bwd_na = lib.fa4fp4_bwd_noalloc
    bwd_na.restype = ctypes.c_int
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    bwd_na.argtypes = [vp] * 11 + [i, vp, vp, i, i, i, i, i, f, i, vp, vp, vp, vp]
    assert bwd_na(*([null] * 11), 0, null, null, 0, 4, 2, 300, 128, 0.0, 1, null, null, null, null) == OK
    # an empty problem with a bad shape or option is still rejected
    assert lib.fa4fp4_quantize(null, 0, 4, 32, 96, 0, 0, null, null, null) == UNSUP
    assert lib.fa4fp4_quantize(null, 0, 4, 0, 64, 0, 0, null, null, null) == INVALID
    assert lib.fa4fp4_quantize(null, 0, 4, 32, 64, 3, 0, null, null, null) == INVALID
    assert lib.fa4fp4_fwd(*n6, 0, 4, 3, 64, 64, 0.0, 0, null, 1, null, null) == UNSUP
    assert lib.fa4fp4_fwd(*n6, 0, 4, 4, 64, 64, 0.0, 0, null, 9, null, null) == INVALID
    assert lib.fa4fp4_fwd_nvfp4(*([null] * 8), 0, 4, 4, 64, 64, 0.0, 0, 5, null, 1, null, null) == INVALID
    assert lib.fa4fp4_bwd(*([null] * 11), 0, null, null, 0, 4, 2, 300, 96, 0.0, 1,
                          null, null, null, null, 0, null) == UNSUP
    assert lib.fa4fp4_bwd(*([null] * 11), 0, null, null, 0, 4, 2, 300, 64, 0.0, 1,
                          null, null, null, null, 0, null) == OK
    assert lib.fa4fp4_quantize_qkv(null, null, null, -1, 4, 2, 64, 128, *n6, null) == INVALID


def test_noalloc_validates_like_bwd(lib):
    """A problem too large for the fixed scratch array still gets the same
    argument errors from fa4fp4_bwd_noalloc as from fa4fp4_bwd (validation
    comes first; nothing is launched)."""
    p, null = ctypes.c_void_p(4096), None
    INVALID, UNSUP, WORKSPACE = 1, 2, 6
    bwd_na = lib.fa4fp4_bwd_noalloc
    bwd_na.restype = ctypes.c_int
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    bwd_na.argtypes = [vp] * 11 + [i, vp, vp, i, i, i, i, i, f, i, vp, vp, vp, vp]
    B, Hq, Hkv, N = 2, 32, 8, 8192
    assert lib.fa4fp4_bwd_workspace_bytes(B, Hq, Hkv, N, 128) > (16 << 20)
    for odt, d, want in ((7, 128, INVALID), (0, 96, UNSUP)):
        got_na = bwd_na(*([p] * 11), odt, p, p, B, Hq, Hkv, N, d, 0.0, 1, p, p, p, null)
        got = lib.fa4fp4_bwd(*([p] * 11), odt, p, p, B, Hq, Hkv, N, d, 0.0, 1, p, p, p, p, 1 << 40, null)
        assert got_na == got == want
    # null gradient pointers: invalid from both
    assert bwd_na(*([p] * 11), 0, p, p, B, Hq, Hkv, N, 128, 0.0, 1, null, p, p, null) == INVALID
    # well-formed but oversized: the scratch limit
    assert bwd_na(*([p] * 11), 0, p, p, B, Hq, Hkv, N, 128, 0.0, 1, p, p, p, null) == WORKSPACE


def test_fwd_host_validation_and_workspace(lib):
    """The host-buffer inference call checks shape, options, pointers,
    alignment and its workspace before it touches the device."""
    p = ctypes.c_void_p(4096)
    odd = ctypes.c_void_p(4097)
    null = None
    OK, INVALID, UNSUP, ALIGN, WS = 0, 1, 2, 3, 6
    fh = lib.fa4fp4_fwd_host
    big = 1 << 40
    # B4 Hq16 Hkv16 N4096 d128: chunks of 8 (batch, kv head) units; staging for
    # two chunks of bf16 Q, K, V (8.4 MB each), of O (f32) and LSE, and of MXFP4
    # Q, K, V^T codes and scales
    want = 2 * 3 * 8 * 4096 * 128 * 2 + 2 * (8 * 4096 * 128 * 4 + 8 * 4096 * 4) + 2 * 3 * (8 * 4096 * 64 + 8 * 4096 * 4)
    assert lib.fa4fp4_fwd_host_workspace_bytes(4, 16, 16, 4096, 128) == want
    assert lib.fa4fp4_fwd_host_workspace_bytes(1, 24, 24, 32760, 128) > 0
    assert lib.fa4fp4_fwd_host_workspace_bytes(1, 4, 3, 300, 128) == 0
    assert lib.fa4fp4_fwd_host_workspace_bytes(1, 4, 2, 300, 96) == 0
    assert lib.fa4fp4_fwd_host_workspace_bytes(0, 4, 2, 300, 128) == 0
    n = lib.fa4fp4_fwd_host_workspace_bytes(2, 8, 2, 300, 64)
    assert fh(null, null, null, 0, 4, 2, 300, 128, 0.0, 1, null, 1, null, null, 0, null) == OK
    assert fh(null, null, null, 0, 4, 2, 300, 96, 0.0, 1, null, 1, null, null, 0, null) == UNSUP
    assert fh(p, p, p, 2, 8, 3, 300, 64, 0.0, 1, p, 1, p, p, big, null) == UNSUP
    assert fh(p, p, p, 2, 8, 2, 0, 64, 0.0, 1, p, 1, p, p, big, null) == INVALID
    assert fh(p, p, p, 2, 8, 2, 300, 64, 0.0, 1, p, 7, p, p, big, null) == INVALID
    assert fh(null, p, p, 2, 8, 2, 300, 64, 0.0, 1, p, 1, p, p, big, null) == INVALID
    assert fh(p, p, p, 2, 8, 2, 300, 64, 0.0, 1, null, 1, p, p, big, null) == INVALID
    assert fh(p, odd, p, 2, 8, 2, 300, 64, 0.0, 1, p, 1, p, p, big, null) == ALIGN
    assert fh(p, p, p, 2, 8, 2, 300, 64, 0.0, 1, p, 1, ctypes.c_void_p(4098), p, big, null) == ALIGN
    assert fh(p, p, p, 2, 8, 2, 300, 64, 0.0, 1, p, 1, p, null, big, null) == WS
    assert fh(p, p, p, 2, 8, 2, 300, 64, 0.0, 1, p, 1, p, p, n - 1, null) == WS
    assert fh(p, p, p, 2, 8, 2, 300, 64, 0.0, 1, p, 1, p, odd, n, null) == ALIGN
