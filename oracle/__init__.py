"""CPU oracle for block-scaled FP4 attention with Direct-P.

TEST INFRASTRUCTURE ONLY: the plain, slow definition the CUDA library is
checked against.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  It shares no code with
the CUDA path; the C source is compiled here with gcc into its own library.

Every function cites the passage of "Hardware-Aware FP4 FlashAttention-4"
(arXiv:2609.04105; gist.science technical summary and the arXiv abstract) it
follows, in ``fa4fp4_oracle.c``.  This module only marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa4fp4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liborc.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE arithmetic: no fast-math, no FMA
    contraction, so x86 and Arm hosts compute the same values)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            fp = ctypes.POINTER(ctypes.c_float)
            u8 = ctypes.POINTER(ctypes.c_uint8)
            i64 = ctypes.POINTER(ctypes.c_int64)
            c_int, c_float, c_long = ctypes.c_int, ctypes.c_float, ctypes.c_long
            lib.orc_e2m1_value.restype = ctypes.c_double
            lib.orc_e4m3_value.restype = ctypes.c_double
            lib.orc_e8m0_value.restype = ctypes.c_double
            lib.orc_round_to_code.argtypes = [ctypes.c_double, c_int]
            lib.orc_block_exponent.argtypes = [c_float, c_int]
            lib.orc_p_block_exponent.argtypes = [c_float]
            lib.orc_quantize.argtypes = [fp, c_int, c_int, c_int, c_int, c_int, c_int, u8, u8]
            lib.orc_dequantize.argtypes = [u8, u8, c_int, c_int, c_int, c_int, c_int, c_int, fp]
            lib.orc_directp_thresholds.argtypes = [fp]
            lib.orc_directp_x.argtypes = [c_float, c_float, c_float]
            lib.orc_directp_x.restype = c_float
            lib.orc_directp_code_of_x.argtypes = [c_float]
            lib.orc_directp_code.argtypes = [c_float, c_float, c_float]
            lib.orc_directp_codes_of_x.argtypes = [fp, c_long, u8]
            lib.orc_fwd.argtypes = [fp, fp, fp, c_int, c_int, c_int, c_int, c_int, c_float, c_int,
                                    c_int, c_long, i64, dp, dp]
            lib.orc_bwd.argtypes = [fp, fp, fp, fp, fp, fp, fp, fp, c_int, c_int, c_int, c_int,
                                    c_int, c_float, c_int, c_int, c_long, i64, dp, c_long, i64,
                                    dp, dp]
            lib.orc_attention_fp64.argtypes = [fp, fp, fp, c_int, c_int, c_int, c_int, c_int,
                                               c_float, c_int, c_long, i64, dp]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def num_threads() -> int:
    return int(_load().orc_num_threads())


# --------------------------------------------------------------------------
# element formats
# --------------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return _load().orc_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return _load().orc_e4m3_value(int(code))


def e8m0_value(byte: int) -> float:
    return _load().orc_e8m0_value(int(byte))


def round_to_code(y: float, fmt: int) -> int:
    """fmt 0 = E2M1, 1 = E4M3: nearest magnitude, ties to even, saturating,
    sign kept."""
    return int(_load().orc_round_to_code(float(y), int(fmt)))


def block_exponent(amax: float, fmt: int) -> int:
    return int(_load().orc_block_exponent(float(amax), int(fmt)))


def p_block_exponent(amax: float) -> int:
    """E8M0 exponent of an E4M3 probability block: the smallest X with
    amax <= 448 * 2^X (no saturation), clamped to [-127, 127]."""
    return int(_load().orc_p_block_exponent(float(amax)))


# --------------------------------------------------------------------------
# quantization
# --------------------------------------------------------------------------

FMT_MXFP4, FMT_MXFP8 = 0, 1
ALONG_D, ALONG_N = 0, 1


def padded_n(N: int) -> int:
    return ((N + 127) // 128) * 128


def qtensor_shapes(B, H, N, d, fmt, axis):
    """(codes shape, scales shape) in bytes of the canonical layouts."""
    if axis == ALONG_D:
        L, R = d, N
    else:
        L, R = padded_n(N), d
    per = L // 2 if fmt == FMT_MXFP4 else L
    return (B, H, R, per), (B, H, R, L // 32)


def quantize(x, fmt: int, axis: int):
    """x: [B,H,N,d] float array (bf16 values).  Returns (codes, scales) as
    uint8 arrays in the canonical layouts (see fa4fp4_oracle.c)."""
    x = _f32(x)
    B, H, N, d = x.shape
    cs, ss = qtensor_shapes(B, H, N, d, fmt, axis)
    codes = np.zeros(cs, dtype=np.uint8)
    scales = np.zeros(ss, dtype=np.uint8)
    _load().orc_quantize(_ptr(x, ctypes.c_float), B, H, N, d, fmt, axis,
                         _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8))
    return codes, scales


def dequantize(codes, scales, shape, fmt: int, axis: int) -> np.ndarray:
    B, H, N, d = shape
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    out = np.zeros((B, H, N, d), dtype=np.float32)
    _load().orc_dequantize(_ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8), B, H, N,
                           d, fmt, axis, _ptr(out, ctypes.c_float))
    return out


def nvfp4_tensor_scale(x) -> float:
    x = _f32(x)
    _load().orc_nvfp4_tensor_scale.restype = ctypes.c_float
    return float(_load().orc_nvfp4_tensor_scale(_ptr(x, ctypes.c_float), ctypes.c_long(x.size)))


def quantize_nvfp4(x):
    """NVFP4 along d: returns (codes [B,H,N,d/2], scales [B,H,N,d/16] E4M3
    bytes, tensor scale float)."""
    x = _f32(x)
    B, H, N, d = x.shape
    ts = nvfp4_tensor_scale(x)
    codes = np.zeros((B, H, N, d // 2), dtype=np.uint8)
    scales = np.zeros((B, H, N, d // 16), dtype=np.uint8)
    _load().orc_quantize_nvfp4(_ptr(x, ctypes.c_float), B, H, N, d, ctypes.c_float(ts),
                               _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8))
    return codes, scales, ts


def dequantize_nvfp4(codes, scales, ts, shape) -> np.ndarray:
    B, H, N, d = shape
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    out = np.zeros((B, H, N, d), dtype=np.float32)
    _load().orc_dequantize_nvfp4(_ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8),
                                 ctypes.c_float(ts), B, H, N, d, _ptr(out, ctypes.c_float))
    return out


# --------------------------------------------------------------------------
# Direct-P
# --------------------------------------------------------------------------

def directp_thresholds() -> np.ndarray:
    T = np.zeros(7, dtype=np.float32)
    _load().orc_directp_thresholds(_ptr(T, ctypes.c_float))
    return T


def directp_x(s: float, m: float, c: float) -> float:
    return float(_load().orc_directp_x(s, m, c))


def directp_code_of_x(x: float) -> int:
    return int(_load().orc_directp_code_of_x(x))


def directp_code(s: float, m: float, c: float) -> int:
    return int(_load().orc_directp_code(s, m, c))


def directp_codes_of_x(x) -> np.ndarray:
    x = _f32(x).ravel()
    out = np.zeros(x.size, dtype=np.uint8)
    _load().orc_directp_codes_of_x(_ptr(x, ctypes.c_float), x.size, _ptr(out, ctypes.c_uint8))
    return out


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

def _rows(rows, total):
    if rows is None:
        rows = np.arange(total, dtype=np.int64)
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int64))


def fwd(Q, K, V, softmax_scale: float = 0.0, causal: bool = False, mode: int = 0, rows=None):
    """Forward for selected query rows ((b*Hq+h)*N+i).  Q [B,Hq,N,d],
    K/V [B,Hkv,N,d] float arrays (dequantized values).  Returns (O [r,d],
    LSE [r]) in float64.  mode 0 = Direct-P, mode 1 = exact exponentials,
    mode 2 = FP8 P/V route (P rounded through MXFP8 per 32 keys; V given as
    the dequantized MXFP8 values)."""
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    B, Hq, N, d = Q.shape
    Hkv = K.shape[1]
    rows = _rows(rows, B * Hq * N)
    O = np.zeros((len(rows), d), dtype=np.float64)
    L = np.zeros(len(rows), dtype=np.float64)
    _load().orc_fwd(_ptr(Q, ctypes.c_float), _ptr(K, ctypes.c_float), _ptr(V, ctypes.c_float),
                    B, Hq, Hkv, N, d, float(softmax_scale), int(bool(causal)), int(mode),
                    len(rows), _ptr(rows, ctypes.c_int64), _ptr(O, ctypes.c_double),
                    _ptr(L, ctypes.c_double))
    return O, L


def bwd(Q4, K4, Q8, K8, V8, O, dO, LSE, softmax_scale: float = 0.0, causal: bool = False,
        mode: int = 0, qrows=None, krows=None):
    """Gradients for selected rows.  All tensors logical [B,H,N,d] floats;
    LSE [B,Hq,N].  Returns (dQ [nq,d], dK [nk,d], dV [nk,d]) float64."""
    Q4, K4, Q8, K8, V8, O, dO = (_f32(a) for a in (Q4, K4, Q8, K8, V8, O, dO))
    LSE = _f32(LSE)
    B, Hq, N, d = Q4.shape
    Hkv = K4.shape[1]
    qrows = _rows(qrows, B * Hq * N)
    krows = _rows(krows, B * Hkv * N)
    dQ = np.zeros((len(qrows), d), dtype=np.float64)
    dK = np.zeros((len(krows), d), dtype=np.float64)
    dV = np.zeros((len(krows), d), dtype=np.float64)
    f = ctypes.c_float
    _load().orc_bwd(_ptr(Q4, f), _ptr(K4, f), _ptr(Q8, f), _ptr(K8, f), _ptr(V8, f), _ptr(O, f),
                    _ptr(dO, f), _ptr(LSE, f), B, Hq, Hkv, N, d, float(softmax_scale),
                    int(bool(causal)), int(mode), len(qrows), _ptr(qrows, ctypes.c_int64),
                    _ptr(dQ, ctypes.c_double), len(krows), _ptr(krows, ctypes.c_int64),
                    _ptr(dK, ctypes.c_double), _ptr(dV, ctypes.c_double))
    return dQ, dK, dV


def attention_fp64(Q, K, V, softmax_scale: float = 0.0, causal: bool = False, rows=None):
    """Unquantized softmax attention in FP64 (error report only)."""
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    B, Hq, N, d = Q.shape
    Hkv = K.shape[1]
    rows = _rows(rows, B * Hq * N)
    O = np.zeros((len(rows), d), dtype=np.float64)
    _load().orc_attention_fp64(_ptr(Q, ctypes.c_float), _ptr(K, ctypes.c_float),
                               _ptr(V, ctypes.c_float), B, Hq, Hkv, N, d, float(softmax_scale),
                               int(bool(causal)), len(rows), _ptr(rows, ctypes.c_int64),
                               _ptr(O, ctypes.c_double))
    return O
