"""Thin ctypes binding of the C ABI in include/fa4fp4.h.

Argument marshalling only: torch tensors give device pointers and the current
stream; every step of the computation runs in the CUDA library.  If the
library is not built, or is called on tensors that are not on a CUDA device,
the call raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(HERE, "libfa4fp4.so")

FMT_MXFP4, FMT_MXFP8 = 0, 1
ALONG_D, ALONG_N = 0, 1
OUT_F32, OUT_BF16 = 0, 1
_STATUS_OK = 0


class Fa4Fp4Error(RuntimeError):
    def __init__(self, where: str, status: int):
        msg = library().fa4fp4_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


_lib = None


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libfa4fp4.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {_LIB_PATH} (run __graft_entry__.build())")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa4fp4_status_string.restype = ctypes.c_char_p
        lib.fa4fp4_status_string.argtypes = [i]
        lib.fa4fp4_qtensor_bytes.restype = sz
        lib.fa4fp4_qtensor_bytes.argtypes = [i, i, i, i, i, i, ctypes.POINTER(sz)]
        lib.fa4fp4_quantize.restype = i
        lib.fa4fp4_quantize.argtypes = [vp, i, i, i, i, i, i, vp, vp, vp]
        lib.fa4fp4_quantize_qkv.restype = i
        lib.fa4fp4_quantize_qkv.argtypes = [vp, vp, vp, i, i, i, i, i] + [vp] * 7
        lib.fa4fp4_fwd_fp8pv.restype = i
        lib.fa4fp4_fwd_fp8pv.argtypes = [vp] * 6 + [i, i, i, i, i, f, i, vp, i, vp, vp]
        lib.fa4fp4_quantize_nvfp4.restype = i
        lib.fa4fp4_quantize_nvfp4.argtypes = [vp, i, i, i, i, vp, vp, vp, vp]
        lib.fa4fp4_fwd_nvfp4.restype = i
        lib.fa4fp4_fwd_nvfp4.argtypes = [vp] * 8 + [i, i, i, i, i, f, i, i, vp, i, vp, vp]
        lib.fa4fp4_fwd.restype = i
        lib.fa4fp4_fwd.argtypes = [vp] * 6 + [i, i, i, i, i, f, i, vp, i, vp, vp]
        lib.fa4fp4_fwd_qbf16.restype = i
        lib.fa4fp4_fwd_qbf16.argtypes = [vp] * 5 + [i, i, i, i, i, f, i, i, vp, i, vp, vp]
        lib.fa4fp4_quantize_kv.restype = i
        lib.fa4fp4_quantize_kv.argtypes = [vp, vp, i, i, i, i, vp, vp, vp, vp, vp]
        lib.fa4fp4_fwd_host_workspace_bytes.restype = sz
        lib.fa4fp4_fwd_host_workspace_bytes.argtypes = [i, i, i, i, i]
        lib.fa4fp4_fwd_host.restype = i
        lib.fa4fp4_fwd_host.argtypes = [vp, vp, vp, i, i, i, i, i, f, i, vp, i, vp, vp, sz, vp]
        lib.fa4fp4_bwd_workspace_bytes.restype = sz
        lib.fa4fp4_bwd_workspace_bytes.argtypes = [i, i, i, i, i]
        lib.fa4fp4_bwd.restype = i
        lib.fa4fp4_bwd.argtypes = [vp] * 11 + [i, vp, vp, i, i, i, i, i, f, i, vp, vp, vp, vp, sz, vp]
        lib.fa4bf16_fwd.restype = i
        lib.fa4bf16_fwd.argtypes = [vp, vp, vp, i, i, i, i, i, f, i, vp, i, vp, vp]
        lib.fa4fp4_directp_codes.restype = i
        lib.fa4fp4_directp_codes.argtypes = [vp, ctypes.c_int64, f, f, i, vp, vp]
        lib.fa4fp4_sync_status.restype = i
        lib.fa4fp4_sync_status.argtypes = [vp]
        _lib = lib
    return _lib


def library():
    return load_library()


def _check(where: str, status: int):
    if status != _STATUS_OK:
        raise Fa4Fp4Error(where, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("fa4fp4: tensors must be contiguous CUDA tensors")


def padded_n(N: int) -> int:
    return (N + 127) // 128 * 128


@dataclass
class QTensor:
    """A block-quantized tensor: codes + E8M0 scales in the canonical layout
    of include/fa4fp4.h, logical shape (B, H, N, d)."""
    codes: torch.Tensor
    scales: torch.Tensor
    shape: tuple
    fmt: int
    axis: int


def qtensor_shapes(B, H, N, d, fmt, axis):
    L, R = (d, N) if axis == ALONG_D else (padded_n(N), d)
    per = L // 2 if fmt == FMT_MXFP4 else L
    return (B, H, R, per), (B, H, R, L // 32)


def _numel(shape) -> int:
    n = 1
    for x in shape:
        n *= x
    return n


def _expect_qt(name: str, t: QTensor, fmt: int, axis: int, shape: tuple):
    """The library reads exactly qtensor_shapes(...) bytes of codes and scales:
    refuse a tensor of another format, axis or size before any launch."""
    if not isinstance(t, QTensor):
        raise ValueError(f"{name}: expected a QTensor")
    kind = ("MXFP4" if fmt == FMT_MXFP4 else "MXFP8") + (" along d" if axis == ALONG_D else " along N")
    if t.fmt != fmt or t.axis != axis:
        raise ValueError(f"{name}: expected {kind}")
    cs, ss = qtensor_shapes(*shape, fmt, axis)
    if (tuple(t.shape) != tuple(shape) or t.codes.dtype != torch.uint8 or t.scales.dtype != torch.uint8
            or t.codes.numel() != _numel(cs) or t.scales.numel() != _numel(ss)):
        raise ValueError(f"{name}: codes/scales are not those of a {kind} tensor of shape {tuple(shape)}")


def _expect(name: str, t, shape: tuple, dtypes):
    if t is None:
        return
    if tuple(t.shape) != tuple(shape) or t.dtype not in dtypes:
        raise ValueError(f"{name}: expected shape {tuple(shape)} and dtype in {[str(x) for x in dtypes]}, "
                         f"got {tuple(t.shape)} {t.dtype}")


def _expect_out(out, lse, B, Hq, N, d, out_dtype):
    if out_dtype not in (OUT_F32, OUT_BF16):
        raise ValueError("out_dtype must be OUT_F32 or OUT_BF16")
    _expect("out", out, (B, Hq, N, d), (torch.bfloat16,) if out_dtype == OUT_BF16 else (torch.float32,))
    _expect("lse", lse, (B, Hq, N), (torch.float32,))


def qtensor_alloc(B, H, N, d, fmt, axis, device="cuda") -> QTensor:
    cs, ss = qtensor_shapes(B, H, N, d, fmt, axis)
    return QTensor(torch.empty(cs, dtype=torch.uint8, device=device),
                   torch.empty(ss, dtype=torch.uint8, device=device), (B, H, N, d), fmt, axis)


def quantize(x: torch.Tensor, fmt: int = FMT_MXFP4, axis: int = ALONG_D, out: QTensor | None = None) -> QTensor:
    """Block-quantize a bf16 [B,H,N,d] CUDA tensor (fa4fp4_quantize)."""
    if x.dtype != torch.bfloat16 or x.dim() != 4:
        raise ValueError("quantize expects a bf16 [B,H,N,d] tensor")
    B, H, N, d = x.shape
    if out is not None:
        _expect_qt("out", out, fmt, axis, (B, H, N, d))
        _cuda(out.codes, out.scales)
    _cuda(x)
    q = out if out is not None else qtensor_alloc(B, H, N, d, fmt, axis, x.device)
    _check("fa4fp4_quantize", load_library().fa4fp4_quantize(
        _ptr(x), B, H, N, d, fmt, axis, _ptr(q.codes), _ptr(q.scales), _stream(x.device)))
    return q


def quantize_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out=None):
    """Q, K (MXFP4 along d) and V (MXFP4 along N) in one launch
    (fa4fp4_quantize_qkv).  Returns (q4, k4, vt) as quantize would."""
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or t.dim() != 4:
            raise ValueError("quantize_qkv expects bf16 [B,H,N,d] tensors")
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, N, d) or v.shape != k.shape:
        raise ValueError("quantize_qkv: k and v must be [B,Hkv,N,d] with q's B, N, d")
    if out is not None:
        _expect_qt("out[0] (q)", out[0], FMT_MXFP4, ALONG_D, (B, Hq, N, d))
        _expect_qt("out[1] (k)", out[1], FMT_MXFP4, ALONG_D, (B, Hkv, N, d))
        _expect_qt("out[2] (v)", out[2], FMT_MXFP4, ALONG_N, (B, Hkv, N, d))
        _cuda(*_qt_buffers(*out))
    _cuda(q, k, v)
    if out is None:
        out = (qtensor_alloc(B, Hq, N, d, FMT_MXFP4, ALONG_D, q.device),
               qtensor_alloc(B, Hkv, N, d, FMT_MXFP4, ALONG_D, q.device),
               qtensor_alloc(B, Hkv, N, d, FMT_MXFP4, ALONG_N, q.device))
    q4, k4, vt = out
    _check("fa4fp4_quantize_qkv", load_library().fa4fp4_quantize_qkv(
        _ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, N, d, _ptr(q4.codes), _ptr(q4.scales), _ptr(k4.codes),
        _ptr(k4.scales), _ptr(vt.codes), _ptr(vt.scales), _stream(q.device)))
    return q4, k4, vt


def fwd(q: QTensor, k: QTensor, vt: QTensor, causal: bool = False, softmax_scale: float = 0.0,
        out_dtype: int = OUT_BF16, with_lse: bool = True, out=None, lse=None):
    """Direct-P FP4 forward (fa4fp4_fwd).  Returns (o, lse or None)."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    _expect_qt("q", q, FMT_MXFP4, ALONG_D, (B, Hq, N, d))
    _expect_qt("k", k, FMT_MXFP4, ALONG_D, (B, Hkv, N, d))
    _expect_qt("vt", vt, FMT_MXFP4, ALONG_N, (B, Hkv, N, d))
    _expect_out(out, lse if with_lse else None, B, Hq, N, d, out_dtype)
    dev = q.codes.device
    if out is None:
        out = torch.empty((B, Hq, N, d), dtype=torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32, device=dev)
    if with_lse and lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    _cuda(q.codes, q.scales, k.codes, k.scales, vt.codes, vt.scales, out, lse)
    _check("fa4fp4_fwd", load_library().fa4fp4_fwd(
        _ptr(q.codes), _ptr(q.scales), _ptr(k.codes), _ptr(k.scales), _ptr(vt.codes), _ptr(vt.scales),
        B, Hq, Hkv, N, d, float(softmax_scale), int(bool(causal)), _ptr(out), out_dtype,
        _ptr(lse) if with_lse else None, _stream(dev)))
    return out, (lse if with_lse else None)


def quantize_kv(k: torch.Tensor, v: torch.Tensor, out=None):
    """K (MXFP4 along d) and V (MXFP4 along N) in one launch
    (fa4fp4_quantize_kv).  Returns (k4, vt) as quantize would."""
    for t in (k, v):
        if t.dtype != torch.bfloat16 or t.dim() != 4:
            raise ValueError("quantize_kv expects bf16 [B,H,N,d] tensors")
    if v.shape != k.shape:
        raise ValueError("quantize_kv: k and v must have the same shape")
    B, Hkv, N, d = k.shape
    if out is not None:
        _expect_qt("out[0] (k)", out[0], FMT_MXFP4, ALONG_D, (B, Hkv, N, d))
        _expect_qt("out[1] (v)", out[1], FMT_MXFP4, ALONG_N, (B, Hkv, N, d))
        _cuda(*_qt_buffers(*out))
    _cuda(k, v)
    if out is None:
        out = (qtensor_alloc(B, Hkv, N, d, FMT_MXFP4, ALONG_D, k.device),
               qtensor_alloc(B, Hkv, N, d, FMT_MXFP4, ALONG_N, k.device))
    k4, vt = out
    _check("fa4fp4_quantize_kv", load_library().fa4fp4_quantize_kv(
        _ptr(k), _ptr(v), B, Hkv, N, d, _ptr(k4.codes), _ptr(k4.scales), _ptr(vt.codes), _ptr(vt.scales),
        _stream(k.device)))
    return k4, vt


def fwd_qbf16(q: torch.Tensor, k: QTensor, vt: QTensor, causal: bool = False, softmax_scale: float = 0.0,
              out_dtype: int = OUT_BF16, with_lse: bool = True, out=None, lse=None):
    """Forward with bf16 Q quantized to MXFP4 in the kernel's prologue
    (fa4fp4_fwd_qbf16).  vt MXFP4 along N gives Direct-P, MXFP8 along N the
    FP8 P/V route.  Returns (o, lse or None), identical to quantize(q)
    followed by fwd (fwd_fp8pv)."""
    if q.dtype != torch.bfloat16 or q.dim() != 4:
        raise ValueError("fwd_qbf16 expects a bf16 [B,H,N,d] q")
    if not isinstance(vt, QTensor) or vt.fmt not in (FMT_MXFP4, FMT_MXFP8):
        raise ValueError("vt: expected an MXFP4 or MXFP8 QTensor blocked along N")
    fp8pv = 1 if vt.fmt == FMT_MXFP8 else 0
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    _expect_qt("k", k, FMT_MXFP4, ALONG_D, (B, Hkv, N, d))
    _expect_qt("vt", vt, vt.fmt, ALONG_N, (B, Hkv, N, d))
    _expect_out(out, lse if with_lse else None, B, Hq, N, d, out_dtype)
    dev = q.device
    if out is None:
        out = torch.empty((B, Hq, N, d), dtype=torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32, device=dev)
    if with_lse and lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    _cuda(q, k.codes, k.scales, vt.codes, vt.scales, out, lse)
    _check("fa4fp4_fwd_qbf16", load_library().fa4fp4_fwd_qbf16(
        _ptr(q), _ptr(k.codes), _ptr(k.scales), _ptr(vt.codes), _ptr(vt.scales), B, Hq, Hkv, N, d,
        float(softmax_scale), int(bool(causal)), fp8pv, _ptr(out), out_dtype, _ptr(lse) if with_lse else None,
        _stream(dev)))
    return out, (lse if with_lse else None)


def fwd_fp8pv(q: QTensor, k: QTensor, v8t: QTensor, causal: bool = False, softmax_scale: float = 0.0,
              out_dtype: int = OUT_BF16, with_lse: bool = True, out=None, lse=None):
    """FP8 P/V route of the forward (fa4fp4_fwd_fp8pv): MXFP4 Q/K, V as MXFP8
    blocked along N.  Returns (o, lse or None)."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    _expect_qt("q", q, FMT_MXFP4, ALONG_D, (B, Hq, N, d))
    _expect_qt("k", k, FMT_MXFP4, ALONG_D, (B, Hkv, N, d))
    _expect_qt("v8t", v8t, FMT_MXFP8, ALONG_N, (B, Hkv, N, d))
    _expect_out(out, lse if with_lse else None, B, Hq, N, d, out_dtype)
    dev = q.codes.device
    if out is None:
        out = torch.empty((B, Hq, N, d), dtype=torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32, device=dev)
    if with_lse and lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    _cuda(q.codes, q.scales, k.codes, k.scales, v8t.codes, v8t.scales, out, lse)
    _check("fa4fp4_fwd_fp8pv", load_library().fa4fp4_fwd_fp8pv(
        _ptr(q.codes), _ptr(q.scales), _ptr(k.codes), _ptr(k.scales), _ptr(v8t.codes), _ptr(v8t.scales),
        B, Hq, Hkv, N, d, float(softmax_scale), int(bool(causal)), _ptr(out), out_dtype,
        _ptr(lse) if with_lse else None, _stream(dev)))
    return out, (lse if with_lse else None)


@dataclass
class NvTensor:
    """NVFP4 tensor: E2M1 codes [B,H,N,d/2], E4M3 scales [B,H,N,d/16], and the
    FP32 tensor scale in a one-element device tensor."""
    codes: torch.Tensor
    scales: torch.Tensor
    ts: torch.Tensor
    shape: tuple


def _expect_nv(name: str, t: NvTensor, shape: tuple):
    B, H, N, d = shape
    if not isinstance(t, NvTensor):
        raise ValueError(f"{name}: expected an NvTensor")
    if (tuple(t.shape) != tuple(shape) or t.codes.dtype != torch.uint8 or t.scales.dtype != torch.uint8
            or t.codes.numel() != B * H * N * d // 2 or t.scales.numel() != B * H * N * d // 16
            or t.ts.dtype != torch.float32 or t.ts.numel() < 1):
        raise ValueError(f"{name}: codes/scales/ts are not those of an NVFP4 tensor of shape {tuple(shape)}")


def quantize_nvfp4(x: torch.Tensor, out: NvTensor | None = None) -> NvTensor:
    """NVFP4 along d of a bf16 [B,H,N,d] CUDA tensor (fa4fp4_quantize_nvfp4)."""
    if x.dtype != torch.bfloat16 or x.dim() != 4:
        raise ValueError("quantize_nvfp4 expects a bf16 [B,H,N,d] tensor")
    B, H, N, d = x.shape
    if out is not None:
        _expect_nv("out", out, (B, H, N, d))
        _cuda(out.codes, out.scales, out.ts)
    _cuda(x)
    if out is None:
        out = NvTensor(torch.empty((B, H, N, d // 2), dtype=torch.uint8, device=x.device),
                       torch.empty((B, H, N, d // 16), dtype=torch.uint8, device=x.device),
                       torch.empty(1, dtype=torch.float32, device=x.device), (B, H, N, d))
    _check("fa4fp4_quantize_nvfp4", load_library().fa4fp4_quantize_nvfp4(
        _ptr(x), B, H, N, d, _ptr(out.codes), _ptr(out.scales), _ptr(out.ts), _stream(x.device)))
    return out


def fwd_nvfp4(q: NvTensor, k: NvTensor, vt: QTensor, causal: bool = False, softmax_scale: float = 0.0,
              out_dtype: int = OUT_BF16, with_lse: bool = True, out=None, lse=None):
    """Forward with NVFP4 Q/K (fa4fp4_fwd_nvfp4).  vt MXFP4 along N gives
    Direct-P, MXFP8 along N the FP8 P/V route.  Returns (o, lse or None)."""
    if not isinstance(vt, QTensor) or vt.fmt not in (FMT_MXFP4, FMT_MXFP8):
        raise ValueError("vt: expected an MXFP4 or MXFP8 QTensor blocked along N")
    fp8pv = 1 if vt.fmt == FMT_MXFP8 else 0
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    _expect_nv("q", q, (B, Hq, N, d))
    _expect_nv("k", k, (B, Hkv, N, d))
    _expect_qt("vt", vt, vt.fmt, ALONG_N, (B, Hkv, N, d))
    _expect_out(out, lse if with_lse else None, B, Hq, N, d, out_dtype)
    dev = q.codes.device
    if out is None:
        out = torch.empty((B, Hq, N, d), dtype=torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32, device=dev)
    if with_lse and lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    _cuda(q.codes, q.scales, q.ts, k.codes, k.scales, k.ts, vt.codes, vt.scales, out, lse)
    _check("fa4fp4_fwd_nvfp4", load_library().fa4fp4_fwd_nvfp4(
        _ptr(q.codes), _ptr(q.scales), _ptr(q.ts), _ptr(k.codes), _ptr(k.scales), _ptr(k.ts),
        _ptr(vt.codes), _ptr(vt.scales), B, Hq, Hkv, N, d, float(softmax_scale), int(bool(causal)), fp8pv,
        _ptr(out), out_dtype, _ptr(lse) if with_lse else None, _stream(dev)))
    return out, (lse if with_lse else None)


def _expect_bwd_inputs(q4, k4, q8c, k8c, v8r, o, dout, lse):
    B, Hq, N, d = q4.shape
    Hkv = k4.shape[1]
    _expect_qt("q4", q4, FMT_MXFP4, ALONG_D, (B, Hq, N, d))
    _expect_qt("k4", k4, FMT_MXFP4, ALONG_D, (B, Hkv, N, d))
    _expect_qt("q8c", q8c, FMT_MXFP8, ALONG_N, (B, Hq, N, d))
    _expect_qt("k8c", k8c, FMT_MXFP8, ALONG_N, (B, Hkv, N, d))
    _expect_qt("v8r", v8r, FMT_MXFP8, ALONG_D, (B, Hkv, N, d))
    _expect("o", o, (B, Hq, N, d), (torch.float32, torch.bfloat16))
    _expect("dout", dout, (B, Hq, N, d), (torch.bfloat16,))
    _expect("lse", lse, (B, Hq, N), (torch.float32,))
    return B, Hq, Hkv, N, d


def _qt_buffers(*qts):
    return [b for t in qts for b in (t.codes, t.scales)]


def _expect_grads(dq, dk, dv, B, Hq, Hkv, N, d):
    _expect("dq", dq, (B, Hq, N, d), (torch.float32,))
    _expect("dk", dk, (B, Hkv, N, d), (torch.float32,))
    _expect("dv", dv, (B, Hkv, N, d), (torch.float32,))


def fwd_host_workspace_bytes(B, Hq, Hkv, N, d) -> int:
    return int(load_library().fa4fp4_fwd_host_workspace_bytes(B, Hq, Hkv, N, d))


def _host(*ts):
    for t in ts:
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError("fa4fp4: host buffers must be contiguous CPU tensors (page-locked for overlap)")


def fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
             softmax_scale: float = 0.0, out_dtype: int = OUT_BF16, with_lse: bool = True, out=None, lse=None,
             workspace: torch.Tensor | None = None, device=None):
    """The inference step on host buffers (fa4fp4_fwd_host): bf16 CPU q, k, v
    in, CPU o (and lse) out, quantization and the Direct-P forward on the
    current CUDA device and stream.  Returns (o, lse or None); they hold the
    result once the stream has reached the end of the call."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("fwd_host expects [B,H,N,d] tensors")
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    _expect("q", q, (B, Hq, N, d), (torch.bfloat16,))
    _expect("k", k, (B, Hkv, N, d), (torch.bfloat16,))
    _expect("v", v, (B, Hkv, N, d), (torch.bfloat16,))
    _expect_out(out, lse if with_lse else None, B, Hq, N, d, out_dtype)
    _host(q, k, v, out, lse if with_lse else None)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    pin = q.is_pinned()
    if out is None:
        out = torch.empty((B, Hq, N, d), dtype=torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32,
                          pin_memory=pin)
    if with_lse and lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, pin_memory=pin)
    ws_bytes = fwd_host_workspace_bytes(B, Hq, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    elif workspace.dtype != torch.uint8:
        raise ValueError("workspace: expected a uint8 tensor")
    _cuda(workspace)
    _check("fa4fp4_fwd_host", load_library().fa4fp4_fwd_host(
        _ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, N, d, float(softmax_scale), int(bool(causal)), _ptr(out), out_dtype,
        _ptr(lse) if with_lse else None, _ptr(workspace), workspace.numel(), _stream(workspace.device)))
    return out, (lse if with_lse else None)


def bwd_workspace_bytes(B, Hq, Hkv, N, d) -> int:
    return int(load_library().fa4fp4_bwd_workspace_bytes(B, Hq, Hkv, N, d))


def bwd(q4: QTensor, k4: QTensor, q8c: QTensor, k8c: QTensor, v8r: QTensor, o: torch.Tensor,
        dout: torch.Tensor, lse: torch.Tensor, causal: bool = True, softmax_scale: float = 0.0,
        workspace: torch.Tensor | None = None):
    """Quantized backward (fa4fp4_bwd).  Returns (dq, dk, dv) in float32."""
    B, Hq, Hkv, N, d = _expect_bwd_inputs(q4, k4, q8c, k8c, v8r, o, dout, lse)
    if workspace is not None and workspace.dtype != torch.uint8:
        raise ValueError("workspace: expected a uint8 tensor")
    dev = dout.device
    dq = torch.empty((B, Hq, N, d), dtype=torch.float32, device=dev)
    dk = torch.empty((B, Hkv, N, d), dtype=torch.float32, device=dev)
    dv = torch.empty((B, Hkv, N, d), dtype=torch.float32, device=dev)
    ws_bytes = bwd_workspace_bytes(B, Hq, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    o_dtype = OUT_BF16 if o.dtype == torch.bfloat16 else OUT_F32
    _cuda(*_qt_buffers(q4, k4, q8c, k8c, v8r), o, dout, lse, workspace)
    _check("fa4fp4_bwd", load_library().fa4fp4_bwd(
        _ptr(q4.codes), _ptr(q4.scales), _ptr(k4.codes), _ptr(k4.scales), _ptr(q8c.codes), _ptr(q8c.scales),
        _ptr(k8c.codes), _ptr(k8c.scales), _ptr(v8r.codes), _ptr(v8r.scales), _ptr(o), o_dtype, _ptr(dout),
        _ptr(lse), B, Hq, Hkv, N, d, float(softmax_scale), int(bool(causal)), _ptr(dq), _ptr(dk), _ptr(dv),
        _ptr(workspace), workspace.numel(), _stream(dev)))
    return dq, dk, dv


def bf16_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
             softmax_scale: float = 0.0, out_dtype: int = OUT_BF16, with_lse: bool = True, out=None, lse=None):
    """BF16 FlashAttention forward (fa4bf16_fwd).  Returns (o, lse or None)."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("bf16_fwd expects [B,H,N,d] tensors")
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    _expect("q", q, (B, Hq, N, d), (torch.bfloat16,))
    _expect("k", k, (B, Hkv, N, d), (torch.bfloat16,))
    _expect("v", v, (B, Hkv, N, d), (torch.bfloat16,))
    _expect_out(out, lse if with_lse else None, B, Hq, N, d, out_dtype)
    _cuda(q, k, v)
    if out is None:
        out = torch.empty((B, Hq, N, d), dtype=torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32, device=q.device)
    if with_lse and lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    _check("fa4bf16_fwd", load_library().fa4bf16_fwd(
        _ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, N, d, float(softmax_scale), int(bool(causal)), _ptr(out),
        out_dtype, _ptr(lse) if with_lse else None, _stream(q.device)))
    return out, (lse if with_lse else None)


def directp_codes(s: torch.Tensor, m: float, c: float, native_exp: bool = False) -> torch.Tensor:
    """Direct-P code of each FP32 score against max m (fa4fp4_directp_codes);
    native_exp selects the native-exponential route instead of the exact
    threshold classifier."""
    _cuda(s)
    if s.dtype != torch.float32:
        raise ValueError("directp_codes expects float32 scores")
    out = torch.empty(s.shape, dtype=torch.uint8, device=s.device)
    _check("fa4fp4_directp_codes", load_library().fa4fp4_directp_codes(
        _ptr(s), s.numel(), float(m), float(c), int(bool(native_exp)), _ptr(out), _stream(s.device)))
    return out


def watchdog_selftest(limit_ns: int = 50_000_000, device=None):
    """Launch the library's watchdog self-test (a bounded wait that nothing
    satisfies); the next sync_status() raises with FA4FP4_ERR_DEVICE_TIMEOUT."""
    lib = load_library()
    fn = lib.fa4fp4_watchdog_selftest
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_int64, ctypes.c_void_p]
    _check("fa4fp4_watchdog_selftest", fn(int(limit_ns), _stream(device)))


def sync_status(device=None):
    """Synchronize the current stream and raise on a device watchdog error."""
    _check("fa4fp4_sync_status", load_library().fa4fp4_sync_status(_stream(device)))


def bwd_noalloc(q4: QTensor, k4: QTensor, q8c: QTensor, k8c: QTensor, v8r: QTensor, o: torch.Tensor,
                dout: torch.Tensor, lse: torch.Tensor, causal: bool = True, softmax_scale: float = 0.0,
                dq=None, dk=None, dv=None):
    """fa4fp4_bwd_noalloc: the backward for callers that cannot allocate device
    memory.  The C entry point takes no workspace and allocates nothing; its
    scratch is a fixed array inside the library (FA4FP4_BWD_NOALLOC_SCRATCH_BYTES),
    so problems whose workspace would be larger are rejected.  Calls that
    overlap on the GPU share that array and race.  Pass dq/dk/dv to avoid the
    output allocations made here on the caller's behalf."""
    lib = load_library()
    fn = lib.fa4fp4_bwd_noalloc
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.restype = i
    fn.argtypes = [vp] * 11 + [i, vp, vp, i, i, i, i, i, f, i, vp, vp, vp, vp]
    B, Hq, Hkv, N, d = _expect_bwd_inputs(q4, k4, q8c, k8c, v8r, o, dout, lse)
    _expect_grads(dq, dk, dv, B, Hq, Hkv, N, d)
    dev = dout.device
    dq = dq if dq is not None else torch.empty((B, Hq, N, d), dtype=torch.float32, device=dev)
    dk = dk if dk is not None else torch.empty((B, Hkv, N, d), dtype=torch.float32, device=dev)
    dv = dv if dv is not None else torch.empty((B, Hkv, N, d), dtype=torch.float32, device=dev)
    o_dtype = OUT_BF16 if o.dtype == torch.bfloat16 else OUT_F32
    _cuda(*_qt_buffers(q4, k4, q8c, k8c, v8r), o, dout, lse, dq, dk, dv)
    _check("fa4fp4_bwd_noalloc", fn(
        _ptr(q4.codes), _ptr(q4.scales), _ptr(k4.codes), _ptr(k4.scales), _ptr(q8c.codes), _ptr(q8c.scales),
        _ptr(k8c.codes), _ptr(k8c.scales), _ptr(v8r.codes), _ptr(v8r.scales), _ptr(o), o_dtype, _ptr(dout),
        _ptr(lse), B, Hq, Hkv, N, d, float(softmax_scale), int(bool(causal)), _ptr(dq), _ptr(dk), _ptr(dv),
        _stream(dev)))
    return dq, dk, dv
