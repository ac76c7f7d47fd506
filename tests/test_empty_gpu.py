"""Empty problems (B == 0 or H == 0) through the Python binding: every call
returns empty outputs without an error, and leaves the device usable."""
import pytest
import torch

from gpu_util import require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,Hq,Hkv", [(0, 4, 2), (2, 0, 0)])
def test_empty_batch_or_heads(B, Hq, Hkv):
    fa = require_gpu()
    N, d = 300, 128
    q = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((B, Hkv, N, d), dtype=torch.bfloat16, device="cuda")
    q4, k4, vt = fa.quantize_qkv(q, k, k.clone())
    o, lse = fa.fwd(q4, k4, vt, causal=True)
    assert o.shape == (B, Hq, N, d) and lse.shape == (B, Hq, N)
    v8 = fa.quantize(k, fa.FMT_MXFP8, fa.ALONG_N)
    o8, _ = fa.fwd_fp8pv(q4, k4, v8)
    assert o8.numel() == 0
    qn, kn = fa.quantize_nvfp4(q), fa.quantize_nvfp4(k)
    on, _ = fa.fwd_nvfp4(qn, kn, vt)
    assert on.numel() == 0
    ob, _ = fa.bf16_fwd(q, k, k)
    assert ob.numel() == 0
    q8c = fa.quantize(q, fa.FMT_MXFP8, fa.ALONG_N)
    k8c = fa.quantize(k, fa.FMT_MXFP8, fa.ALONG_N)
    v8r = fa.quantize(k, fa.FMT_MXFP8, fa.ALONG_D)
    dq, dk, dv = fa.bwd(q4, k4, q8c, k8c, v8r, o, o, lse, causal=True)
    assert dq.shape == (B, Hq, N, d) and dk.shape == (B, Hkv, N, d) and dv.shape == (B, Hkv, N, d)
    fa.sync_status()
    # the device still runs a non-empty problem afterwards
    x = torch.randn((1, 1, 64, 64), device="cuda").to(torch.bfloat16)
    x4 = fa.quantize(x)
    xt = fa.quantize(x, fa.FMT_MXFP4, fa.ALONG_N)
    o1, _ = fa.fwd(x4, x4, xt)
    fa.sync_status()
    assert torch.isfinite(o1.float()).all()
