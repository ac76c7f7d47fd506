"""Synthetic extreme-logit inputs (scaled scores up to ~2000, far above the
pages' "logits > 500" regime): every forward path stays finite and matches the
oracle.  The rows' maxima jump by hundreds between key tiles, so the eager
rescale factors underflow to zero (the exact limit of 2^(c (m_old - m_new)))."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, require_gpu

pytestmark = pytest.mark.gpu


def extreme_inputs(N=640, d=128, seed=3):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(1, 2, N, d, generator=g) * 6.0
    k = torch.randn(1, 2, N, d, generator=g) * 6.0
    # key tiles grow in magnitude along N: each later tile raises the row max
    k = k * (1.0 + torch.arange(N).float().div(128).floor().view(1, 1, N, 1))
    v = torch.randn(1, 2, N, d, generator=g)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


@pytest.mark.parametrize("path", ["directp", "fp8pv", "nvfp4"])
@pytest.mark.parametrize("causal", [False, True])
def test_extreme_logits(path, causal):
    fa = require_gpu()
    q, k, v = extreme_inputs()
    qf, kf, vf = (t.float().numpy() for t in (q, k, v))
    d = q.shape[-1]
    if path == "nvfp4":
        qn, kn = fa.quantize_nvfp4(q.cuda()), fa.quantize_nvfp4(k.cuda())
        vt = fa.quantize(v.cuda(), fa.FMT_MXFP4, fa.ALONG_N)
        o, lse = fa.fwd_nvfp4(qn, kn, vt, causal=causal, out_dtype=fa.OUT_F32)
        cq, sq, tq = oracle.quantize_nvfp4(qf)
        ck, sk, tk = oracle.quantize_nvfp4(kf)
        Qd = oracle.dequantize_nvfp4(cq, sq, 1.0, qf.shape)
        Kd = oracle.dequantize_nvfp4(ck, sk, 1.0, kf.shape)
        scale = float(np.float32(np.float32(np.float32(1 / np.sqrt(d)) * np.float32(tq)) * np.float32(tk)))
        Vd, mode = oracle.dequantize(*oracle.quantize(vf, 0, 1), vf.shape, 0, 1), 0
    else:
        q4, k4 = fa.quantize(q.cuda()), fa.quantize(k.cuda())
        Qd = oracle.dequantize(*oracle.quantize(qf, 0, 0), qf.shape, 0, 0)
        Kd = oracle.dequantize(*oracle.quantize(kf, 0, 0), kf.shape, 0, 0)
        scale = 0.0
        if path == "fp8pv":
            v8 = fa.quantize(v.cuda(), fa.FMT_MXFP8, fa.ALONG_N)
            o, lse = fa.fwd_fp8pv(q4, k4, v8, causal=causal, out_dtype=fa.OUT_F32)
            Vd, mode = oracle.dequantize(*oracle.quantize(vf, 1, 1), vf.shape, 1, 1), 2
        else:
            vt = fa.quantize(v.cuda(), fa.FMT_MXFP4, fa.ALONG_N)
            o, lse = fa.fwd(q4, k4, vt, causal=causal, out_dtype=fa.OUT_F32)
            Vd, mode = oracle.dequantize(*oracle.quantize(vf, 0, 1), vf.shape, 0, 1), 0
    fa.sync_status()
    o, lse = o.cpu().numpy().reshape(-1, d), lse.cpu().numpy().reshape(-1)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    Oo, Lo = oracle.fwd(Qd, Kd, Vd, softmax_scale=scale, causal=causal, mode=mode)
    assert np.max(Lo) > 500          # the regime under test
    assert_close(o, Oo, f"extreme logits {path}")
    assert np.max(np.abs(lse - Lo) / np.maximum(1.0, np.abs(Lo))) < 1e-5
