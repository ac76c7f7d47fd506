"""Synthetic extreme-logit inputs (scaled scores up to ~2000, far above the
pages' "logits > 500" regime): every forward path stays finite and matches the
oracle.  The rows' maxima jump by hundreds between key tiles, so the eager
rescale factors underflow to zero (the exact limit of 2^(c (m_old - m_new)))."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, rel_l2, require_gpu
from precision_attention_fa4fp4_gb300.inputs import Workload, extreme_logit_inputs, make_inputs

pytestmark = pytest.mark.gpu


def extreme_inputs():
    return extreme_logit_inputs()


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
        Qd = oracle.dequantize_nvfp4(cq, sq, tq, qf.shape)
        Kd = oracle.dequantize_nvfp4(ck, sk, tk, kf.shape)
        scale = 0.0
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


@pytest.mark.parametrize("path", ["directp", "fp8pv"])
@pytest.mark.parametrize("causal", [False, True])
def test_softmax_path_error_no_worse_at_extreme_logits(path, causal):
    """Range guarding (the technical summary's sampled anchor for logits above
    500) is not built.  Evidence that it is not needed here: the error of the
    GPU's softmax path against exact FP64 softmax attention on the same
    quantized operands is no larger at logits of several hundred than at
    N(0,1) logits of the same shape.  (Against FP64 attention on the raw bf16
    inputs both regimes are dominated by the FP4 error of Q and K, which the
    logit scale amplifies; an anchor would not change that.)"""
    fa = require_gpu()
    errs = {}
    for regime in ("extreme", "normal"):
        if regime == "extreme":
            q, k, v = extreme_inputs()
        else:
            q, k, v = make_inputs(Workload("normal_640", 1, 2, 2, 640, 128, causal=causal), seed=3)
        qf, kf, vf = (t.float().numpy() for t in (q, k, v))
        q4, k4 = fa.quantize(q.cuda()), fa.quantize(k.cuda())
        Qd = oracle.dequantize(*oracle.quantize(qf, 0, 0), qf.shape, 0, 0)
        Kd = oracle.dequantize(*oracle.quantize(kf, 0, 0), kf.shape, 0, 0)
        if path == "fp8pv":
            o, lse = fa.fwd_fp8pv(q4, k4, fa.quantize(v.cuda(), fa.FMT_MXFP8, fa.ALONG_N), causal=causal,
                                  out_dtype=fa.OUT_F32)
            Vd = oracle.dequantize(*oracle.quantize(vf, 1, 1), vf.shape, 1, 1)
        else:
            o, lse = fa.fwd(q4, k4, fa.quantize(v.cuda(), fa.FMT_MXFP4, fa.ALONG_N), causal=causal,
                            out_dtype=fa.OUT_F32)
            Vd = oracle.dequantize(*oracle.quantize(vf, 0, 1), vf.shape, 0, 1)
        fa.sync_status()
        o = o.cpu().numpy().reshape(-1, q.shape[-1])
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse.cpu().numpy()))
        exact_q = oracle.attention_fp64(Qd, Kd, Vd, causal=causal)
        errs[regime] = rel_l2(o, exact_q)
    assert errs["extreme"] <= errs["normal"], errs
