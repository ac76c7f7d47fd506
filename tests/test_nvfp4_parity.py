"""NVFP4 Q/K on the GPU vs the oracle.

Quantization: codes, E4M3 block scales and the FP32 tensor scale bit-exact.
Forward: the oracle runs on the plain definition, deq = E2M1 x E4M3 x the
FP32 tensor scale, with the softmax scale 1/sqrt(d).  (The kernel folds the
two tensor scales into the softmax scale; the CPU tests pin that this moves
O and LSE by FP32 rounding only.)  Tolerances as for the MXFP4 forward.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, require_gpu, round_like
from precision_attention_fa4fp4_gb300.inputs import TINY, TRAIN_8B, VIDEO_DIT, Workload, make_inputs, sample_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(1, 2, 1, 64), (2, 3, 33, 128), (1, 4, 300, 64), (1, 2, 1000, 128)])
def test_quantize_nvfp4_bit_exact(shape):
    fa = require_gpu()
    g = torch.Generator().manual_seed(sum(shape))
    x = torch.randn(shape, generator=g) * torch.exp2(torch.randint(-6, 6, shape[:3] + (shape[3] // 16,), generator=g).float()).repeat_interleave(16, -1)
    x = x.to(torch.bfloat16)
    x[0, 0, 0, :16] = 0.0
    got = fa.quantize_nvfp4(x.cuda())
    fa.sync_status()
    co, so, tso = oracle.quantize_nvfp4(x.float().numpy())
    assert np.float32(got.ts.item()) == np.float32(tso)
    assert np.array_equal(got.scales.cpu().numpy(), so)
    assert np.array_equal(got.codes.cpu().numpy(), co)


def test_quantize_nvfp4_full_size_outliers():
    fa = require_gpu()
    q, _, _ = make_inputs(VIDEO_DIT)
    got = fa.quantize_nvfp4(q.cuda())
    fa.sync_status()
    co, so, tso = oracle.quantize_nvfp4(q.float().numpy())
    assert np.float32(got.ts.item()) == np.float32(tso)
    assert np.array_equal(got.scales.cpu().numpy(), so) and np.array_equal(got.codes.cpu().numpy(), co)


def check(w: Workload, fp8pv: bool, out_bf16=False, rows=None, seed=0):
    fa = require_gpu()
    q, k, v = make_inputs(w, seed=seed)
    qn, kn = fa.quantize_nvfp4(q.cuda()), fa.quantize_nvfp4(k.cuda())
    vt = fa.quantize(v.cuda(), fa.FMT_MXFP8 if fp8pv else fa.FMT_MXFP4, fa.ALONG_N)
    o, lse = fa.fwd_nvfp4(qn, kn, vt, causal=w.causal, out_dtype=fa.OUT_BF16 if out_bf16 else fa.OUT_F32)
    fa.sync_status()
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    qf, kf, vf = (t.float().numpy() for t in (q, k, v))
    cq, sq, tq = oracle.quantize_nvfp4(qf)
    ck, sk, tk = oracle.quantize_nvfp4(kf)
    Qd = oracle.dequantize_nvfp4(cq, sq, tq, qf.shape)
    Kd = oracle.dequantize_nvfp4(ck, sk, tk, kf.shape)
    fmt = 1 if fp8pv else 0
    Vd = oracle.dequantize(*oracle.quantize(vf, fmt, 1), vf.shape, fmt, 1)
    rows = np.arange(w.B * w.Hq * w.N) if rows is None else np.asarray(rows)
    Oo, Lo = oracle.fwd(Qd, Kd, Vd, causal=w.causal, rows=rows, mode=2 if fp8pv else 0)
    name = w.name + (" NVFP4 Q/K + FP8 P/V" if fp8pv else " NVFP4 Q/K")
    assert_close(o.reshape(-1, w.d)[rows], round_like(Oo, out_bf16), name + " O")
    assert np.max(np.abs(lse.reshape(-1)[rows] - Lo)) < 1e-3, name + " LSE"


@pytest.mark.parametrize("fp8pv", [False, True])
def test_tiny(fp8pv):
    check(TINY, fp8pv, out_bf16=True)


@pytest.mark.parametrize("fp8pv", [False, True])
@pytest.mark.parametrize("N,d,causal", [(1, 64, False), (129, 128, True), (300, 64, True), (1000, 128, False)])
def test_ragged(N, d, causal, fp8pv):
    check(Workload(f"nv_ragged_n{N}_d{d}", 1, 4, 2, N, d, causal=causal), fp8pv, seed=N)


def test_video_dit_outliers_sampled():
    check(VIDEO_DIT, False, rows=sample_rows(VIDEO_DIT, tiles_per_head=3, heads=[0, 23]))


def test_train_causal_gqa_sampled():
    check(TRAIN_8B, True, rows=sample_rows(TRAIN_8B, tiles_per_head=2, heads=[0, 37]))
