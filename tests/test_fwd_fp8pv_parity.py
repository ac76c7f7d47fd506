"""FP8 P/V route of the forward on the GPU vs the oracle (mode 2) on the same
seeded inputs: MXFP4 Q/K, V through MXFP8 along N, P through MXFP8 per 32 keys.

Tolerance as for the Direct-P forward: rel-L2 <= 1e-3 and max-abs <= 1e-2 on O
after the oracle's O is rounded to the kernel's output dtype; LSE to 1e-3.
The kernel's p uses the hardware exponential and the oracle fl32(2^x); an E4M3
code differs only where p*2^-X lies within a few ulp of a rounding midpoint.
"""
import numpy as np
import pytest

import oracle
from gpu_util import assert_close, require_gpu, round_like
from precision_attention_fa4fp4_gb300.inputs import TINY, TRAIN_8B, FWD_4K, Workload, make_inputs, sample_rows

pytestmark = pytest.mark.gpu


def oracle_operands(q, k, v):
    qf, kf, vf = (t.float().numpy() for t in (q, k, v))
    Qd = oracle.dequantize(*oracle.quantize(qf, 0, 0), qf.shape, 0, 0)
    Kd = oracle.dequantize(*oracle.quantize(kf, 0, 0), kf.shape, 0, 0)
    V8 = oracle.dequantize(*oracle.quantize(vf, 1, 1), vf.shape, 1, 1)
    return Qd, Kd, V8


def gpu_fwd(fa, q, k, v, causal, out_bf16):
    q4, k4 = fa.quantize(q.cuda()), fa.quantize(k.cuda())
    v8 = fa.quantize(v.cuda(), fa.FMT_MXFP8, fa.ALONG_N)
    o, lse = fa.fwd_fp8pv(q4, k4, v8, causal=causal, out_dtype=fa.OUT_BF16 if out_bf16 else fa.OUT_F32)
    fa.sync_status()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check(w: Workload, out_bf16=True, rows=None, seed=0):
    fa = require_gpu()
    q, k, v = make_inputs(w, seed=seed)
    o, lse = gpu_fwd(fa, q, k, v, w.causal, out_bf16)
    Qd, Kd, V8 = oracle_operands(q, k, v)
    rows = np.arange(w.B * w.Hq * w.N) if rows is None else np.asarray(rows)
    Oo, Lo = oracle.fwd(Qd, Kd, V8, causal=w.causal, rows=rows, mode=2)
    assert_close(o.reshape(-1, w.d)[rows], round_like(Oo, out_bf16), w.name + " O (FP8 P/V)")
    assert np.max(np.abs(lse.reshape(-1)[rows] - Lo)) < 1e-3, w.name + " LSE (FP8 P/V)"


@pytest.mark.parametrize("out_bf16", [True, False])
def test_tiny(out_bf16):
    check(TINY, out_bf16)


@pytest.mark.parametrize("N", [1, 33, 127, 128, 129, 300, 1000])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged(N, d, causal):
    check(Workload(f"ragged_n{N}_d{d}", 1, 4, 2, N, d, causal=causal), out_bf16=False, seed=N)


def test_noncausal_4k_sampled():
    check(FWD_4K, True, rows=sample_rows(FWD_4K, tiles_per_head=3, heads=range(0, 64, 9)))


def test_train_causal_gqa_sampled():
    check(TRAIN_8B, False, rows=sample_rows(TRAIN_8B, tiles_per_head=3, heads=[0, 37]))


def test_closer_to_exact_than_direct_p():
    """On the training shape's sampled rows, the FP8 route's O is closer to
    exact softmax attention over the same quantized Q/K than Direct-P's."""
    fa = require_gpu()
    w = Workload("acc_n2048_d128", 1, 4, 2, 2048, 128, causal=True)
    q, k, v = make_inputs(w, seed=5)
    rows = sample_rows(w, tiles_per_head=4, heads=[0, 3])
    o8, _ = gpu_fwd(fa, q, k, v, True, False)
    q4, k4 = fa.quantize(q.cuda()), fa.quantize(k.cuda())
    vt = fa.quantize(v.cuda(), fa.FMT_MXFP4, fa.ALONG_N)
    o4, _ = fa.fwd(q4, k4, vt, causal=True, out_dtype=fa.OUT_F32)
    fa.sync_status()
    qf, kf, vf = (t.float().numpy() for t in (q, k, v))
    Qd = oracle.dequantize(*oracle.quantize(qf, 0, 0), qf.shape, 0, 0)
    Kd = oracle.dequantize(*oracle.quantize(kf, 0, 0), kf.shape, 0, 0)
    Oe, _ = oracle.fwd(Qd, Kd, vf, causal=True, rows=rows, mode=1)
    e8 = np.linalg.norm(o8.reshape(-1, 128)[rows] - Oe) / np.linalg.norm(Oe)
    e4 = np.linalg.norm(o4.float().cpu().numpy().reshape(-1, 128)[rows] - Oe) / np.linalg.norm(Oe)
    assert e8 < e4 / 2, (e8, e4)
