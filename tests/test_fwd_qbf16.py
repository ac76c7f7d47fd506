"""The forward with bf16 Q quantized in its prologue (fa4fp4_fwd_qbf16) and
the K/V-only quantize launch (fa4fp4_quantize_kv).

The prologue quantizes Q with the same block routine as fa4fp4_quantize, so
the result must equal, bit for bit, fa4fp4_quantize of Q followed by
fa4fp4_fwd (or fa4fp4_fwd_fp8pv); on the 4K workload it is also checked
against the oracle like the other forwards (rel-L2 <= 1e-3, max-abs <= 1e-2
after rounding the oracle to bf16, LSE to 1e-3)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, require_gpu, round_like
from precision_attention_fa4fp4_gb300.inputs import FWD_4K, TRAIN_8B, Workload, make_inputs, sample_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fp8pv", [False, True])
@pytest.mark.parametrize("N,d,causal,Hq,Hkv", [(1, 64, False, 2, 2), (129, 128, True, 4, 2), (300, 64, True, 6, 2),
                                               (1000, 128, False, 8, 1), (256, 128, True, 2, 2)])
def test_bit_identical_to_quantize_then_fwd(N, d, causal, Hq, Hkv, fp8pv):
    fa = require_gpu()
    w = Workload(f"qbf16_n{N}_d{d}", 2, Hq, Hkv, N, d, causal=causal)
    q, k, v = (t.cuda() for t in make_inputs(w, seed=N + d))
    k4 = fa.quantize(k)
    vt = fa.quantize(v, fa.FMT_MXFP8 if fp8pv else fa.FMT_MXFP4, fa.ALONG_N)
    for out_dtype in (fa.OUT_F32, fa.OUT_BF16):
        o1, l1 = fa.fwd_qbf16(q, k4, vt, causal=causal, out_dtype=out_dtype)
        q4 = fa.quantize(q)
        f = fa.fwd_fp8pv if fp8pv else fa.fwd
        o2, l2 = f(q4, k4, vt, causal=causal, out_dtype=out_dtype)
        fa.sync_status()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("N,d", [(1, 64), (300, 128), (1000, 64)])
def test_quantize_kv_bytes(N, d):
    fa = require_gpu()
    _, k, v = (t.cuda() for t in make_inputs(Workload("kv", 2, 2, 3, N, d), seed=N))
    k4, vt = fa.quantize_kv(k, v)
    k4r, vtr = fa.quantize(k), fa.quantize(v, fa.FMT_MXFP4, fa.ALONG_N)
    fa.sync_status()
    for a, b in ((k4.codes, k4r.codes), (k4.scales, k4r.scales), (vt.codes, vtr.codes), (vt.scales, vtr.scales)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("w", [FWD_4K, TRAIN_8B], ids=lambda w: w.name)
def test_full_size_against_the_oracle(w):
    fa = require_gpu()
    q, k, v = make_inputs(w, seed=0)
    k4, vt = fa.quantize_kv(k.cuda(), v.cuda())
    o, lse = fa.fwd_qbf16(q.cuda(), k4, vt, causal=w.causal, out_dtype=fa.OUT_BF16)
    fa.sync_status()
    rows = sample_rows(w, tiles_per_head=2, heads=[0, w.B * w.Hq - 1]).numpy()
    qf, kf, vf = (t.float().numpy() for t in (q, k, v))
    Qd = oracle.dequantize(*oracle.quantize(qf, 0, 0), qf.shape, 0, 0)
    Kd = oracle.dequantize(*oracle.quantize(kf, 0, 0), kf.shape, 0, 0)
    Vd = oracle.dequantize(*oracle.quantize(vf, 0, 1), vf.shape, 0, 1)
    Oo, Lo = oracle.fwd(Qd, Kd, Vd, causal=w.causal, rows=rows)
    assert_close(o.float().cpu().numpy().reshape(-1, w.d)[rows], round_like(Oo, True), w.name + " O")
    assert np.max(np.abs(lse.cpu().numpy().reshape(-1)[rows] - Lo)) < 1e-3
