"""Direct-P FP4 forward on the GPU vs the oracle on the same seeded inputs.

Tolerance: rel-L2 <= 1e-3 and max-abs <= 1e-2 on O after
the oracle's O is rounded to the kernel's output dtype; LSE to 1e-3 absolute.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, require_gpu, round_like
from precision_attention_fa4fp4_gb300.inputs import (FWD_4K, SWEEP, TINY, TRAIN_8B, VIDEO_DIT,
                                                     Workload, make_inputs, sample_rows)

pytestmark = pytest.mark.gpu


def oracle_operands(q, k, v):
    qf, kf, vf = (t.float().numpy() for t in (q, k, v))
    Qd = oracle.dequantize(*oracle.quantize(qf, 0, 0), qf.shape, 0, 0)
    Kd = oracle.dequantize(*oracle.quantize(kf, 0, 0), kf.shape, 0, 0)
    Vd = oracle.dequantize(*oracle.quantize(vf, 0, 1), vf.shape, 0, 1)
    return Qd, Kd, Vd


def gpu_fwd(fa, q, k, v, causal, out_bf16):
    q4, k4 = fa.quantize(q.cuda()), fa.quantize(k.cuda())
    vt = fa.quantize(v.cuda(), fa.FMT_MXFP4, fa.ALONG_N)
    o, lse = fa.fwd(q4, k4, vt, causal=causal, out_dtype=fa.OUT_BF16 if out_bf16 else fa.OUT_F32)
    fa.sync_status()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check(w: Workload, out_bf16=True, rows=None, seed=0):
    fa = require_gpu()
    q, k, v = make_inputs(w, seed=seed)
    o, lse = gpu_fwd(fa, q, k, v, w.causal, out_bf16)
    Qd, Kd, Vd = oracle_operands(q, k, v)
    rows = np.arange(w.B * w.Hq * w.N) if rows is None else np.asarray(rows)
    Oo, Lo = oracle.fwd(Qd, Kd, Vd, causal=w.causal, rows=rows)
    d = w.d
    assert_close(o.reshape(-1, d)[rows], round_like(Oo, out_bf16), w.name + " O")
    assert np.max(np.abs(lse.reshape(-1)[rows] - Lo)) < 1e-3, w.name + " LSE"


@pytest.mark.parametrize("out_bf16", [True, False])
def test_tiny(out_bf16):
    check(TINY, out_bf16)


@pytest.mark.parametrize("N", [1, 33, 127, 128, 129, 300, 1000])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged(N, d, causal):
    check(Workload(f"ragged_n{N}_d{d}", 1, 4, 2, N, d, causal=causal), out_bf16=False, seed=N)


@pytest.mark.parametrize("B,Hq,Hkv", [(2, 3, 3), (1, 8, 1), (2, 6, 2)], ids=["mha", "mqa", "gqa3"])
@pytest.mark.parametrize("causal", [False, True])
def test_head_groupings(B, Hq, Hkv, causal):
    """kv head = h / (Hq / Hkv) for MHA, MQA and groups of three, across batches."""
    check(Workload(f"heads_b{B}_hq{Hq}_hkv{Hkv}", B, Hq, Hkv, 300, 128, causal=causal), out_bf16=True,
          seed=B * 100 + Hq * 10 + Hkv)


def test_noncausal_4k_sampled():
    check(FWD_4K, True, rows=sample_rows(FWD_4K, tiles_per_head=3, heads=range(0, 64, 9)))


def test_video_dit_sampled():
    # FP32 output: with outlier channels |O| reaches [2,4), where one bf16 ulp
    # (0.0156) alone exceeds the 1e-2 max-abs bar.
    check(VIDEO_DIT, False, rows=sample_rows(VIDEO_DIT, tiles_per_head=4, heads=[0, 23]))


def check_heads(w: Workload, bh_list, tiles_per_head=3, out_bf16=True, seed=0):
    """The GPU runs the whole problem; the oracle quantizes and runs only the
    sampled (batch, head) pairs of an MHA workload (heads are independent
    problems), on `tiles_per_head` query tiles of each, first and last
    included."""
    assert w.Hq == w.Hkv
    fa = require_gpu()
    q, k, v = make_inputs(w, seed=seed)
    o, lse = gpu_fwd(fa, q, k, v, w.causal, out_bf16)
    sel = lambda t: t.reshape(w.B * w.Hq, w.N, w.d)[bh_list].reshape(1, len(bh_list), w.N, w.d)
    Qd, Kd, Vd = oracle_operands(sel(q), sel(k), sel(v))
    sub = Workload(w.name + "_heads", 1, len(bh_list), len(bh_list), w.N, w.d, causal=w.causal)
    rows = sample_rows(sub, tiles_per_head=tiles_per_head).numpy()
    Oo, Lo = oracle.fwd(Qd, Kd, Vd, causal=w.causal, rows=rows)
    full = np.asarray(bh_list)[rows // w.N] * w.N + rows % w.N
    assert_close(o.reshape(-1, w.d)[full], round_like(Oo, out_bf16), w.name + " O")
    assert np.max(np.abs(lse.reshape(-1)[full] - Lo)) < 1e-3, w.name + " LSE"


@pytest.mark.parametrize("w", [SWEEP[0], SWEEP[6 + 3]], ids=lambda w: w.name)
def test_sweep_points_sampled(w):
    check(w, True, rows=sample_rows(w, tiles_per_head=3, heads=[0, w.B * w.Hq - 1]))


@pytest.mark.parametrize("w", [SWEEP[2], SWEEP[3], SWEEP[4], SWEEP[5], SWEEP[11]], ids=lambda w: w.name)
def test_sweep_long_points_sampled(w):
    """d = 64 from N = 4096 up, and both N = 32768 points (256 key tiles: the
    longest chains of running-max rescales), in the sweep's launch shape."""
    check_heads(w, [0, w.B * w.Hq - 1], tiles_per_head=3)


def test_train_causal_gqa_sampled():
    check(TRAIN_8B, False, rows=sample_rows(TRAIN_8B, tiles_per_head=3, heads=[0, 37]))
