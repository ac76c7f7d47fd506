"""The BF16 reference forward vs unquantized FP64 attention.

Tolerance derived from the arithmetic: Q, K, V are bf16 (exact inputs); the
only rounding is P -> bf16 for the P V product (relative <= 2^-9 per
element, independent signs) plus FP32 accumulation, so O's relative L2 error
is about 2^-9/sqrt(3) ~ 1.1e-3; the bar is 3e-3 with FP32 output.
"""
import numpy as np
import pytest

import oracle
from gpu_util import assert_close, require_gpu
from precision_attention_fa4fp4_gb300.inputs import FWD_4K, SWEEP, TINY, TRAIN_8B, VIDEO_DIT, Workload, make_inputs, sample_rows

pytestmark = pytest.mark.gpu
TOL = 3e-3


def check(w, rows=None, seed=0):
    fa = require_gpu()
    q, k, v = make_inputs(w, seed=seed)
    o, lse = fa.bf16_fwd(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, out_dtype=fa.OUT_F32)
    fa.sync_status()
    rows = np.arange(w.B * w.Hq * w.N) if rows is None else np.asarray(rows)
    qf, kf, vf = (t.float().numpy() for t in (q, k, v))
    Oo = oracle.attention_fp64(qf, kf, vf, causal=w.causal, rows=rows)
    _, Le = oracle.fwd(qf, kf, vf, causal=w.causal, mode=1, rows=rows)
    assert_close(o.cpu().numpy().reshape(-1, w.d)[rows], Oo, w.name, rel=TOL)
    assert np.max(np.abs(lse.cpu().numpy().reshape(-1)[rows] - Le)) < 1e-3


def test_tiny():
    check(TINY)


@pytest.mark.parametrize("N", [1, 129, 300])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged(N, d, causal):
    check(Workload(f"bf16_n{N}_d{d}", 1, 4, 2, N, d, causal=causal), seed=N)


def test_4k_sampled():
    check(FWD_4K, rows=sample_rows(FWD_4K, tiles_per_head=3, heads=[0, 33]))


def test_train_causal_gqa_sampled():
    check(TRAIN_8B, rows=sample_rows(TRAIN_8B, tiles_per_head=3, heads=[5]))


def test_video_dit_sampled():
    """Outlier channels (logit std ~11): peaked rows, ragged N = 32760."""
    check(VIDEO_DIT, rows=sample_rows(VIDEO_DIT, tiles_per_head=3, heads=[0, 23]))


@pytest.mark.parametrize("w", [SWEEP[0], SWEEP[5], SWEEP[11]], ids=lambda w: w.name)
def test_sweep_points_sampled(w):
    check(w, rows=sample_rows(w, tiles_per_head=2, heads=[w.B * w.Hq - 1]))


@pytest.mark.parametrize("B,Hq,Hkv", [(2, 3, 3), (1, 8, 1), (2, 6, 2)], ids=["mha", "mqa", "gqa3"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [257, 300])
def test_head_groupings(B, Hq, Hkv, causal, N):
    """kv head = h / (Hq / Hkv) across batches; N = 257 and 300 leave the last
    pair of query tiles with one partial tile (the other past N)."""
    check(Workload(f"bf16_heads_b{B}_hq{Hq}_hkv{Hkv}_n{N}", B, Hq, Hkv, N, 128, causal=causal),
          seed=B * 100 + Hq * 10 + Hkv + N)
