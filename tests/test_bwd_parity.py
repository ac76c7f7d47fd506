"""Quantized backward on the GPU vs the oracle on the same inputs.

Both sides take the same backward inputs: the seeded Q, K, V, dO (each side
makes its own MXFP4/MXFP8 views, bit-identical), and O and LSE as the GPU
forward wrote them (the forward is checked against the oracle on its own), so
the comparison sees the backward's arithmetic alone.  Tolerance: rel-L2 <=
1e-3 and max-abs <= 1e-2 on dQ, dK, dV (FP32).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, require_gpu
from precision_attention_fa4fp4_gb300.inputs import TRAIN_8B, Workload, extreme_logit_inputs, make_inputs

pytestmark = pytest.mark.gpu


def gpu_grads(fa, q, k, v, do, causal, o_bf16=False):
    """GPU forward + backward; returns (dq, dk, dv, O as the backward read it,
    LSE) as float arrays."""
    q, k, v, do = (t.cuda() for t in (q, k, v, do))
    q4, k4 = fa.quantize(q), fa.quantize(k)
    vt = fa.quantize(v, fa.FMT_MXFP4, fa.ALONG_N)
    q8c = fa.quantize(q, fa.FMT_MXFP8, fa.ALONG_N)
    k8c = fa.quantize(k, fa.FMT_MXFP8, fa.ALONG_N)
    v8r = fa.quantize(v, fa.FMT_MXFP8, fa.ALONG_D)
    o, lse = fa.fwd(q4, k4, vt, causal=causal, out_dtype=fa.OUT_BF16 if o_bf16 else fa.OUT_F32)
    dq, dk, dv = fa.bwd(q4, k4, q8c, k8c, v8r, o, do, lse, causal=causal)
    fa.sync_status()
    return (dq.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy(), o.float().cpu().numpy(),
            lse.cpu().numpy())


def oracle_views(q, k, v):
    qf, kf, vf = (t.float().numpy() for t in (q, k, v))
    Q4 = oracle.dequantize(*oracle.quantize(qf, 0, 0), qf.shape, 0, 0)
    K4 = oracle.dequantize(*oracle.quantize(kf, 0, 0), kf.shape, 0, 0)
    V4 = oracle.dequantize(*oracle.quantize(vf, 0, 1), vf.shape, 0, 1)
    Q8 = oracle.dequantize(*oracle.quantize(qf, 1, 1), qf.shape, 1, 1)
    K8 = oracle.dequantize(*oracle.quantize(kf, 1, 1), kf.shape, 1, 1)
    V8 = oracle.dequantize(*oracle.quantize(vf, 1, 0), vf.shape, 1, 0)
    return Q4, K4, V4, Q8, K8, V8


def check(w: Workload, qrows=None, krows=None, seed=0, o_bf16=False):
    fa = require_gpu()
    q, k, v, do = make_inputs(w, seed=seed, with_dout=True)
    dq, dk, dv, O, L = gpu_grads(fa, q, k, v, do, w.causal, o_bf16)
    Q4, K4, V4, Q8, K8, V8 = oracle_views(q, k, v)
    dQ, dK, dV = oracle.bwd(Q4, K4, Q8, K8, V8, O, do.float().numpy(), L, causal=w.causal,
                            qrows=qrows, krows=krows)
    qsel = np.arange(w.B * w.Hq * w.N) if qrows is None else np.asarray(qrows)
    ksel = np.arange(w.B * w.Hkv * w.N) if krows is None else np.asarray(krows)
    assert_close(dq.reshape(-1, w.d)[qsel], dQ, w.name + " dQ")
    assert_close(dk.reshape(-1, w.d)[ksel], dK, w.name + " dK")
    assert_close(dv.reshape(-1, w.d)[ksel], dV, w.name + " dV")


@pytest.mark.parametrize("N", [64, 200, 300])
@pytest.mark.parametrize("causal", [True, False])
def test_small(N, causal):
    check(Workload(f"bwd_n{N}", 1, 4, 2, N, 128, causal=causal, qk_std=128 ** -0.25), seed=N)


@pytest.mark.parametrize("N", [1, 64, 129, 300, 1000])
@pytest.mark.parametrize("causal", [True, False])
def test_d64(N, causal):
    """Head dimension 64: GQA groups of two, ragged N (one key, partial key
    tiles, partial 64-query steps)."""
    check(Workload(f"bwd_d64_n{N}", 1, 4, 2, N, 64, causal=causal, qk_std=64 ** -0.25), seed=N + 64)


def test_d64_mqa_two_batches_bf16_o():
    check(Workload("bwd_d64_b2_mqa_n257", 2, 4, 1, 257, 64, causal=True, qk_std=64 ** -0.25), seed=5,
          o_bf16=True)


def test_train_causal_gqa_sampled():
    """Causal GQA training shape: the kv head (b=1, hk=5) in full for dK/dV on
    its first and last key tiles, dQ on two query tiles of its first head."""
    w = TRAIN_8B
    b, hk = 1, 5
    heads = [b * w.Hq + hk * 4 + u for u in range(4)]
    kbase = (b * w.Hkv + hk) * w.N
    krows = np.concatenate([kbase + np.arange(0, 128), kbase + np.arange(w.N - 128, w.N)])
    qbase = heads[0] * w.N
    qrows = np.concatenate([qbase + np.arange(0, 128), qbase + np.arange(4096, 4224)])
    check(w, qrows=qrows, krows=krows)


def test_train_causal_gqa_sampled_middle_tile_other_batch():
    """The same shape on batch 0, kv head 2: dK/dV on a middle key tile (keys
    4096-4223, half the queries above the diagonal), dQ on a middle and the
    last query tile of the group's third query head."""
    w = TRAIN_8B
    b, hk = 0, 2
    heads = [b * w.Hq + hk * 4 + u for u in range(4)]
    kbase = (b * w.Hkv + hk) * w.N
    krows = kbase + np.arange(4096, 4224)
    qbase = heads[2] * w.N
    qrows = np.concatenate([qbase + np.arange(2560, 2688), qbase + np.arange(w.N - 128, w.N)])
    check(w, qrows=qrows, krows=krows)


def test_causal_gqa_partial_cta_group():
    """Six (batch, kv head) pairs: the causal backward orders its CTAs in groups
    of four pairs, so the last group holds two; ragged N (three key tiles)."""
    check(Workload("bwd_b2_hq6_hkv3_n300", 2, 6, 3, 300, 128, causal=True, qk_std=128 ** -0.25), seed=7)


@pytest.mark.parametrize("causal", [True, False])
def test_o_in_bf16(causal):
    """O handed to the backward in bf16 (the preprocess widens it for D)."""
    check(Workload("bwd_bf16o_n300", 1, 4, 2, 300, 128, causal=causal, qk_std=128 ** -0.25), seed=11,
          o_bf16=True)


def test_mqa_causal():
    """One kv head shared by eight query heads: dK and dV sum over all eight."""
    check(Workload("bwd_mqa_n200", 1, 8, 1, 200, 128, causal=True, qk_std=128 ** -0.25), seed=13)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("qk_std", [1.0, 0.5])
def test_unit_std_qk(d, qk_std):
    """Q and K drawn with a larger spread than the training workload's
    (logits of std ~1 after scaling): more peaked rows, a wider range of P
    and dS inside each MXFP8 block."""
    check(Workload(f"bwd_std{qk_std}_d{d}", 1, 4, 2, 200, d, causal=True, qk_std=qk_std), seed=0)


@pytest.mark.parametrize("causal", [True, False])
def test_extreme_logits(causal):
    """Scaled logits of several hundred (LSE > 500): the score accumulators
    start at -LSE log2 e / c of magnitude ~10^4, so their sums cancel to the
    offset that P is taken from; the gradients must still match the oracle."""
    fa = require_gpu()
    q, k, v = extreme_logit_inputs()
    g = torch.Generator().manual_seed(17)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    dq, dk, dv, O, L = gpu_grads(fa, q, k, v, do, causal)
    assert np.max(L) > 500
    Q4, K4, V4, Q8, K8, V8 = oracle_views(q, k, v)
    dQ, dK, dV = oracle.bwd(Q4, K4, Q8, K8, V8, O, do.float().numpy(), L, causal=causal)
    d = q.shape[-1]
    for nm, got, want in (("dQ", dq, dQ), ("dK", dk, dK), ("dV", dv, dV)):
        # K is scaled up to 5x here, so dQ and dK reach ~10^2: the max-abs bar
        # is taken relative to the largest gradient (rel-L2 as everywhere)
        want = want.reshape(-1, d)
        assert_close(got.reshape(-1, d), want, f"extreme logits {nm}",
                     mabs=1e-2 * max(1.0, float(np.max(np.abs(want)))))


@pytest.mark.parametrize("d,N,o_bf16", [(128, 300, False), (64, 129, True), (128, 1, False)])
def test_preprocess_views_match_the_quantizer(d, N, o_bf16):
    """The two MXFP8 views of dO that the backward's preprocess leaves in its
    workspace are byte for byte what the quantizer gives for blocks along d
    and along N (padded tokens included)."""
    fa = require_gpu()
    w = Workload(f"prep_d{d}_n{N}", 2, 4, 2, N, d, causal=True, qk_std=d ** -0.25)
    q, k, v, do = (t.cuda() for t in make_inputs(w, seed=N + d, with_dout=True))
    q4, k4 = fa.quantize(q), fa.quantize(k)
    vt = fa.quantize(v, fa.FMT_MXFP4, fa.ALONG_N)
    q8c, k8c = fa.quantize(q, fa.FMT_MXFP8, fa.ALONG_N), fa.quantize(k, fa.FMT_MXFP8, fa.ALONG_N)
    v8r = fa.quantize(v, fa.FMT_MXFP8, fa.ALONG_D)
    o, lse = fa.fwd(q4, k4, vt, causal=True, out_dtype=fa.OUT_BF16 if o_bf16 else fa.OUT_F32)
    ws = torch.zeros(fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, N, d), dtype=torch.uint8, device="cuda")
    fa.bwd(q4, k4, q8c, k8c, v8r, o, do, lse, causal=True, workspace=ws)
    torch.cuda.synchronize()
    fa.sync_status()
    row = fa.quantize(do, fa.FMT_MXFP8, fa.ALONG_D)
    col = fa.quantize(do, fa.FMT_MXFP8, fa.ALONG_N)
    up = lambda x: (x + 255) // 256 * 256
    off = 0
    for t in (row.codes, row.scales, col.codes, col.scales):
        n = t.numel()
        assert torch.equal(ws[off:off + n], t.reshape(-1).view(torch.uint8)), f"view piece at {off}"
        off += up(n)
