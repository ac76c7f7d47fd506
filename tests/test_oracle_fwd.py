"""Pins of the oracle's tiled forward (Methodology 1 of the technical summary
of "Hardware-Aware FP4 FlashAttention-4").

mode 1 (exact exponentials, identity quantizers) is pinned to brute-force
softmax attention in numpy; mode 0 (Direct-P) to closed-form limits and
invariants that hold for the method exactly.
"""
import numpy as np
import pytest
import torch

import oracle


def brute_softmax_attention(Q, K, V, scale, causal):
    """Textbook softmax(scale*QK^T)V in FP64, K/V heads repeated for GQA."""
    B, Hq, N, d = Q.shape
    rep = Hq // K.shape[1]
    K = np.repeat(K.astype(np.float64), rep, axis=1)
    V = np.repeat(V.astype(np.float64), rep, axis=1)
    S = scale * np.einsum("bhid,bhjd->bhij", Q.astype(np.float64), K)
    if causal:
        S = np.where(np.tril(np.ones((N, N), bool)), S, -np.inf)
    mx = S.max(-1, keepdims=True)
    P = np.exp(S - mx)
    l = P.sum(-1, keepdims=True)
    return np.einsum("bhij,bhjd->bhid", P / l, V), (mx + np.log(l))[..., 0]


def rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("N", [1, 5, 127, 128, 129, 300])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2)])
def test_mode1_equals_brute_force(N, causal, Hq, Hkv):
    d = 64
    Q, K, V = rand((1, Hq, N, d), 1), rand((1, Hkv, N, d), 2), rand((1, Hkv, N, d), 3)
    O, L = oracle.fwd(Q, K, V, causal=causal, mode=1)
    Ob, Lb = brute_softmax_attention(Q, K, V, 1 / np.sqrt(d), causal)
    np.testing.assert_allclose(O, Ob.reshape(-1, d), rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Lb.reshape(-1), rtol=0, atol=1e-12)


def quantized_inputs(Q, K, V):
    shp_q, shp_k = Q.shape, K.shape
    qc, qs = oracle.quantize(Q, 0, oracle.ALONG_D)
    kc, ks = oracle.quantize(K, 0, oracle.ALONG_D)
    vc, vs = oracle.quantize(V, 0, oracle.ALONG_N)
    return (oracle.dequantize(qc, qs, shp_q, 0, oracle.ALONG_D),
            oracle.dequantize(kc, ks, shp_k, 0, oracle.ALONG_D),
            oracle.dequantize(vc, vs, shp_k, 0, oracle.ALONG_N))


def test_hard_attention_limit_and_ties():
    """If each row's max score beats every other by more than ln(24)/scale
    (and the max sits in the first key tile), every other key gets code 0 and
    O_i is exactly the argmax key's V row; two tied maxima give their mean."""
    d, N = 64, 300
    rng = np.random.default_rng(0)
    K = np.zeros((1, 1, N, d), np.float32)
    K[0, 0] = np.sign(rng.standard_normal((N, d))) * 0.5        # E2M1-exact entries
    Q = np.zeros((1, 1, 64, d), np.float32)
    targets = rng.integers(0, 128, 64)
    Q[0, 0] = 4.0 * K[0, 0, targets]                            # q.k_target = 4*d*0.25 = 64
    V = rand((1, 1, N, d), 9)
    Qd, Kd, Vd = quantized_inputs(np.concatenate([Q, np.zeros((1, 1, N - 64, d), np.float32)], 2), K, V)
    scale = 1 / np.sqrt(d)
    S = Qd[0, 0, :64] @ Kd[0, 0].T
    top2 = np.sort(S, axis=1)[:, -2:]
    assert np.all(scale * (top2[:, 1] - top2[:, 0]) > np.log(24) + 0.01)
    O, _ = oracle.fwd(Qd, Kd, Vd, rows=np.arange(64))
    assert np.array_equal(O, Vd[0, 0, targets].astype(np.float64))
    # tie: duplicate the target key of row 0 into key 7 (tile 0)
    K2 = Kd.copy()
    K2[0, 0, 7] = K2[0, 0, targets[0]]
    if targets[0] != 7:
        O2, _ = oracle.fwd(Qd, K2, Vd, rows=np.arange(1))
        want = (Vd[0, 0, targets[0]].astype(np.float64) + Vd[0, 0, 7]) / 2
        np.testing.assert_allclose(O2[0], want, rtol=0, atol=1e-15)


def test_permutation_within_tile_invariance():
    d, N = 64, 300
    Qd, Kd, Vd = quantized_inputs(rand((1, 2, N, d), 4), rand((1, 2, N, d), 5), rand((1, 2, N, d), 6))
    O, L = oracle.fwd(Qd, Kd, Vd)
    rng = np.random.default_rng(1)
    perm = np.concatenate([rng.permutation(np.arange(t, min(N, t + 128))) for t in range(0, N, 128)])
    Op, Lp = oracle.fwd(Qd, Kd[:, :, perm], Vd[:, :, perm])
    np.testing.assert_allclose(Op, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lp, L, rtol=0, atol=1e-12)


def test_any_permutation_when_max_in_first_tile():
    """With Q >= 0 and a dominant positive key 0, every row's max is in tile 0,
    every code is taken against the final max, and key order is irrelevant."""
    d, N = 64, 384
    rng = np.random.default_rng(2)
    Q = np.abs(rand((1, 1, N, d), 7))
    K = rand((1, 1, N, d), 8) * 0.25
    K[0, 0, 0] = 2.0
    Qd, Kd, Vd = quantized_inputs(Q, K, rand((1, 1, N, d), 9))
    O, L = oracle.fwd(Qd, Kd, Vd)
    perm = np.concatenate([[0], 1 + rng.permutation(N - 1)])
    Op, Lp = oracle.fwd(Qd, Kd[:, :, perm], Vd[:, :, perm])
    np.testing.assert_allclose(Op, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lp, L, rtol=0, atol=1e-12)
    # and the tiled result equals Direct-P against the global max (brute force)
    c = np.float32(np.float32(1 / np.sqrt(d)) * np.float32(np.log2(np.e)))
    S = (Qd[0, 0].astype(np.float64) @ Kd[0, 0].T.astype(np.float64)).astype(np.float32)
    m = S.max(1, keepdims=True)
    codes = np.array([[oracle.directp_code(float(s), float(mm), float(c)) for s in row]
                      for row, mm in zip(S[:8], m[:8, 0])])
    vals = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])[codes]
    want = vals @ Vd[0, 0].astype(np.float64) / vals.sum(1, keepdims=True)
    np.testing.assert_allclose(O[:8], want, rtol=0, atol=1e-12)


def test_constant_v():
    d, N = 64, 300
    v = np.array([0.5, -1.0, 3.0, 0.0] * (d // 4), np.float32)
    V = np.broadcast_to(v, (1, 2, N, d)).copy()
    Qd, Kd, Vd = quantized_inputs(rand((1, 2, N, d), 10, 2.0), rand((1, 2, N, d), 11, 2.0), V)
    assert np.array_equal(Vd[0, 0, 0], v)
    O, L = oracle.fwd(Qd, Kd, Vd)
    np.testing.assert_allclose(O, np.broadcast_to(v, O.shape), rtol=0, atol=1e-6)
    # l >= 6 (the running max's key carries code 7) -> LSE >= scale * max s
    S = np.einsum("bhid,bhjd->bhij", Qd.astype(np.float64), Kd.astype(np.float64))
    assert np.all(L >= (S.max(-1).reshape(-1) / np.sqrt(d)) - 1e-9)


@pytest.mark.parametrize("mode", [0, 2])
def test_causal_first_row_and_future_independence(mode):
    d, N = 64, 260
    Qd, Kd, Vd = quantized_inputs(rand((1, 1, N, d), 12), rand((1, 1, N, d), 13), rand((1, 1, N, d), 14))
    O, _ = oracle.fwd(Qd, Kd, Vd, causal=True, mode=mode)
    assert np.array_equal(O[0], Vd[0, 0, 0].astype(np.float64))
    i = 140
    K2, V2 = Kd.copy(), Vd.copy()
    K2[:, :, i + 1:] = rand((1, 1, N - i - 1, d), 15)
    V2[:, :, i + 1:] = rand((1, 1, N - i - 1, d), 16)
    O2, _ = oracle.fwd(Qd, K2, V2, causal=True, rows=np.arange(i + 1), mode=mode)
    assert np.array_equal(O2, O[: i + 1])


@pytest.mark.parametrize("mode", [0, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_repeated_mha(causal, mode):
    d, N = 64, 200
    Qd, Kd, Vd = quantized_inputs(rand((2, 4, N, d), 17), rand((2, 2, N, d), 18), rand((2, 2, N, d), 19))
    O, L = oracle.fwd(Qd, Kd, Vd, causal=causal, mode=mode)
    Om, Lm = oracle.fwd(Qd, np.repeat(Kd, 2, 1), np.repeat(Vd, 2, 1), causal=causal, mode=mode)
    assert np.array_equal(O, Om) and np.array_equal(L, Lm)


def test_directp_close_to_softmax():
    """Direct-P is an approximation of softmax: its LSE is within the E2M1
    quantization error of the exact one (which also pins the l/6 factor), and
    its output stays well correlated with exact attention."""
    d, N = 64, 256
    Q, K, V = rand((1, 2, N, d), 20), rand((1, 2, N, d), 21), rand((1, 2, N, d), 22)
    Qd, Kd, Vd = quantized_inputs(Q, K, V)
    O, L = oracle.fwd(Qd, Kd, Vd)
    O1, L1 = oracle.fwd(Qd, Kd, Vd, mode=1)
    # E2M1 drops keys below 1/24 of the running max, so l/6 under-counts the
    # exact mass a little; a missing or doubled factor 6 would be off by ln 6.
    assert np.max(np.abs(L - L1)) < 0.9 and np.mean(np.abs(L - L1)) < 0.2
    cos = np.sum(O * O1, 1) / np.linalg.norm(O, axis=1) / np.linalg.norm(O1, axis=1)
    assert cos.mean() > 0.9


# ---------------------------------------------------------------------------
# mode 2: the FP8 P/V training route (P through MXFP8 per 32 keys)
# ---------------------------------------------------------------------------

def test_fp8pv_constant_v():
    """The normalizer is summed from the same rounded P the product uses, so a
    constant V row comes back unchanged (a normalizer from the unrounded p
    would scale it by sum(p8)/sum(p))."""
    d, N = 64, 300
    v = np.array([0.5, -1.0, 3.0, 0.0] * (d // 4), np.float32)
    V = np.broadcast_to(v, (1, 2, N, d)).copy()
    Qd, Kd, _ = quantized_inputs(rand((1, 2, N, d), 30, 2.0), rand((1, 2, N, d), 31, 2.0), V)
    O, L = oracle.fwd(Qd, Kd, V, mode=2)
    np.testing.assert_allclose(O, np.broadcast_to(v, O.shape), rtol=0, atol=1e-12)
    # the max key has x = 0, p = 1, exact in E4M3 under its block scale: l >= 1
    S = np.einsum("bhid,bhjd->bhij", Qd.astype(np.float64), Kd.astype(np.float64))
    assert np.all(L >= (S.max(-1).reshape(-1) / np.sqrt(d)) - 1e-9)


def test_fp8pv_equal_scores():
    """q = 0: every score is 0, every p is exactly 1 (exact in E4M3), so O is
    the mean of the V rows and LSE = ln N."""
    d, N = 64, 300
    V = rand((1, 1, N, d), 32)
    O, L = oracle.fwd(np.zeros((1, 1, N, d), np.float32), rand((1, 1, N, d), 33), V, mode=2)
    np.testing.assert_allclose(O, np.broadcast_to(V[0, 0].astype(np.float64).mean(0), O.shape), rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, np.log(N), rtol=0, atol=1e-12)


def test_fp8pv_scale_per_32_keys():
    """Keys 0-31 have p = 1, keys 32-63 have p ~ 2^-25.5 and V ~ 2^25.5, the rest
    p = 0.  With one E8M0 scale per 32 keys the small block keeps its own scale
    and contributes ~1 to O[0] (O ~ 2, as exact softmax); under one scale per
    row it would flush to 0 (O = 1)."""
    d, N, scale = 64, 128, 0.125
    c = np.float32(np.float32(scale) * np.float32(np.log2(np.e)))
    Q = np.zeros((1, 1, N, d), np.float32)
    Q[0, 0, 0, 0] = 1.0
    K = np.zeros((1, 1, N, d), np.float32)
    K[0, 0, 32:64, 0] = np.float32(-25.5 / float(c))
    K[0, 0, 64:, 0] = -1000.0
    V = np.zeros((1, 1, N, d), np.float32)
    V[0, 0, :32, 0] = 1.0
    V[0, 0, 32:64, 0] = np.float32(2.0 ** 25.5)
    O2, _ = oracle.fwd(Q, K, V, softmax_scale=scale, mode=2, rows=np.arange(1))
    O1, _ = oracle.fwd(Q, K, V, softmax_scale=scale, mode=1, rows=np.arange(1))
    assert abs(O1[0, 0] - 2.0) < 1e-5
    assert abs(O2[0, 0] - O1[0, 0]) < 0.05          # E4M3 rounding of 2^8.5 -> 352
    assert abs(O2[0, 0] - 1.0) > 0.9                 # not flushed


def test_fp8pv_block_max_above_1_75_not_saturated():
    """Keys 0-31 have p = 1 (the max, V = 0), keys 32-63 p ~ 0.95 (V = 1 in
    channel 0), c = 1.  The second block's maximum has significand 1.9: its
    exponent is the least X with 0.95 <= 448 * 2^X, X = -8, so p scales to
    243.2 and rounds to the E4M3 value 240: O[0] = (240/256) / (1 + 240/256)
    and LSE = ln(32 + 32 * 240/256).  (Under the OCP exponent, X = -9, it
    would saturate to 448/512 = 0.875.)"""
    d, N = 64, 64
    scale = float(np.float32(np.log(2.0)))          # c = fl32(scale * log2 e) = 1
    Q = np.zeros((1, 1, N, d), np.float32)
    Q[0, 0, 0, 0] = 1.0
    K = np.zeros((1, 1, N, d), np.float32)
    K[0, 0, 32:, 0] = np.float32(np.log2(0.95))
    V = np.zeros((1, 1, N, d), np.float32)
    V[0, 0, 32:, 0] = 1.0
    O, L = oracle.fwd(Q, K, V, softmax_scale=scale, mode=2, rows=np.arange(1))
    p8 = 240.0 / 256.0
    assert abs(O[0, 0] - p8 / (1 + p8)) < 1e-12
    np.testing.assert_array_equal(O[0, 1:], 0)
    assert abs(L[0] - np.log(32 + 32 * p8)) < 1e-6


def test_fp8pv_permutation_within_32_key_blocks():
    d, N = 64, 300
    Qd, Kd, Vd = quantized_inputs(rand((1, 2, N, d), 34), rand((1, 2, N, d), 35), rand((1, 2, N, d), 36))
    O, L = oracle.fwd(Qd, Kd, Vd, mode=2)
    rng = np.random.default_rng(3)
    perm = np.concatenate([rng.permutation(np.arange(t, min(N, t + 32))) for t in range(0, N, 32)])
    Op, Lp = oracle.fwd(Qd, Kd[:, :, perm], Vd[:, :, perm], mode=2)
    np.testing.assert_allclose(Op, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lp, L, rtol=0, atol=1e-12)


def test_fp8pv_close_to_softmax():
    """E4M3 P (3 mantissa bits, per-32 scales): close to exact softmax on the
    same dequantized inputs, and closer than the E2M1 Direct-P codes."""
    d, N = 64, 512
    Qd, Kd, Vd = quantized_inputs(rand((1, 2, N, d), 37), rand((1, 2, N, d), 38), rand((1, 2, N, d), 39))
    O1, L1 = oracle.fwd(Qd, Kd, Vd, mode=1)
    O2, L2 = oracle.fwd(Qd, Kd, Vd, mode=2)
    O0, _ = oracle.fwd(Qd, Kd, Vd, mode=0)
    e2 = np.linalg.norm(O2 - O1) / np.linalg.norm(O1)
    e0 = np.linalg.norm(O0 - O1) / np.linalg.norm(O1)
    assert e2 < 0.08 and e2 < e0 / 2
    assert np.max(np.abs(L2 - L1)) < 0.05     # a stray factor (Direct-P's 6) would be ln 6


def test_nvfp4_qk_scores_beat_mxfp4_on_outlier_channels():
    """On the outlier-channel workload's distribution (4 of 128 channels x8 in
    Q and K), NVFP4 Q/K (a scale per 16 plus a tensor scale) give scores
    closer to the bf16 scores than MXFP4 (a power-of-two scale per 32)."""
    from precision_attention_fa4fp4_gb300.inputs import VIDEO_DIT, Workload, make_inputs
    w = Workload("outliers_small", 1, 2, 2, 512, 128, n_outliers=VIDEO_DIT.n_outliers)
    q, k, _ = (t.float().numpy() for t in make_inputs(w))
    S = np.einsum("bhid,bhjd->bhij", q.astype(np.float64), k.astype(np.float64))

    def scores(qd, kd):
        return np.einsum("bhid,bhjd->bhij", qd.astype(np.float64), kd.astype(np.float64))

    mx = scores(oracle.dequantize(*oracle.quantize(q, 0, 0), q.shape, 0, 0),
                oracle.dequantize(*oracle.quantize(k, 0, 0), k.shape, 0, 0))
    cq, sq, tq = oracle.quantize_nvfp4(q)
    ck, sk, tk = oracle.quantize_nvfp4(k)
    nv = scores(oracle.dequantize_nvfp4(cq, sq, tq, q.shape), oracle.dequantize_nvfp4(ck, sk, tk, k.shape))
    e_mx = np.linalg.norm(mx - S) / np.linalg.norm(S)
    e_nv = np.linalg.norm(nv - S) / np.linalg.norm(S)
    assert e_nv < e_mx, (e_nv, e_mx)


@pytest.mark.parametrize("N", [1, 77, 300])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (6, 2)])
def test_attention_fp64_equals_brute_force(N, causal, Hq, Hkv):
    """The unquantized FP64 reference (used for the error report and the BF16
    kernel's parity) is textbook softmax attention: it equals the numpy brute
    force to 1e-12, with the causal mask and GQA head sharing."""
    d = 64
    Q, K, V = rand((2, Hq, N, d), 41, 2.0), rand((2, Hkv, N, d), 42, 2.0), rand((2, Hkv, N, d), 43)
    O = oracle.attention_fp64(Q, K, V, causal=causal)
    Ob, _ = brute_softmax_attention(Q, K, V, 1 / np.sqrt(d), causal)
    np.testing.assert_allclose(O, Ob.reshape(-1, d), rtol=0, atol=1e-12)
    # an explicit softmax scale and a row subset
    rows = np.array([0, N - 1, Hq * N + N // 2])
    O2 = oracle.attention_fp64(Q, K, V, softmax_scale=0.3, causal=causal, rows=rows)
    Ob2, _ = brute_softmax_attention(Q, K, V, np.float32(0.3), causal)
    np.testing.assert_allclose(O2, Ob2.reshape(-1, d)[rows], rtol=0, atol=1e-12)


@pytest.mark.parametrize("mode", [0, 2])
@pytest.mark.parametrize("N,d,causal,outliers", [(300, 64, True, 0), (1000, 128, False, 0), (700, 128, False, 4)])
def test_nvfp4_folded_tensor_scales_match_plain_definition(N, d, causal, outliers, mode):
    """NVFP4 Q/K by the plain definition: s = fl32(deq(Q).deq(K)) with the
    FP32 tensor scales inside deq, softmax scale 1/sqrt(d).  Folding the two
    tensor scales into the softmax scale instead, fl32(fl32(scale*ts_q)*ts_k)
    on scores of the E2M1 x E4M3 values alone, moves the scores by FP32
    rounding only; O and LSE stay within the parity bar (rel-L2 1e-3,
    max-abs 1e-2, LSE 1e-3) of the plain form, for Direct-P and the FP8 P/V
    route."""
    from precision_attention_fa4fp4_gb300.inputs import Workload, make_inputs
    w = Workload("nv_fold", 1, 4, 2, N, d, causal=causal, n_outliers=outliers)
    q, k, v = (t.float().numpy() for t in make_inputs(w, seed=5))
    cq, sq, tq = oracle.quantize_nvfp4(q)
    ck, sk, tk = oracle.quantize_nvfp4(k)
    fmt = 1 if mode == 2 else 0
    Vd = oracle.dequantize(*oracle.quantize(v, fmt, 1), v.shape, fmt, 1)
    # plain definition
    Qt, Kt = oracle.dequantize_nvfp4(cq, sq, tq, q.shape), oracle.dequantize_nvfp4(ck, sk, tk, k.shape)
    Op, Lp = oracle.fwd(Qt, Kt, Vd, causal=causal, mode=mode)
    # folded form
    Qu, Ku = oracle.dequantize_nvfp4(cq, sq, 1.0, q.shape), oracle.dequantize_nvfp4(ck, sk, 1.0, k.shape)
    s0 = np.float32(1 / np.sqrt(d))
    folded = np.float32(np.float32(s0 * np.float32(tq)) * np.float32(tk))
    Of, Lf = oracle.fwd(Qu, Ku, Vd, softmax_scale=float(folded), causal=causal, mode=mode)
    rel = np.linalg.norm(Of - Op) / np.linalg.norm(Op)
    assert rel <= 1e-3 and np.max(np.abs(Of - Op)) <= 1e-2 and np.max(np.abs(Lf - Lp)) <= 1e-3
    # the tensor scales are really inside the plain scores (a dropped ts would
    # shift every LSE by orders of magnitude of the logit scale)
    Ox, Lx = oracle.fwd(Qu, Ku, Vd, causal=causal, mode=mode)
    assert np.max(np.abs(Lx - Lp)) > 0.05
