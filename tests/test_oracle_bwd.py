"""Pins of the oracle's backward (Methodology 2, "Quantized Causal Backward",
of the technical summary of "Hardware-Aware FP4 FlashAttention-4"; FP8
gradient operands per the arXiv abstract).

mode 1 (identity quantizers) is pinned to the analytic gradient of softmax
attention and to central finite differences of the brute-force forward;
mode 0 is pinned by the GQA group-sum identity and by the FP8 error bound on
inputs whose own views are exactly representable.
"""
import numpy as np
import pytest

import oracle
from test_oracle_fwd import brute_softmax_attention, rand


def analytic_grads(Q, K, V, dO, scale, causal):
    B, Hq, N, d = Q.shape
    rep = Hq // K.shape[1]
    Kr = np.repeat(K.astype(np.float64), rep, 1)
    Vr = np.repeat(V.astype(np.float64), rep, 1)
    Q = Q.astype(np.float64)
    dO = dO.astype(np.float64)
    S = scale * np.einsum("bhid,bhjd->bhij", Q, Kr)
    if causal:
        S = np.where(np.tril(np.ones((N, N), bool)), S, -np.inf)
    P = np.exp(S - S.max(-1, keepdims=True))
    P /= P.sum(-1, keepdims=True)
    O = P @ Vr
    dV = np.einsum("bhij,bhid->bhjd", P, dO)
    dP = dO @ Vr.transpose(0, 1, 3, 2)
    D = (dO * O).sum(-1, keepdims=True)
    dS = P * (dP - D)
    dQ = scale * dS @ Kr
    dK = scale * np.einsum("bhij,bhid->bhjd", dS, Q)
    sh = (B, K.shape[1], rep, N, d)
    return dQ, dK.reshape(sh).sum(2), dV.reshape(sh).sum(2)


def run_mode1(Q, K, V, dO, causal):
    d = Q.shape[-1]
    O, L = brute_softmax_attention(Q, K, V, 1 / np.sqrt(d), causal)
    return oracle.bwd(Q, K, Q, K, V, O.astype(np.float32), dO, L.astype(np.float32),
                      causal=causal, mode=1), O, L


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [33, 130])
def test_mode1_equals_analytic(causal, N):
    d = 32
    Q, K, V, dO = rand((1, 4, N, d), 1), rand((1, 2, N, d), 2), rand((1, 2, N, d), 3), rand((1, 4, N, d), 4)
    # the oracle reads O and LSE as FP32 inputs, so build the reference from
    # the same rounded O (D = rowsum(dO*O))
    (dQ, dK, dV), O, L = run_mode1(Q, K, V, dO, causal)
    aQ, aK, aV = analytic_grads(Q, K, V, dO, 1 / np.sqrt(d), causal)
    tol = 1e-5    # O and LSE pass through FP32 on their way in
    np.testing.assert_allclose(dQ, aQ.reshape(-1, d), atol=tol, rtol=0)
    np.testing.assert_allclose(dK, aK.reshape(-1, d), atol=tol, rtol=0)
    np.testing.assert_allclose(dV, aV.reshape(-1, d), atol=tol, rtol=0)


def test_analytic_matches_finite_differences():
    """Central differences of f = sum(dO * attention(Q,K,V)) in FP64."""
    N, d = 20, 16
    Q, K, V, dO = (rand((1, 2, N, d), s).astype(np.float64) for s in (5, 6, 7, 8))
    K, V = K[:, :1], V[:, :1]
    scale = 1 / np.sqrt(d)
    for causal in (False, True):
        aQ, aK, aV = analytic_grads(Q, K, V, dO, scale, causal)

        def f(Q_, K_, V_):
            return float((brute_softmax_attention(Q_, K_, V_, scale, causal)[0] * dO).sum())
        h = 1e-6
        rng = np.random.default_rng(0)
        for _ in range(12):
            idx = tuple(rng.integers(0, n) for n in (1, 1, N, d))
            for X, G, which in ((Q, aQ, 0), (K, aK, 1), (V, aV, 2)):
                iq = (idx[0], rng.integers(0, X.shape[1]), idx[2], idx[3])
                Xp, Xm = X.copy(), X.copy()
                Xp[iq] += h
                Xm[iq] -= h
                args_p = [Q, K, V]
                args_m = [Q, K, V]
                args_p[which], args_m[which] = Xp, Xm
                fd = (f(*args_p) - f(*args_m)) / (2 * h)
                assert abs(fd - G[iq]) < 1e-7


def quantized_views(Q, K, V, dO):
    """The method's operands: FP4 Q/K (along d), FP8 column views of Q/K (along
    N), FP8 row view of V (along d)."""
    sh_q, sh_k = Q.shape, K.shape
    Q4 = oracle.dequantize(*oracle.quantize(Q, 0, 0), sh_q, 0, 0)
    K4 = oracle.dequantize(*oracle.quantize(K, 0, 0), sh_k, 0, 0)
    Q8 = oracle.dequantize(*oracle.quantize(Q, 1, 1), sh_q, 1, 1)
    K8 = oracle.dequantize(*oracle.quantize(K, 1, 1), sh_k, 1, 1)
    V8 = oracle.dequantize(*oracle.quantize(V, 1, 0), sh_k, 1, 0)
    return Q4, K4, Q8, K8, V8


@pytest.mark.parametrize("causal", [False, True])
def test_mode0_gqa_is_group_sum(causal):
    N, d = 100, 32
    Q, K, V, dO = rand((1, 4, N, d), 9), rand((1, 2, N, d), 10), rand((1, 2, N, d), 11), rand((1, 4, N, d), 12)
    Q4, K4, Q8, K8, V8 = quantized_views(Q, K, V, dO)
    O, L = oracle.fwd(Q4, K4, V8, causal=causal)
    O = O.reshape(Q.shape).astype(np.float32)
    L = L.reshape(Q.shape[:3]).astype(np.float32)
    dQ, dK, dV = oracle.bwd(Q4, K4, Q8, K8, V8, O, dO, L, causal=causal)
    rep = lambda a: np.repeat(a, 2, 1)
    dQm, dKm, dVm = oracle.bwd(Q4, rep(K4), Q8, rep(K8), rep(V8), O, dO, L, causal=causal)
    assert np.array_equal(dQ, dQm)
    dKm = dKm.reshape(1, 2, 2, N, d).sum(2).reshape(-1, d)
    dVm = dVm.reshape(1, 2, 2, N, d).sum(2).reshape(-1, d)
    np.testing.assert_allclose(dK, dKm, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dV, dVm, rtol=0, atol=1e-12)


def e2m1_exact(shape, seed):
    """Entries E2M1 values times one power of two per row of 32: exactly
    representable by every MXFP4 and MXFP8 view."""
    rng = np.random.default_rng(seed)
    mags = np.array([0.5, 1, 1.5, 2, 3, 4, 6])
    return (rng.choice(mags, shape) * rng.choice([-1.0, 1.0], shape) * 0.25).astype(np.float32)


def test_mode0_within_fp8_bound():
    """On inputs whose FP4/FP8 views are exact, mode 0 differs from mode 1
    only by the E4M3 rounding of P, dS and the dO views (half-ulp 2^-4
    relative per element), so the relative L2 gap stays a few percent."""
    N, d = 96, 32
    Q, K = e2m1_exact((1, 2, N, d), 1), e2m1_exact((1, 2, N, d), 2)
    V, dO = e2m1_exact((1, 2, N, d), 3), e2m1_exact((1, 2, N, d), 4)
    Q4, K4, Q8, K8, V8 = quantized_views(Q, K, V, dO)
    assert np.array_equal(Q4, Q) and np.array_equal(Q8, Q) and np.array_equal(V8, V)
    O, L = brute_softmax_attention(Q, K, V, 1 / np.sqrt(d), True)
    O, L = O.astype(np.float32), L.astype(np.float32)
    g0 = oracle.bwd(Q, K, Q, K, V, O, dO, L, causal=True, mode=0)
    g1 = oracle.bwd(Q, K, Q, K, V, O, dO, L, causal=True, mode=1)
    for a, b in zip(g0, g1):
        rel = np.linalg.norm(a - b) / np.linalg.norm(b)
        assert 1e-4 < rel < 0.06


# ---------------------------------------------------------------------------
# The MXFP8 block axes of the quantized backward (Methodology 2, "Gradient
# Formats": row- and column-oriented FP8 views; the block runs along the
# contraction axis of the product each operand feeds).  In every case below
# one operand holds a value 2^-20 of its neighbour along the WRONG axis and
# equal values along the stated one: blocked along the stated axis it is
# exact, blocked along the other it shares an E8M0 scale with a value 2^20
# larger and flushes to zero (E4M3's smallest subnormal is 2^-9 of the
# block's scale, and the scale puts the block maximum in [224, 512)).  The
# expected gradients are written out by hand; softmax_scale = fl32(ln 2)
# makes c = 1, so P = 2^s exactly with LSE = 0.
# ---------------------------------------------------------------------------

AX_N, AX_D = 64, 64
TINY = 2.0 ** -20


def axis_case(which):
    N, d = AX_N, AX_D
    z = lambda: np.zeros((1, 1, N, d), np.float32)
    Q4, K4, Q8, K8, V8, O, dO = z(), z(), z(), z(), z(), z(), z()
    LSE = np.zeros((1, 1, N), np.float32)
    if which == "P_along_queries":
        # s_i,n = a_n: P_i,0 = 1, P_i,1 = 2^-20, P = 0 for n >= 2 (equal down
        # each key's column of queries, 2^20 apart along a query's row)
        Q4[..., 0] = 1.0
        K4[0, 0, :, 0] = -200.0
        K4[0, 0, 0, 0], K4[0, 0, 1, 0] = 0.0, -20.0
        dO[:] = 1.0
    elif which == "dO_for_dV_along_queries":
        # P = 1; dO_i = (1, 2^-20, 0, ...) for every query i
        dO[..., 0], dO[..., 1] = 1.0, TINY
    elif which == "dO_for_dP_along_d_and_dS_for_dQ_along_keys":
        # P = 1, D = 0; dO row 1 = 2^-20 * ones, every other row ones; V = ones:
        # dP_1,n = 64 * 2^-20 for every key (equal along the row), 2^20 below
        # row 0 down each column
        dO[:] = 1.0
        dO[0, 0, 1] = TINY
        V8[:] = 1.0
        K8[:] = 1.0
    elif which == "dS_for_dK_along_queries":
        # P = 1, D = 0; dO = ones; V_0 = ones, V_1 = 2^-20 * ones: dS_i,1 =
        # 2^-14 for every query (equal down the column), 2^20 below dS_i,0
        dO[:] = 1.0
        V8[0, 0, 0] = 1.0
        V8[0, 0, 1] = TINY
        Q8[:] = 1.0
    return Q4, K4, Q8, K8, V8, O, dO, LSE


SCALE_C1 = float(np.float32(np.log(2.0)))


@pytest.mark.parametrize("which", ["P_along_queries", "dO_for_dV_along_queries",
                                   "dO_for_dP_along_d_and_dS_for_dQ_along_keys", "dS_for_dK_along_queries"])
def test_mxfp8_block_axes(which):
    args = axis_case(which)
    dQ, dK, dV = oracle.bwd(*args, softmax_scale=SCALE_C1, causal=False, mode=0)
    N, d = AX_N, AX_D
    ones = np.ones(d)
    if which == "P_along_queries":
        # dV_n = sum_i P_i,n dO_i: key 0 -> 64, key 1 -> 64 * 2^-20
        np.testing.assert_array_equal(dV[0], 64 * ones)
        np.testing.assert_array_equal(dV[1], 64 * TINY * ones)
        np.testing.assert_array_equal(dV[2:], 0)
    elif which == "dO_for_dV_along_queries":
        want = np.zeros(d)
        want[0], want[1] = 64.0, 64 * TINY
        np.testing.assert_array_equal(dV, np.broadcast_to(want, dV.shape))
    elif which == "dO_for_dP_along_d_and_dS_for_dQ_along_keys":
        # dQ_1 = scale * sum_n dS_1,n K_n = scale * 64 keys * 64 * 2^-20
        np.testing.assert_array_equal(dQ[1], SCALE_C1 * 64 * 64 * TINY * ones)
        np.testing.assert_array_equal(dQ[0], SCALE_C1 * 64 * 64 * ones)
    elif which == "dS_for_dK_along_queries":
        # dK_1 = scale * sum_i dS_i,1 Q_i = scale * 64 queries * 2^-14
        np.testing.assert_array_equal(dK[1], SCALE_C1 * 64 * 64 * TINY * ones)
        np.testing.assert_array_equal(dK[0], SCALE_C1 * 64 * 64 * ones)
        np.testing.assert_array_equal(dK[2:], 0)


def test_p_one_ulp_below_one_keeps_its_value():
    """P of every query against key 0 is fl32(2^(-2^-22)) = 1 - 3*2^-24, a
    probability 1 computed a few ulps low.  The probability blocks' exponent
    (the least X with amax <= 448 * 2^X) scales it to 256 - 3*2^-16, which
    rounds to 256: dV_0 = sum over 64 queries of 1 * dO = 64 exactly.  (The
    OCP exponent, one lower, would scale it to 512 - 3*2^-15 and saturate it
    to 448: dV_0 = 56.)"""
    N, d = 64, 64
    z = lambda: np.zeros((1, 1, N, d), np.float32)
    Q4, K4, Q8, K8, V8, O, dO = z(), z(), z(), z(), z(), z(), z()
    Q4[..., 0] = 1.0
    K4[0, 0, :, 0] = -200.0
    K4[0, 0, 0, 0] = -(2.0 ** -22)
    dO[:] = 1.0
    p = np.float32(2.0 ** -(2.0 ** -22))
    assert p == np.float32(1 - 3 * 2.0 ** -24) and p < 1
    dQ, dK, dV = oracle.bwd(Q4, K4, Q8, K8, V8, O, dO, np.zeros((1, 1, N), np.float32),
                            softmax_scale=SCALE_C1, causal=False, mode=0)
    np.testing.assert_array_equal(dV[0], 64 * np.ones(d))
    np.testing.assert_array_equal(dV[1:], 0)
    np.testing.assert_array_equal(dQ, 0)
    np.testing.assert_array_equal(dK, 0)
