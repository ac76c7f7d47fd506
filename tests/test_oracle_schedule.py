"""Pin of the oracle's running-max schedule (technical summary of
"Hardware-Aware FP4 FlashAttention-4", Methodology 1: Direct Mapping and
Consistent Normalization).

The Direct-P codes of a key tile are taken against the running maximum that
includes that tile, they are never re-rounded later, and O and l are rescaled
by alpha = 2^(c*(m_old - m_new)) as soon as the maximum grows.  A two-tile row
whose second tile raises the maximum by an integer Delta gives O and LSE that
follow from the E2M1 magnitudes alone; codes taken against the previous
tile's maximum (stale), a rescale skipped for small growth (lazy), or codes
taken against the final maximum of the row (two-pass) each give different
numbers, worked out below beside the expected ones.
"""
import math

import numpy as np
import pytest

import oracle

D = 64


def two_tile_row(c: float, gap: float):
    """One query row over two 128-key tiles.

    q = e_0 and k_n = (score_n, 0, ..., 0), so s_n = score_n exactly.  Scores
    are integers times `gap` (= 1/c), so every offset c*(s - m) is an exact
    integer and x = fmaf(s, c, -fl32(m*c)) carries no rounding.
      tile 0: keys 0..5 at offsets 0, -1, -2, -3, -4, -5 (units of gap) from
              its maximum m0 = 0; the other keys at -100 (code 0);
      tile 1: keys 128..131 at +2, +1, 0, -1 (new maximum m1 = 2*gap);
              the other keys at -100.
    V: key n of the six (and four) scored keys carries a one-hot row on its
    own channel; every code-0 key carries 1.0 on channel 63 (it must add
    nothing)."""
    N = 256
    Q = np.zeros((1, 1, N, D), np.float32)
    Q[0, 0, 0, 0] = 1.0
    K = np.zeros((1, 1, N, D), np.float32)
    K[0, 0, :, 0] = -100.0 * gap
    V = np.zeros((1, 1, N, D), np.float32)
    V[0, 0, :, 63] = 1.0
    for j, off in enumerate([0, -1, -2, -3, -4, -5]):
        K[0, 0, j, 0] = off * gap
        V[0, 0, j, 63] = 0.0
        V[0, 0, j, j] = 1.0
    for j, off in enumerate([2, 1, 0, -1]):
        K[0, 0, 128 + j, 0] = off * gap
        V[0, 0, 128 + j, 63] = 0.0
        V[0, 0, 128 + j, 6 + j] = 1.0
    return Q, K, V


# E2M1 value of 6*2^x at integer offsets x (RNE on the grid 0, .5, 1, 1.5, 2,
# 3, 4, 6): 0 -> 6, -1 -> 3, -2 -> 1.5, -3 -> 0.75 ties to the even code 1.0,
# -4 -> 0.375 -> 0.5, -5 -> 0.1875 -> 0; positive offsets saturate at 6.
VAL = {0: 6.0, -1: 3.0, -2: 1.5, -3: 1.0, -4: 0.5, -5: 0.0}


def expected(scheme: str):
    """Per-channel weights (before division by l), l and the final max in
    units of gap, for the method (eager) and for the three wrong schedules."""
    w = np.zeros(D)
    if scheme == "eager":
        # tile 0 against m0 = 0, then alpha = 2^-2 when m grows to 2
        for j, off in enumerate([0, -1, -2, -3, -4, -5]):
            w[j] = 0.25 * VAL[off]
        for j, off in enumerate([0, -1, -2, -3]):          # 2,1,0,-1 minus m1 = 2
            w[6 + j] = VAL[off]
    elif scheme == "stale":
        # tile 1's codes against m0 = 0 (offsets +2, +1 saturate to 6)
        for j, off in enumerate([0, -1, -2, -3, -4, -5]):
            w[j] = 0.25 * VAL[off]
        for j, off in enumerate([2, 1, 0, -1]):
            w[6 + j] = VAL[min(off, 0)]
    elif scheme == "lazy":
        # no rescale for a growth of 2: everything against m0 = 0
        for j, off in enumerate([0, -1, -2, -3, -4, -5]):
            w[j] = VAL[off]
        for j, off in enumerate([2, 1, 0, -1]):
            w[6 + j] = VAL[min(off, 0)]
    elif scheme == "two_pass":
        # every code against the row's final max 2
        for j, off in enumerate([0, -1, -2, -3, -4, -5]):
            w[j] = VAL.get(off - 2, 0.0)
        for j, off in enumerate([0, -1, -2, -3]):
            w[6 + j] = VAL[off]
    l = w.sum()
    m = 0 if scheme == "lazy" else 2
    return w, l, m


def test_hand_derived_expected_values():
    """The numbers the method gives, written out: l = 0.25*(6+3+1.5+1+0.5) +
    (6+3+1.5+1) = 3 + 11.5 = 14.5."""
    w, l, m = expected("eager")
    assert l == 14.5 and m == 2
    assert list(w[:10]) == [1.5, 0.75, 0.375, 0.25, 0.125, 0.0, 6.0, 3.0, 1.5, 1.0]


@pytest.mark.parametrize("c", [1.0, 0.5, 2.0])
def test_running_max_schedule(c):
    # softmax_scale chosen so that c = fl32(scale*log2 e) is exactly 1, 1/2 or 2
    scale = np.float32(c * math.log(2.0))
    assert np.float32(np.float64(scale) * 1.4426950408889634) == np.float32(c)
    gap = 1.0 / c
    Q, K, V = two_tile_row(c, gap)
    O, L = oracle.fwd(Q, K, V, softmax_scale=float(scale), rows=np.arange(1))
    w, l, m = expected("eager")
    np.testing.assert_allclose(O[0], w / l, rtol=0, atol=1e-15)
    # LSE = scale*m + ln(l/6), m = 2*gap in score units
    assert abs(L[0] - (float(scale) * m * gap + math.log(l / 6.0))) < 1e-12
    # the schedules that the method excludes give other outputs
    for wrong in ("stale", "lazy", "two_pass"):
        w2, l2, _ = expected(wrong)
        assert np.max(np.abs(w2 / l2 - w / l)) > 0.01, wrong
