"""Pins of the oracle's Direct-P map (Methodology 1, "Direct Mapping").

The map is pinned against RNE_E2M1(6*2^x) evaluated independently in FP64
(numpy exp2 + binade round-half-even), against thresholds derived from the
closed form log2(midpoint/6), and against the worked example with c = 1.
"""
import json
import os
from fractions import Fraction

import numpy as np

import oracle
from test_oracle_formats import rne_e2m1

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "directp_thresholds.json")
E2M1_MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def code_of_value(v: np.ndarray) -> np.ndarray:
    return np.searchsorted(np.array(E2M1_MAGS), v)


def independent_thresholds():
    """T_k = smallest FP32 x whose RNE_E2M1(6*2^x) reaches magnitude k.
    The switching point is log2(mu_k/6), mu_k the midpoint below magnitude k;
    the midpoint itself rounds to the even neighbour, which is magnitude k
    only for mu = 0.75 (-> 1.0), 1.75 (-> 2.0) and 3.5 (-> 4.0)."""
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    inclusive = [False, True, False, True, False, True, False]
    out = []
    for mu, inc in zip(mids, inclusive):
        r = np.log2(mu / 6.0)
        t = np.float32(r)
        if float(t) < r or (float(t) == r and not inc):
            t = np.nextafter(t, np.float32(1))
        out.append(t)
    return np.array(out, dtype=np.float32)


def test_thresholds_closed_form_and_golden():
    T = oracle.directp_thresholds()
    assert np.array_equal(T, independent_thresholds())
    assert T[1] == np.float32(-3.0)                 # the one exact tie
    with open(GOLDEN) as f:
        g = json.load(f)
    assert [float(np.float32(t)) for t in g["T_fp32"]] == [float(t) for t in T]
    # distance of each threshold's neighbourhood from the real switching point
    # is far above FP64 evaluation error, so the bisection's predicate was exact
    for k, t in enumerate(T):
        if k == 1:
            continue
        r = np.log2([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0][k] / 6.0)
        assert min(abs(float(t) - r), abs(float(np.nextafter(t, np.float32(-1))) - r)) > 1e-12


def test_threshold_map_equals_rne_of_6exp2_dense():
    x = np.linspace(-6.0, 0.0, 10_000_001, dtype=np.float64).astype(np.float32)
    T = oracle.directp_thresholds()
    nb = []
    for t in T:
        v = t
        for _ in range(4):
            v = np.nextafter(v, np.float32(-10))
        for _ in range(9):
            nb.append(v)
            v = np.nextafter(v, np.float32(10))
    x = np.concatenate([x, np.array(nb, dtype=np.float32),
                        np.array([0.0, -0.0, 1e-30, -1e-30, -50.0, -np.inf], np.float32)])
    ours = oracle.directp_codes_of_x(x)
    want = code_of_value(rne_e2m1(6.0 * np.exp2(x.astype(np.float64))))
    assert np.array_equal(ours, want)


def test_worked_example_unit_c():
    """c = 1, integer gaps m - s: 6*2^-gap -> 6, 3, 1.5, 1.0 (0.75 ties to
    even), 0.5, then 0."""
    want = {0: 7, 1: 5, 2: 3, 3: 2, 4: 1, 5: 0, 6: 0, 9: 0}
    for gap, code in want.items():
        assert oracle.directp_code(10.0 - gap, 10.0, 1.0) == code


def _rn32(q: Fraction) -> np.float32:
    """Correctly rounded FP32 of a rational (ties to even)."""
    f = np.float32(float(q))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - q),
                                     int(np.frombuffer(c.tobytes(), np.uint32)[0]) & 1))
    return best


def test_x_is_single_rounding_fma():
    g = np.random.default_rng(11)
    for _ in range(3000):
        s = np.float32(g.standard_normal() * 20)
        m = np.float32(abs(g.standard_normal()) * 20 + float(s))
        c = np.float32(g.uniform(0.01, 0.3))
        mc = _rn32(Fraction(float(m)) * Fraction(float(c)))
        want = _rn32(Fraction(float(s)) * Fraction(float(c)) - Fraction(float(mc)))
        assert oracle.directp_x(float(s), float(m), float(c)) == float(want)
