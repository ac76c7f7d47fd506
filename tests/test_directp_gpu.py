"""The device Direct-P classifier vs the oracle's map, bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu


def test_every_fp32_offset_in_range():
    """All FP32 x in [-6, 0.5] with |x| >= 2^-8 (every threshold lies in
    [-4.59, -0.26]; smaller |x| are code 7), plus specials (m=0, c=1 makes
    x = s exactly)."""
    fa = require_gpu()
    lo = np.float32(-6.0)
    neg = np.arange(np.float32(2.0 ** -8).view(np.int32), lo.view(np.int32) + 1, dtype=np.int32)
    pos = np.arange(np.float32(2.0 ** -8).view(np.int32), np.float32(0.5).view(np.int32) + 1, dtype=np.int32)
    x = np.concatenate([-(neg.view(np.float32)), pos.view(np.float32),
                        np.array([0.0, -0.0, -np.inf, -100.0, 1e-30, -1e-30], np.float32)])
    got = fa.directp_codes(torch.from_numpy(x).cuda(), 0.0, 1.0).cpu().numpy()
    want = oracle.directp_codes_of_x(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} codes differ, e.g. x={x[bad[:5]]} gpu={got[bad[:5]]} oracle={want[bad[:5]]}"


def test_random_scores_and_maxima():
    fa = require_gpu()
    rng = np.random.default_rng(0)
    for _ in range(20):
        m = np.float32(rng.standard_normal() * 30)
        c = np.float32(rng.uniform(0.05, 0.3))
        s = (m - np.abs(rng.standard_normal(100000)) * 40).astype(np.float32)
        got = fa.directp_codes(torch.from_numpy(s).cuda(), float(m), float(c)).cpu().numpy()
        want = np.array([oracle.directp_code(float(v), float(m), float(c)) for v in s[:3000]])
        assert np.array_equal(got[:3000], want)


def test_native_exponential_route_is_exact():
    """The forward's route (ex2 of fmaf(s, c, log2 6 - eps - mc) + bracketed
    RNE to E2M1, threshold count where the bracket is ambiguous) must equal
    the exact threshold map for every FP32 offset in [-6, -2^-8] (with m = 0
    and c = 1 the offset is the score itself; the bracket's width depends on
    mc, which the random tests below vary)."""
    fa = require_gpu()
    neg = np.arange(np.float32(2.0 ** -8).view(np.int32), np.float32(6.0).view(np.int32) + 1, dtype=np.int32)
    x = np.concatenate([-(neg.view(np.float32)),
                        np.array([0.0, -0.0, -np.inf, -100.0, 1e-30, 0.25, -1e-30], np.float32)])
    got = fa.directp_codes(torch.from_numpy(x).cuda(), 0.0, 1.0, native_exp=True).cpu().numpy()
    want = oracle.directp_codes_of_x(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} codes differ, e.g. x={x[bad[:5]]} gpu={got[bad[:5]]} oracle={want[bad[:5]]}"


@pytest.mark.parametrize("m_std", [3.0, 30.0, 300.0])
def test_native_route_random_scores_and_maxima(m_std):
    """Scores below a random maximum m: |m c| small (the narrowest bracket),
    moderate and large (the bracket widens with the unit in the last place of
    m c, which the rounding of klo adds to the offset)."""
    fa = require_gpu()
    rng = np.random.default_rng(1)
    for _ in range(10):
        m = np.float32(rng.standard_normal() * m_std)
        c = np.float32(rng.uniform(0.05, 0.3))
        s = (m - np.abs(rng.standard_normal(200003)) * 40).astype(np.float32)
        got = fa.directp_codes(torch.from_numpy(s).cuda(), float(m), float(c), native_exp=True).cpu().numpy()
        x = np.array([oracle.directp_x(float(v), float(m), float(c)) for v in s[:20000]], np.float32)
        assert np.array_equal(got[:20000], oracle.directp_codes_of_x(x))
