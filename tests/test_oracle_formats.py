"""Pins of the oracle's element formats and block quantization.

Each check compares the oracle with something other than itself: the format
definitions (bit fields), a library conversion (torch float8_e4m3fn), an
independent binade-wise round-half-even, or an invariant of the OCP MX rule.
"""
import math

import numpy as np
import pytest
import torch

import oracle

E2M1_MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # E2M1 (bias 1, 1 mantissa bit)


def test_e2m1_table_and_roundtrip():
    for c in range(16):
        v = oracle.e2m1_value(c)
        mag = E2M1_MAGS[c & 7]
        assert abs(v) == mag
        assert np.signbit(v) == bool(c & 8)
        assert oracle.round_to_code(v, 0) == c        # every code re-encodes to itself
    assert oracle.round_to_code(-0.0, 0) == 0x8       # negative zero keeps its sign


def test_e4m3_table_matches_torch():
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(ours))
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(lib[~nan], ours[~nan])
    assert np.array_equal(np.signbit(lib[~nan]), np.signbit(ours[~nan]))
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.round_to_code(oracle.e4m3_value(c), 1) == c
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(1) == 2.0 ** -9


def test_e8m0():
    for b in range(255):
        assert oracle.e8m0_value(b) == 2.0 ** (b - 127)
    assert np.isnan(oracle.e8m0_value(255))


# ---------------------------------------------------------------------------
# independent rounding: round-half-even per binade (numpy rint), saturating
# ---------------------------------------------------------------------------

def rne_e2m1(y: np.ndarray) -> np.ndarray:
    a = np.abs(y)
    q = np.where(a < 2, np.rint(a * 2) / 2, np.where(a < 4, np.rint(a), 2 * np.rint(a / 2)))
    return np.copysign(np.minimum(q, 6.0), y)


def rne_e4m3(y: np.ndarray) -> np.ndarray:
    a = np.abs(y)
    _, e = np.frexp(a)                       # a = f * 2^e, f in [0.5, 1)
    e = np.maximum(e - 1, -6)                # binade exponent, subnormals share -6
    step = np.ldexp(1.0, e - 3)
    q = np.rint(a / step) * step
    return np.copysign(np.minimum(q, 448.0), y)


def all_finite_bf16() -> np.ndarray:
    bits = np.arange(65536, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    return v[np.isfinite(v)]


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("X", [-127, -40, -3, 0, 7, 100, 117])
def test_quantize_exhaustive_bf16(fmt, X):
    """All finite bf16 values that keep the block exponent at X, each in a
    block whose amax is pinned by an anchor 2^(X+emax)."""
    emax = 2 if fmt == 0 else 8
    if X + emax > 127:
        pytest.skip("anchor not representable")
    anchor = np.float32(np.ldexp(1.0, X + emax))
    v = all_finite_bf16()
    v = v[np.abs(v.astype(np.float64)) < 2.0 * float(anchor)]
    nblk = -(-v.size // 31)
    pad = np.zeros(nblk * 31, dtype=np.float32)
    pad[: v.size] = v
    x = np.concatenate([np.full((nblk, 1), anchor, np.float32), pad.reshape(nblk, 31)], axis=1)
    x = x.reshape(1, 1, nblk, 32)
    codes, scales = oracle.quantize(x, fmt, oracle.ALONG_D)
    assert np.all(scales == X + 127)
    deq = oracle.dequantize(codes, scales, x.shape, fmt, oracle.ALONG_D).astype(np.float64)
    y = np.ldexp(x.astype(np.float64), -X)
    want = (rne_e2m1(y) if fmt == 0 else rne_e4m3(y)) * np.ldexp(1.0, X)
    assert np.array_equal(deq, want)
    assert np.array_equal(np.signbit(deq), np.signbit(want))


def test_e4m3_rounding_matches_torch_in_range():
    g = torch.Generator().manual_seed(3)
    y = (torch.rand(200000, generator=g, dtype=torch.float64) * 2 - 1) * 460
    y = y.to(torch.float32)
    lib = y.to(torch.float8_e4m3fn).to(torch.float64).numpy()
    ok = np.abs(y.numpy()) <= 448
    ours = np.array([oracle.e4m3_value(oracle.round_to_code(float(t), 1)) for t in y.numpy()[ok][:20000]])
    assert np.array_equal(ours, lib[ok][:20000])


@pytest.mark.parametrize("fmt,lo,hi", [(0, 4.0, 8.0), (1, 256.0, 512.0)])
def test_block_exponent_closed_form(fmt, lo, hi):
    g = np.random.default_rng(0)
    a = np.float32(np.abs(g.standard_normal(5000)) * np.exp2(g.integers(-60, 60, 5000))) + np.float32(1e-30)
    for amax in a:
        X = oracle.block_exponent(float(amax), fmt)
        r = float(amax) * 2.0 ** -X
        assert lo <= r < hi
    assert oracle.block_exponent(0.0, fmt) == -127


def test_p_block_exponent_is_smallest_unsaturated():
    """The probability blocks' exponent is the least X with amax <= 448 * 2^X
    (checked by exact double comparisons, and against the OCP exponent: the
    same below a significand of 1.75, one more above it)."""
    g = np.random.default_rng(1)
    a = np.float32(np.abs(g.standard_normal(5000)) * np.exp2(g.integers(-60, 60, 5000))) + np.float32(1e-30)
    edge = np.float32([1.0, np.nextafter(np.float32(1), np.float32(0)), 0.875, 0.95, 1.75, 0.5,
                       np.nextafter(np.float32(0.875), np.float32(1)), 448.0, 449.0])
    for amax in np.concatenate([a, edge]):
        X = oracle.p_block_exponent(float(amax))
        assert float(amax) <= math.ldexp(448.0, X) and float(amax) > math.ldexp(448.0, X - 1)
        frac = math.frexp(float(amax))[0] * 2     # significand in [1, 2)
        assert X == oracle.block_exponent(float(amax), 1) + (1 if frac > 1.75 else 0)
    # one ulp below 1 takes the exponent of 1 (1 - 2^-24 scales to 256 - 2^-16,
    # which rounds to the E4M3 value 256)
    assert oracle.p_block_exponent(float(edge[1])) == oracle.p_block_exponent(1.0) == -8
    assert oracle.p_block_exponent(0.0) == -127


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("axis", [0, 1])
def test_quantize_scale_and_sign_invariants(fmt, axis):
    g = torch.Generator().manual_seed(5)
    x = torch.randn(2, 3, 77, 64, generator=g).to(torch.bfloat16).float().numpy()
    c0, s0 = oracle.quantize(x, fmt, axis)
    for k in (-5, 1, 9):
        c1, s1 = oracle.quantize(np.ldexp(x, k).astype(np.float32), fmt, axis)
        assert np.array_equal(c1, c0)
        valid = s0 > 0    # all-zero padding blocks are clamped at -127
        assert np.array_equal(s1[valid].astype(int), s0[valid].astype(int) + k)
    cn, sn = oracle.quantize(-x, fmt, axis)
    flip = 0x88 if fmt == 0 else 0x80
    if axis == 1:
        # padded positions hold +0 on both sides
        Np = oracle.padded_n(x.shape[2])
        mask = np.zeros(c0.shape, dtype=np.uint8)
        per = 2 if fmt == 0 else 1
        cols = x.shape[2] // per
        mask[..., :cols] = flip
        if fmt == 0 and x.shape[2] % 2:
            mask[..., cols] = 0x08
        assert Np > x.shape[2]
        assert np.array_equal(cn, c0 ^ mask)
    else:
        assert np.array_equal(cn, c0 ^ flip)
    assert np.array_equal(sn, s0)


@pytest.mark.parametrize("fmt", [0, 1])
def test_along_n_is_along_d_of_the_transpose(fmt):
    """Quantizing along N equals quantizing the zero-padded transpose along d."""
    g = torch.Generator().manual_seed(7)
    B, H, N, d = 1, 2, 200, 64
    x = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).float().numpy()
    cN, sN = oracle.quantize(x, fmt, oracle.ALONG_N)
    Np = oracle.padded_n(N)
    xt = np.zeros((B, H, d, Np), dtype=np.float32)
    xt[:, :, :, :N] = np.swapaxes(x, 2, 3)
    cD, sD = oracle.quantize(xt, fmt, oracle.ALONG_D)
    assert np.array_equal(cN, cD) and np.array_equal(sN, sD)
    back = oracle.dequantize(cN, sN, x.shape, fmt, oracle.ALONG_N)
    want = np.swapaxes(oracle.dequantize(cD, sD, xt.shape, fmt, oracle.ALONG_D), 2, 3)[:, :, :N]
    assert np.array_equal(back, want)


def test_nibble_order():
    """Element 2i sits in the low nibble, 2i+1 in the high nibble."""
    x = np.zeros((1, 1, 1, 32), dtype=np.float32)
    x[0, 0, 0, 0] = 4.0      # amax 4 -> X = 0
    x[0, 0, 0, 1] = 0.5
    codes, scales = oracle.quantize(x, 0, oracle.ALONG_D)
    assert scales[0, 0, 0, 0] == 127
    assert codes[0, 0, 0, 0] == (0x6 | (0x1 << 4))


# ---------------------------------------------------------------------------
# NVFP4 (E2M1, one E4M3 scale per 16 along d, one FP32 scale per tensor)
# ---------------------------------------------------------------------------

def nvfp4_reference(x):
    """The reading's steps in numpy FP32 with the independent round-half-even
    helpers above: ts = amax/2688; sb = RNE_E4M3(amax_b / (6 ts));
    y = x / (sb ts); RNE_E2M1(y) * sb * ts."""
    x = np.asarray(x, np.float32)
    amax = np.float32(np.abs(x).max())
    ts = np.float32(amax / np.float32(2688.0)) if amax > 0 else np.float32(1.0)
    blocks = x.reshape(-1, 16)
    ab = np.abs(blocks).max(1).astype(np.float32)
    sb = rne_e4m3((ab / np.float32(np.float32(6.0) * ts)).astype(np.float64)).astype(np.float32)
    den = (sb * ts).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = (blocks / den[:, None]).astype(np.float32)
    q = np.where(den[:, None] == 0, 0.0, rne_e2m1(y.astype(np.float64)))
    return (q * sb[:, None].astype(np.float64) * np.float64(ts)).reshape(x.shape), sb, ts


def test_nvfp4_matches_independent_steps():
    g = np.random.default_rng(4)
    x = g.standard_normal((2, 3, 50, 64)) * np.exp2(g.integers(-10, 10, (2, 3, 50, 4)).repeat(16, -1))
    x = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).float().numpy()
    x[0, 0, 0, :16] = 0.0                      # an all-zero block: scale 0, codes 0
    codes, scales, ts = oracle.quantize_nvfp4(x)
    want, sb, ts_ref = nvfp4_reference(x)
    assert np.float32(ts) == ts_ref
    assert np.array_equal(np.array([oracle.e4m3_value(int(c)) for c in scales.reshape(-1)]), sb.astype(np.float64))
    got = oracle.dequantize_nvfp4(codes, scales, ts, x.shape)      # FP32 values
    assert np.array_equal(got, want.astype(np.float32))
    assert scales.reshape(-1)[0] == 0 and np.all(codes[0, 0, 0, :8] == 0)


def test_nvfp4_invariants():
    g = torch.Generator().manual_seed(9)
    x = torch.randn(1, 2, 33, 128, generator=g).to(torch.bfloat16).float().numpy()
    c0, s0, t0 = oracle.quantize_nvfp4(x)
    for k in (-7, 3):
        c1, s1, t1 = oracle.quantize_nvfp4(np.ldexp(x, k).astype(np.float32))
        assert np.array_equal(c1, c0) and np.array_equal(s1, s0) and t1 == np.ldexp(t0, k)
    cn, sn, tn = oracle.quantize_nvfp4(-x)
    assert np.array_equal(cn, c0 ^ 0x88) and np.array_equal(sn, s0) and tn == t0
    # the largest element lands on the top of the grid: 6 * 448 * ts = amax
    deq = oracle.dequantize_nvfp4(c0, s0, t0, x.shape)
    i = np.unravel_index(np.abs(x).argmax(), x.shape)
    assert abs(deq[i] - x[i]) <= abs(x[i]) * 2.0 ** -3


def test_nvfp4_grid_tops():
    """Properties that fix the two constants: in every block the largest
    element lands on the top of the E2M1 grid (6, within the E4M3 rounding of
    the block scale: 2^-4 relative for normal scales), and the tensor's
    largest block carries the largest E4M3 scale (448)."""
    g = np.random.default_rng(12)
    x = g.standard_normal((1, 2, 64, 128)) * np.exp2(g.integers(-5, 5, (1, 2, 64, 8)).repeat(16, -1))
    x = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).float().numpy()
    codes, scales, ts = oracle.quantize_nvfp4(x)
    sb = np.array([oracle.e4m3_value(int(c)) for c in scales.reshape(-1)])
    amax_b = np.abs(x.reshape(-1, 16)).max(1).astype(np.float64)
    normal = sb >= 2.0 ** -6
    top = amax_b[normal] / (sb[normal] * ts)
    assert np.all(top >= 6 / (1 + 2.0 ** -4) - 1e-9) and np.all(top <= 6 / (1 - 2.0 ** -4) + 1e-9)
    assert sb[np.argmax(amax_b)] == 448.0 and sb.max() == 448.0
