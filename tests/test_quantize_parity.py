"""GPU quantization vs the oracle: codes and scales bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import require_gpu
from precision_attention_fa4fp4_gb300.inputs import FWD_4K, VIDEO_DIT, make_inputs

pytestmark = pytest.mark.gpu


def gpu_quant(fa, x_bf16, fmt, axis):
    q = fa.quantize(x_bf16.cuda(), fmt, axis)
    fa.sync_status()
    return q.codes.cpu().numpy(), q.scales.cpu().numpy()


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("N,d", [(1, 64), (31, 128), (33, 64), (129, 128), (300, 64), (1000, 128)])
def test_random_shapes(fmt, axis, N, d):
    fa = require_gpu()
    g = torch.Generator().manual_seed(N * 7 + d)
    x = (torch.randn(2, 3, N, d, generator=g) * torch.exp2(torch.randint(-8, 8, (2, 3, N, 1), generator=g).float()))
    x = x.to(torch.bfloat16)
    x[0, 0, 0, :5] = torch.tensor([0.0, -0.0, 1e-40, -1e-3, 3e38]).to(torch.bfloat16)
    c, s = gpu_quant(fa, x, fmt, axis)
    co, so = oracle.quantize(x.float().numpy(), fmt, axis)
    assert np.array_equal(s, so)
    assert np.array_equal(c, co)


@pytest.mark.parametrize("fmt", [0, 1])
def test_all_bf16_values(fmt):
    """Every finite bf16 value, in blocks anchored at several exponents."""
    fa = require_gpu()
    bits = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    vals = bits[np.isfinite(bits)]
    blocks = []
    emax = 2 if fmt == 0 else 8
    for X in (-127, -60, -3, 0, 5, 60, 117):
        anchor = np.float32(np.ldexp(1.0, X + emax))
        v = vals[np.abs(vals.astype(np.float64)) < 2.0 * float(anchor)]
        n = -(-v.size // 31)
        pad = np.zeros(n * 31, np.float32)
        pad[: v.size] = v
        blocks.append(np.concatenate([np.full((n, 1), anchor, np.float32), pad.reshape(n, 31)], 1))
    x = np.concatenate(blocks, 0)
    rows = x.shape[0] // 4 * 4
    x = x[:rows].reshape(1, 1, rows, 32)
    x = np.concatenate([x, x], axis=3)        # d = 64
    xt = torch.from_numpy(x).to(torch.bfloat16)
    c, s = gpu_quant(fa, xt, fmt, 0)
    co, so = oracle.quantize(x, fmt, 0)
    assert np.array_equal(s, so)
    mism = np.nonzero(c != co)
    assert mism[0].size == 0, f"{mism[0].size} code bytes differ, e.g. gpu {c[mism][:8]} oracle {co[mism][:8]}"


@pytest.mark.parametrize("w", [FWD_4K, VIDEO_DIT], ids=lambda w: w.name)
def test_full_size_q_k_v(w):
    fa = require_gpu()
    q, k, v = make_inputs(w)
    for x, fmt, axis in ((q, 0, 0), (k, 0, 0), (v, 0, 1), (v, 1, 0), (k, 1, 1)):
        c, s = gpu_quant(fa, x, fmt, axis)
        co, so = oracle.quantize(x.float().numpy(), fmt, axis)
        assert np.array_equal(s, so) and np.array_equal(c, co), (fmt, axis)


@pytest.mark.parametrize("N,d", [(1, 64), (33, 128), (129, 64), (300, 128), (1000, 64)])
def test_quantize_qkv_one_launch(N, d):
    """The fused call writes exactly what the oracle (and three separate
    quantize calls) give: Q and K along d, V along N, GQA head counts."""
    fa = require_gpu()
    g = torch.Generator().manual_seed(N + d)
    q = torch.randn(2, 4, N, d, generator=g).to(torch.bfloat16)
    k = (torch.randn(2, 2, N, d, generator=g) * 3).to(torch.bfloat16)
    v = (torch.randn(2, 2, N, d, generator=g) * torch.exp2(torch.randint(-6, 6, (2, 2, N, 1), generator=g).float())).to(torch.bfloat16)
    q4, k4, vt = fa.quantize_qkv(q.cuda(), k.cuda(), v.cuda())
    fa.sync_status()
    for got, x, axis in ((q4, q, 0), (k4, k, 0), (vt, v, 1)):
        co, so = oracle.quantize(x.float().numpy(), 0, axis)
        assert np.array_equal(got.scales.cpu().numpy(), so), axis
        assert np.array_equal(got.codes.cpu().numpy(), co), axis


@pytest.mark.parametrize("w", [FWD_4K, VIDEO_DIT], ids=lambda w: w.name)
def test_quantize_qkv_full_size(w):
    fa = require_gpu()
    q, k, v = make_inputs(w)
    outs = fa.quantize_qkv(q.cuda(), k.cuda(), v.cuda())
    fa.sync_status()
    for got, x, axis in zip(outs, (q, k, v), (0, 0, 1)):
        co, so = oracle.quantize(x.float().numpy(), 0, axis)
        assert np.array_equal(got.scales.cpu().numpy(), so), axis
        assert np.array_equal(got.codes.cpu().numpy(), co), axis
