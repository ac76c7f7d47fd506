"""The inference step on host buffers (fa4fp4_fwd_host) against the device
path it chains (fa4fp4_quantize_qkv + fa4fp4_fwd) on the same data: the
outputs must be bit-identical, whatever the chunking.  One case is also
compared with the oracle (rel-L2 <= 1e-3, LSE to 1e-3 absolute).

The shapes give 3, 4, 5 and 7 chunks, so both staging sets and both compute
streams are reused, and one shape has chunks that cross a batch boundary;
two calls in a row share one workspace; pageable host tensors work too (their
copies do not overlap)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, require_gpu
from precision_attention_fa4fp4_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu


def device_path(fa, q, k, v, causal, out_dtype):
    qg, kg, vg = (t.cuda() for t in (q, k, v))
    q4, k4, vt = fa.quantize_qkv(qg, kg, vg)
    o, lse = fa.fwd(q4, k4, vt, causal=causal, out_dtype=out_dtype)
    return o.cpu(), lse.cpu()


def host_path(fa, q, k, v, causal, out_dtype, with_lse=True, pin=True, workspace=None):
    if pin:
        q, k, v = (t.pin_memory() for t in (q, k, v))
    o, lse = fa.fwd_host(q, k, v, causal=causal, out_dtype=out_dtype, with_lse=with_lse, workspace=workspace)
    torch.cuda.synchronize()
    fa.sync_status()
    return o, lse


@pytest.mark.parametrize("w,out_dtype,with_lse", [
    (Workload("host_b2_hq8_hkv2_n300", 2, 8, 2, 300, 128, causal=True), 0, True),
    (Workload("host_b1_hq6_hkv3_n257_d64", 1, 6, 3, 257, 64), 1, False),
    (Workload("host_b3_h4_n130", 3, 4, 4, 130, 128), 0, True),
    (Workload("host_b3_hq6_hkv3_n100_d64", 3, 6, 3, 100, 64, causal=True), 1, True),
])
def test_matches_device_path(w, out_dtype, with_lse):
    fa = require_gpu()
    q, k, v = make_inputs(w, seed=21)
    o_ref, l_ref = device_path(fa, q, k, v, w.causal, out_dtype)
    o, lse = host_path(fa, q, k, v, w.causal, out_dtype, with_lse)
    assert not o.is_cuda
    assert torch.equal(o, o_ref)
    if with_lse:
        assert torch.equal(lse, l_ref)
    else:
        assert lse is None


def test_two_calls_share_a_workspace_and_pageable_buffers():
    fa = require_gpu()
    w = Workload("host_b2_h4_n200", 2, 4, 2, 200, 64, causal=True)
    ws = torch.empty(fa.fwd_host_workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.d), dtype=torch.uint8, device="cuda")
    inputs = [make_inputs(w, seed=s) for s in (31, 32)]
    pinned = [tuple(t.pin_memory() for t in x) for x in inputs]
    outs = [fa.fwd_host(*x, causal=True, out_dtype=0, workspace=ws) for x in pinned]   # both enqueued
    torch.cuda.synchronize()
    fa.sync_status()
    for x, (o, lse) in zip(inputs, outs):
        o_ref, l_ref = device_path(fa, *x, True, 0)
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    o, lse = host_path(fa, *inputs[0], True, 0, pin=False)
    assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])


def test_against_oracle():
    fa = require_gpu()
    w = Workload("host_b2_hq8_hkv4_n333", 2, 8, 4, 333, 128, causal=True, qk_std=1.0)
    q, k, v = make_inputs(w, seed=41)
    o, lse = host_path(fa, q, k, v, True, 0)
    qf, kf, vf = (t.float().numpy() for t in (q, k, v))
    Qd = oracle.dequantize(*oracle.quantize(qf, 0, 0), qf.shape, 0, 0)
    Kd = oracle.dequantize(*oracle.quantize(kf, 0, 0), kf.shape, 0, 0)
    Vd = oracle.dequantize(*oracle.quantize(vf, 0, 1), vf.shape, 0, 1)
    rows = np.concatenate([np.arange(0, 40), np.arange(w.B * w.Hq * w.N - 300, w.B * w.Hq * w.N)])
    Oo, Lo = oracle.fwd(Qd, Kd, Vd, causal=True, rows=rows)
    assert_close(o.numpy().reshape(-1, w.d)[rows], Oo, w.name + " O")
    assert np.max(np.abs(lse.numpy().reshape(-1)[rows] - Lo)) <= 1e-3
