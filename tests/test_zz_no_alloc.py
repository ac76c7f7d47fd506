"""fa4fp4_bwd_noalloc: the backward for callers that cannot allocate device
memory (plugins whose host framework owns every device allocation, runtimes
that forbid allocation after start-up).  It must give the same gradients as fa4fp4_bwd with a
caller workspace, call after call, although every call reuses the same fixed
scratch array inside the library.

Collected last on purpose (file name), so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest

from gpu_util import assert_close, require_gpu
from precision_attention_fa4fp4_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu


def operands(fa, w, seed):
    q, k, v, do = (t.cuda() for t in make_inputs(w, seed=seed, with_dout=True))
    q4, k4 = fa.quantize(q), fa.quantize(k)
    vt = fa.quantize(v, fa.FMT_MXFP4, fa.ALONG_N)
    q8c = fa.quantize(q, fa.FMT_MXFP8, fa.ALONG_N)
    k8c = fa.quantize(k, fa.FMT_MXFP8, fa.ALONG_N)
    v8r = fa.quantize(v, fa.FMT_MXFP8, fa.ALONG_D)
    o, lse = fa.fwd(q4, k4, vt, causal=w.causal, out_dtype=fa.OUT_F32)
    return q4, k4, q8c, k8c, v8r, o, do, lse


def test_noalloc_matches_workspace_backward_twice():
    fa = require_gpu()
    shapes = [Workload("noalloc_a", 1, 4, 2, 300, 128, causal=True, qk_std=128 ** -0.25),
              Workload("noalloc_b", 2, 2, 1, 777, 128, causal=False, qk_std=128 ** -0.25)]
    for call, w in enumerate(shapes):          # two calls in a row, different sizes
        args = operands(fa, w, seed=10 + call)
        ref = fa.bwd(*args, causal=w.causal)
        got = fa.bwd_noalloc(*args, causal=w.causal)
        fa.sync_status()
        for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
            assert_close(a.cpu().numpy(), b.cpu().numpy(), f"{w.name} call {call} {name}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    fa = require_gpu()
    lib = fa.load_library()
    limit = 16 << 20
    assert fa.bwd_workspace_bytes(2, 32, 8, 8192, 128) > limit
    w = Workload("noalloc_big", 1, 64, 8, 2048, 128, causal=True)
    assert fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.d) > limit
    args = operands(fa, w, seed=3)
    with pytest.raises(fa.Fa4Fp4Error) as e:
        fa.bwd_noalloc(*args, causal=True)
    assert e.value.status == 6     # FA4FP4_ERR_WORKSPACE
    assert lib is not None
