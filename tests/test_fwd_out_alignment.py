"""The forward's epilogue writes 32-byte words when O is 32-byte aligned and
16-byte words otherwise (the ABI requires 16): both give the same bytes."""
import pytest
import torch

from gpu_util import require_gpu
from precision_attention_fa4fp4_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("route", ["directp", "fp8pv"])
@pytest.mark.parametrize("out_bf16", [True, False])
@pytest.mark.parametrize("d", [64, 128])
def test_output_16_byte_aligned_only(route, out_bf16, d):
    fa = require_gpu()
    w = Workload(f"align_d{d}", 1, 4, 2, 300, d, causal=True)
    q, k, v = (t.cuda() for t in make_inputs(w, seed=23))
    q4, k4 = fa.quantize(q), fa.quantize(k)
    dtype = torch.bfloat16 if out_bf16 else torch.float32
    odt = fa.OUT_BF16 if out_bf16 else fa.OUT_F32
    if route == "fp8pv":
        vt = fa.quantize(v, fa.FMT_MXFP8, fa.ALONG_N)
        run = lambda out: fa.fwd_fp8pv(q4, k4, vt, causal=True, out_dtype=odt, out=out)
    else:
        vt = fa.quantize(v, fa.FMT_MXFP4, fa.ALONG_N)
        run = lambda out: fa.fwd(q4, k4, vt, causal=True, out_dtype=odt, out=out)
    shape = (w.B, w.Hq, w.N, w.d)
    o32, _ = run(torch.empty(shape, dtype=dtype, device="cuda"))
    step = 16 // o32.element_size()
    buf = torch.empty(o32.numel() + step, dtype=dtype, device="cuda")
    o16 = buf[step:].view(shape)                       # 16-byte aligned, not 32
    assert o32.data_ptr() % 32 == 0 and o16.data_ptr() % 32 == 16
    run(o16)
    torch.cuda.synchronize()
    fa.sync_status()
    assert torch.equal(o16, o32)
