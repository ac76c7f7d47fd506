"""The Python binding refuses, before any launch, quantized tensors of the
wrong format, axis or size and outputs of the wrong shape or dtype: the
library would otherwise read or write past the buffers.  CPU tensors only;
a call whose arguments pass these checks stops at the CUDA-tensor check."""
import pytest
import torch

from precision_attention_fa4fp4_gb300 import api

B, Hq, Hkv, N, d = 1, 4, 2, 300, 128


def qt(H, fmt, axis, n=N):
    return api.qtensor_alloc(B, H, n, d, fmt, axis, device="cpu")


def fwd_inputs():
    return (qt(Hq, api.FMT_MXFP4, api.ALONG_D), qt(Hkv, api.FMT_MXFP4, api.ALONG_D),
            qt(Hkv, api.FMT_MXFP4, api.ALONG_N))


def bwd_inputs():
    q4, k4, _ = fwd_inputs()
    return dict(q4=q4, k4=k4, q8c=qt(Hq, api.FMT_MXFP8, api.ALONG_N), k8c=qt(Hkv, api.FMT_MXFP8, api.ALONG_N),
                v8r=qt(Hkv, api.FMT_MXFP8, api.ALONG_D), o=torch.zeros(B, Hq, N, d),
                dout=torch.zeros(B, Hq, N, d, dtype=torch.bfloat16), lse=torch.zeros(B, Hq, N))


def test_valid_arguments_reach_the_device_check():
    q4, k4, vt = fwd_inputs()
    with pytest.raises(ValueError, match="CUDA tensors"):
        api.fwd(q4, k4, vt)
    with pytest.raises(ValueError, match="CUDA tensors"):
        api.bwd(**bwd_inputs())


def test_fwd_refuses_wrong_v_layout_and_sizes():
    q4, k4, vt = fwd_inputs()
    with pytest.raises(ValueError, match="vt: expected MXFP4 along N"):
        api.fwd(q4, k4, qt(Hkv, api.FMT_MXFP4, api.ALONG_D))
    with pytest.raises(ValueError, match="vt: codes/scales"):
        api.fwd(q4, k4, qt(Hkv, api.FMT_MXFP4, api.ALONG_N, n=N - 1))
    short = api.QTensor(vt.codes[..., :-1].contiguous(), vt.scales, vt.shape, vt.fmt, vt.axis)
    with pytest.raises(ValueError, match="vt: codes/scales"):
        api.fwd(q4, k4, short)
    with pytest.raises(ValueError, match="k: expected MXFP4 along d"):
        api.fwd(q4, qt(Hkv, api.FMT_MXFP8, api.ALONG_D), vt)


def test_fwd_refuses_wrong_outputs():
    q4, k4, vt = fwd_inputs()
    with pytest.raises(ValueError, match="out: expected"):
        api.fwd(q4, k4, vt, out_dtype=api.OUT_BF16, out=torch.zeros(B, Hq, N, d))
    with pytest.raises(ValueError, match="lse: expected"):
        api.fwd(q4, k4, vt, lse=torch.zeros(B, Hq, N + 1))
    with pytest.raises(ValueError, match="out_dtype"):
        api.fwd(q4, k4, vt, out_dtype=7)


def test_fp8pv_and_nvfp4_refuse_wrong_v():
    q4, k4, vt = fwd_inputs()
    with pytest.raises(ValueError, match="v8t: expected MXFP8 along N"):
        api.fwd_fp8pv(q4, k4, vt)
    nq = api.NvTensor(torch.zeros(B, Hq, N, d // 2, dtype=torch.uint8), torch.zeros(B, Hq, N, d // 16, dtype=torch.uint8),
                      torch.ones(1), (B, Hq, N, d))
    nk = api.NvTensor(torch.zeros(B, Hkv, N, d // 2, dtype=torch.uint8),
                      torch.zeros(B, Hkv, N, d // 16, dtype=torch.uint8), torch.ones(1), (B, Hkv, N, d))
    with pytest.raises(ValueError, match="vt: expected MXFP4 along N"):
        api.fwd_nvfp4(nq, nk, qt(Hkv, api.FMT_MXFP4, api.ALONG_D))
    bad = api.NvTensor(nk.codes, nk.scales[..., :-1].contiguous(), nk.ts, nk.shape)
    with pytest.raises(ValueError, match="k: codes/scales/ts"):
        api.fwd_nvfp4(nq, bad, vt)
    with pytest.raises(ValueError, match="CUDA tensors"):
        api.fwd_nvfp4(nq, nk, vt)


def test_bwd_refuses_wrong_views_and_gradients():
    for key, wrong, msg in [("q8c", qt(Hq, api.FMT_MXFP8, api.ALONG_D), "q8c: expected MXFP8 along N"),
                            ("v8r", qt(Hkv, api.FMT_MXFP8, api.ALONG_N), "v8r: expected MXFP8 along d"),
                            ("dout", torch.zeros(B, Hq, N, d), "dout: expected"),
                            ("lse", torch.zeros(B, Hq, N, dtype=torch.float64), "lse: expected"),
                            ("o", torch.zeros(B, Hq, N, d, dtype=torch.float16), "o: expected")]:
        args = bwd_inputs()
        args[key] = wrong
        with pytest.raises(ValueError, match=msg):
            api.bwd(**args)
    with pytest.raises(ValueError, match="dq: expected"):
        api.bwd_noalloc(**bwd_inputs(), dq=torch.zeros(B, Hq, N, d // 2))


def test_quantize_and_bf16_refuse_mismatches():
    x = torch.zeros(B, Hkv, N, d, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="out: expected MXFP8 along N"):
        api.quantize(x, api.FMT_MXFP8, api.ALONG_N, out=qt(Hkv, api.FMT_MXFP4, api.ALONG_N))
    q = torch.zeros(B, Hq, N, d, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="out\\[2\\] \\(v\\): expected"):
        api.quantize_qkv(q, x, x, out=(qt(Hq, 0, 0), qt(Hkv, 0, 0), qt(Hkv, 0, 0)))
    with pytest.raises(ValueError, match="v: expected"):
        api.bf16_fwd(q, x, x.float())


def test_quantize_nvfp4_refuses_wrong_out():
    x = torch.zeros(B, Hkv, N, d, dtype=torch.bfloat16)
    bad = api.NvTensor(torch.zeros(B, Hkv, N, d // 2, dtype=torch.uint8),
                       torch.zeros(B, Hkv, N, d // 32, dtype=torch.uint8), torch.ones(1), (B, Hkv, N, d))
    with pytest.raises(ValueError, match="out: codes/scales/ts"):
        api.quantize_nvfp4(x, out=bad)


def test_fwd_qbf16_and_quantize_kv_check_buffers():
    _, k4, vt = fwd_inputs()
    q = torch.zeros(B, Hq, N, d, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensors"):
        api.fwd_qbf16(q, k4, vt)
    with pytest.raises(ValueError, match="bf16"):
        api.fwd_qbf16(q.float(), k4, vt)
    with pytest.raises(ValueError, match="vt: expected"):
        api.fwd_qbf16(q, k4, qt(Hkv, api.FMT_MXFP4, api.ALONG_D))
    with pytest.raises(ValueError, match="k: codes/scales"):
        api.fwd_qbf16(q, qt(Hkv, api.FMT_MXFP4, api.ALONG_D, n=N - 1), vt)
    k = torch.zeros(B, Hkv, N, d, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensors"):
        api.quantize_kv(k, k)
    with pytest.raises(ValueError, match="same shape"):
        api.quantize_kv(k, torch.zeros(B, Hkv, N - 1, d, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="out\\[1\\]"):
        api.quantize_kv(k, k, out=(qt(Hkv, api.FMT_MXFP4, api.ALONG_D), qt(Hkv, api.FMT_MXFP4, api.ALONG_D)))
