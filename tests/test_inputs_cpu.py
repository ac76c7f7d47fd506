"""The seeded input generators shared by the oracle's and the CUDA path's
callers: deterministic, in the documented draw order, with the workloads'
shapes, FLOP counts and outlier channels."""
import torch

from precision_attention_fa4fp4_gb300.inputs import (FWD_4K, SWEEP, TINY, TRAIN_8B, VIDEO_DIT, Workload,
                                                      make_inputs, outlier_channels, sample_rows)


def test_deterministic_and_seed_dependent():
    a = make_inputs(TINY, seed=3, with_dout=True)
    b = make_inputs(TINY, seed=3, with_dout=True)
    c = make_inputs(TINY, seed=4, with_dout=True)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert not any(torch.equal(x, y) for x, y in zip(a, c))
    assert all(x.dtype == torch.bfloat16 for x in a)


def test_draw_order_and_scaling():
    w = Workload("t", 1, 4, 2, 40, 64, qk_std=0.5)
    q, k, v, do = make_inputs(w, seed=7, with_dout=True)
    g = torch.Generator().manual_seed(7)
    draws = [torch.randn(s, generator=g) for s in ((1, 4, 40, 64), (1, 2, 40, 64), (1, 2, 40, 64), (1, 4, 40, 64))]
    assert torch.equal(q, (draws[0] * 0.5).to(torch.bfloat16))
    assert torch.equal(k, (draws[1] * 0.5).to(torch.bfloat16))
    assert torch.equal(v, draws[2].to(torch.bfloat16))
    assert torch.equal(do, draws[3].to(torch.bfloat16))


def test_outlier_channels_scale_q_and_k_only():
    ch = outlier_channels(128, 4)
    assert len(set(ch)) == 4 and all(0 <= c < 128 for c in ch)
    w = Workload("t", 1, 2, 2, 64, 128, n_outliers=4)
    plain = Workload("t", 1, 2, 2, 64, 128)
    q, k, v = make_inputs(w)
    q0, k0, v0 = make_inputs(plain)
    assert torch.equal(v, v0)
    rest = [c for c in range(128) if c not in ch]
    assert torch.equal(q[..., rest], q0[..., rest]) and torch.equal(k[..., rest], k0[..., rest])
    # a power-of-two factor commutes with rounding to bf16
    assert torch.equal(q[..., ch], (q0[..., ch].float() * 8).to(torch.bfloat16))
    assert torch.equal(k[..., ch], (k0[..., ch].float() * 8).to(torch.bfloat16))


def test_workload_shapes_and_flops():
    assert (FWD_4K.B, FWD_4K.Hq, FWD_4K.N, FWD_4K.d, FWD_4K.causal) == (4, 16, 4096, 128, False)
    assert abs(FWD_4K.fwd_flops - 5.50e11) / 5.50e11 < 1e-3
    assert (TRAIN_8B.Hq, TRAIN_8B.Hkv, TRAIN_8B.N, TRAIN_8B.causal) == (32, 8, 8192, True)
    assert abs(TRAIN_8B.fwd_flops - 1.10e12) / 1.10e12 < 1e-2 and TRAIN_8B.bwd_flops == 2.5 * TRAIN_8B.fwd_flops
    assert abs(VIDEO_DIT.fwd_flops - 1.32e13) / 1.32e13 < 1e-2 and VIDEO_DIT.N % 128 != 0
    assert len(SWEEP) == 12 and {w.d for w in SWEEP} == {64, 128}


def test_sample_rows_include_first_and_last_tile():
    w = Workload("t", 1, 2, 2, 1000, 64)          # 8 tiles, the last one partial (104 rows)
    rows = sample_rows(w, tiles_per_head=4)
    per_head = [r for r in rows.tolist() if r < w.N]
    assert 0 in per_head and w.N - 1 in per_head
    assert len(rows) == len(set(rows.tolist()))
    assert all(0 <= r < w.B * w.Hq * w.N for r in rows.tolist())
    small = Workload("s", 1, 1, 1, 200, 64)        # fewer tiles than asked: every row
    assert sample_rows(small, tiles_per_head=8).tolist() == list(range(200))
