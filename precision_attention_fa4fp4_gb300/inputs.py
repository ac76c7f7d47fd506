"""Seeded synthetic inputs for the attention workloads.

This module holds no arithmetic of the method: it only draws random numbers.
It is the one piece both the CUDA path's callers (tests, benchmark) and the
oracle's callers share.

Recipe (identical on every host): a torch CPU ``Generator`` seeded with
``seed``; float32 standard-normal draws in the order Q, K, V, dO, each
multiplied by its standard deviation and cast to bfloat16 (round to nearest
even).  Optional outlier channels (video-DiT-shaped workload): the first
``n_outliers`` entries of ``torch.randperm(d)`` drawn from a separate
generator seeded 0, multiplied by ``outlier_scale`` in Q and K before the cast.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, mask and input distribution."""
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: bool = False
    qk_std: float = 1.0
    n_outliers: int = 0
    outlier_scale: float = 8.0

    @property
    def fwd_flops(self) -> float:
        """4*B*H*N^2*d for a noncausal forward, half of it for causal."""
        f = 4.0 * self.B * self.Hq * self.N * self.N * self.d
        return f / 2 if self.causal else f

    @property
    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops


# The workloads the library is specified and measured on.
TINY = Workload("tiny_b1_h2_n256_d64", 1, 2, 2, 256, 64)
FWD_4K = Workload("noncausal_b4_h16_n4096_d128", 4, 16, 16, 4096, 128)
VIDEO_DIT = Workload("videodit_b1_h24_n32760_d128_outliers", 1, 24, 24, 32760, 128, n_outliers=4)
SWEEP = tuple(Workload(f"sweep_b2_h32_n{n}_d{d}", 2, 32, 32, n, d)
              for d in (64, 128) for n in (1024, 2048, 4096, 8192, 16384, 32768))
TRAIN_8B = Workload("causal_gqa_b2_hq32_hkv8_n8192_d128", 2, 32, 8, 8192, 128, causal=True,
                    qk_std=128 ** -0.25)


def outlier_channels(d: int, n: int) -> list[int]:
    g = torch.Generator().manual_seed(0)
    return torch.randperm(d, generator=g)[:n].tolist()


def make_inputs(w: Workload, seed: int = 0, with_dout: bool = False):
    """Return bf16 CPU tensors (Q [B,Hq,N,d], K [B,Hkv,N,d], V [B,Hkv,N,d]
    [, dO [B,Hq,N,d]])."""
    g = torch.Generator().manual_seed(seed)
    shape_q = (w.B, w.Hq, w.N, w.d)
    shape_kv = (w.B, w.Hkv, w.N, w.d)
    q = torch.randn(shape_q, generator=g, dtype=torch.float32) * w.qk_std
    k = torch.randn(shape_kv, generator=g, dtype=torch.float32) * w.qk_std
    v = torch.randn(shape_kv, generator=g, dtype=torch.float32)
    if w.n_outliers:
        ch = outlier_channels(w.d, w.n_outliers)
        q[..., ch] *= w.outlier_scale
        k[..., ch] *= w.outlier_scale
    out = [q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)]
    if with_dout:
        out.append(torch.randn(shape_q, generator=g, dtype=torch.float32).to(torch.bfloat16))
    return tuple(out)


def sample_rows(w: Workload, tiles_per_head: int = 8, heads=None, seed: int = 1) -> torch.Tensor:
    """Deterministic sample of query rows ((b*Hq+h)*N + i): ``tiles_per_head``
    128-row tiles per sampled (b,h), always including the first and the last
    (possibly partial) tile."""
    g = torch.Generator().manual_seed(seed)
    ntiles = (w.N + 127) // 128
    if heads is None:
        heads = range(w.B * w.Hq)
    rows = []
    for bh in heads:
        if ntiles <= tiles_per_head:
            tiles = list(range(ntiles))
        else:
            mid = torch.randperm(ntiles - 2, generator=g)[: tiles_per_head - 2] + 1
            tiles = sorted([0, ntiles - 1] + mid.tolist())
        for t in tiles:
            lo, hi = t * 128, min(w.N, t * 128 + 128)
            rows.extend(bh * w.N + i for i in range(lo, hi))
    return torch.tensor(rows, dtype=torch.int64)


def extreme_logit_inputs(N: int = 640, d: int = 128, seed: int = 3):
    """Synthetic inputs whose scaled logits reach several hundred (far above
    500): Q and K N(0, 36), K's 128-key tile t multiplied by t + 1, so every
    later key tile raises the row maximum by a large step; V N(0, 1).
    bf16 CPU tensors [1, 2, N, d]."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(1, 2, N, d, generator=g) * 6.0
    k = torch.randn(1, 2, N, d, generator=g) * 6.0
    k = k * (1.0 + torch.arange(N).float().div(128).floor().view(1, 1, N, 1))
    v = torch.randn(1, 2, N, d, generator=g)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)
