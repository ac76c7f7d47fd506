"""Benchmark: FP4 Direct-P attention forward TFLOP/s (noncausal, d=128) and its
speedup over the library's own BF16 FlashAttention forward, on one GB300.

Workload (one step): bf16 Q, K, V of shape [4,16,4096,128] resident in HBM ->
fa4fp4_quantize Q, K (MXFP4 along d) and V (MXFP4 along N) -> fa4fp4_fwd
(Direct-P, noncausal) -> O bf16 + LSE.  FLOPs per step: 4*B*H*N^2*d.
L2 is flushed (a 256 MiB write) before every timed step; each step is timed
with CUDA events on the launching stream.

Also reported: the forward kernel alone (the roofline line), the BF16 kernel on
the same inputs, the quantize launch against HBM bandwidth, the causal GQA
training config (forward + backward, with roofline fractions), the video-DiT
and sweep workloads (TFLOP/s and roofline fraction per point), each forward
path's error against FP64 softmax attention on sampled rows of every workload
and on extreme-logit inputs, and an end-to-end figure through host buffers.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun every rank runs its own copy of the workload (independent
problems, no data-path collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from precision_attention_fa4fp4_gb300.inputs import FWD_4K, SWEEP, TRAIN_8B, VIDEO_DIT, make_inputs  # noqa: E402

METRIC = "FP4 attention fwd TFLOP/s (noncausal, d=128) and speedup vs own BF16 kernel"
FP4_OVER_BF16 = 13.5 / 2.25     # nominal dense FP4 : BF16 tensor rate on GB300
FP8_OVER_BF16 = 4.5 / 2.25
# DRAM read + write of one fwd_fp4_kernel<128> launch on the 4K workload, from
# one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum), with the
# SHA-256 of the kernel's sources at that capture: its .cu file, the shared
# device header and its parameter block in the host header.  The figure is
# reported only while those are unchanged; after any edit it reads null until
# the kernel is captured again.
FWD_FP4_TRAFFIC = {"bytes": 78.42e6, "sources_sha256": "c0a99da7312cca3a06820a4a49d5fba8ae2618136eec1f45c0ad11e13a20541e"}
FWD_FP4_SOURCES = ("csrc/fwd_fp4.cu", "csrc/common.cuh")


def fwd_sources_sha256() -> str:
    import hashlib
    import re
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "precision_attention_fa4fp4_gb300")
    for rel in FWD_FP4_SOURCES:
        with open(os.path.join(pkg, rel), "rb") as f:
            h.update(f.read())
    with open(os.path.join(pkg, "csrc", "internal.h")) as f:
        h.update(re.search(r"struct FwdFp4Params \{.*?\n\};", f.read(), re.S).group(0).encode())
    return h.hexdigest()


def fwd_traffic_bytes():
    if FWD_FP4_TRAFFIC["bytes"] is None or FWD_FP4_TRAFFIC["sources_sha256"] != fwd_sources_sha256():
        return None
    return FWD_FP4_TRAFFIC["bytes"]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            mp = json.load(f)
        return {"bf16": float(mp["bf16_tflops"]), "bf16_sustained": float(mp["bf16_tflops_sustained"]),
                "hbm": float(mp["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


# ----------------------------------------------------------------------------
# distributed plumbing (barrier + max over ranks only)
# ----------------------------------------------------------------------------
def dist_setup(ngpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world, sync_cuda: bool = True):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if sync_cuda:
        torch.cuda.synchronize()


def max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """The slowest rank's time (every rank gets it)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: float, world: int, max_ms: float) -> float:
    """Weak scaling: every rank processes its own copy of the workload (its
    own seeded inputs, no exchange); the job's rate is all ranks' work over
    the slowest rank's time."""
    return world * flops_per_rank / (max_ms * 1e-3) / 1e12


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        load = [s for s in sm if s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# the timed loops
# ----------------------------------------------------------------------------
class Flusher:
    def __init__(self, dev):
        self.buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.buf.zero_()


def time_steps(step, warmup, steps, flush, world, inner=None):
    """Returns (per-step ms list, per-step inner-kernel ms list or None).  With
    `inner`, the step gets three events: it records [2] before its first
    launch, [0] and [1] around the inner kernel; the per-step time of the
    launches before the inner kernel ([2] to [0]) is kept in time_steps.pre."""
    for _ in range(warmup):
        flush()
        step(None)
    barrier(world)
    outer, inner_ms = [], []
    evs = []
    for _ in range(steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ie = [torch.cuda.Event(enable_timing=True) for _ in range(3)] if inner else None
        e0.record()
        step(ie)
        e1.record()
        evs.append((e0, e1, ie))
    barrier(world)
    time_steps.pre = []
    for e0, e1, ie in evs:
        outer.append(e0.elapsed_time(e1))
        if ie:
            inner_ms.append(ie[0].elapsed_time(ie[1]))
            time_steps.pre.append(ie[2].elapsed_time(ie[0]))
    return outer, (inner_ms if inner else None)


def run_ours(args, rank, world, local):
    import precision_attention_fa4fp4_gb300 as fa
    fa.load_library()
    dev = torch.device("cuda", local)
    w = FWD_4K
    q, k, v = (t.to(dev) for t in make_inputs(w, seed=rank))
    B, H, N, d = w.B, w.Hq, w.N, w.d
    q4 = fa.qtensor_alloc(B, H, N, d, fa.FMT_MXFP4, fa.ALONG_D, dev)
    k4 = fa.qtensor_alloc(B, H, N, d, fa.FMT_MXFP4, fa.ALONG_D, dev)
    vt = fa.qtensor_alloc(B, H, N, d, fa.FMT_MXFP4, fa.ALONG_N, dev)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    flush = Flusher(dev)

    def step(ie):
        if ie:
            ie[2].record()
        fa.quantize_qkv(q, k, v, out=(q4, k4, vt))
        if ie:
            ie[0].record()
        fa.fwd(q4, k4, vt, causal=False, out_dtype=fa.OUT_BF16, out=o, lse=lse)
        if ie:
            ie[1].record()

    def step_bf16(ie):
        fa.bf16_fwd(q, k, v, causal=False, out_dtype=fa.OUT_BF16, out=o, lse=lse)

    k4q, vtq = fa.qtensor_alloc(B, H, N, d, fa.FMT_MXFP4, fa.ALONG_D, dev), fa.qtensor_alloc(
        B, H, N, d, fa.FMT_MXFP4, fa.ALONG_N, dev)

    def step_fused_q(ie):
        # the same inference step with Q quantized in the forward's prologue:
        # one launch for K and V, then the forward on bf16 Q
        fa.quantize_kv(k, v, out=(k4q, vtq))
        fa.fwd_qbf16(q, k4q, vtq, causal=False, out_dtype=fa.OUT_BF16, out=o, lse=lse)

    def step_fwd_only(ie):
        fa.fwd(q4, k4, vt, causal=False, out_dtype=fa.OUT_BF16, out=o, lse=lse)

    # clocks are sampled across every timed loop below (main step, kernel-only,
    # BF16, end to end, training shape)
    clocks = ClockSampler(local) if rank == 0 else None
    t0 = time.time()
    step_ms, fwd_ms = time_steps(step, args.warmup, args.steps, flush, world, inner=True)
    wall = time.time() - t0
    fa.sync_status()
    flops = w.fwd_flops
    ms = max_over_ranks(statistics.mean(step_ms), world)
    fwd_mean = max_over_ranks(statistics.mean(fwd_ms), world)
    quant_mean = max_over_ranks(statistics.mean(time_steps.pre), world)
    # algorithmic HBM bytes of the quantize launch: bf16 Q, K, V read; E2M1
    # codes (half a byte per element) and one E8M0 byte per 32 elements written
    nel = q.numel() + k.numel() + v.numel()
    quant_bytes = 2 * nel + nel // 2 + nel // 32

    # kernel-only forward (L2 flushed) and the BF16 denominator
    fwd_only, _ = time_steps(step_fwd_only, args.warmup, args.steps, flush, world)
    bf16_ms, _ = time_steps(step_bf16, args.warmup, args.steps, flush, world)
    fa.sync_status()
    fwd_only_ms = max_over_ranks(statistics.mean(fwd_only), world)
    bf16_mean = max_over_ranks(statistics.mean(bf16_ms), world)
    fused_ms, _ = time_steps(step_fused_q, args.warmup, args.steps, flush, world)
    fa.sync_status()
    fused_mean = max_over_ranks(statistics.mean(fused_ms), world)

    # end to end through host buffers: pinned bf16 Q/K/V in, O (bf16) + LSE out
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    ho = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True)]
    hl = [torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)]
    qd, kd, vd = ([torch.empty_like(t)] for t in (q, k, v))
    od = [torch.empty_like(o)]
    ld = [torch.empty_like(lse)]

    def compute(b):
        fa.quantize_qkv(qd[b], kd[b], vd[b], out=(q4, k4, vt))
        fa.fwd(q4, k4, vt, causal=False, out_dtype=fa.OUT_BF16, out=od[b], lse=ld[b])

    def step_e2e(ie):
        # one stream, copies in series with the compute
        for dst, src in ((qd[0], hq), (kd[0], hk), (vd[0], hv)):
            dst.copy_(src, non_blocking=True)
        compute(0)
        ho[0].copy_(od[0], non_blocking=True)
        hl[0].copy_(ld[0], non_blocking=True)

    e2e_serial, _ = time_steps(step_e2e, args.warmup, args.steps, flush, world)
    e2e_serial_mean = max_over_ranks(statistics.mean(e2e_serial), world)

    # end to end through the C ABI on host buffers: one fa4fp4_fwd_host call
    # per step (bf16 Q, K, V in from pinned host memory, O and LSE out to it;
    # inside the call the copies of one chunk overlap the compute of another)
    ho_h, hl_h = ho[0], hl[0]
    ws_host = torch.empty(fa.fwd_host_workspace_bytes(B, H, H, N, d), dtype=torch.uint8, device=dev)

    def host_step():
        fa.fwd_host(hq, hk, hv, causal=False, out_dtype=fa.OUT_BF16, out=ho_h, lse=hl_h, workspace=ws_host)

    for _ in range(args.warmup):
        host_step()
    torch.cuda.synchronize(dev)
    fa.sync_status()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        host_step()
    e1.record()
    torch.cuda.synchronize(dev)
    fa.sync_status()
    barrier(world)
    e2e_mean = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    # the host link's copy rate on this machine, for the bound of that number
    link = torch.empty(hq.numel() * 3, dtype=torch.bfloat16, device=dev)
    hlink = torch.cat([hq.reshape(-1), hk.reshape(-1), hv.reshape(-1)]).pin_memory()
    link.copy_(hlink, non_blocking=True)
    torch.cuda.synchronize(dev)
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0.record()
    for _ in range(3):
        link.copy_(hlink, non_blocking=True)
    l1.record()
    torch.cuda.synchronize(dev)
    h2d_gbs = hlink.numel() * 2 * 3 / (l0.elapsed_time(l1) * 1e-3) / 1e9
    # the step's inputs in and its outputs out at the same time, on two streams
    s_a, s_b = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    outd = torch.empty(ho_h.numel() * ho_h.element_size() + hl_h.numel() * 4, dtype=torch.uint8, device=dev)
    outh = torch.empty(outd.numel(), dtype=torch.uint8, pin_memory=True)
    torch.cuda.synchronize(dev)
    l0.record()
    for st_ in (s_a, s_b):
        st_.wait_event(l0)
    for _ in range(3):
        with torch.cuda.stream(s_a):
            link.copy_(hlink, non_blocking=True)
        with torch.cuda.stream(s_b):
            outh.copy_(outd, non_blocking=True)
    for st_ in (s_a, s_b):
        torch.cuda.current_stream(dev).wait_stream(st_)
    l1.record()
    torch.cuda.synchronize(dev)
    both_ms = l0.elapsed_time(l1) / 3
    del link, hlink, outd, outh
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho[0].numel() * ho[0].element_size() + hl[0].numel() * hl[0].element_size()

    # causal GQA training shape: forward + backward (if the backward is built)
    train = None
    try:
        train = run_train(fa, dev, args, world)
    except Exception as e:  # reported, not hidden
        train = {"error": f"{type(e).__name__}: {e}"}

    pk = peaks()
    fp4_peak = pk["bf16"] * FP4_OVER_BF16
    if isinstance(train, dict):
        if "fwd_tflops" in train:
            train["fwd_frac"] = round(train["fwd_tflops"] / fp4_peak, 4)
        if "fwd_fp8pv_tflops" in train:
            train["fwd_fp8pv_frac"] = round(train["fwd_fp8pv_tflops"] / (pk["bf16"] * FP8_OVER_BF16), 4)
        if "bwd_tflops" in train:
            train["bwd_frac"] = round(train["bwd_tflops"] / (pk["bf16"] * FP8_OVER_BF16), 4)
            train["bwd_peak"] = round(pk["bf16"] * FP8_OVER_BF16, 1)

    workloads = None
    if not args.no_sweep:
        try:
            workloads = run_workloads(fa, dev, 3)
            for row in workloads:
                row["fp4_frac"] = round(row["fp4_tflops"] / fp4_peak, 4)
                row["bf16_frac"] = round(row["bf16_tflops"] / pk["bf16"], 4)
        except Exception as e:
            workloads = {"error": f"{type(e).__name__}: {e}"}
    clock_info = clocks.stop() if clocks else None

    accuracy = None
    if not args.no_accuracy:
        try:
            accuracy = accuracy_report(fa, dev)
        except Exception as e:
            accuracy = {"error": f"{type(e).__name__}: {e}"}

    achieved = flops / (fwd_mean * 1e-3) / 1e12
    result = {
        "metric": METRIC,
        "value": round(whole_job_tflops(flops, world, ms), 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e2m1",
        "data": "synthetic (seeded bf16 N(0,1) Q/K/V)",
        "config": {"workload": w.name, "B": w.B, "H": w.Hq, "N": w.N, "d": w.d, "causal": False,
                   "step": "quantize Q,K,V (MXFP4, one launch) + Direct-P FP4 forward, bf16 O + LSE",
                   "l2": "flushed (256 MiB write) before every timed step",
                   "parallelism": f"independent problems x{world}"},
        "speedup_vs_bf16": round(bf16_mean / ms, 3),
        "speedup_vs_bf16_kernel_only": round(bf16_mean / fwd_only_ms, 3),
        "fwd_kernel_tflops": round(flops / (fwd_only_ms * 1e-3) / 1e12, 2),
        "bf16_kernel_tflops": round(flops / (bf16_mean * 1e-3) / 1e12, 2),
        "quantize_ms": round(quant_mean, 4),
        "step_q_in_prologue": {"ms_per_step": round(fused_mean, 4),
                               "tflops": round(flops / (fused_mean * 1e-3) / 1e12, 2),
                               "what": "quantize K, V (one launch) + forward on bf16 Q, quantized in its prologue"},
        "quantize_roofline": {"kernel": "quant_qkv_kernel", "bound": "hbm",
                              "achieved": round(quant_bytes / (quant_mean * 1e-3) / 1e9, 1),
                              "peak": pk["hbm"], "unit": "GB/s",
                              "frac": round(quant_bytes / (quant_mean * 1e-3) / 1e9 / pk["hbm"], 4),
                              "algorithmic_bytes": quant_bytes},
        "roofline": {"kernel": "fwd_fp4_kernel<128>", "bound": "tensor", "achieved": round(achieved, 1),
                     "peak": round(fp4_peak, 1), "unit": "TFLOP/s", "frac": round(achieved / fp4_peak, 4),
                     "traffic": fwd_traffic_bytes(),
                     "peak_source": f"{pk['source']} bf16 burst {pk['bf16']} TFLOP/s x nominal FP4/BF16 ratio 6"},
        "e2e": {"value": round(whole_job_tflops(flops, world, e2e_mean), 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_mean, 4),
                "mode": "one fa4fp4_fwd_host call per step (C ABI, pinned host buffers): the call cuts the "
                        "problem into 9 chunks of (batch, head) units (8 x 8, 7, 1) and overlaps each chunk's copy "
                        "in and copy out with other chunks' quantize + forward on two compute streams",
                "link": {"h2d_gbs": round(h2d_gbs, 1), "h2d_bound_ms": round(h2d / h2d_gbs / 1e6, 4),
                         "both_ms": round(both_ms, 4), "frac": round(max(h2d / h2d_gbs / 1e6, both_ms) / e2e_mean, 3),
                         "what": "measured host-to-device copy rate; both_ms: the step's input copy and output "
                                 "copy run at the same time on two streams; the step cannot be shorter than the "
                                 "larger of the two (frac = that bound / ms_per_step)"},
                "serial_ms_per_step": round(e2e_serial_mean, 4),
                "serial_what": "torch copies in, quantize + forward, copies out, all in series on one stream"},
        "gpu_launches": 2 * args.steps,
        "timed_wall_s": round(wall, 3),
        "clocks": clock_info,
        "train": train,
        "workloads": workloads,
        "accuracy": accuracy,
    }
    return result


# ----------------------------------------------------------------------------
# error against unquantized FP64 attention (reported, not gated)
# ----------------------------------------------------------------------------
def fp64_attention_rows(q, k, v, rows, causal):
    """Textbook softmax(QK^T/sqrt(d))V in FP64 on the host for the selected
    query rows ((b*Hq+h)*N+i) of the raw bf16 inputs (K/V head h/(Hq/Hkv))."""
    B, Hq, N, d = q.shape
    group = Hq // k.shape[1]
    rows = torch.as_tensor(rows, dtype=torch.int64)
    out = torch.empty((len(rows), d), dtype=torch.float64)
    bh = rows // N
    for u in torch.unique(bh).tolist():
        sel = (bh == u).nonzero().flatten()
        b, h = divmod(u, Hq)
        i = rows[sel] % N
        kk = k[b, h // group].double()
        s = (q[b, h, i].double() @ kk.T) / (d ** 0.5)
        if causal:
            s = s.masked_fill(torch.arange(N).view(1, N) > i.view(-1, 1), float("-inf"))
        out[sel] = torch.softmax(s, dim=-1) @ v[b, h // group].double()
    return out


def error_vs_fp64(o, ref):
    o = o.double()
    rel = float(torch.linalg.norm(o - ref) / torch.linalg.norm(ref))
    cos = torch.nn.functional.cosine_similarity(o, ref, dim=1)
    return {"rel_l2": round(rel, 5), "cosine": round(float(cos.mean()), 5)}


def accuracy_report(fa, dev):
    """Each forward path's output (FP32) on sampled rows of every workload
    against FP64 softmax attention on the same raw bf16 inputs."""
    from precision_attention_fa4fp4_gb300.inputs import TINY, extreme_logit_inputs, sample_rows
    cases = [(TINY, None), (FWD_4K, [0, 63]), (VIDEO_DIT, [0, 23]), (SWEEP[0], [0]), (SWEEP[11], [63]),
             (TRAIN_8B, [0, 37])]
    report = []
    for w, heads in cases + [("extreme_logits", False), ("extreme_logits", True)]:
        if w == "extreme_logits":
            causal = heads
            q, k, v = extreme_logit_inputs()
            name, rows = f"extreme_logits_n640_d128{'_causal' if causal else ''}", torch.arange(q.numel() // q.shape[-1])
        else:
            causal = w.causal
            q, k, v = make_inputs(w, seed=0)
            name = w.name
            rows = (torch.arange(w.B * w.Hq * w.N) if heads is None
                    else sample_rows(w, tiles_per_head=2, heads=heads))
        ref = fp64_attention_rows(q, k, v, rows, causal)
        qd, kd, vd = (t.to(dev) for t in (q, k, v))
        d = q.shape[-1]
        q4, k4 = fa.quantize(qd), fa.quantize(kd)
        vt = fa.quantize(vd, fa.FMT_MXFP4, fa.ALONG_N)
        o, _ = fa.fwd(q4, k4, vt, causal=causal, out_dtype=fa.OUT_F32)
        row = {"workload": name, "rows": len(rows),
               "directp": error_vs_fp64(o.reshape(-1, d)[rows.to(dev)].cpu(), ref)}
        del o
        v8 = fa.quantize(vd, fa.FMT_MXFP8, fa.ALONG_N)
        o, _ = fa.fwd_fp8pv(q4, k4, v8, causal=causal, out_dtype=fa.OUT_F32)
        row["fp8pv"] = error_vs_fp64(o.reshape(-1, d)[rows.to(dev)].cpu(), ref)
        del o, v8
        qn, kn = fa.quantize_nvfp4(qd), fa.quantize_nvfp4(kd)
        o, _ = fa.fwd_nvfp4(qn, kn, vt, causal=causal, out_dtype=fa.OUT_F32)
        row["nvfp4_qk"] = error_vs_fp64(o.reshape(-1, d)[rows.to(dev)].cpu(), ref)
        del o, qn, kn
        o, _ = fa.bf16_fwd(qd, kd, vd, causal=causal, out_dtype=fa.OUT_F32)
        row["bf16"] = error_vs_fp64(o.reshape(-1, d)[rows.to(dev)].cpu(), ref)
        fa.sync_status()
        report.append(row)
        del o, q4, k4, vt, qd, kd, vd
        torch.cuda.empty_cache()
    return {"reference": "FP64 softmax attention on the raw bf16 inputs (host); rel-L2 over the sampled rows, "
                         "mean cosine per row; every path with FP32 output",
            "rows": report}


def run_workloads(fa, dev, steps):
    """Kernel-only FP4 and BF16 forward TFLOP/s on the sweep and video-DiT
    workloads (inputs quantized beforehand, L2 flushed before every launch)."""
    flush = Flusher(dev)
    out = []
    for w in (VIDEO_DIT,) + SWEEP:
        q, k, v = (t.to(dev) for t in make_inputs(w, seed=0))
        q4, k4 = fa.quantize(q), fa.quantize(k)
        vt = fa.quantize(v, fa.FMT_MXFP4, fa.ALONG_N)
        o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        f_ms, _ = time_steps(lambda ie: fa.fwd(q4, k4, vt, out=o, lse=lse), 2, steps, flush, 1)
        b_ms, _ = time_steps(lambda ie: fa.bf16_fwd(q, k, v, out=o, lse=lse), 2, steps, flush, 1)
        fa.sync_status()
        fm, bm = statistics.mean(f_ms), statistics.mean(b_ms)
        row = {"workload": w.name, "fp4_tflops": round(w.fwd_flops / (fm * 1e-3) / 1e12, 1),
               "bf16_tflops": round(w.fwd_flops / (bm * 1e-3) / 1e12, 1), "speedup": round(bm / fm, 3)}
        if w is VIDEO_DIT:
            # NVFP4 Q/K (the pages' Q/K format) on the outlier-channel workload
            qn, kn = fa.quantize_nvfp4(q), fa.quantize_nvfp4(k)
            n_ms, _ = time_steps(lambda ie: fa.fwd_nvfp4(qn, kn, vt, out=o, lse=lse), 2, steps, flush, 1)
            fa.sync_status()
            row["fp4_nvfp4_qk_tflops"] = round(w.fwd_flops / (statistics.mean(n_ms) * 1e-3) / 1e12, 1)
            del qn, kn
        out.append(row)
        del q, k, v, q4, k4, vt, o, lse
        torch.cuda.empty_cache()
    return out


def run_train(fa, dev, args, world):
    w = TRAIN_8B
    q, k, v, do = (t.to(dev) for t in make_inputs(w, seed=0, with_dout=True))
    B, Hq, Hkv, N, d = w.B, w.Hq, w.Hkv, w.N, w.d
    q4, k4 = fa.quantize(q), fa.quantize(k)
    vt = fa.quantize(v, fa.FMT_MXFP4, fa.ALONG_N)
    q8c = fa.quantize(q, fa.FMT_MXFP8, fa.ALONG_N)
    k8c = fa.quantize(k, fa.FMT_MXFP8, fa.ALONG_N)
    v8r = fa.quantize(v, fa.FMT_MXFP8, fa.ALONG_D)
    o = torch.empty((B, Hq, N, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    flush = Flusher(dev)

    def fwd_step(ie):
        fa.fwd(q4, k4, vt, causal=True, out_dtype=fa.OUT_F32, out=o, lse=lse)

    f_ms, _ = time_steps(fwd_step, args.warmup, args.steps, flush, world)
    fa.sync_status()
    out = {"workload": w.name, "fwd_ms": round(statistics.mean(f_ms), 4),
           "fwd_tflops": round(w.fwd_flops / (statistics.mean(f_ms) * 1e-3) / 1e12, 2)}

    # the FP8 P/V training route of the forward (E4M3 P and V, MXFP8 scales)
    v8n = fa.quantize(v, fa.FMT_MXFP8, fa.ALONG_N)
    o8 = torch.empty_like(o)
    lse8 = torch.empty_like(lse)

    def fwd8_step(ie):
        fa.fwd_fp8pv(q4, k4, v8n, causal=True, out_dtype=fa.OUT_F32, out=o8, lse=lse8)

    f8_ms, _ = time_steps(fwd8_step, args.warmup, args.steps, flush, world)
    fa.sync_status()
    out["fwd_fp8pv_ms"] = round(statistics.mean(f8_ms), 4)
    out["fwd_fp8pv_tflops"] = round(w.fwd_flops / (statistics.mean(f8_ms) * 1e-3) / 1e12, 2)
    ws = torch.empty(max(fa.bwd_workspace_bytes(B, Hq, Hkv, N, d), 16), dtype=torch.uint8, device=dev)
    try:
        fa.bwd(q4, k4, q8c, k8c, v8r, o, do, lse, causal=True, workspace=ws)
        fa.sync_status()
    except Exception as e:
        out["bwd"] = f"unavailable: {e}"
        return out

    def bwd_step(ie):
        fa.bwd(q4, k4, q8c, k8c, v8r, o, do, lse, causal=True, workspace=ws)

    b_ms, _ = time_steps(bwd_step, args.warmup, args.steps, flush, world)
    fa.sync_status()
    bm = statistics.mean(b_ms)
    out.update({"bwd_ms": round(bm, 4), "bwd_tflops": round(w.bwd_flops / (bm * 1e-3) / 1e12, 2)})

    # the whole attention training step of the pages' retained route: every
    # quantization from the bf16 tensors, the FP8 P/V forward, the backward
    def train_step(ie):
        fa.quantize(q, fa.FMT_MXFP4, fa.ALONG_D, out=q4)
        fa.quantize(k, fa.FMT_MXFP4, fa.ALONG_D, out=k4)
        fa.quantize(v, fa.FMT_MXFP8, fa.ALONG_N, out=v8n)
        fa.quantize(q, fa.FMT_MXFP8, fa.ALONG_N, out=q8c)
        fa.quantize(k, fa.FMT_MXFP8, fa.ALONG_N, out=k8c)
        fa.quantize(v, fa.FMT_MXFP8, fa.ALONG_D, out=v8r)
        fa.fwd_fp8pv(q4, k4, v8n, causal=True, out_dtype=fa.OUT_F32, out=o8, lse=lse8)
        fa.bwd(q4, k4, q8c, k8c, v8r, o8, do, lse8, causal=True, workspace=ws)

    t_ms, _ = time_steps(train_step, args.warmup, args.steps, flush, world)
    fa.sync_status()
    tm_ = statistics.mean(t_ms)
    out["step"] = {"ms": round(tm_, 4), "tflops": round((w.fwd_flops + w.bwd_flops) / (tm_ * 1e-3) / 1e12, 2),
                   "launches": 11,
                   "what": "6 quantize launches (MXFP4 Q, K; MXFP8 V along N; MXFP8 Q, K along N, V along d) + "
                           "FP8 P/V forward + backward (preprocess, 2 dO quantizations, main); FLOP = forward + "
                           "backward convention"}
    return out


# ----------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample
# ----------------------------------------------------------------------------
def oracle_sample(heads: int = 8, rows_tiles: int = 32):
    """Quantize the first `heads` (batch, head) pairs of the 4K workload (all
    64 = the whole workload) and run the oracle forward for `rows_tiles`
    128-query tiles of each.  Returns (seconds, flops, threads)."""
    import numpy as np
    import oracle
    w = FWD_4K
    q, k, v = make_inputs(w, seed=0)
    sel = lambda t: t.reshape(1, w.B * w.Hq, w.N, w.d)[:, :heads]
    qf, kf, vf = (sel(t).float().numpy() for t in (q, k, v))
    oracle.build()
    t0 = time.time()
    shp = qf.shape
    Qd = oracle.dequantize(*oracle.quantize(qf, 0, 0), shp, 0, 0)
    Kd = oracle.dequantize(*oracle.quantize(kf, 0, 0), shp, 0, 0)
    Vd = oracle.dequantize(*oracle.quantize(vf, 0, 1), shp, 0, 1)
    rows = np.concatenate([h * w.N + np.arange(rows_tiles * 128) for h in range(heads)])
    oracle.fwd(Qd, Kd, Vd, rows=rows)
    dt = time.time() - t0
    flops = 4.0 * len(rows) * w.N * w.d
    return dt, flops, oracle.num_threads()


def oracle_tiny_full():
    """The tiny workload (B1 H2 N256 d64) in full: oracle quantize of Q/K/V
    and the Direct-P forward of every row.  Returns (seconds, flops)."""
    import oracle
    from precision_attention_fa4fp4_gb300.inputs import TINY
    q, k, v = (t.float().numpy() for t in make_inputs(TINY, seed=0))
    oracle.build()
    reps = 20
    t0 = time.time()
    for _ in range(reps):
        Qd = oracle.dequantize(*oracle.quantize(q, 0, 0), q.shape, 0, 0)
        Kd = oracle.dequantize(*oracle.quantize(k, 0, 0), k.shape, 0, 0)
        Vd = oracle.dequantize(*oracle.quantize(v, 0, 1), v.shape, 0, 1)
        oracle.fwd(Qd, Kd, Vd)
    return (time.time() - t0) / reps, TINY.fwd_flops


def cpu_baseline_entry():
    dt, flops, thr = oracle_sample(heads=FWD_4K.B * FWD_4K.Hq, rows_tiles=32)
    tdt, tflops = oracle_tiny_full()
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
            "sample": "the whole 4K workload (all 64 batch-heads): oracle MXFP4 quantize of Q/K/V and the "
                      f"Direct-P forward of every query row ({flops / 1e9:.1f} GFLOP in {dt:.1f} s)",
            "tiny_full": {"workload": "tiny_b1_h2_n256_d64", "ms": round(tdt * 1e3, 3),
                          "tflops": round(tflops / tdt / 1e12, 6),
                          "what": "whole workload: quantize Q/K/V + Direct-P forward, mean of 20 runs"}}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    times = []
    for _ in range(args.warmup):
        oracle_sample(heads=1, rows_tiles=32)
    flops = None
    thr = 1
    for _ in range(args.steps):
        dt, flops, thr = oracle_sample(heads=1, rows_tiles=32)
        times.append(dt)
    mean = statistics.mean(times)
    val = flops / mean / 1e12
    return {"impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded bf16 N(0,1) Q/K/V)",
            "config": {"workload": FWD_4K.name, "B": FWD_4K.B, "H": FWD_4K.Hq, "N": FWD_4K.N, "d": FWD_4K.d,
                       "causal": False, "step": "CPU oracle on a bounded sample (see cpu_baseline.sample)"},
            "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                             "sample": "4K workload, head 0 of batch 0: oracle quantize of Q/K/V + Direct-P forward of all 4096 query rows"},
            "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the per-workload kernel table")
    ap.add_argument("--no-accuracy", action="store_true", help="skip the error report against FP64 attention")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    rank, world, local = dist_setup(args.gpus)
    res = run_ours(args, rank, world, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline_entry()
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
