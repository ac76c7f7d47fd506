"""The bench's multi-rank path on CPU: two gloo ranks in separate processes.

What runs on the GPU under torchrun is one independent copy of the workload
per rank (weak scaling, no data-path collective); the host logic around it is
the barrier, the max over ranks of the timed region, the whole-job aggregate,
rank-dependent input seeds, and a reference arm that runs on rank 0 only.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    from precision_attention_fa4fp4_gb300.inputs import TINY, make_inputs
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # every rank waits at the barrier; the slowest rank's time wins
        bench.barrier(world, sync_cuda=False)
        t = bench.max_over_ranks(1.0 + rank, world, device="cpu")
        # each rank's inputs are its own (seed = rank), so no rank repeats another's work
        x = make_inputs(TINY, seed=rank)[0].float()
        xs = [torch.zeros_like(x) for _ in range(world)]
        dist.all_gather(xs, x)
        distinct = not torch.equal(xs[0], xs[1])
        ref = bench.run_reference(type("A", (), {"warmup": 0, "steps": 0})(), rank, world) if rank != 0 else None
        q.put((rank, t, distinct, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict((r, (t, distinct, ref)) for r, t, distinct, ref in (q.get(timeout=120) for _ in range(world)))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 2.0          # max over ranks
    assert out[0][1] and out[1][1]                # rank-seeded inputs differ
    assert out[1][2] is None                      # the reference arm does no work off rank 0


def test_whole_job_aggregate():
    sys.path.insert(0, ROOT)
    import bench
    # two ranks each doing 1e12 FLOP, slowest in 10 ms: 200 TFLOP/s for the job
    assert abs(bench.whole_job_tflops(1e12, 2, 10.0) - 200.0) < 1e-9
    assert bench.max_over_ranks(3.5, 1) == 3.5
