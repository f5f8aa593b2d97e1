"""The multi-GPU path of bench.py on CPU: two gloo ranks, no GPU.

With N > 1 every rank runs an independent replica of the layer on its own
batch of tokens (weak scaling, no data-path collective); the only collective
is the max over ranks of the step time, and the whole-job value counts every
replica's tokens over that slowest step.  These tests run that host logic as
two processes with the gloo backend.
"""
import math
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import moe_synth  # noqa: E402


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, step_ms, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.reduce_max(step_ms[rank], world)
        dist.barrier()
        q.put((rank, ms, bench.job_value(world, 128, ms)))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_whole_job_value():
    world, port = 2, _free_port()
    step_ms = [1.5, 2.0]   # rank 1 is the slower replica
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, step_ms, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in got:
        assert ms == max(step_ms), rank                 # every rank sees the slowest step
        assert math.isclose(value, world * 128 / (max(step_ms) / 1e3))


def test_one_rank_needs_no_collective():
    assert bench.reduce_max(3.25, 1) == 3.25
    assert math.isclose(bench.job_value(1, 4096, 2.0), 4096 / 2e-3)


def test_replicas_share_weights_not_tokens():
    wl = moe_synth.WORKLOADS["tiny"]
    a = moe_synth.make_inputs(wl, batch=0)
    b = moe_synth.make_inputs(wl, batch=1)
    for name in ("w1", "w1_sf", "w2", "w2_sf"):
        assert torch.equal(a[name], b[name]), name       # one layer, replicated
    assert not torch.equal(a["x"], b["x"])                # each rank its own batch
    assert not torch.equal(a["topk_idx"], b["topk_idx"])


def test_reference_arm_runs_on_rank_zero_only():
    class Args:
        steps, warmup, gpus = 1, 0, 2
    assert bench.run_reference(Args(), moe_synth.WORKLOADS["tiny"], rank=1, world=2) is None
