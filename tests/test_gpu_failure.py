"""Failure detection on the GPU without a GPU fault.

A test hook (moe_test_arm_timeout) makes one forward's GEMM wait for a
pipeline stage that its producer never fills, or the multi-CTA dispatch's
grid-wide barrier wait for an arrival that never comes, with every wait
limited to a few milliseconds: the bounded wait must give up, the kernel must
drain its copies, free its tensor memory and return, the forward's later
kernels must skip (per-forward abort word), the host must read
MOE_ERR_DEVICE_TIMEOUT, and the next forward on the same context must be
correct again.  Nothing faults, traps or hangs.
"""
import time

import pytest
import torch

import moe_synth
from gpu_util import new_layer, to_dev

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_ffn_gb300 import build
    build.build()
    import moe_expert_ffn_gb300 as mod
    return mod


@pytest.mark.parametrize("mode", ["two", "fused", "split"], ids=["two_launches", "one_launch", "split_launch"])
@pytest.mark.parametrize("which", [1, 2], ids=["l1", "l2"])
def test_timeout_is_reported_and_context_recovers(m, which, mode, monkeypatch):
    # one_launch: both GEMMs in one kernel, where L2 tiles of other CTAs also
    # wait (bounded) for the M block the withheld stage belongs to; split: the
    # first CTA of the L1 (or of the L2) CTA set withholds its stage, and the
    # L2 CTAs waiting on that M block give up too
    monkeypatch.setenv("MOE_FUSED", "1" if mode == "fused" else "0")
    monkeypatch.setenv("MOE_SPLIT", "1" if mode == "split" else "0")
    wl = moe_synth.custom(T=96, H=512, I=256, E=4, k=2, seed=71)
    inp = to_dev(moe_synth.make_inputs(wl), DEV)
    layer = new_layer(m, wl, DEV)
    layer.transform_weights(inp["w1"], inp["w1_sf"], inp["w2"], inp["w2_sf"])
    args = (inp["x"], inp["x_sf"], inp["topk_idx"], inp["topk_weights"])
    y0 = layer.forward(*args).clone()
    assert layer.device_status() == m.MOE_OK

    layer.arm_timeout_test(which, 20000)          # 20 ms limit per wait
    t0 = time.monotonic()
    layer.forward(*args)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert layer.device_status() == m.MOE_ERR_DEVICE_TIMEOUT
    assert elapsed < 5.0, elapsed                  # gave up, did not wait the default 2 s per wait

    # the status read cleared the error word; the context is usable and exact again
    y1 = layer.forward(*args)
    assert layer.device_status() == m.MOE_OK
    assert torch.equal(y1, y0)


def test_arm_rejects_bad_arguments(m):
    wl = moe_synth.WORKLOADS["tiny"]
    layer = new_layer(m, wl, DEV)
    for which, lim in ((0, 1000), (4, 1000), (1, 0)):
        with pytest.raises(m.MoEError):
            layer.arm_timeout_test(which, lim)


@pytest.mark.parametrize("fused", ["0", "1"], ids=["dispatch_kernel", "one_launch"])
def test_dispatch_barrier_timeout_is_reported_and_skips_the_forward(m, fused, monkeypatch):
    # 8192 routed pairs: the dispatch runs over 8 CTAs with a grid-wide
    # barrier (or, in the one-launch forward, over every CTA); the hook makes
    # CTA 0 withhold its arrival
    monkeypatch.setenv("MOE_FUSED", fused)
    wl = moe_synth.custom(T=2048, H=256, I=128, E=64, k=4, seed=72, routing="zipf")
    inp = to_dev(moe_synth.make_inputs(wl), DEV)
    layer = new_layer(m, wl, DEV)
    layer.transform_weights(inp["w1"], inp["w1_sf"], inp["w2"], inp["w2_sf"])
    args = (inp["x"], inp["x_sf"], inp["topk_idx"], inp["topk_weights"])
    y0 = layer.forward(*args).clone()
    assert layer.device_status() == m.MOE_OK

    layer.arm_timeout_test(3, 20000)
    t0 = time.monotonic()
    layer.forward(*args)
    torch.cuda.synchronize()
    assert time.monotonic() - t0 < 5.0
    assert layer.device_status() == m.MOE_ERR_DEVICE_TIMEOUT

    y1 = layer.forward(*args)
    assert layer.device_status() == m.MOE_OK
    assert torch.equal(y1, y0)


def test_forward_after_a_timeout_runs_without_reading_the_status(m):
    # the abort word is per forward: the forward after a timed-out one runs in
    # full even though the sticky status bit has not been read yet
    wl = moe_synth.custom(T=96, H=512, I=256, E=4, k=2, seed=73)
    inp = to_dev(moe_synth.make_inputs(wl), DEV)
    layer = new_layer(m, wl, DEV)
    layer.transform_weights(inp["w1"], inp["w1_sf"], inp["w2"], inp["w2_sf"])
    args = (inp["x"], inp["x_sf"], inp["topk_idx"], inp["topk_weights"])
    y0 = layer.forward(*args).clone()
    assert layer.device_status() == m.MOE_OK
    layer.arm_timeout_test(1, 20000)
    layer.forward(*args)
    y1 = layer.forward(*args)
    torch.cuda.synchronize()
    assert torch.equal(y1, y0)
    assert layer.device_status() == m.MOE_ERR_DEVICE_TIMEOUT



@pytest.mark.parametrize("which", [1, 2], ids=["l1", "l2"])
def test_fp4_timeout_is_reported_and_context_recovers(m, which):
    # the block-scaled FP4-weight GEMMs: MMA issuer, scale writers and
    # epilogue all leave through the abort flag
    wl = moe_synth.custom(T=96, H=512, I=256, E=4, k=2, seed=74, wfmt=1)
    inp = to_dev(moe_synth.make_inputs(wl), DEV)
    layer = new_layer(m, wl, DEV, wfmt=1)
    layer.transform_weights(inp["w1"], inp["w1_sf"], inp["w2"], inp["w2_sf"])
    args = (inp["x"], inp["x_sf"], inp["topk_idx"], inp["topk_weights"])
    y0 = layer.forward(*args).clone()
    assert layer.device_status() == m.MOE_OK
    layer.arm_timeout_test(which, 20000)
    t0 = time.monotonic()
    layer.forward(*args)
    torch.cuda.synchronize()
    assert time.monotonic() - t0 < 5.0
    assert layer.device_status() == m.MOE_ERR_DEVICE_TIMEOUT
    y1 = layer.forward(*args)
    assert layer.device_status() == m.MOE_OK
    assert torch.equal(y1, y0)


def test_first_forward_of_a_context_times_out_in_dispatch(m):
    # a context whose very first forward stops at the dispatch barrier: the
    # later steps skip instead of reading tables no forward has written, and
    # the second forward equals the forward of a fresh context
    wl = moe_synth.custom(T=2048, H=256, I=128, E=64, k=4, seed=75, routing="zipf")
    inp = to_dev(moe_synth.make_inputs(wl), DEV)
    args = (inp["x"], inp["x_sf"], inp["topk_idx"], inp["topk_weights"])
    ref = new_layer(m, wl, DEV)
    ref.transform_weights(inp["w1"], inp["w1_sf"], inp["w2"], inp["w2_sf"])
    y_ref = ref.forward(*args).clone()
    assert ref.device_status() == m.MOE_OK
    layer = new_layer(m, wl, DEV)
    layer.transform_weights(inp["w1"], inp["w1_sf"], inp["w2"], inp["w2_sf"])
    layer.arm_timeout_test(3, 20000)
    layer.forward(*args)
    torch.cuda.synchronize()
    assert layer.device_status() == m.MOE_ERR_DEVICE_TIMEOUT
    y1 = layer.forward(*args)
    assert layer.device_status() == m.MOE_OK
    assert torch.equal(y1, y_ref)
