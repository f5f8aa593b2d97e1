"""bench.py's host logic on CPU: the work model behind every roofline figure,
the roofline arithmetic, the launch count, and the reference arm's JSON line.

The work-model values are checked against the layer's sizes worked out by
hand (FLOPs 6·P·H·I over routed pairs; FP8 weights H·I bytes per matrix plus
one f32 per 128x128 block), not against the formula in bench.py.
"""
import math
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import moe_synth  # noqa: E402


def _counts(wl):
    idx, _ = moe_synth.make_routing(wl)
    return torch.bincount(idx.flatten()[idx.flatten() >= 0], minlength=wl.E).tolist()


def test_decode_work_model():
    wl = moe_synth.WORKLOADS["decode"]
    counts = _counts(wl)
    wm = bench.work_model(wl, counts)
    assert wm["pairs"] == 128 * 8
    n = sum(1 for c in counts if c > 0)
    assert wm["n_touched"] == n and 240 <= n <= 256    # uniform routing of 1024 pairs over 256 experts
    # per expert: W1 2·2048·7168 codes + 32·56 scales, W2 7168·2048 codes + 56·16 scales
    per_expert = (29_360_128 + 7_168) + (14_680_064 + 3_584)
    assert per_expert == 44_050_944
    weights = n * per_expert
    lay = wm["bytes"]["layer"]
    assert weights < lay < weights + 4_000_000           # plus x, its scales, routing and y (3.7 MB)
    assert wm["flops"]["layer"] == 6 * 1024 * 7168 * 2048
    assert wm["flops"]["l1"] + wm["flops"]["l2"] == wm["flops"]["layer"]


def test_prefill_and_wide_flops():
    pre = moe_synth.WORKLOADS["prefill"]
    wide = moe_synth.WORKLOADS["wide"]
    assert math.isclose(bench.work_model(pre, _counts(pre))["flops"]["layer"], 2.886e12, rel_tol=1e-3)
    assert math.isclose(bench.work_model(wide, _counts(wide))["flops"]["layer"], 1.443e12, rel_tol=1e-3)


def test_roofline_bound_and_fraction():
    peaks = {"hbm_gbs": 6777.6, "bf16_tflops": 1861.9}
    dec = moe_synth.WORKLOADS["decode"]
    wide = moe_synth.WORKLOADS["wide"]
    r = bench.roofline_for("layer", bench.work_model(dec, _counts(dec)), 1.6e-3, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert math.isclose(r["frac"], r["achieved"] / 6777.6)
    w = bench.roofline_for("layer", bench.work_model(wide, _counts(wide)), 0.8e-3, peaks)
    assert w["bound"] == "tensor" and w["unit"] == "TFLOP/s"
    assert math.isclose(w["peak"], 2 * 1861.9)           # FP8 dense = 2 x bf16
    assert math.isclose(w["achieved"], 1.443e12 / 0.8e-3 / 1e12, rel_tol=1e-3)


def test_launches_per_forward():
    os.environ.pop("MOE_L1_A", None)
    assert bench.launches_per_forward(moe_synth.WORKLOADS["decode"]) == 4   # rows gathered inside L1
    assert bench.launches_per_forward(moe_synth.WORKLOADS["prefill"]) == 5  # plus the pool copy


def test_reference_line_contract():
    class Args:
        steps, warmup, gpus = 1, 0, 1
    out = bench.run_reference(Args(), moe_synth.WORKLOADS["tiny"], rank=0, world=1)
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline",
                "e2e", "gpu_launches"):
        assert key in out, key
    assert out["impl"] == "reference" and out["value"] > 0 and out["unit"] == "tokens/s"
    assert out["config"]["workload"] == "tiny"
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["cores"] >= 1
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["e2e"]["value"] == out["value"]
