#!/usr/bin/env python3
"""Throughput of the MegaMoE expert layer on GB300 (one JSON line on stdout).

A step is one forward of the whole layer (dispatch -> L1 GEMM + SwiGLU +
requant -> L2 GEMM -> combine) over one batch of T synthetic tokens of the
chosen workload (default: prefill, T=4096 H=7168 I=2048 E=256 k=8, Zipf-skewed
routing: the largest configuration of the layer that fits one GPU).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

With N > 1 (under torchrun) every rank runs an independent replica on its own
batch (weak scaling, no data-path collective); the timed region is bracketed
by a barrier and the max time over ranks is reported.  `--impl reference`
times the CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s at 1 GB300; achieved fraction of FP8-tensor / HBM roofline"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0          # nominal dense ratio (4.5 / 2.25 PFLOP/s)
NOMINAL_HBM_GBS = 7900.0     # HBM3e nominal, for context beside the measured copy peak
# Context figures measured on the GB300s (not the roofline denominators,
# which come from MEASURED_PEAKS.json): an FP8 E4M3 8192^3 GEMM through
# torch._scaled_mm (cuBLAS) at a median 1462 MHz under the power cap, and the
# tcgen05 kind::f8f6f4 issue rate per SM per clock.
CUBLAS_FP8_TFLOPS = 3371.2
TCGEN05_FP8_MAC_PER_CLK_SM = 8192
# A read-only HBM stream (16-byte loads over 8 GiB, best of 10, CUDA events):
# the ceiling of a read-mostly kernel, which the read+write copy peak
# understates.
READ_STREAM_GBS = 7049.0
STAGES = ("dispatch", "l1", "l2", "combine")
KERNELS = {"dispatch": "dispatch_kernel", "l1": "l1_kernel", "l2": "l2_kernel", "combine": "combine_kernel"}
KERNELS_FP4 = dict(KERNELS, l1="fp4_gemm_kernel_l1", l2="fp4_gemm_kernel_l2")


def kernel_name(stage, wl):
    """The library kernel that runs a stage of this workload (the dispatch
    over several CTAs for batches of 8192 routed pairs or more)."""
    if stage == "dispatch" and wl.T * wl.k >= 8192:
        return "dispatch_mc_kernel"
    return (KERNELS_FP4 if wl.wfmt == 1 else KERNELS)[stage]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="prefill")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--experts", type=int, default=None,
                    help="override E (smaller profiling cases; not a bench line)")
    ap.add_argument("--tokens", type=int, default=None, help="override T")
    return ap.parse_args()


# --------------------------------------------------------------------------- peaks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            pk = json.load(fh)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# --------------------------------------------------------------------------- work model
def work_model(wl, counts):
    """Algorithmic bytes and flops per forward, per stage and for the layer.

    Weight bytes count only touched experts (count > 0) with their canonical
    f32 block scales; activations count what each kernel must read or write."""
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    n_touch = int(sum(1 for c in counts if c > 0))
    P = int(sum(counts))
    if wl.wfmt == 0:   # FP8 codes + f32 128x128 block scales
        w1 = 2 * I * H + (2 * I // 128) * (H // 128) * 4
        w2 = H * I + (H // 128) * (I // 128) * 4
        x = T * H + T * (H // 128) * 4
    else:              # packed E2M1 + UE8M0 per 32
        w1 = 2 * I * H // 2 + 2 * I * H // 32
        w2 = H * I // 2 + H * I // 32
        x = T * H + T * (H // 32)
    routing = T * k * 8
    y = T * H * 2
    acts = P * I + P * (I // 64) * 4
    l2o = P * H * 2
    return {
        "n_touched": n_touch, "pairs": P,
        "bytes": {
            "dispatch": T * k * 4 + P * 8 + E * 12,
            "l1": n_touch * w1 + x + P * 8 + acts,
            "l2": n_touch * w2 + acts + l2o,
            "combine": l2o + y + T * k * 4,
            "layer": n_touch * (w1 + w2) + x + routing + y,
        },
        "flops": {"dispatch": 0, "l1": 2 * P * 2 * I * H, "l2": 2 * P * H * I, "combine": 0,
                  "layer": 6 * P * H * I},
    }


def roofline_for(stage, wm, seconds, peaks, traffic=None):
    b, f = wm["bytes"][stage], wm["flops"][stage]
    tens = peaks["bf16_tflops"] * FP8_OVER_BF16 * 1e12
    hbm = peaks["hbm_gbs"] * 1e9
    if f / tens > b / hbm:
        ach = f / seconds / 1e12
        peak = tens / 1e12
        out = {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s"}
    else:
        ach = b / seconds / 1e9
        peak = hbm / 1e9
        out = {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s"}
    out["frac"] = ach / peak
    out["traffic"] = traffic
    return out


def alt_fractions(roof, clk):
    """The achieved figure against other denominators, for context: HBM-bound
    kernels against the nominal bandwidth and a measured read-only stream
    (the measured copy peak counts the bytes of a read+write copy, so a
    read-mostly stream can pass 1.0 of it),
    tensor-bound ones against a measured cuBLAS FP8 GEMM and against the
    tcgen05 FP8 issue rate at the clock sampled during the timed region."""
    a = roof["achieved"]
    if roof["bound"] == "hbm":
        out = {"vs_nominal_hbm": a / NOMINAL_HBM_GBS, "vs_read_stream": a / READ_STREAM_GBS}
    else:
        out = {"vs_cublas_fp8": a / CUBLAS_FP8_TFLOPS}
        if clk and clk.get("sm_mhz"):
            rate = TCGEN05_FP8_MAC_PER_CLK_SM * 2 * 152 * clk["sm_mhz"] * 1e6 / 1e12
            out["vs_tcgen05_rate_at_clock"] = a / rate
    out["above_measured_peak"] = roof["frac"] > 1.0
    return out


def launches_per_forward(wl):
    """Library kernels per forward: dispatch, L1, L2, combine, plus the pool
    copy when token rows are not gathered inside L1 (the library's rule:
    gather when T*k <= 4E, unless MOE_L1_A overrides it)."""
    mode = os.environ.get("MOE_L1_A", "")
    gather = (mode == "gather") if mode in ("gather", "pool") else wl.T * wl.k <= 4 * wl.E
    return 4 if gather else 5


def profiled_traffic(stage, wl):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload (a line `traffic_bytes_per_launch: N`), or None."""
    path = os.path.join(ROOT, "profiles", f"{kernel_name(stage, wl)}_{wl.name}.md")
    try:
        with open(path) as fh:
            for line in fh:
                if line.strip().startswith("traffic_bytes_per_launch:"):
                    v = line.split(":", 1)[1].strip()
                    return None if v in ("", "null", "None") else float(v)
    except OSError:
        pass
    return None


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """Polls NVML (SM clock, max clock, throttle reasons) in a thread."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x2: "applications_clocks_setting", 0x1: "gpu_idle"}

    def __init__(self, torch_device_index=0, period_s=0.005):
        self.ok = False
        self.samples = []
        self.period = period_s
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            handle_ok = False
            try:
                import torch
                p = torch.cuda.get_device_properties(torch_device_index)
                bus = f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0".encode()
                handle_ok = self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.h)) == 0
            except Exception:
                handle_ok = False
            if not handle_ok and self.nvml.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
            self.max_mhz = mx.value
            self.ok = True
        except OSError:
            pass

    def _one(self):
        mhz = ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz))
        fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        fn(self.h, ctypes.byref(reasons))
        self.samples.append((mhz.value, reasons.value))

    def _loop(self):
        while not self._stop.is_set():
            self._one()
            time.sleep(self.period)

    def start(self):
        if not self.ok:
            return
        self._stop = threading.Event()
        self._one()
        self._t = threading.Thread(target=self._loop, daemon=True)
        self._t.start()

    def stop(self):
        if not self.ok:
            return None
        self._stop.set()
        self._t.join()
        self._one()
        busy = [s for s in self.samples if not (s[1] & 0x1)] or self.samples
        reasons = 0
        for _, r in busy:
            reasons |= r
        return {"sm_mhz": statistics.median(m for m, _ in busy), "sm_max_mhz": self.max_mhz,
                "reasons": [n for b, n in self.REASONS.items() if reasons & b and b != 0x1],
                "samples": len(busy)}


# --------------------------------------------------------------------------- oracle (CPU)
def cpu_sample_inputs(wl, n_tokens, seed_offset=0):
    """Inputs for `n_tokens` tokens of the workload with only the experts they
    route to (ids remapped), generated on the host."""
    import torch
    import moe_synth
    inp = moe_synth.make_inputs(wl, device="cpu", weights=False)
    g = torch.Generator().manual_seed(1234 + seed_offset)
    tokens = torch.randperm(wl.T, generator=g)[:n_tokens].sort().values
    idx = inp["topk_idx"][tokens]
    used = torch.unique(idx[idx >= 0])
    remap = torch.full((wl.E,), -1, dtype=torch.int32)
    remap[used] = torch.arange(used.numel(), dtype=torch.int32)
    w1, w1_sf, w2, w2_sf = moe_synth.make_weights(wl, "cpu", experts=used.tolist())
    return {"x": inp["x"][tokens].contiguous(), "x_sf": inp["x_sf"][tokens].contiguous(),
            "topk_idx": torch.where(idx >= 0, remap[idx.clamp_min(0).long()], idx).contiguous(),
            "topk_weights": inp["topk_weights"][tokens].contiguous(),
            "w1": w1, "w1_sf": w1_sf, "w2": w2, "w2_sf": w2_sf}


def time_oracle(inp, wfmt=0):
    import oracle
    t0 = time.perf_counter()
    oracle.forward(inp, wfmt=wfmt)
    return time.perf_counter() - t0


# --------------------------------------------------------------------------- replicas
def reduce_max(x: float, world: int, device=None) -> float:
    """The largest of every rank's x (the slowest replica sets the step time).

    `device` is where the collective's tensor lives: the rank's GPU under
    NCCL, None (host memory) under gloo."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every replica's tokens over the slowest step."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


def run_reference(args, wl, rank, world):
    """The reference arm: the CPU oracle, on a bounded token sample per step."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    threads = oracle.num_threads()
    n_tok = max(1, min(wl.T, threads))
    inp = cpu_sample_inputs(wl, n_tok)
    for _ in range(args.warmup):
        time_oracle(inp, wl.wfmt)
    times = [time_oracle(inp, wl.wfmt) for _ in range(args.steps)]
    total = sum(times)
    value = n_tok * args.steps / total
    sample = (f"{n_tok} tokens x {wl.k} slots of the {wl.name} workload per step "
              f"(H={wl.H}, I={wl.I}), experts they route to only")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, DeepSeek-V3-shaped)",
        "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# --------------------------------------------------------------------------- our arm
def run_ours(args, wl, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import moe_expert_ffn_gb300 as m
    import moe_synth
    from moe_expert_ffn_gb300 import build as mbuild

    mbuild.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp = moe_synth.make_inputs(wl, device=dev, batch=rank)
    layer = m.MoELayer(wl.T, wl.H, wl.I, wl.E, wl.k, wfmt=wl.wfmt, device=dev)
    layer.transform_weights(inp["w1"], inp["w1_sf"], inp["w2"], inp["w2_sf"])
    del inp["w1"], inp["w2"]
    y = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        layer.forward(inp["x"], inp["x_sf"], inp["topk_idx"], inp["topk_weights"], y=y)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if layer.device_status() != m.MOE_OK:
        raise RuntimeError("device error during warm-up")
    counts, _, _ = layer.get_dispatch(wl.T)
    counts = counts.cpu().tolist()

    # ---- timed region (device)
    clocks = ClockSampler(local_rank)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    layer.profile_begin(args.steps)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    ms = ev0.elapsed_time(ev1) / args.steps
    stage_ms, nfw = layer.profile_end()
    if layer.device_status() != m.MOE_OK:
        raise RuntimeError("device error in the timed region")
    ms = reduce_max(ms, world, dev)

    # ---- end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e:
        hx = inp["x"].cpu().pin_memory()
        hsf = inp["x_sf"].cpu().pin_memory()
        hidx = inp["topk_idx"].cpu().pin_memory()
        hw = inp["topk_weights"].cpu().pin_memory()
        hy = torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
        for _ in range(args.warmup):
            layer.forward_host(hx, hsf, hidx, hw, y=hy)
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            layer.forward_host(hx, hsf, hidx, hw, y=hy)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        e_ms = reduce_max(e0.elapsed_time(e1) / args.steps, world, dev)
        h2d = hx.numel() + hsf.numel() * 4 + hidx.numel() * 4 + hw.numel() * 4
        e2e = {"value": job_value(world, wl.T, e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": hy.numel() * 2, "ms_per_step": e_ms}

    if rank != 0:
        return None

    peaks = load_peaks()
    wm = work_model(wl, counts)
    per_launch = {s: stage_ms[s] / max(nfw, 1) for s in STAGES}
    dom = max(("l1", "l2", "combine", "dispatch"), key=lambda s: per_launch[s])
    roof = roofline_for(dom, wm, per_launch[dom] / 1e3, peaks, profiled_traffic(dom, wl))
    roof["kernel"] = kernel_name(dom, wl)
    roof["peak_source"] = f"{peaks['source']} ({'HBM copy' if roof['bound'] == 'hbm' else 'bf16 cuBLAS x2 for FP8'})"
    roof["frac_alt"] = alt_fractions(roof, clk)
    layer_roof = roofline_for("layer", wm, ms / 1e3, peaks)
    tens = peaks["bf16_tflops"] * FP8_OVER_BF16 * 1e12
    t_roof = max(wm["flops"]["layer"] / tens, wm["bytes"]["layer"] / (peaks["hbm_gbs"] * 1e9))

    out = {
        "metric": METRIC, "value": job_value(world, wl.T, ms), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3 (fp32 accumulate)" if wl.wfmt == 0 else "fp8_e4m3 x fp4_e2m1, ue8m0 block scales (fp32 accumulate)",
        "data": "synthetic (seeded, DeepSeek-V3-shaped, random-init weights)",
        "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
                   "touched_experts": wm["n_touched"], "parallelism": f"dp{world} (independent replicas)",
                   "l2_cache": f"inputs larger than L2: touched expert weights "
                               f"{wm['bytes']['layer'] / 1e9:.2f} GB per step"},
        "tflops": wm["flops"]["layer"] / (ms / 1e3) / 1e12,
        "layer_roofline": {"t_roofline_ms": t_roof * 1e3, "frac": t_roof / (ms / 1e3),
                           "frac_alt": alt_fractions(layer_roof, clk),
                           "bound": layer_roof["bound"], "achieved": layer_roof["achieved"],
                           "unit": layer_roof["unit"]},
        "roofline": roof,
        "stage_ms": per_launch,
        "gpu_launches": launches_per_forward(wl) * args.steps,
        "e2e": e2e,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        threads = oracle.num_threads()
        n_tok = max(1, min(wl.T, 6 * threads))       # about 10-15 s of host work
        cin = cpu_sample_inputs(wl, n_tok, seed_offset=1)
        dt = time_oracle(cin, wl.wfmt)
        out["cpu_baseline"] = {"value": n_tok / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
                               "sample": f"{n_tok} tokens x {wl.k} slots of the {wl.name} workload "
                                         f"({dt:.1f} s wall on the host cores)"}
    return out


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    import moe_synth
    if args.workload not in moe_synth.WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}")
    wl = moe_synth.WORKLOADS[args.workload]
    if args.experts or args.tokens:
        import dataclasses
        E = args.experts or wl.E
        T = args.tokens or wl.T
        wl = dataclasses.replace(wl, E=E, T=T, name=f"{wl.name}_T{T}_E{E}")
    if args.impl == "reference":
        out = run_reference(args, wl, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        out = run_ours(args, wl, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
