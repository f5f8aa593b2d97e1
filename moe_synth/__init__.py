"""Seeded synthetic inputs for the MegaMoE expert layer.

The one module that both the CUDA path's tests/benchmark and the CPU oracle
draw their inputs from.  It holds none of the layer's arithmetic: it only
draws random numbers and packs them into the input formats the layer takes
(FP8 E4M3 codes with their scales, E2M1 nibbles with UE8M0 scales, top-k
routing).  Format conversions of inputs use PyTorch's own casts where PyTorch
has one.

Workloads (shapes of the DeepSeek-V3-style configurations the pages test,
MegaMoE SM90 Implementation Design (Final), §20.2, and PR357 Green-Context
Split MegaMoE code review, §8):

    tiny     T=32   H=256  I=128   E=8   k=2  uniform routing          seed 0
    decode   T=128  H=7168 I=2048  E=256 k=8  uniform routing          seed 1
    prefill  T=4096 H=7168 I=2048  E=256 k=8  Zipf(1.2)-skewed routing seed 2
    wide     T=2048 H=4096 I=14336 E=8   k=2  uniform routing          seed 3
    fp4      T=1024 H=7168 I=2048  E=256 k=8  16 experts forced empty  seed 4
             (FP4 E2M1 weights, UE8M0 per-1x32 scales everywhere)

Recipe: x = bf16 N(0,1) -> FP8 E4M3 with per-1x128 f32 scales amax/448 (fp4:
per-1x32 UE8M0 scales 2^ceil(log2(amax/448))); router logits N(0,1) [T,E]
(prefill: + log p_pi(e), p_r ~ r^-1.2 over a seeded permutation pi; fp4: 16
seeded experts' logits = -inf) -> softmax -> top-k -> weights renormalised to
sum 1; W1 [E,2I,H] ~ N(0,1/H), W2 [E,H,I] ~ N(0,1/I) -> FP8 E4M3 with 128x128
f32 block scales amax/448 (fp4: E2M1 with per-1x32 UE8M0 scales
2^ceil(log2(amax/6)), two codes per byte, low nibble = even k).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    seed: int
    routing: str = "uniform"      # "uniform" | "zipf"
    wfmt: int = 0                 # 0: FP8 weights, f32 block scales; 1: FP4 E2M1 weights, UE8M0
    n_empty: int = 0              # experts forced empty (logits = -inf)
    zipf_alpha: float = 1.2

    @property
    def pairs(self) -> int:
        return self.T * self.k


WORKLOADS = {
    "tiny": Workload("tiny", 32, 256, 128, 8, 2, 0),
    "decode": Workload("decode", 128, 7168, 2048, 256, 8, 1),
    "prefill": Workload("prefill", 4096, 7168, 2048, 256, 8, 2, routing="zipf"),
    "wide": Workload("wide", 2048, 4096, 14336, 8, 2, 3),
    "fp4": Workload("fp4", 1024, 7168, 2048, 256, 8, 4, wfmt=1, n_empty=16),
}


def custom(T, H, I, E, k, seed=0, routing="uniform", wfmt=0, n_empty=0, name="custom") -> Workload:
    return Workload(name, T, H, I, E, k, seed, routing=routing, wfmt=wfmt, n_empty=n_empty)


def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + stream)
    return g


# ---- input format packing --------------------------------------------------
def _pow2_scale_exponent(ratio: torch.Tensor) -> torch.Tensor:
    """Exponent e of the smallest power of two 2^e >= ratio (ratio > 0), int32."""
    m, e = torch.frexp(ratio)
    e = e.to(torch.int32)
    e = torch.where(m == 0.5, e - 1, e)
    e = torch.where(ratio > 0, e, torch.full_like(e, -127))
    return e.clamp(-127, 127)


def _to_e4m3_codes(v: torch.Tensor) -> torch.Tensor:
    return v.to(torch.float8_e4m3fn).view(torch.uint8)


def pack_fp8_rows_f32(xf: torch.Tensor, group: int = 128):
    """[R, K] float -> (codes uint8 [R,K], f32 scales [R,K/group]) with amax/448."""
    R, K = xf.shape
    g = xf.view(R, K // group, group)
    amax = g.abs().amax(dim=2)
    sf = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = _to_e4m3_codes(g / sf.unsqueeze(2)).view(R, K)
    return q, sf.to(torch.float32).contiguous()


def pack_fp8_rows_ue8m0(xf: torch.Tensor, group: int = 32):
    """[R, K] float -> (codes uint8 [R,K], UE8M0 codes uint8 [R,K/group])."""
    R, K = xf.shape
    g = xf.view(R, K // group, group)
    amax = g.abs().amax(dim=2)
    e = _pow2_scale_exponent(amax / 448.0)
    sf = torch.ldexp(torch.ones_like(amax), e.to(amax.dtype))
    q = _to_e4m3_codes(g / sf.unsqueeze(2)).view(R, K)
    return q, (e + 127).to(torch.uint8).contiguous()


def pack_fp8_blocks(w: torch.Tensor, block: int = 128):
    """[N, K] float -> (codes uint8 [N,K], f32 scales [N/128, K/128]) with amax/448."""
    N, K = w.shape
    g = w.view(N // block, block, K // block, block)
    amax = g.abs().amax(dim=(1, 3))
    sf = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = _to_e4m3_codes(g / sf[:, None, :, None]).view(N, K)
    return q, sf.to(torch.float32).contiguous()


_E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def pack_e2m1_rows(w: torch.Tensor, group: int = 32):
    """[N, K] float -> (packed uint8 [N, K/2] low nibble = even k, UE8M0 uint8 [N, K/32])."""
    N, K = w.shape
    g = w.view(N, K // group, group)
    amax = g.abs().amax(dim=2)
    e = _pow2_scale_exponent(amax / 6.0)
    sf = torch.ldexp(torch.ones_like(amax), e.to(amax.dtype))
    v = (g / sf.unsqueeze(2)).view(N, K)
    grid = torch.tensor(_E2M1_GRID, device=w.device, dtype=v.dtype)
    mag = torch.argmin((v.abs().unsqueeze(-1) - grid).abs(), dim=-1).to(torch.uint8)
    nib = mag | ((v < 0).to(torch.uint8) << 3)
    packed = nib[:, 0::2] | (nib[:, 1::2] << 4)
    return packed.contiguous(), (e + 127).to(torch.uint8).contiguous()


# ---- the pieces of one workload --------------------------------------------
def make_routing(wl: Workload, device="cpu"):
    """topk_idx int32 [T,k], topk_weights f32 [T,k] (softmax -> top-k -> renormalise)."""
    g = _gen(device, wl.seed, 1)
    logits = torch.randn(wl.T, wl.E, generator=g, device=device, dtype=torch.float32)
    if wl.routing == "zipf":
        perm = torch.randperm(wl.E, generator=g, device=device)
        ranks = torch.arange(1, wl.E + 1, device=device, dtype=torch.float32)
        logp = -wl.zipf_alpha * torch.log(ranks)
        logp = logp - torch.logsumexp(logp, 0)
        bias = torch.empty(wl.E, device=device, dtype=torch.float32)
        bias[perm] = logp
        logits = logits + bias
    if wl.n_empty:
        empty = torch.randperm(wl.E, generator=g, device=device)[: wl.n_empty]
        logits[:, empty] = -math.inf
    probs = torch.softmax(logits, dim=-1)
    vals, idx = torch.topk(probs, wl.k, dim=-1)
    w = vals / vals.sum(dim=-1, keepdim=True)
    return idx.to(torch.int32).contiguous(), w.to(torch.float32).contiguous()


def make_acts(wl: Workload, device="cpu"):
    g = _gen(device, wl.seed, 2)
    x = torch.randn(wl.T, wl.H, generator=g, device=device, dtype=torch.float32)
    x = x.to(torch.bfloat16).to(torch.float32)
    if wl.wfmt == 0:
        return pack_fp8_rows_f32(x, 128)
    return pack_fp8_rows_ue8m0(x, 32)


def make_expert_weights(wl: Workload, e: int, device="cpu"):
    """Canonical weights of expert e alone (each expert has its own random stream)."""
    H, I = wl.H, wl.I
    g = _gen(device, wl.seed, 1000 + e)
    a = torch.randn(2 * I, H, generator=g, device=device, dtype=torch.float32) * (1.0 / math.sqrt(H))
    b = torch.randn(H, I, generator=g, device=device, dtype=torch.float32) * (1.0 / math.sqrt(I))
    if wl.wfmt == 0:
        return pack_fp8_blocks(a) + pack_fp8_blocks(b)
    return pack_e2m1_rows(a) + pack_e2m1_rows(b)


def make_weights(wl: Workload, device="cpu", experts=None):
    """Canonical (non-interleaved) W1 [E,2I,H] (gate rows [0,I), up rows [I,2I)) and W2 [E,H,I].

    With ``experts`` (a list of expert ids) only those experts are generated,
    stacked in that order."""
    E, H, I = wl.E, wl.H, wl.I
    ids = list(range(E)) if experts is None else [int(e) for e in experts]
    n = len(ids)
    if wl.wfmt == 0:
        w1 = torch.empty(n, 2 * I, H, dtype=torch.uint8, device=device)
        w1_sf = torch.empty(n, 2 * I // 128, H // 128, dtype=torch.float32, device=device)
        w2 = torch.empty(n, H, I, dtype=torch.uint8, device=device)
        w2_sf = torch.empty(n, H // 128, I // 128, dtype=torch.float32, device=device)
    else:
        w1 = torch.empty(n, 2 * I, H // 2, dtype=torch.uint8, device=device)
        w1_sf = torch.empty(n, 2 * I, H // 32, dtype=torch.uint8, device=device)
        w2 = torch.empty(n, H, I // 2, dtype=torch.uint8, device=device)
        w2_sf = torch.empty(n, H, I // 32, dtype=torch.uint8, device=device)
    for i, e in enumerate(ids):
        w1[i], w1_sf[i], w2[i], w2_sf[i] = make_expert_weights(wl, e, device)
    return w1, w1_sf, w2, w2_sf


def make_inputs(wl: Workload, device="cpu", weights: bool = True, batch: int = 0) -> dict:
    """All inputs of one forward.  ``batch`` selects an independent batch of
    tokens and routing (same weights), e.g. one per data-parallel replica."""
    if batch:
        wl = dataclasses.replace(wl, seed=wl.seed + 7919 * batch)
    x, x_sf = make_acts(wl, device)
    idx, w = make_routing(wl, device)
    out = {"x": x, "x_sf": x_sf, "topk_idx": idx, "topk_weights": w}
    if weights:
        base = dataclasses.replace(wl, seed=wl.seed - 7919 * batch) if batch else wl
        out["w1"], out["w1_sf"], out["w2"], out["w2_sf"] = make_weights(base, device)
    return out
