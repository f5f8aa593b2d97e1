"""Helpers shared by the GPU parity tests (CUDA path vs the CPU oracle)."""
import numpy as np
import torch

import moe_synth

# Tolerances of the whole layer: normalised L2 error and max |error| relative
# to the RMS of the oracle's y.  Sources of mismatch: FP32 (tensor core +
# promotion) vs double accumulation, and the rare FP8 code of the L2
# activations that lands on the other side of a rounding boundary.
REL_L2 = 2e-3
MAX_ABS_RMS = 3e-2


def bf16_bits_to_float(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).astype(np.uint16).view(np.int16)).view(
        torch.bfloat16).float()


def compare_y(got: torch.Tensor, ref: torch.Tensor):
    """Returns (rel_l2, max_abs / rms(ref)); both must be within tolerance."""
    got = got.float().cpu()
    ref = ref.float().cpu()
    diff = got - ref
    rel = (diff.norm() / ref.norm().clamp_min(1e-30)).item()
    rms = ref.pow(2).mean().sqrt().clamp_min(1e-30)
    mx = (diff.abs().max() / rms).item()
    return rel, mx


def assert_y_close(got, ref, what=""):
    rel, mx = compare_y(got, ref)
    assert rel <= REL_L2, f"{what}: normalised L2 {rel:.3e} > {REL_L2}"
    assert mx <= MAX_ABS_RMS, f"{what}: max|err|/rms {mx:.3e} > {MAX_ABS_RMS}"
    return rel, mx


def new_layer(m, wl, device, **kw):
    layer = m.MoELayer(wl.T, wl.H, wl.I, wl.E, wl.k, device=device, **kw)
    return layer


def to_dev(inp: dict, device) -> dict:
    return {n: t.to(device) for n, t in inp.items()}


def sub_inputs(inp_dev: dict, tokens) -> dict:
    """CPU inputs restricted to `tokens` and the experts they use (ids remapped),
    so the oracle need not see the full weight set."""
    tok = torch.as_tensor(tokens, dtype=torch.long, device=inp_dev["x"].device)
    idx = inp_dev["topk_idx"][tok]
    used = torch.unique(idx[idx >= 0])
    remap = torch.full((inp_dev["w1"].shape[0],), -1, dtype=torch.int32, device=idx.device)
    remap[used] = torch.arange(used.numel(), dtype=torch.int32, device=idx.device)
    new_idx = torch.where(idx >= 0, remap[idx.clamp_min(0).long()], idx)
    out = {
        "x": inp_dev["x"][tok].cpu(), "x_sf": inp_dev["x_sf"][tok].cpu(),
        "topk_idx": new_idx.cpu().contiguous(), "topk_weights": inp_dev["topk_weights"][tok].cpu(),
    }
    for n in ("w1", "w1_sf", "w2", "w2_sf"):
        out[n] = inp_dev[n][used].cpu().contiguous()
    return out


def stratified_tokens(oc, oo, og, k, T, top=3, every_touched=0, seed=0, blocks=True):
    """Tokens whose pairs reach chosen tiles of a full-size forward.

    From the oracle's dispatch (counts oc, offsets oo, gather og): for each of
    the `top` largest experts, one pair in every 128-row M block (when
    `blocks`) and the expert's last pair; with `every_touched` = n, one pair of
    every n-th touched expert; plus the first and the last token.  Returns the
    sorted tokens and a description of what they cover."""
    rng = np.random.default_rng(seed)
    tok = {0, T - 1}
    order = np.argsort(-oc, kind="stable")[:top]
    covered = []
    for e in order:
        e = int(e)
        lo, hi = int(oo[e]), int(oo[e + 1])
        if hi <= lo:
            continue
        nb = (hi - lo + 127) // 128
        if blocks:
            for b in range(nb):
                r = lo + 128 * b + int(rng.integers(0, min(128, hi - lo - 128 * b)))
                tok.add(int(og[r]) // k)
        tok.add(int(og[hi - 1]) // k)
        covered.append(f"expert {e} ({hi - lo} pairs: {'all ' + str(nb) if blocks else 'last of ' + str(nb)} M blocks"
                       f" + last pair)")
    if every_touched:
        touched = np.nonzero(oc > 0)[0]
        for e in touched[::every_touched]:
            lo, hi = int(oo[e]), int(oo[e + 1])
            tok.add(int(og[lo + int(rng.integers(0, hi - lo))]) // k)
        covered.append(f"one pair of every {every_touched}th of {len(touched)} touched experts")
    return np.array(sorted(tok), dtype=np.int32), "; ".join(covered)
