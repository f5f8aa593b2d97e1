"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Dispatch maps bit-exact; L2 activations (FP8 codes and scales) stage by
stage; y within the layer tolerance (normalised L2 <= 2e-3, max |err| <=
3e-2 * rms(y_ref)) on small cases the oracle finishes in seconds (several
tiles, ragged tails) and on sampled tokens of the full-size workloads.
"""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_util import assert_y_close, bf16_bits_to_float, compare_y, new_layer, stratified_tokens, sub_inputs, to_dev

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


def _run(m, wl, inp, **kw):
    layer = new_layer(m, wl, DEV, **kw)
    g = to_dev(inp, DEV)
    layer.transform_weights(g["w1"], g["w1_sf"], g["w2"], g["w2_sf"])
    y = layer.forward(g["x"], g["x_sf"], g["topk_idx"], g["topk_weights"])
    torch.cuda.synchronize()
    assert layer.device_status() == m.MOE_OK
    return layer, g, y


SMALL = [
    moe_synth.WORKLOADS["tiny"],
    moe_synth.custom(T=200, H=512, I=384, E=6, k=4, seed=31, name="ragged"),
    moe_synth.custom(T=300, H=256, I=256, E=3, k=2, seed=32, name="nmajor"),
    moe_synth.custom(T=50, H=384, I=128, E=40, k=3, seed=33, name="sparse"),
    # full 32-row groups next to the half-empty last column block (H % 256 == 128)
    moe_synth.custom(T=300, H=384, I=256, E=3, k=2, seed=34, name="halfblock"),
    # Zipf routing: experts of 3-5 M blocks (N-major walk), of 2 (M-major)
    # and of one, and an empty one, in one launch
    moe_synth.custom(T=600, H=256, I=256, E=32, k=4, seed=35, routing="zipf", name="skewed"),
    # 8192 pairs: the dispatch runs over 8 CTAs, hot experts spanning them
    moe_synth.custom(T=2048, H=256, I=128, E=64, k=4, seed=36, routing="zipf", name="multi_cta_dispatch"),
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_dispatch_bit_exact(m, orc, wl):
    inp = moe_synth.make_inputs(wl)
    layer, g, _ = _run(m, wl, inp)
    counts, offsets, gather = layer.get_dispatch(wl.T)
    st, oc, oo, og = orc.dispatch(inp["topk_idx"], wl.E)
    assert st == orc.OK
    assert np.array_equal(counts.cpu().numpy(), oc)
    assert np.array_equal(offsets.cpu().numpy(), oo)
    assert np.array_equal(gather.cpu().numpy()[: oo[-1]], og)


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_y_matches_oracle(m, orc, wl):
    inp = moe_synth.make_inputs(wl)
    _, _, y = _run(m, wl, inp)
    ref = bf16_bits_to_float(orc.forward(inp))
    rel, mx = assert_y_close(y, ref, wl.name)
    print(f"{wl.name}: rel L2 {rel:.2e}, max/rms {mx:.2e}")


def test_l2_activations_stage_by_stage(m, orc):
    wl = moe_synth.custom(T=64, H=512, I=256, E=4, k=2, seed=34)
    inp = moe_synth.make_inputs(wl)
    layer, g, _ = _run(m, wl, inp)
    _, offsets, gather = layer.get_dispatch(wl.T)
    acts, sf, out = layer.get_intermediates(wl.T)
    acts, sf, out, gather = acts.cpu().numpy(), sf.cpu().numpy(), out.cpu(), gather.cpu().numpy()
    idx, w = inp["topk_idx"].numpy(), inp["topk_weights"].numpy()
    code_mismatch = total = 0
    for r in range(0, int(offsets[-1]), 7):
        pair = int(gather[r])
        t, j = divmod(pair, wl.k)
        pr = orc.pair(inp, t, int(idx[t, j]), float(w[t, j]))
        np.testing.assert_allclose(sf[r], pr["sf"], rtol=1e-5, atol=0)
        code_mismatch += int((acts[r] != pr["q"]).sum())
        total += wl.I
        ob = bf16_bits_to_float(pr["ob"])
        rel, _ = compare_y(out[r:r + 1], ob[None])
        assert rel <= 1e-3, (r, rel)
    assert code_mismatch <= 0.01 * total, (code_mismatch, total)


def _crafted_counts(T, k, E, counts, seed):
    """topk_idx [T, k] with distinct experts per token and the given per-expert counts."""
    assert sum(counts) == T * k and len(counts) == E and max(counts) <= T
    # experts sorted, slots filled column by column: a run of <= T equal ids
    # never puts one expert in two slots of a token; then shuffle the tokens
    ids = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(counts)])
    idx = ids.reshape(k, T).T.copy()
    np.random.default_rng(seed).shuffle(idx)
    assert all(len(set(r)) == k for r in idx.tolist())
    return torch.from_numpy(idx)


# L1 on CTA pairs (256-row blocks): experts whose counts leave the second CTA
# empty (<= 128), ragged in either half, exactly one or two blocks, several
# blocks (N-major), plus the generic small cases
PAIR_CASES = SMALL[1:3] + [moe_synth.custom(T=600, H=512, I=256, E=8, k=2, seed=37, name="pair_counts")]
PAIR_COUNTS = {"pair_counts": [1, 127, 128, 129, 255, 256, 257, 47]}


@pytest.mark.parametrize("a_mode", ["pool", "gather"])
@pytest.mark.parametrize("wl", PAIR_CASES, ids=lambda w: w.name)
def test_l1_cta_pairs_match_oracle(m, orc, wl, a_mode, monkeypatch):
    monkeypatch.setenv("MOE_L1_PAIR", "1")
    monkeypatch.setenv("MOE_L1_A", a_mode)
    inp = moe_synth.make_inputs(wl)
    if wl.name in PAIR_COUNTS:
        inp["topk_idx"] = _crafted_counts(wl.T, wl.k, wl.E, PAIR_COUNTS[wl.name], wl.seed)
    layer, g, y = _run(m, wl, inp)
    ref = bf16_bits_to_float(orc.forward(inp))
    rel, mx = assert_y_close(y, ref, f"{wl.name}/pairs/{a_mode}")
    # the L1 output itself: scales and FP8 codes of sampled rows
    _, offsets, gather = layer.get_dispatch(wl.T)
    acts, sf, _ = layer.get_intermediates(wl.T)
    acts, sf, gather = acts.cpu().numpy(), sf.cpu().numpy(), gather.cpu().numpy()
    idx, w = inp["topk_idx"].numpy(), inp["topk_weights"].numpy()
    mism = total = 0
    for r in range(0, int(offsets[-1]), 11):
        t, j = divmod(int(gather[r]), wl.k)
        pr = orc.pair(inp, t, int(idx[t, j]), float(w[t, j]))
        np.testing.assert_allclose(sf[r], pr["sf"], rtol=1e-5, atol=0)
        mism += int((acts[r] != pr["q"]).sum())
        total += wl.I
    assert mism <= 0.01 * total, (mism, total)
    print(f"{wl.name}/pairs/{a_mode}: rel L2 {rel:.2e}, max/rms {mx:.2e}")


# The whole FP8 forward in one cooperative launch (MOE_FUSED=1: dispatch,
# pool copy, both GEMMs, combine, with grid barriers between the phases): the
# same arithmetic as the separate kernels, so y must be bit-identical to
# theirs, and the dispatch maps equal to the oracle's.  Small cases plus an
# expert mix where many M blocks finish their L1 tiles at different times.
FUSED_CASES = SMALL + [moe_synth.custom(T=600, H=512, I=256, E=8, k=2, seed=38, name="fused_counts")]


@pytest.mark.parametrize("wl", FUSED_CASES, ids=lambda w: w.name)
def test_fused_launch_matches_two_launches(m, orc, wl, monkeypatch):
    inp = moe_synth.make_inputs(wl)
    if wl.name == "fused_counts":
        inp["topk_idx"] = _crafted_counts(wl.T, wl.k, wl.E, [1, 127, 128, 129, 255, 256, 257, 47], wl.seed)
    monkeypatch.setenv("MOE_FUSED", "0")
    _, _, y2 = _run(m, wl, inp)
    monkeypatch.setenv("MOE_FUSED", "1")
    layer, _, y1 = _run(m, wl, inp)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    counts, offsets, gather = layer.get_dispatch(wl.T)
    st, oc, oo, og = orc.dispatch(inp["topk_idx"], wl.E)
    assert np.array_equal(counts.cpu().numpy(), oc) and np.array_equal(offsets.cpu().numpy(), oo)
    assert np.array_equal(gather.cpu().numpy()[: oo[-1]], og)
    ref = bf16_bits_to_float(orc.forward(inp))
    rel, mx = assert_y_close(y1, ref, f"{wl.name}/fused")
    print(f"{wl.name}/fused: bit-identical to the separate kernels, rel L2 {rel:.2e}")


def test_fused_launch_inactive_slots_bad_ids_and_stats(m, orc, monkeypatch):
    """The one-launch dispatch skips inactive slots, reports an out-of-range
    expert id (and skips it), and adds the counts to the caller's statistics."""
    monkeypatch.setenv("MOE_FUSED", "1")
    wl = moe_synth.custom(T=300, H=256, I=128, E=16, k=3, seed=39, name="fused_slots")
    inp = moe_synth.make_inputs(wl)
    inp["topk_idx"][::3, 1] = -1
    inp["topk_idx"][7, :] = -1
    layer = new_layer(m, wl, DEV)
    g = to_dev(inp, DEV)
    layer.transform_weights(g["w1"], g["w1_sf"], g["w2"], g["w2_sf"])
    stats = torch.zeros(wl.E, dtype=torch.int32, device=DEV)
    y = layer.forward(g["x"], g["x_sf"], g["topk_idx"], g["topk_weights"], stats=stats)
    y = layer.forward(g["x"], g["x_sf"], g["topk_idx"], g["topk_weights"], stats=stats)
    torch.cuda.synchronize()
    assert layer.device_status() == m.MOE_OK
    st, oc, oo, og = orc.dispatch(inp["topk_idx"], wl.E)
    assert np.array_equal(stats.cpu().numpy(), 2 * oc)
    assert torch.all(y[7] == 0)
    assert_y_close(y, bf16_bits_to_float(orc.forward(inp)), "fused inactive slots")
    bad = g["topk_idx"].clone()
    bad[11, 2] = wl.E + 5
    layer.forward(g["x"], g["x_sf"], bad, g["topk_weights"])
    assert layer.device_status() == m.MOE_ERR_BAD_EXPERT


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_fused_launch_full_size(m, name, monkeypatch):
    """Full sizes in the bench's launch configuration: the one-launch y equals
    the two-launch y bit for bit."""
    wl = moe_synth.WORKLOADS[name]
    inp = moe_synth.make_inputs(wl, device=DEV)
    ys = []
    for fused in ("0", "1"):
        monkeypatch.setenv("MOE_FUSED", fused)
        layer = new_layer(m, wl, DEV)
        layer.transform_weights(inp["w1"], inp["w1_sf"], inp["w2"], inp["w2_sf"])
        ys.append(layer.forward(inp["x"], inp["x_sf"], inp["topk_idx"], inp["topk_weights"]).clone())
        torch.cuda.synchronize()
        assert layer.device_status() == m.MOE_OK
        del layer
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))


# Both FP8 GEMMs at the same time on disjoint CTA sets of one cooperative
# launch (MOE_SPLIT=1): L2 tiles start on an M block as soon as its L1 tiles
# are stored, so y must again be bit-identical to the two launches.  The L1
# share is the default and, to make L2 CTAs wait on many M blocks, 8 CTAs.
@pytest.mark.parametrize("l1_sms", ["", "8"], ids=["default_share", "l1_8_ctas"])
@pytest.mark.parametrize("wl", FUSED_CASES, ids=lambda w: w.name)
def test_split_launch_matches_two_launches(m, orc, wl, l1_sms, monkeypatch):
    inp = moe_synth.make_inputs(wl)
    if wl.name == "fused_counts":
        inp["topk_idx"] = _crafted_counts(wl.T, wl.k, wl.E, [1, 127, 128, 129, 255, 256, 257, 47], wl.seed)
    monkeypatch.setenv("MOE_SPLIT", "0")
    _, _, y2 = _run(m, wl, inp)
    monkeypatch.setenv("MOE_SPLIT", "1")
    if l1_sms:
        monkeypatch.setenv("MOE_SPLIT_L1_SMS", l1_sms)
    _, _, y1 = _run(m, wl, inp)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    ref = bf16_bits_to_float(orc.forward(inp))
    rel, mx = assert_y_close(y1, ref, f"{wl.name}/split")
    print(f"{wl.name}/split{l1_sms}: bit-identical to two launches, rel L2 {rel:.2e}")


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_split_launch_full_size(m, name, monkeypatch):
    """Full sizes in the bench's launch configuration: the split launch's y
    equals the two-launch y bit for bit."""
    wl = moe_synth.WORKLOADS[name]
    inp = moe_synth.make_inputs(wl, device=DEV)
    ys = []
    for split in ("0", "1"):
        monkeypatch.setenv("MOE_SPLIT", split)
        layer = new_layer(m, wl, DEV)
        layer.transform_weights(inp["w1"], inp["w1_sf"], inp["w2"], inp["w2_sf"])
        ys.append(layer.forward(inp["x"], inp["x_sf"], inp["topk_idx"], inp["topk_weights"]).clone())
        torch.cuda.synchronize()
        assert layer.device_status() == m.MOE_OK
        del layer
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))


@pytest.mark.parametrize("clamp", [float("inf"), 1.0], ids=["noclamp", "clamp1"])
@pytest.mark.parametrize("fast", [0, 1], ids=["expf", "fastexp"])
@pytest.mark.parametrize("variant", ["single", "pairs", "fp4"])
def test_epilogue_options_match_oracle(m, orc, variant, fast, clamp, monkeypatch):
    """fast_math and the activation clamp in each L1 epilogue (one CTA, CTA
    pairs, FP4 weights): the clamp of 1.0 clips about a third of the gate/up
    values of this case, so its branch is exercised."""
    wfmt = 1 if variant == "fp4" else 0
    monkeypatch.setenv("MOE_L1_PAIR", "1" if variant == "pairs" else "0")
    wl = moe_synth.custom(T=300, H=512, I=256, E=8, k=2, seed=81, wfmt=wfmt, name="opts")
    inp = moe_synth.make_inputs(wl)
    layer, g, y = _run(m, wl, inp, wfmt=wfmt, act_clamp=clamp, fast_math=bool(fast))
    ref = bf16_bits_to_float(orc.forward(inp, wfmt=wfmt, act_clamp=clamp))
    rel, mx = assert_y_close(y, ref, f"{variant}/fast{fast}/clamp{clamp}")
    print(f"{variant} fast={fast} clamp={clamp}: rel L2 {rel:.2e}, max/rms {mx:.2e}")


@pytest.mark.parametrize("variant", ["single", "pairs", "fp4"])
def test_fast_math_within_half_percent_of_expf(m, variant, monkeypatch):
    """The __expf SwiGLU against the expf one on the same inputs (MegaMoE SM90
    Implementation Design (Final), §21 Phase 4, step 4.4: the fast path within
    0.5% of the exact one): normalised L2 difference of y below 5e-3, and the
    L2-activation codes of the two runs mostly equal."""
    wfmt = 1 if variant == "fp4" else 0
    monkeypatch.setenv("MOE_L1_PAIR", "1" if variant == "pairs" else "0")
    wl = moe_synth.custom(T=300, H=512, I=256, E=8, k=2, seed=82, wfmt=wfmt, name="fastexp")
    inp = moe_synth.make_inputs(wl)
    la, _, ya = _run(m, wl, inp, wfmt=wfmt, fast_math=False)
    qa, sa, _ = la.get_intermediates(wl.T)
    lb, _, yb = _run(m, wl, inp, wfmt=wfmt, fast_math=True)
    qb, sb, _ = lb.get_intermediates(wl.T)
    ya, yb = ya.float(), yb.float()
    rel = float((yb - ya).norm() / ya.norm())
    assert rel < 5e-3, rel
    diff = float((qa != qb).float().mean())
    assert diff < 0.02, diff
    print(f"{variant}: fast vs expf rel L2 {rel:.2e}, activation codes differing {diff:.2%}")


def test_zero_tokens_and_inactive_slots(m, orc):
    wl = moe_synth.custom(T=40, H=256, I=128, E=8, k=3, seed=35)
    inp = moe_synth.make_inputs(wl)
    inp["topk_idx"][::3, 1] = -1
    inp["topk_idx"][5, :] = -1
    layer, g, y = _run(m, wl, inp)
    ref = bf16_bits_to_float(orc.forward(inp))
    assert_y_close(y, ref, "inactive slots")
    assert torch.all(y[5] == 0)
    y0 = torch.empty(0, wl.H, dtype=torch.bfloat16, device=DEV)
    layer.forward(g["x"][:0], g["x_sf"][:0], g["topk_idx"][:0], g["topk_weights"][:0], y=y0)
    assert layer.device_status() == m.MOE_OK


def test_repeat_calls_stats_and_token_order(m, orc):
    wl = moe_synth.custom(T=96, H=256, I=256, E=8, k=2, seed=36)
    inp = moe_synth.make_inputs(wl)
    layer, g, y1 = _run(m, wl, inp)
    stats = torch.zeros(wl.E, dtype=torch.int32, device=DEV)
    y2 = layer.forward(g["x"], g["x_sf"], g["topk_idx"], g["topk_weights"], stats=stats)
    y3 = layer.forward(g["x"], g["x_sf"], g["topk_idx"], g["topk_weights"], stats=stats)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(y2, y3)
    counts = torch.bincount(inp["topk_idx"].reshape(-1).long(), minlength=wl.E).int()
    assert torch.equal(stats.cpu(), 2 * counts)
    perm = torch.randperm(wl.T, generator=torch.Generator().manual_seed(3)).to(DEV)
    yp = layer.forward(g["x"][perm].contiguous(), g["x_sf"][perm].contiguous(),
                       g["topk_idx"][perm].contiguous(), g["topk_weights"][perm].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(yp, y1[perm])            # bit-exact: rows are computed independently


def test_forward_host_matches_device(m):
    wl = moe_synth.custom(T=33, H=256, I=128, E=4, k=2, seed=37)
    inp = moe_synth.make_inputs(wl)
    layer, g, y = _run(m, wl, inp)
    pinned = {n: inp[n].pin_memory() for n in ("x", "x_sf", "topk_idx", "topk_weights")}
    # pinned y: the combine stores into it directly; twice, the second over stale contents
    yh = layer.forward_host(pinned["x"], pinned["x_sf"], pinned["topk_idx"], pinned["topk_weights"])
    assert yh.is_pinned()
    assert torch.equal(yh, y.cpu())
    yh.fill_(7.0)
    layer.forward_host(pinned["x"], pinned["x_sf"], pinned["topk_idx"], pinned["topk_weights"], y=yh)
    assert torch.equal(yh, y.cpu())
    # pageable inputs and output: staged in the workspace and copied back
    yp = torch.full((wl.T, wl.H), 7.0, dtype=torch.bfloat16)
    layer.forward_host(inp["x"], inp["x_sf"], inp["topk_idx"], inp["topk_weights"], y=yp)
    assert torch.equal(yp, y.cpu())


GRAPH_CASES = [
    moe_synth.custom(T=50, H=384, I=128, E=40, k=3, seed=81, name="graph_sparse"),           # gather4 A
    moe_synth.custom(T=200, H=512, I=384, E=6, k=4, seed=82, name="graph_pool"),             # pool A
    moe_synth.custom(T=2048, H=256, I=128, E=64, k=4, seed=83, routing="zipf",
                     name="graph_multi_cta_dispatch"),                                        # cooperative dispatch
    moe_synth.custom(T=64, H=256, I=128, E=8, k=2, seed=84, wfmt=1, name="graph_fp4"),
]


@pytest.mark.parametrize("wl", GRAPH_CASES, ids=lambda w: w.name)
def test_cuda_graph_replay_matches_eager(m, wl):
    """One forward captured into a CUDA graph and replayed equals the eager
    forward bit for bit, also after the inputs are rewritten in place (the
    graph keeps the buffers, not their contents)."""
    inp = to_dev(moe_synth.make_inputs(wl), DEV)
    layer = new_layer(m, wl, DEV, wfmt=wl.wfmt)
    layer.transform_weights(inp["w1"], inp["w1_sf"], inp["w2"], inp["w2_sf"])
    args = [inp["x"], inp["x_sf"], inp["topk_idx"], inp["topk_weights"]]
    y_eager = layer.forward(*args).clone()          # also the one-time launch set-up, outside the capture
    torch.cuda.synchronize()
    y_graph = torch.empty_like(y_eager)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=side):
        layer.forward(*args, y=y_graph)
    graph.replay()
    torch.cuda.synchronize()
    assert layer.device_status() == m.MOE_OK
    assert torch.equal(y_graph, y_eager)
    # new tokens and routing in the same buffers: replay against eager
    other = to_dev(moe_synth.make_inputs(wl, weights=False, batch=1), DEV)
    for a, n in zip(args, ("x", "x_sf", "topk_idx", "topk_weights")):
        a.copy_(other[n])
    graph.replay()
    y2 = layer.forward(*args).clone()
    torch.cuda.synchronize()
    assert layer.device_status() == m.MOE_OK
    assert torch.equal(y_graph, y2)
    assert not torch.equal(y2, y_eager)


def test_bad_expert_id_is_reported_and_skipped(m, orc):
    wl = moe_synth.custom(T=16, H=256, I=128, E=4, k=2, seed=38)
    inp = moe_synth.make_inputs(wl)
    layer, g, _ = _run(m, wl, inp)
    bad = g["topk_idx"].clone()
    bad[3, 1] = 77
    layer.forward(g["x"], g["x_sf"], bad, g["topk_weights"])
    assert layer.device_status() == m.MOE_ERR_BAD_EXPERT
    assert layer.device_status() == m.MOE_OK     # cleared after reading
    ref_inp = dict(inp)
    ref_idx = inp["topk_idx"].clone()
    ref_idx[3, 1] = -1
    ref_inp["topk_idx"] = ref_idx
    y = layer.forward(g["x"], g["x_sf"], bad, g["topk_weights"])
    assert_y_close(y, bf16_bits_to_float(orc.forward(ref_inp)), "bad id skipped")
    layer.device_status()


def test_one_expert_takes_everything(m, orc):
    wl = moe_synth.custom(T=700, H=256, I=128, E=4, k=1, seed=39)
    inp = moe_synth.make_inputs(wl)
    inp["topk_idx"][:] = 2
    inp["topk_weights"][:] = 1.0
    _, _, y = _run(m, wl, inp)
    sel = np.arange(0, wl.T, 9, dtype=np.int32)
    ref = bf16_bits_to_float(orc.forward(inp, tokens=sel))
    assert_y_close(y[torch.from_numpy(sel).long().to(DEV)], ref, "one expert")


# Degenerate shapes: one token, top-1 with a single expert (the layer is then
# a dense FFN of that expert), E = 1, and a layer created for more tokens than
# the call passes (the pool and tile tables sized for max_tokens).
EDGE = [
    moe_synth.custom(T=1, H=256, I=128, E=8, k=2, seed=91, name="one_token"),
    moe_synth.custom(T=1, H=256, I=128, E=8, k=8, seed=92, name="one_token_k8"),
    moe_synth.custom(T=77, H=384, I=256, E=1, k=1, seed=93, name="single_expert"),
    moe_synth.custom(T=130, H=256, I=128, E=16, k=1, seed=94, name="top1"),
]


@pytest.mark.parametrize("wl", EDGE, ids=lambda w: w.name)
@pytest.mark.parametrize("wfmt", [0, 1], ids=["fp8", "fp4"])
def test_degenerate_shapes_match_oracle(m, orc, wl, wfmt):
    wl = moe_synth.custom(T=wl.T, H=wl.H, I=wl.I, E=wl.E, k=wl.k, seed=wl.seed, wfmt=wfmt, name=wl.name)
    inp = moe_synth.make_inputs(wl)
    layer, g, y = _run(m, wl, inp, wfmt=wfmt)
    ref = bf16_bits_to_float(orc.forward(inp, wfmt=wfmt))
    assert_y_close(y, ref, f"{wl.name}/{'fp4' if wfmt else 'fp8'}")
    counts, offsets, gather = layer.get_dispatch(wl.T)
    st, oc, oo, og = orc.dispatch(inp["topk_idx"], wl.E)
    assert np.array_equal(counts.cpu().numpy(), oc) and np.array_equal(gather.cpu().numpy()[: oo[-1]], og)


def test_fewer_tokens_than_capacity(m, orc):
    """A layer sized for 512 tokens called with 100 and then 512: each call
    matches the oracle for its own tokens."""
    big = moe_synth.custom(T=512, H=256, I=256, E=8, k=2, seed=95, name="capacity")
    inp = moe_synth.make_inputs(big)
    layer = new_layer(m, big, DEV)
    g = to_dev(inp, DEV)
    layer.transform_weights(g["w1"], g["w1_sf"], g["w2"], g["w2_sf"])
    for T in (100, 512):
        y = layer.forward(g["x"][:T].contiguous(), g["x_sf"][:T].contiguous(), g["topk_idx"][:T].contiguous(),
                          g["topk_weights"][:T].contiguous())
        torch.cuda.synchronize()
        assert layer.device_status() == m.MOE_OK
        sub = {n: (t[:T].contiguous() if n in ("x", "x_sf", "topk_idx", "topk_weights") else t) for n, t in inp.items()}
        assert_y_close(y, bf16_bits_to_float(orc.forward(sub)), f"T={T} of 512")


@pytest.mark.parametrize("name", ["decode", "prefill", "wide"])
def test_full_size_sampled_tokens(m, orc, name):
    wl = moe_synth.WORKLOADS[name]
    inp = moe_synth.make_inputs(wl, device=DEV)
    layer = new_layer(m, wl, DEV)
    layer.transform_weights(inp["w1"], inp["w1_sf"], inp["w2"], inp["w2_sf"])
    y = layer.forward(inp["x"], inp["x_sf"], inp["topk_idx"], inp["topk_weights"])
    torch.cuda.synchronize()
    assert layer.device_status() == m.MOE_OK
    counts, offsets, gather = layer.get_dispatch(wl.T)
    st, oc, oo, og = orc.dispatch(inp["topk_idx"].cpu(), wl.E)
    assert np.array_equal(counts.cpu().numpy(), oc) and np.array_equal(gather.cpu().numpy()[: oo[-1]], og)
    # every M block (and the last pair) of the three largest experts, one pair
    # of every 16th touched expert, the first and the last token
    tokens, covered = stratified_tokens(oc, oo, og, wl.k, wl.T, top=3, every_touched=16, seed=7)
    sub = sub_inputs(inp, tokens)
    ref = bf16_bits_to_float(orc.forward(sub))
    rel, mx = assert_y_close(y[torch.from_numpy(tokens).long().to(DEV)], ref, name)
    print(f"{name}: {len(tokens)} tokens covering {covered}; rel L2 {rel:.2e} max/rms {mx:.2e}")
    assert torch.isfinite(y.float()).all()


def test_largest_batch_sampled_tokens(m, orc):
    """Four times the prefill batch (131072 routed pairs, 1024 M blocks, 16384
    L1 and 28672 L2 tiles): dispatch maps bit-exact and sampled tokens,
    including the first and the last, within the layer tolerance."""
    wl = moe_synth.custom(T=16384, H=7168, I=2048, E=256, k=8, seed=41, name="largest")
    inp = moe_synth.make_inputs(wl, device=DEV)
    layer = new_layer(m, wl, DEV)
    layer.transform_weights(inp["w1"], inp["w1_sf"], inp["w2"], inp["w2_sf"])
    st, oc, oo, og = orc.dispatch(inp["topk_idx"].cpu(), wl.E)
    # the last pair (the last, ragged M block) of the three largest experts,
    # a few random tokens, the first and the last token
    rng = np.random.default_rng(11)
    tokens, covered = stratified_tokens(oc, oo, og, wl.k, wl.T, top=3, blocks=False, seed=11)
    tokens = np.unique(np.concatenate([tokens, rng.choice(wl.T, size=4, replace=False)])).astype(np.int32)
    sub = sub_inputs(inp, tokens)   # the oracle needs only the experts these tokens use
    del inp["w1"], inp["w2"]
    y = layer.forward(inp["x"], inp["x_sf"], inp["topk_idx"], inp["topk_weights"])
    torch.cuda.synchronize()
    assert layer.device_status() == m.MOE_OK
    counts, offsets, gather = layer.get_dispatch(wl.T)
    assert int(oo[-1]) == wl.T * wl.k
    assert np.array_equal(counts.cpu().numpy(), oc) and np.array_equal(gather.cpu().numpy()[: oo[-1]], og)
    ref = bf16_bits_to_float(orc.forward(sub))
    rel, mx = assert_y_close(y[torch.from_numpy(tokens).long().to(DEV)], ref, "largest")
    print(f"largest: tokens {tokens.tolist()} covering {covered}; rel L2 {rel:.2e} max/rms {mx:.2e}")
    assert torch.isfinite(y.float()).all()


FP4 = [
    moe_synth.custom(T=40, H=256, I=128, E=8, k=2, seed=61, wfmt=1, name="fp4_tiny"),
    moe_synth.custom(T=300, H=512, I=384, E=6, k=3, seed=62, wfmt=1, name="fp4_ragged"),
    moe_synth.custom(T=64, H=384, I=256, E=40, k=4, seed=63, wfmt=1, n_empty=8, name="fp4_sparse"),
    moe_synth.custom(T=600, H=256, I=128, E=32, k=4, seed=64, wfmt=1, routing="zipf", name="fp4_skewed"),
]


@pytest.mark.parametrize("wl", FP4, ids=lambda w: w.name)
def test_fp4_weights_y_matches_oracle(m, orc, wl):
    inp = moe_synth.make_inputs(wl)
    _, _, y = _run(m, wl, inp, wfmt=m.MOE_W_FP4_E2M1_UE8M0_32)
    ref = bf16_bits_to_float(orc.forward(inp, wfmt=1))
    rel, mx = assert_y_close(y, ref, wl.name)
    print(f"{wl.name}: rel L2 {rel:.2e}, max/rms {mx:.2e}")


def test_fp4_l2_activations_stage_by_stage(m, orc):
    wl = moe_synth.custom(T=48, H=256, I=256, E=4, k=2, seed=64, wfmt=1)
    inp = moe_synth.make_inputs(wl)
    layer, g, _ = _run(m, wl, inp, wfmt=m.MOE_W_FP4_E2M1_UE8M0_32)
    _, offsets, gather = layer.get_dispatch(wl.T)
    acts, sf, out = layer.get_intermediates(wl.T)
    acts, sf, gather = acts.cpu().numpy(), sf.cpu().numpy(), gather.cpu().numpy()
    idx, w = inp["topk_idx"].numpy(), inp["topk_weights"].numpy()
    mism = total = 0
    for r in range(0, int(offsets[-1]), 5):
        t, j = divmod(int(gather[r]), wl.k)
        pr = orc.pair(inp, t, int(idx[t, j]), float(w[t, j]), wfmt=1)
        assert np.array_equal(sf[r].astype(np.float32), pr["sf"]), r      # UE8M0 codes
        mism += int((acts[r] != pr["q"]).sum())
        total += wl.I
    assert mism <= 0.01 * total, (mism, total)


def test_fp4_full_size_sampled_tokens(m, orc):
    wl = moe_synth.WORKLOADS["fp4"]
    inp = moe_synth.make_inputs(wl, device=DEV)
    layer = new_layer(m, wl, DEV, wfmt=m.MOE_W_FP4_E2M1_UE8M0_32)
    layer.transform_weights(inp["w1"], inp["w1_sf"], inp["w2"], inp["w2_sf"])
    y = layer.forward(inp["x"], inp["x_sf"], inp["topk_idx"], inp["topk_weights"])
    torch.cuda.synchronize()
    assert layer.device_status() == m.MOE_OK
    counts, _, _ = layer.get_dispatch(wl.T)
    assert (counts.cpu().numpy() == 0).sum() >= wl.n_empty
    st, oc, oo, og = orc.dispatch(inp["topk_idx"].cpu(), wl.E)
    assert np.array_equal(counts.cpu().numpy(), oc)
    tokens, covered = stratified_tokens(oc, oo, og, wl.k, wl.T, top=3, every_touched=16, seed=9)
    ref = bf16_bits_to_float(orc.forward(sub_inputs(inp, tokens), wfmt=1))
    rel, mx = assert_y_close(y[torch.from_numpy(tokens).long().to(DEV)], ref, "fp4")
    print(f"fp4: {len(tokens)} tokens covering {covered}; rel L2 {rel:.2e} max/rms {mx:.2e}")
