"""moe_dispatch_noalloc, the dispatch entry point for callers that cannot
allocate device memory (a host runtime that plans every device byte itself
and gives its plugins no workspace), against the dispatch that moe_forward
runs and against the oracle's dispatch, through the C ABI, on two calls in a
row with different routings, and at the largest size the fixed scratch takes.

Dispatch maps are integer results: the comparison is bit-exact.  Collected
last on purpose (file name), so a run that stops at its first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import moe_synth
import oracle as orc

pytestmark = pytest.mark.gpu


def _noalloc_fn(m):
    raw = ctypes.CDLL(m.LIB_PATH)
    fn = raw.moe_dispatch_noalloc
    vp = ctypes.c_void_p
    fn.restype = ctypes.c_int
    fn.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp]
    return fn


def test_noalloc_dispatch_matches_forward_dispatch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_ffn_gb300 import build
    build.build()
    import moe_expert_ffn_gb300 as m
    dev = torch.device("cuda:0")
    fn = _noalloc_fn(m)
    stream = torch.cuda.current_stream(dev)
    wl = moe_synth.custom(T=700, H=256, I=128, E=48, k=6, seed=51)
    layer = m.MoELayer(wl.T, wl.H, wl.I, wl.E, wl.k, device=dev)
    w = moe_synth.make_weights(wl, device=dev)
    layer.transform_weights(*w)
    for call, (seed, T) in enumerate(((52, 700), (53, 333))):
        inp = moe_synth.make_inputs(moe_synth.custom(T=T, H=wl.H, I=wl.I, E=wl.E, k=wl.k, seed=seed),
                                    device=dev, weights=False)
        if call == 1:
            inp["topk_idx"][::5, 2] = -1            # some inactive slots on the second call
        layer.forward(inp["x"], inp["x_sf"], inp["topk_idx"], inp["topk_weights"])
        ref_c, ref_o, ref_g = layer.get_dispatch(T)
        counts = torch.full((wl.E,), -7, dtype=torch.int32, device=dev)
        offsets = torch.full((wl.E + 1,), -7, dtype=torch.int32, device=dev)
        gather = torch.full((T * wl.k,), -7, dtype=torch.int32, device=dev)
        rc = fn(ctypes.c_void_p(inp["topk_idx"].data_ptr()), T, wl.k, wl.E,
                ctypes.c_void_p(counts.data_ptr()), ctypes.c_void_p(offsets.data_ptr()),
                ctypes.c_void_p(gather.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
        assert rc == m.MOE_OK, m.strerror(rc)
        torch.cuda.synchronize(dev)
        P = int(ref_o[-1])
        assert torch.equal(counts, ref_c), f"call {call}: counts"
        assert torch.equal(offsets, ref_o), f"call {call}: offsets"
        assert torch.equal(gather[:P], ref_g[:P]), f"call {call}: gather"
        assert P == int((inp["topk_idx"] >= 0).sum())
        st, oc, oo, og = orc.dispatch(inp["topk_idx"].cpu().numpy(), wl.E)
        assert st == 0
        assert np.array_equal(counts.cpu().numpy(), oc), f"call {call}: counts vs oracle"
        assert np.array_equal(offsets.cpu().numpy(), oo), f"call {call}: offsets vs oracle"
        assert np.array_equal(gather[:P].cpu().numpy(), og), f"call {call}: gather vs oracle"
    assert layer.device_status() == m.MOE_OK
    # sizes beyond the fixed scratch are refused before anything is launched
    big = int(65536 // wl.k) + 1
    rc = fn(ctypes.c_void_p(inp["topk_idx"].data_ptr()), big, wl.k, wl.E,
            ctypes.c_void_p(counts.data_ptr()), ctypes.c_void_p(offsets.data_ptr()),
            ctypes.c_void_p(gather.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    assert rc == m.MOE_ERR_INVALID_ARG


def test_noalloc_dispatch_at_its_limits():
    """E = MOE_NOALLOC_MAX_EXPERTS experts and T*k = MOE_NOALLOC_MAX_PAIRS
    routed pairs with skewed routing (the scan uses every thread, the M-block
    table is near its bound), twice in a row, bit-exact against the oracle;
    one pair or one expert more is refused."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_ffn_gb300 import build
    build.build()
    import moe_expert_ffn_gb300 as m
    dev = torch.device("cuda:0")
    fn = _noalloc_fn(m)
    stream = torch.cuda.current_stream(dev)
    E, k = 1024, 8
    T = 65536 // k
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    gather = torch.empty(T * k, dtype=torch.int32, device=dev)
    for seed in (61, 62):
        wl = moe_synth.custom(T=T, H=128, I=128, E=E, k=k, seed=seed, routing="zipf")
        idx, _ = moe_synth.make_routing(wl, device=dev)
        if seed == 62:
            idx[::7, 3] = -1
        counts.fill_(-7)
        offsets.fill_(-7)
        gather.fill_(-7)
        rc = fn(ctypes.c_void_p(idx.data_ptr()), T, k, E, ctypes.c_void_p(counts.data_ptr()),
                ctypes.c_void_p(offsets.data_ptr()), ctypes.c_void_p(gather.data_ptr()),
                ctypes.c_void_p(stream.cuda_stream))
        assert rc == m.MOE_OK, m.strerror(rc)
        torch.cuda.synchronize(dev)
        st, oc, oo, og = orc.dispatch(idx.cpu().numpy(), E)
        assert st == 0
        P = int(oo[-1])
        assert oc.max() > 10 * oc.mean() and (oc == 0).any()   # skewed, some experts empty
        assert np.array_equal(counts.cpu().numpy(), oc)
        assert np.array_equal(offsets.cpu().numpy(), oo)
        assert np.array_equal(gather[:P].cpu().numpy(), og)
    # one routed pair, or one expert, past the fixed scratch: refused, nothing launched
    args = (ctypes.c_void_p(counts.data_ptr()), ctypes.c_void_p(offsets.data_ptr()),
            ctypes.c_void_p(gather.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    assert fn(ctypes.c_void_p(idx.data_ptr()), 65537, 1, E, *args) == m.MOE_ERR_INVALID_ARG
    assert fn(ctypes.c_void_p(idx.data_ptr()), T, k, E + 1, *args) == m.MOE_ERR_INVALID_ARG
