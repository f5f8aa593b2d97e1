"""Pins of the oracle's expert layer against facts that do not come from it.

* closed form: a one-hot activation row picks one column of W1, so the L1
  output, the SwiGLU, the FP8 requantisation and (with a permutation-matrix
  W2) the L2 output can be written down element by element; gate/up order,
  W2's orientation and the block-scale indexing all show up here;
* k = 1 with weight 1 equals a dense FFN of that expert, computed here in
  matrix form (float64 matmul, PyTorch's FP8/BF16 casts);
* the output does not depend on token order (bit-exact);
* exact power-of-two scalings (top-k weights, W2 scales) scale y exactly;
* an inactive slot (-1) contributes nothing.

Definition followed: MegaMoE SM90 Implementation Design (Final), §3.3, §10.1,
§11.1-§11.2, §15.1, §20.1; PR357 Green-Context Split MegaMoE code review, §6.
"""
import math

import numpy as np
import pytest
import torch

import moe_synth


def _fp8_decode(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _fp8_encode(v32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _bf16_bits(v32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)


def _bf16_value(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).float().numpy()


_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_unpack(packed: np.ndarray) -> np.ndarray:
    lo = packed & 15
    hi = packed >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)
    mag = _GRID[nib & 7]
    return np.where(nib & 8, -mag, mag)


def _ue8m0(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e8m0fnu).to(torch.float64).numpy()


def _np(t):
    return t.numpy() if hasattr(t, "numpy") else t


def dense_ffn(inp, e, w, wfmt=0):
    """Dense quantised FFN of expert e in matrix form, float64 matmuls."""
    x, x_sf = _np(inp["x"]), _np(inp["x_sf"])
    w1, w1_sf, w2, w2_sf = (_np(inp[n]) for n in ("w1", "w1_sf", "w2", "w2_sf"))
    if wfmt == 0:
        X = _fp8_decode(x) * np.repeat(x_sf.astype(np.float64), 128, axis=1)
        W1 = _fp8_decode(w1[e]) * np.kron(w1_sf[e].astype(np.float64), np.ones((128, 128)))
        W2 = _fp8_decode(w2[e]) * np.kron(w2_sf[e].astype(np.float64), np.ones((128, 128)))
        group = 64
    else:
        X = _fp8_decode(x) * np.repeat(_ue8m0(x_sf), 32, axis=1)
        W1 = _e2m1_unpack(w1[e]) * np.repeat(_ue8m0(w1_sf[e]), 32, axis=1)
        W2 = _e2m1_unpack(w2[e]) * np.repeat(_ue8m0(w2_sf[e]), 32, axis=1)
        group = 32
    I = W2.shape[1]
    G = X @ W1[:I].T
    U = X @ W1[I:].T
    A = (G / (1.0 + np.exp(-G)) * U * float(np.float32(w))).astype(np.float32)
    T = A.shape[0]
    Ag = A.reshape(T, I // group, group)
    amax = np.abs(Ag).max(axis=2)
    if wfmt == 0:
        sf = (amax / np.float32(448.0)).astype(np.float32)
    else:
        ratio = (amax / np.float32(448.0)).astype(np.float32)
        m, ex = np.frexp(ratio.astype(np.float64))
        ex = np.where(m == 0.5, ex - 1, ex)
        ex = np.clip(np.where(ratio > 0, ex, -127), -127, 127)
        sf = np.ldexp(np.float32(1.0), ex).astype(np.float32)
    safe = np.where(sf == 0, np.float32(1.0), sf).astype(np.float32)
    quot = (Ag / safe[:, :, None]).astype(np.float32)
    q = _fp8_encode(quot)
    q = np.where((amax == 0)[:, :, None], 0, q).astype(np.uint8)
    AD = (_fp8_decode(q) * sf[:, :, None].astype(np.float64)).reshape(T, I)
    O = AD @ W2.T
    # combine of a single slot: the FP32 accumulator starts at +0
    ob = _bf16_value(_bf16_bits(O.astype(np.float32)))
    return _bf16_bits(np.float32(0.0) + ob)


def _k1_inputs(wl, e_of_token):
    inp = moe_synth.make_inputs(wl)
    inp["topk_idx"] = torch.tensor(e_of_token, dtype=torch.int32).view(-1, 1)
    inp["topk_weights"] = torch.ones(wl.T, 1, dtype=torch.float32)
    return inp


@pytest.mark.parametrize("H,I,E,wfmt", [(256, 128, 2, 0), (384, 256, 3, 0), (256, 128, 2, 1)])
def test_k1_weight1_equals_dense_ffn(orc, H, I, E, wfmt):
    wl = moe_synth.custom(T=5, H=H, I=I, E=E, k=1, seed=21 + H, wfmt=wfmt)
    e_of_token = [t % E for t in range(wl.T)]
    inp = _k1_inputs(wl, e_of_token)
    y = orc.forward(inp, wfmt=wfmt)
    for t in range(wl.T):
        sub = dict(inp)
        sub["x"], sub["x_sf"] = inp["x"][t:t + 1], inp["x_sf"][t:t + 1]
        ref = dense_ffn(sub, e_of_token[t], 1.0, wfmt)[0]
        assert np.array_equal(y[t], ref), (t, np.flatnonzero(y[t] != ref)[:8])


def test_one_hot_closed_form(orc):
    H, I = 128, 128
    h0 = 37
    x = np.zeros((1, H), np.uint8)
    x[0, h0] = 0x38                                    # 1.0 in E4M3
    x_sf = np.ones((1, 1), np.float32) * 0.75
    rng = np.random.default_rng(4)
    w1 = rng.integers(0, 0x7E, size=(1, 2 * I, H)).astype(np.uint8)
    w1 |= (rng.integers(0, 2, size=w1.shape) << 7).astype(np.uint8)
    w1_sf = np.array([[[0.5], [0.25]]], np.float32)    # gate block, up block
    perm = rng.permutation(I)                          # o[h] = ad[perm^-1(h)]
    w2 = np.zeros((1, H, I), np.uint8)
    w2[0, perm, np.arange(I)] = 0x38
    w2_sf = np.array([[[2.0]]], np.float32)
    wt = np.float32(0.8125)
    inp = {"x": x, "x_sf": x_sf, "topk_idx": np.zeros((1, 1), np.int32),
           "topk_weights": np.array([[wt]], np.float32),
           "w1": w1, "w1_sf": w1_sf, "w2": w2, "w2_sf": w2_sf}
    # by hand
    a = np.zeros(I, np.float32)
    for i in range(I):
        g = _fp8_decode(w1[0, i, h0:h0 + 1])[0] * 0.5 * 0.75
        u = _fp8_decode(w1[0, I + i, h0:h0 + 1])[0] * 0.25 * 0.75
        a[i] = np.float32(g / (1.0 + math.exp(-g)) * u * float(wt))
    ad = np.zeros(I)
    for b in range(I // 64):
        grp = a[b * 64:(b + 1) * 64]
        sf = np.float32(np.abs(grp).max()) / np.float32(448.0)
        q = _fp8_encode(grp / sf)
        ad[b * 64:(b + 1) * 64] = _fp8_decode(q) * float(sf)
    o = np.zeros(H)
    o[perm] = ad * 2.0
    ob = _bf16_value(_bf16_bits(o.astype(np.float32)))
    ref = _bf16_bits(np.float32(0.0) + ob)            # combine accumulator starts at +0
    assert np.array_equal(orc.forward(inp)[0], ref)
    pr = orc.pair(inp, 0, 0, float(wt))
    assert np.array_equal(pr["a"], a)


def test_token_order_invariance(orc):
    wl = moe_synth.custom(T=24, H=256, I=128, E=6, k=3, seed=5)
    inp = moe_synth.make_inputs(wl)
    y = orc.forward(inp)
    perm = torch.randperm(wl.T, generator=torch.Generator().manual_seed(1))
    pinp = dict(inp)
    for n in ("x", "x_sf", "topk_idx", "topk_weights"):
        pinp[n] = inp[n][perm].contiguous()
    yp = orc.forward(pinp)
    assert np.array_equal(yp, y[perm.numpy()])


def test_power_of_two_scalings_are_exact(orc):
    wl = moe_synth.custom(T=12, H=256, I=128, E=4, k=2, seed=6)
    inp = moe_synth.make_inputs(wl)
    y = _bf16_value(orc.forward(inp))
    s1 = dict(inp); s1["topk_weights"] = inp["topk_weights"] * 4.0
    assert np.array_equal(_bf16_value(orc.forward(s1)), y * 4.0)
    s2 = dict(inp); s2["w2_sf"] = inp["w2_sf"] * 0.5
    assert np.array_equal(_bf16_value(orc.forward(s2)), y * 0.5)


def test_inactive_slot_contributes_nothing_and_slots_sum_in_fp32(orc):
    wl = moe_synth.custom(T=6, H=256, I=128, E=4, k=2, seed=8)
    inp = moe_synth.make_inputs(wl)
    idx = inp["topk_idx"].clone()
    idx[:, 1] = -1
    one = dict(inp); one["topk_idx"] = idx
    y1 = orc.forward(one)
    for t in range(wl.T):
        e0 = int(idx[t, 0]); w0 = float(inp["topk_weights"][t, 0])
        ob = _bf16_value(orc.pair(inp, t, e0, w0)["ob"])
        assert np.array_equal(y1[t], _bf16_bits(np.float32(0.0) + ob))
    y2 = orc.forward(inp)
    for t in range(wl.T):
        obs = [orc.pair(inp, t, int(inp["topk_idx"][t, j]), float(inp["topk_weights"][t, j]))["ob"]
               for j in range(2)]
        acc = np.float32(0) + _bf16_value(obs[0]).astype(np.float32)
        acc = (acc + _bf16_value(obs[1]).astype(np.float32)).astype(np.float32)
        assert np.array_equal(y2[t], _bf16_bits(acc))
    none = dict(inp); none["topk_idx"] = torch.full_like(idx, -1)
    assert not orc.forward(none).any()


def test_activation_clamp_bounds_gate_and_up(orc):
    wl = moe_synth.custom(T=4, H=256, I=128, E=2, k=1, seed=12)
    inp = moe_synth.make_inputs(wl)
    c = 0.05
    pr = orc.pair(inp, 0, int(inp["topk_idx"][0, 0]), 1.0, act_clamp=c)
    bound = c / (1 + math.exp(-c)) * c
    assert np.abs(pr["a"]).max() <= bound * (1 + 1e-6)
    free = orc.pair(inp, 0, int(inp["topk_idx"][0, 0]), 1.0)
    assert np.abs(free["a"]).max() > bound
