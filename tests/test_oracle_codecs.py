"""Pins of the oracle's number formats against facts outside the oracle.

E4M3 / BF16 / UE8M0 decoding and rounding are checked against PyTorch's own
casts (a library routine, used here as an external reference only); E2M1 is
checked against the OCP MX grid fixture and by properties (round trip,
nearest-value bracketing, ties to even).  Formats: MegaMoE SM90 Implementation
Design (Final), §2.1 "Scale Factor Format" and "FP4 Tensor Core (E2M1)".
"""
import math
import os
import struct

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f32(x):
    return struct.unpack("<f", struct.pack("<f", x))[0]


def test_e4m3_decode_all_codes_match_torch(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = orc.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])
    assert orc.e4m3_decode(0x7E) == 448.0 and orc.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_round_trip_every_code(orc):
    for c in range(256):
        v = orc.e4m3_decode(c)
        if math.isnan(v):
            assert orc.e4m3_encode(v) == 0x7F
        else:
            assert orc.e4m3_encode(v) == c, c


def test_e4m3_encode_matches_torch_rne_including_ties(orc):
    rng = np.random.default_rng(7)
    vals = list(rng.uniform(-463.0, 463.0, 3000)) + list(rng.normal(0, 1e-2, 1000))
    vals += list(rng.normal(0, 1e-3, 500))
    # exact midpoints between neighbouring codes (ties go to the even code)
    pos = [orc.e4m3_decode(c) for c in range(0x7F)]
    vals += [(pos[i] + pos[i + 1]) / 2 for i in range(len(pos) - 1)]
    vals += [-(pos[i] + pos[i + 1]) / 2 for i in range(len(pos) - 1)]
    vals = [_f32(v) for v in vals]
    ref = torch.tensor(vals, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(v) for v in vals], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates(orc):
    assert orc.e4m3_encode(1e6) == 0x7E
    assert orc.e4m3_encode(-1e6) == 0xFE
    assert orc.e4m3_encode(float("inf")) == 0x7E
    assert orc.e4m3_encode(float("nan")) == 0x7F
    assert orc.e4m3_encode(470.0) == 0x7E


def test_bf16_encode_matches_torch(orc):
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    bits = bits[(bits & 0x7F800000) != 0x7F800000]            # finite
    ties = (rng.integers(0, 2 ** 16, 2000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    ties = ties[(ties & 0x7F800000) != 0x7F800000]
    allb = np.concatenate([bits, ties]).astype(np.uint32)
    f = allb.view(np.float32)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([orc.bf16_encode(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, ref)
    for h in (0x3F80, 0xC2F7, 0x0001, 0x7F7F):
        ref_v = torch.from_numpy(np.array([h], np.uint16).view(np.int16)).view(torch.bfloat16).float().item()
        assert orc.bf16_decode(h) == ref_v


def test_ue8m0_decode_all_codes_match_torch(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    for c in range(255):
        assert orc.ue8m0_decode(c) == ref[c], c
    assert math.isnan(orc.ue8m0_decode(255))


def test_ue8m0_for_amax_is_the_smallest_covering_power_of_two(orc):
    from fractions import Fraction
    rng = np.random.default_rng(11)
    amaxes = list(rng.lognormal(0, 4, 2000).astype(np.float32))
    amaxes += [448.0 * 2.0 ** e for e in range(-20, 20)]          # exact powers of two
    for qmax in (448.0, 6.0):
        for a in amaxes:
            code = orc.ue8m0_for_amax(float(a), qmax)
            e = code - 127
            r = Fraction(float(np.float32(np.float32(a) / np.float32(qmax))))
            if -127 < e < 127:
                assert Fraction(2) ** (e - 1) < r <= Fraction(2) ** e, (a, qmax, e)
    assert orc.ue8m0_for_amax(0.0, 448.0) == 0


def _golden_e2m1():
    out = {}
    with open(os.path.join(GOLDEN, "e2m1_grid.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            c, v = line.split()
            out[int(c)] = float(v)
    return out


def test_e2m1_decode_matches_ocp_grid(orc):
    grid = _golden_e2m1()
    for c in range(16):
        mag = grid[c & 7]
        v = orc.e2m1_decode(c)
        assert v == (-mag if c & 8 else mag) or (mag == 0 and v == 0)


def test_e2m1_decode_matches_e4m3_bit_remap(orc):
    # E2M1 (bias 1) embeds in E4M3 (bias 7): exponent + 6, mantissa << 2;
    # the subnormal 0.5 is the E4M3 normal 2^-1.  Decoded by torch's FP8 cast.
    for c in range(16):
        s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
        if e == 0 and m == 0:
            f8 = 0
        elif e == 0:
            f8 = (6 << 3)
        else:
            f8 = ((e + 6) << 3) | (m << 2)
        f8 |= s << 7
        ref = torch.tensor([f8], dtype=torch.uint8).view(torch.float8_e4m3fn).float().item()
        assert orc.e2m1_decode(c) == ref, c


def test_e2m1_encode_nearest_and_ties_to_even(orc):
    grid = sorted(_golden_e2m1().items(), key=lambda kv: kv[1])
    for c in range(16):
        if c == 8:
            continue
        assert orc.e2m1_encode(orc.e2m1_decode(c)) == c
    rng = np.random.default_rng(5)
    for v in rng.uniform(-7, 7, 4000).astype(np.float32):
        c = orc.e2m1_encode(float(v))
        dv = orc.e2m1_decode(c)
        best = min(abs(abs(float(v)) - g) for _, g in grid)
        assert abs(abs(dv) - min(abs(float(v)), 6.0)) <= best + 1e-12 or abs(v) > 6
        assert math.copysign(1, dv) == math.copysign(1, v) or dv == 0
    # exact midpoints: 0.25 -> 0 (even), 0.75 -> 1.0 (code 2), 1.25 -> 1.0, 1.75 -> 2.0,
    # 2.5 -> 2.0, 3.5 -> 4.0, 5.0 -> 4.0
    expect = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for v, c in expect.items():
        assert orc.e2m1_encode(v) == c, v
        assert orc.e2m1_encode(-v) == (c | 8 if c else 8) or (c == 0 and orc.e2m1_encode(-v) in (0, 8))
    assert orc.e2m1_encode(100.0) == 7 and orc.e2m1_encode(-100.0) == 15
