"""Pins of the oracle's L1-output quantisers (MegaMoE SM90 Implementation Design
(Final), §10.1 steps 4-6 and §21 Phase 4 step 4.7; FP4-weight configuration:
PR357 Green-Context Split MegaMoE code review, §6.1 "SwiGLU/quant").

Checked: idempotence of the dequantised values, the half-ulp error bound,
the codes against PyTorch's FP8 cast of the same binary32 quotient, and the
degenerate all-zero group.
"""
import numpy as np
import torch


def _dq(orc, q, sf):
    return np.array([orc.e4m3_decode(int(c)) for c in q]) * float(sf)


def _groups(seed, n=200, size=64):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        scale = float(np.exp(rng.uniform(-12, 8)))
        g = (rng.standard_normal(size) * scale).astype(np.float32)
        if i % 7 == 0:
            g[rng.integers(0, size, 5)] = 0.0
        out.append(g)
    return out


def test_fp8_group_codes_match_torch_cast_of_quotient(orc):
    for g in _groups(1):
        sf, q = orc.quant_fp8_group(g)
        assert np.float32(sf) == np.float32(np.abs(g).max()) / np.float32(448.0)
        quot = torch.from_numpy(g) / torch.tensor(sf, dtype=torch.float32)
        ref = quot.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(q, ref)


def test_fp8_group_idempotent_on_dequantised_values(orc):
    for g in _groups(2):
        sf, q = orc.quant_fp8_group(g)
        d1 = _dq(orc, q, sf).astype(np.float32)
        sf2, q2 = orc.quant_fp8_group(d1)
        d2 = _dq(orc, q2, sf2).astype(np.float32)
        assert np.array_equal(d1, d2)
        assert np.array_equal(q, q2)


def test_fp8_group_error_within_half_ulp(orc):
    for g in _groups(3):
        sf, q = orc.quant_fp8_group(g)
        d = _dq(orc, q, sf)
        for v, dv in zip(g.astype(np.float64), d):
            a = abs(v) / sf
            # E4M3 spacing around |a|: 2^(floor(log2 a) - 3) for normals, 2^-9 below 2^-6
            ulp = 2.0 ** -9 if a < 2.0 ** -6 else 2.0 ** (np.floor(np.log2(a)) - 3)
            assert abs(v - dv) <= 0.5 * ulp * sf * (1 + 1e-6) + 1e-30
        amax_pos = int(np.argmax(np.abs(g)))
        assert abs(orc.e4m3_decode(int(q[amax_pos]))) == 448.0


def test_fp8_group_all_zero(orc):
    sf, q = orc.quant_fp8_group(np.zeros(64, np.float32))
    assert sf == 0.0 and not q.any()


def test_ue8m0_group_idempotent_and_bounded(orc):
    for g in _groups(4, size=32):
        code, q = orc.quant_fp8_ue8m0_group(g)
        sf = orc.ue8m0_decode(code)
        d1 = _dq(orc, q, sf).astype(np.float32)
        code2, q2 = orc.quant_fp8_ue8m0_group(d1)
        d2 = _dq(orc, q2, orc.ue8m0_decode(code2)).astype(np.float32)
        assert np.array_equal(d1, d2)
        assert np.abs(d1).max() <= 448.0 * sf
        amax = np.abs(g).max()
        assert amax / 448.0 <= sf * (1 + 1e-6)
        assert amax / 448.0 > sf / 2 * (1 - 1e-6)
    code, q = orc.quant_fp8_ue8m0_group(np.zeros(32, np.float32))
    assert code == 0 and not q.any()
