"""Pins of the oracle's dispatch (MegaMoE SM90 Implementation Design (Final),
§9.2 "Dispatch Pull Path" and §21 Phase 2 steps 2.3-2.4; PR357 Green-Context
Split MegaMoE code review, §6.1 "Dispatch metadata").

Brute force: the gather map equals the (token, slot) pairs sorted by
(expert, token, slot).  Invariants: counts sum to the number of active pairs,
every active pair appears exactly once, offsets are the exclusive prefix.
"""
import numpy as np
import pytest

import moe_synth


def _brute(idx, E):
    T, k = idx.shape
    pairs = [(int(idx[t, j]), t, j) for t in range(T) for j in range(k) if idx[t, j] >= 0]
    pairs.sort()
    count = np.array([sum(1 for p in pairs if p[0] == e) for e in range(E)], np.int32)
    gather = np.array([t * k + j for _, t, j in pairs], np.int32)
    return count, gather


@pytest.mark.parametrize("T,k,E,seed", [(1, 1, 1, 0), (7, 3, 5, 1), (64, 8, 16, 2), (300, 2, 8, 3), (0, 4, 4, 4)])
def test_dispatch_matches_brute_force(orc, T, k, E, seed):
    rng = np.random.default_rng(seed)
    idx = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    st, count, offset, gather = orc.dispatch(idx, E)
    assert st == orc.OK
    bc, bg = _brute(idx, E)
    assert np.array_equal(count, bc)
    assert np.array_equal(gather, bg)
    assert offset[0] == 0 and np.array_equal(np.diff(offset), count)
    assert count.sum() == (idx >= 0).sum()
    assert sorted(gather.tolist()) == sorted(int(p) for p in np.flatnonzero(idx.reshape(-1) >= 0))


def test_dispatch_routing_from_generator(orc):
    wl = moe_synth.custom(T=200, H=128, I=128, E=16, k=4, seed=9)
    idx, w = moe_synth.make_routing(wl)
    st, count, offset, gather = orc.dispatch(idx, wl.E)
    assert st == orc.OK
    assert count.sum() == wl.T * wl.k                       # counts sum to T*k
    assert len(set(gather.tolist())) == wl.T * wl.k         # each pair exactly once
    bc, bg = _brute(idx.numpy(), wl.E)
    assert np.array_equal(gather, bg)
    assert np.allclose(w.sum(1).numpy(), 1.0, atol=1e-6)


def test_dispatch_reports_bad_expert_and_skips_it(orc):
    idx = np.array([[0, 5], [1, -1]], np.int32)
    st, count, offset, gather = orc.dispatch(idx, 4)
    assert st == orc.EBADEXPERT
    assert count.tolist() == [1, 1, 0, 0]
    assert gather.tolist() == [0, 2]


def test_skewed_and_forced_empty_routing_shapes():
    wl = moe_synth.WORKLOADS["prefill"]
    idx, _ = moe_synth.make_routing(moe_synth.custom(T=wl.T, H=128, I=128, E=wl.E, k=wl.k,
                                                     seed=wl.seed, routing="zipf"))
    cnt = np.bincount(idx.numpy().reshape(-1), minlength=wl.E)
    assert cnt.max() > 10 * cnt.mean() and (cnt == 0).sum() >= 1
    wl4 = moe_synth.WORKLOADS["fp4"]
    idx4, _ = moe_synth.make_routing(moe_synth.custom(T=wl4.T, H=128, I=128, E=wl4.E, k=wl4.k,
                                                      seed=wl4.seed, n_empty=wl4.n_empty))
    cnt4 = np.bincount(idx4.numpy().reshape(-1), minlength=wl4.E)
    assert (cnt4 == 0).sum() >= wl4.n_empty
