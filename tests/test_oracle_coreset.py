"""Pins for the oracle's block coreset.

What pins it: a hand-worked fixture (tests/golden/coreset_small.json), the
top_p = 1 reduction to the union of all candidates, nesting in top_p, the
covering bounds of the cut, brute force over every subset on tiny blocks,
order independence and request independence.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def random_routing(rng, T, E, k, sharp=1.0):
    z = rng.normal(scale=sharp, size=(T, E))
    idx, mass, _ = oracle.route_from_logits(z, k)
    return idx, mass.astype(np.float32)


def test_golden_small():
    g = json.load(open(os.path.join(GOLDEN, "coreset_small.json")))
    idx = np.array(g["idx"])
    mass = np.array(g["mass"])
    for case in g["cases"]:
        cs = oracle.coreset_select(idx, mass, case["top_p"], g["tokens_per_req"])
        assert cs.sel[0] == case["sel"], case
        np.testing.assert_array_equal(cs.survive.astype(int), case["survive"])
        np.testing.assert_allclose(cs.gate_rr, case["gate_rr"], rtol=1e-15)


def test_top_p_one_is_union_of_candidates():
    rng = np.random.default_rng(5)
    idx, mass = random_routing(rng, 32, 64, 8)
    cs = oracle.coreset_select(idx, mass, 1.0, 32)
    assert set(cs.sel[0]) == set(np.unique(idx).tolist())
    assert cs.survive.all()
    np.testing.assert_allclose(cs.gate_rr, mass / mass.astype(np.float64).sum(1, keepdims=True), rtol=1e-7)


@pytest.mark.parametrize("seed", range(5))
def test_nesting_and_cover_bounds(seed):
    rng = np.random.default_rng(seed)
    idx, mass = random_routing(rng, 16, 40, 4, sharp=2.0)
    prev = set()
    for tp in [0.05, 0.2, 0.5, 0.7, 0.9, 0.97, 1.0]:
        cs = oracle.coreset_select(idx, mass, tp, 16)
        S = cs.sel[0]
        assert prev <= set(S)
        prev = set(S)
        agg = cs.agg[0]
        if cs.target[0] is not None:
            cum = [sum(agg[e] for e in S[:m]) for m in range(len(S) + 1)]
            assert cum[-1] >= cs.target[0] > cum[-2]
            total = sum(agg.values())
            assert cs.target[0] == min(max(math.ceil(float(np.float32(tp)) * float(total)), 1), total)


def brute_force_coreset(idx, mass, top_p):
    """Minimum-cardinality set of candidate experts whose mass reaches the target,
    maximum mass among those, then the lexicographically smallest id tuple."""
    q = oracle.mass_to_fixed(mass)
    agg = {}
    for t in range(idx.shape[0]):
        for j in range(idx.shape[1]):
            agg[int(idx[t, j])] = agg.get(int(idx[t, j]), 0) + int(q[t, j])
    cands = sorted(agg)
    total = sum(agg.values())
    if top_p >= 1.0:
        return set(cands)
    target = min(max(math.ceil(float(np.float32(top_p)) * float(total)), 1), total)
    for m in range(1, len(cands) + 1):
        best = None
        for sub in itertools.combinations(cands, m):
            s = sum(agg[e] for e in sub)
            if s >= target:
                key = (-s, sub)
                if best is None or key < best:
                    best = key
        if best is not None:
            return set(best[1])
    raise AssertionError


@pytest.mark.parametrize("seed", range(40))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(100 + seed)
    T, E, k = int(rng.integers(1, 4)), int(rng.integers(3, 9)), int(rng.integers(1, 4))
    k = min(k, E)
    if seed % 3 == 0:
        # force equal aggregated masses to exercise the tie-break
        idx = np.array([rng.permutation(E)[:k] for _ in range(T)])
        mass = np.full((T, k), 0.125, np.float32)
    else:
        idx, mass = random_routing(rng, T, E, k, sharp=1.5)
    for tp in [0.1, 0.3, 0.5, 0.75, 0.9, 1.0]:
        cs = oracle.coreset_select(idx, mass, tp, T)
        assert set(cs.sel[0]) == brute_force_coreset(idx, mass, tp)


def test_order_independence():
    rng = np.random.default_rng(7)
    idx, mass = random_routing(rng, 32, 128, 8)
    a = oracle.coreset_select(idx, mass, 0.7, 32)
    perm = rng.permutation(32)
    b = oracle.coreset_select(idx[perm], mass[perm], 0.7, 32)
    assert a.sel[0] == b.sel[0]
    np.testing.assert_array_equal(a.survive[perm], b.survive)
    # permuting candidates within a token also changes nothing
    cperm = rng.permutation(8)
    c = oracle.coreset_select(idx[:, cperm], mass[:, cperm], 0.7, 32)
    assert a.sel[0] == c.sel[0]


def test_requests_are_independent():
    rng = np.random.default_rng(8)
    idx, mass = random_routing(rng, 4 * 8, 32, 4)
    tps = [0.9, 0.5, 1.0, 0.7]
    joint = oracle.coreset_select(idx, mass, tps, 8)
    for r in range(4):
        sl = slice(8 * r, 8 * r + 8)
        alone = oracle.coreset_select(idx[sl], mass[sl], tps[r], 8)
        assert joint.sel[r] == alone.sel[0]
        np.testing.assert_array_equal(joint.survive[sl], alone.survive)
        np.testing.assert_array_equal(joint.gate_rr[sl], alone.gate_rr)


def test_degenerate_cases():
    idx = np.array([[0, 1], [1, 2]])
    # all-zero mass: keep every candidate
    cs = oracle.coreset_select(idx, np.zeros((2, 2), np.float32), 0.5, 2)
    assert set(cs.sel[0]) == {0, 1, 2}
    # tiny top_p keeps exactly the top-ranked expert
    cs = oracle.coreset_select(idx, np.array([[0.25, 0.5], [0.5, 0.125]], np.float32), 1e-9, 2)
    assert cs.sel[0] == [1]
    # a token whose candidates are all pruned gets zero gates
    idx = np.array([[0, 1], [2, 3]])
    cs = oracle.coreset_select(idx, np.array([[0.5, 0.4], [0.01, 0.01]], np.float32), 0.9, 2)
    assert cs.sel[0] == [0, 1]
    assert not cs.survive[1].any() and (cs.gate_rr[1] == 0).all()
    for bad in [0.0, -0.1, float("nan")]:
        with pytest.raises(ValueError):
            oracle.coreset_select(idx, np.ones((2, 2), np.float32), bad, 2)


def test_fixed_point_is_exact():
    m = np.array([2.0 ** -30, 0.1, 1.0, 3e-20], np.float32)
    q = oracle.mass_to_fixed(m)
    assert q[0] == 2 ** 24 and q[2] == 2 ** 54
    assert q[1] == int(float(np.float32(0.1)) * 2 ** 54)
    assert q[3] == round(float(np.float32(3e-20)) * 2 ** 54)
