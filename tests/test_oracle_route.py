"""Pins for the oracle's router (logits, softmax, top-k, masses, gates).

What pins it: brute-force full sorts, explicit double loops, closed forms of the
two-expert softmax, and a library top-k (torch, float64) on tie-free inputs.
"""
import math

import numpy as np
import pytest

import oracle


def test_router_logits_explicit_loops():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(3, 5))
    Wr = rng.normal(size=(4, 5))
    z = oracle.router_logits(x, Wr)
    for t in range(3):
        for e in range(4):
            assert z[t, e] == pytest.approx(sum(x[t, h] * Wr[e, h] for h in range(5)), abs=1e-12)


def test_softmax_closed_forms():
    z = np.array([[0.3, -1.2], [5.0, 5.0], [1e3, 0.0]])
    p = oracle.softmax(z)
    for row, (a, b) in zip(p, z):
        assert row[0] == pytest.approx(1.0 / (1.0 + math.exp(b - a)), rel=1e-14)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=1e-15)
    np.testing.assert_allclose(oracle.softmax(z + 7.5), p, rtol=1e-13)


def test_topk_brute_force_and_library():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(2)
    z = rng.normal(size=(20, 37))
    idx = oracle.topk_by_logit(z, 6)
    for t in range(20):
        assert list(idx[t]) == sorted(range(37), key=lambda e: -z[t, e])[:6]
    lib = torch.topk(torch.tensor(z, dtype=torch.float64), 6, dim=1).indices.numpy()
    np.testing.assert_array_equal(idx, lib)


def test_topk_ties_go_to_lower_index():
    z = np.array([[1.0, 3.0, 3.0, 2.0, 3.0, 0.0]])
    assert list(oracle.topk_by_logit(z, 4)[0]) == [1, 2, 4, 3]
    z = np.zeros((1, 8))
    assert list(oracle.topk_by_logit(z, 3)[0]) == [0, 1, 2]


def test_route_masses_and_gates():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(5, 16))
    Wr = rng.normal(scale=0.3, size=(12, 16))
    idx, mass, gate, z = oracle.route(x, Wr, 4)
    p = oracle.softmax(z)
    for t in range(5):
        for j in range(4):
            assert mass[t, j] == p[t, idx[t, j]]
        # gate ratios are the logit differences exponentiated, and gates sum to 1
        assert gate[t].sum() == pytest.approx(1.0, rel=1e-14)
        assert gate[t, 0] / gate[t, 1] == pytest.approx(math.exp(z[t, idx[t, 0]] - z[t, idx[t, 1]]), rel=1e-12)
        # masses are non-increasing along the ranking
        assert np.all(np.diff(mass[t]) <= 0)


def test_route_from_logits_matches_route():
    rng = np.random.default_rng(4)
    x = rng.normal(size=(4, 8))
    Wr = rng.normal(size=(10, 8))
    idx, mass, gate, z = oracle.route(x, Wr, 3)
    i2, m2, g2 = oracle.route_from_logits(z, 3)
    np.testing.assert_array_equal(idx, i2)
    np.testing.assert_array_equal(mass, m2)
    np.testing.assert_array_equal(gate, g2)


def test_round_bf16_known_values():
    # 1 + 2^-8 is exactly halfway between bf16 neighbours 1 and 1 + 2^-7: ties to even -> 1
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.140625, 1.0 + 2 ** -9])
    out = oracle.round_bf16(v)
    np.testing.assert_array_equal(out, [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 3.140625, 1.0])
