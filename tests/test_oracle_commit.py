"""Pins for the oracle's confidence, argmax and LowConfidence commit and round loop.

What pins it: the hand-worked fixture tests/golden/commit_small.json, the
closed form of a two-logit softmax, scipy's softmax, the loop invariants (at
least one commit per round, committed tokens never change, at most P rounds,
block size 1 resolves in one round) and the toy estimate (1-p)^n for the
probability that a round needs the fallback when positions pass the
threshold independently with probability p.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_golden_commit():
    g = json.load(open(os.path.join(GOLDEN, "commit_small.json")))
    for c in g["cases"]:
        res = oracle.lowconfidence_commit(np.array(c["conf"]), np.array(c["choice"]), np.array(c["tokens"]),
                                          np.array(c["masked"], bool), g["threshold"], g["P"])
        assert res.tokens.tolist() == c["out_tokens"], c["name"]
        assert res.masked.astype(int).tolist() == c["out_masked"], c["name"]
        assert res.accept.astype(int).tolist() == c["accept"], c["name"]
        assert int(res.fallback[0]) == c["fallback"] and int(res.n_committed[0]) == c["n_committed"]


def test_confidence_closed_form_and_library():
    special = pytest.importorskip("scipy.special")
    L = np.array([[2.0, -1.0], [0.5, 0.5], [-3.0, 4.0]])
    conf, choice = oracle.confidence_and_choice(L)
    for row, c in zip(L, conf):
        assert c == pytest.approx(1.0 / (1.0 + math.exp(-abs(row[0] - row[1]))), rel=1e-14)
    assert choice.tolist() == [0, 0, 1]
    rng = np.random.default_rng(0)
    L = rng.normal(scale=4, size=(5, 1000))
    conf, choice = oracle.confidence_and_choice(L)
    np.testing.assert_allclose(conf, special.softmax(L, axis=1).max(1), rtol=1e-12)
    np.testing.assert_array_equal(choice, L.argmax(1))
    L[2, 17] = L[2, 900] = L[2].max() + 1.0
    assert oracle.confidence_and_choice(L)[1][2] == 17


@pytest.mark.parametrize("seed", range(20))
def test_round_invariants(seed):
    rng = np.random.default_rng(seed)
    R, P = 3, 32
    tokens = rng.integers(0, 100, R * P).astype(np.int32)
    masked = rng.random(R * P) < 0.6
    conf = rng.random(R * P) ** 0.2
    choice = rng.integers(0, 1000, R * P).astype(np.int32)
    res = oracle.lowconfidence_commit(conf, choice, tokens, masked, 0.95, P)
    for r in range(R):
        sl = slice(r * P, (r + 1) * P)
        m = masked[sl]
        if m.any():
            assert res.n_committed[r] >= 1
        assert res.n_committed[r] == res.accept[sl].sum()
        assert not (res.accept[sl] & ~m).any()
        np.testing.assert_array_equal(res.tokens[sl][~m], tokens[sl][~m])
        qualifies = m & (conf[sl] >= 0.95)
        assert res.fallback[r] == (m.any() and not qualifies.any())
        if res.fallback[r]:
            p = int(np.flatnonzero(res.accept[sl])[0])
            assert conf[sl][p] == conf[sl][m].max()
        else:
            np.testing.assert_array_equal(res.accept[sl], qualifies)
        np.testing.assert_array_equal(res.tokens[sl][res.accept[sl]], choice[sl][res.accept[sl]])


def test_loop_resolves_within_P_rounds_and_never_rewrites():
    rng = np.random.default_rng(1)
    P, R = 32, 2
    seen = {}

    def logits_fn(tokens, masked, rnd):
        L = rng.normal(scale=rng.uniform(0.5, 12.0), size=(R * P, 64))
        for p, tok in seen.items():
            assert tokens[p] == tok and not masked[p]
        return L

    tokens, rounds, hist = oracle.lowconfidence_loop(logits_fn, R * P, P, 0.95)
    for res in hist:
        for p in np.flatnonzero(res.accept):
            seen[int(p)] = int(res.tokens[p])
        assert (res.n_committed >= 1).all() or not hist[-1].masked.any()
    assert rounds <= P
    assert not hist[-1].masked.any()


def test_block_size_one_resolves_in_one_round():
    rng = np.random.default_rng(2)
    _, rounds, _ = oracle.lowconfidence_loop(lambda t, m, r: rng.normal(size=(5, 50)), 5, 1, 0.95)
    assert rounds == 1


def test_all_fallback_takes_exactly_P_rounds():
    # uniform logits: confidence 1/V everywhere, far below the threshold
    _, rounds, hist = oracle.lowconfidence_loop(lambda t, m, r: np.zeros((8, 16)), 8, 8, 0.95)
    assert rounds == 8 and all(h.fallback[0] and h.n_committed[0] == 1 for h in hist)
    # ties on confidence: the lowest masked position goes first
    assert [int(np.flatnonzero(h.accept)[0]) for h in hist] == list(range(8))


@pytest.mark.parametrize("p", [0.05, 0.1, 0.3])
def test_fallback_rate_matches_toy_estimate(p):
    rng = np.random.default_rng(3)
    n, trials = 32, 20000
    passes = rng.random((trials, n)) < p
    conf = np.where(passes, 0.99, rng.uniform(0.1, 0.9, (trials, n)))
    fb = 0
    commits = 0
    for t in range(trials):
        res = oracle.lowconfidence_commit(conf[t], np.zeros(n, np.int32), np.zeros(n, np.int32),
                                          np.ones(n, bool), 0.95, n)
        fb += int(res.fallback[0])
        commits += int(res.n_committed[0])
    q = (1 - p) ** n
    assert abs(fb / trials - q) < 5 * math.sqrt(q * (1 - q) / trials) + 1e-4
    assert abs(commits / trials - (n * p + q)) < 5 * math.sqrt(n * p * (1 - p) / trials) + 0.01
