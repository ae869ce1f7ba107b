"""Pins for the oracle's expert FFN, RMSNorm and the block-size-1 reduction.

What pins it: SiLU against scipy's logistic function, SwiGLU against explicit
loops and torch float64, a dense all-experts computation masked by the gates,
zero weights, RMSNorm's closed form, and the reduction of a one-token block at
top_p = 1 to an ordinary top-k MoE written separately.
"""
import numpy as np
import pytest

import oracle


def make_layer(rng, H, E, I, Is, std=0.3):
    Wr = rng.normal(scale=std, size=(E, H))
    ex = [(rng.normal(scale=std, size=(I, H)), rng.normal(scale=std, size=(I, H)),
           rng.normal(scale=std, size=(H, I))) for _ in range(E)]
    sh = (rng.normal(scale=std, size=(Is, H)), rng.normal(scale=std, size=(Is, H)),
          rng.normal(scale=std, size=(H, Is)))
    return oracle.MoELayer(Wr=Wr, expert=lambda e: ex[e], shared=lambda: sh), ex, sh


def test_silu_against_library():
    special = pytest.importorskip("scipy.special")
    a = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(oracle.silu(a), a * special.expit(a), rtol=1e-13, atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert oracle.silu(np.array([-1000.0]))[0] == 0.0


def test_swiglu_explicit_loops_and_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    H, I = 6, 4
    x = rng.normal(size=(2, H))
    Wg, Wu, Wd = rng.normal(size=(I, H)), rng.normal(size=(I, H)), rng.normal(size=(H, I))
    y = oracle.swiglu_expert(x, Wg, Wu, Wd)
    for t in range(2):
        act = []
        for i in range(I):
            g = sum(Wg[i, h] * x[t, h] for h in range(H))
            u = sum(Wu[i, h] * x[t, h] for h in range(H))
            act.append(g / (1 + np.exp(-g)) * u)
        for h in range(H):
            assert y[t, h] == pytest.approx(sum(Wd[h, i] * act[i] for i in range(I)), rel=1e-12, abs=1e-12)
    tx = torch.tensor(x)
    ty = (torch.nn.functional.silu(tx @ torch.tensor(Wg).T) * (tx @ torch.tensor(Wu).T)) @ torch.tensor(Wd).T
    np.testing.assert_allclose(y, ty.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("top_p", [1.0, 0.8, 0.5])
def test_sparse_equals_dense_masked(top_p):
    rng = np.random.default_rng(1)
    H, E, k, I, Is, T = 12, 9, 3, 5, 4, 6
    layer, ex, sh = make_layer(rng, H, E, I, Is)
    x = rng.normal(size=(T, H))
    idx, mass, _, _ = oracle.route(x, layer.Wr, k)
    cs = oracle.coreset_select(idx, mass, top_p, T)
    out = oracle.moe_ffn(x, layer, idx, cs.gate_rr)
    dense = np.zeros((T, H))
    all_y = np.stack([oracle.swiglu_expert(x, *ex[e]) for e in range(E)], 1)  # [T, E, H]
    for t in range(T):
        w = np.zeros(E)
        for j in range(k):
            w[idx[t, j]] += cs.gate_rr[t, j]
        dense[t] = w @ all_y[t] + oracle.swiglu_expert(x[t:t + 1], *sh)[0]
    np.testing.assert_allclose(out, dense, rtol=1e-12, atol=1e-12)


def test_zero_weights():
    rng = np.random.default_rng(2)
    H, E, k, I, Is, T = 8, 5, 2, 4, 4, 3
    layer, ex, sh = make_layer(rng, H, E, I, Is)
    zero = tuple(np.zeros_like(w) for w in sh)
    lz = oracle.MoELayer(Wr=layer.Wr, expert=lambda e: tuple(np.zeros_like(w) for w in ex[e]), shared=lambda: zero)
    x = rng.normal(size=(T, H))
    idx, mass, gate, _ = oracle.route(x, layer.Wr, k)
    assert np.all(oracle.moe_ffn(x, lz, idx, gate) == 0.0)
    # zero routed experts: only the shared expert remains
    ls = oracle.MoELayer(Wr=layer.Wr, expert=lz.expert, shared=layer.shared)
    np.testing.assert_allclose(oracle.moe_ffn(x, ls, idx, gate), oracle.swiglu_expert(x, *sh), rtol=1e-14)


@pytest.mark.parametrize("seed", range(4))
def test_block_size_one_is_plain_topk_moe(seed):
    rng = np.random.default_rng(10 + seed)
    H, E, k, I, Is, T = 16, 12, 4, 6, 5, 7
    layer, _, _ = make_layer(rng, H, E, I, Is)
    x = rng.normal(size=(T, H))
    idx, mass, _, _ = oracle.route(x, layer.Wr, k)
    cs = oracle.coreset_select(idx, mass.astype(np.float32), 1.0, 1)   # every token is its own block
    out = oracle.moe_ffn(x, layer, idx, cs.gate_rr)
    ref = oracle.plain_topk_moe(x, layer, k)
    # gates differ only by the fp32 rounding of the masses the coreset is fed
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-6 * np.abs(ref).max())
    cs64 = oracle.coreset_select(idx, mass, 1.0, 1)
    np.testing.assert_allclose(cs64.gate_rr, mass / mass.sum(1, keepdims=True), rtol=1e-15)


def test_rmsnorm_closed_form():
    h = np.array([[3.0, 4.0], [1e-3, -1e-3]])
    out = oracle.rmsnorm(h, 1e-6)
    np.testing.assert_allclose(out[0], h[0] / np.sqrt(12.5 + 1e-6), rtol=1e-15)
    np.testing.assert_allclose(out[1], h[1] / np.sqrt(1e-6 + 1e-6), rtol=1e-15)
    big = np.random.default_rng(3).normal(size=(4, 2048)) * 5
    np.testing.assert_allclose(np.sqrt((oracle.rmsnorm(big) ** 2).mean(1)), 1.0, rtol=1e-6)
