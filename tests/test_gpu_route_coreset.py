"""GPU parity of the router and the block coreset against the fp64 oracle.

Integer outputs are compared bit-exactly: on fed inputs (generator-made logits,
top-k indices and masses, identical on both sides) without exception, and on
computed logits wherever the oracle's own decision margin is outside the
float32 accumulation error (the test asserts the inputs have such margins)."""
import numpy as np
import pytest
import torch

import moe_expert_step_gb300 as ms
import oracle
import synth
from synth import workloads as W
from tests.helpers import (aligned, coreset_margin, dot_error_bound, match_topk, max_rel, np_, router_kind, t,
                           topk_margin_ok)

pytestmark = pytest.mark.gpu


def dims_of(cfg, **over):
    d = dict(H=cfg.H, E=cfg.E, k=cfg.k, I=cfg.I, Is=cfg.Is, V=cfg.V, P=cfg.P,
             dtype=ms.BF16 if cfg.dtype == "bf16" else ms.F32)
    d.update(over)
    return ms.ModelDims(**d)


def route_gpu(d, x, Wr, logits_in=None):
    T = x.shape[0] if x is not None else logits_in.shape[0]
    R = -(-T // d.P)
    ws = ms.workspace(d, R)
    idx = torch.empty((T, d.k), dtype=torch.int32, device="cuda")
    mass = torch.empty((T, d.k), dtype=torch.float32, device="cuda")
    gate = torch.empty_like(mass)
    logits = torch.empty((T, d.E), dtype=torch.float32, device="cuda")
    if logits_in is None:
        ms.moe_block_route(d, x, Wr, idx, mass, gate, ws, logits=logits)
    else:
        ms.moe_route_from_logits(d, logits_in, idx, mass, gate, ws)
        logits = logits_in
    torch.cuda.synchronize()
    assert ms.read_device_error(ws) == ms.OK
    return np_(idx), np_(mass), np_(gate), np_(logits)


@pytest.mark.parametrize("E,k,T", [(256, 8, 32), (16, 4, 8), (100, 7, 45), (1024, 32, 3), (8, 8, 5)])
def test_topk_from_fed_logits_exact(E, k, T):
    cfg = W.LAYER
    d = dims_of(cfg, E=E, k=k, P=32, H=2048)
    key = synth.tensor_key(0, "fed_logits", E, k, T)
    z = synth.host_normal(key, 0, T * E, 1.5, "f32").reshape(T, E)
    z[0, :4] = z[0].max() + 1.0       # a 4-way exact tie at the top: lowest ids first
    if E > 20:
        z[1, 10] = z[1, 17] = z[1, 3]   # ties elsewhere in the ranking
    idx, mass, gate, _ = route_gpu(d, None, None, logits_in=t(z))
    oi, om, og = oracle.route_from_logits(z.astype(np.float64), k)
    np.testing.assert_array_equal(idx, oi)
    assert max_rel(mass, om) < 1e-5
    assert max_rel(gate, og) < 1e-5


@pytest.mark.parametrize("cfg_name,T", [("tiny_fp32", 8), ("clover_layer", 32), ("clover_layer", 71),
                                        ("clover_layer", 300), ("clover_layer", 517)])
def test_route_matches_oracle(cfg_name, T):
    """Computed logits; T = 300 and 517 take the 16- and 32-token router tiles, with ragged tails."""
    cfg = W.CONFIGS[cfg_name]
    d = dims_of(cfg)
    lay = W.device_layer(cfg, 0)
    xa = W.host_activations(cfg, "x_route", T)
    x = W.to_device(xa, cfg.dtype)
    idx, mass, gate, logits = route_gpu(d, x, lay["Wr"])
    ol = W.HostLayer(cfg, 0)
    xo = synth.as_f64(xa, cfg.dtype)
    oi, om, og, oz = oracle.route(xo, ol.Wr, cfg.k)
    assert max_rel(logits, oz) < 1e-5
    eps = dot_error_bound(xo, ol.Wr, router_kind(cfg.H, cfg.E, cfg.dtype))
    ok = topk_margin_ok(oz, eps, cfg.k)
    assert ok.mean() > 0.99
    perm = match_topk(idx[ok], oi[ok], oz[ok], cfg.k, eps[ok])
    assert max_rel(aligned(mass[ok], perm), om[ok]) < 1e-4 and max_rel(aligned(gate[ok], perm), og[ok]) < 1e-4
    assert max_rel(mass, om) < 1e-4 and max_rel(gate, og) < 1e-4


def fed_routing(E, k, T, key):
    """Distinct random experts per token with descending fp32 masses (generator-made)."""
    u = synth.np_uniform01(key, 0, T * E).reshape(T, E)
    idx = np.argsort(u, axis=1)[:, :k].astype(np.int32)
    m = synth.np_uniform01(key ^ 0x55, 0, T * k).reshape(T, k) ** 3 * 0.3
    m = -np.sort(-m, axis=1)
    return idx, m.astype(np.float32)


def coreset_gpu(d, R, top_p, idx, mass):
    ws = ms.workspace(d, R)
    T = idx.shape[0]
    n_sel = torch.empty(R, dtype=torch.int32, device="cuda")
    sel = torch.empty((R, d.E), dtype=torch.int32, device="cuda")
    survive = torch.empty((T, d.k), dtype=torch.uint8, device="cuda")
    gate_rr = torch.empty((T, d.k), dtype=torch.float32, device="cuda")
    ms.coreset_select(d, R, t(np.asarray(top_p, np.float32)), t(idx), t(mass), n_sel, sel, survive, gate_rr, ws)
    torch.cuda.synchronize()
    err = ms.read_device_error(ws)
    return np_(n_sel), np_(sel), np_(survive).astype(bool), np_(gate_rr), err


@pytest.mark.parametrize("E,k,P,R", [(256, 8, 32, 1), (256, 8, 32, 4), (256, 8, 32, 16), (16, 4, 8, 1),
                                     (64, 6, 7, 3), (1024, 32, 5, 2), (300, 8, 1, 9)])
@pytest.mark.parametrize("tp", [1.0, 0.9, 0.7, 0.3, 1e-6])
def test_coreset_fed_exact(E, k, P, R, tp):
    d = ms.ModelDims(H=2048, E=E, k=k, I=512, Is=512, V=1024, P=P, dtype=ms.BF16)
    idx, mass = fed_routing(E, k, R * P, synth.tensor_key(0, "fed_route", E, k, P, R))
    tps = [tp if r % 2 == 0 else min(1.0, tp + 0.15) for r in range(R)]
    n_sel, sel, survive, gate_rr, err = coreset_gpu(d, R, tps, idx, mass)
    assert err == ms.OK
    cs = oracle.coreset_select(idx, mass, tps, P)
    np.testing.assert_array_equal(n_sel, cs.n_sel)
    for r in range(R):
        assert list(sel[r, :n_sel[r]]) == cs.sel[r]
    np.testing.assert_array_equal(survive, cs.survive)
    np.testing.assert_allclose(gate_rr, cs.gate_rr, rtol=2e-6, atol=1e-7)


def test_coreset_edge_cases():
    d = ms.ModelDims(H=2048, E=32, k=4, I=512, Is=512, V=1024, P=4, dtype=ms.BF16)
    # every token picks the same experts; masses tie exactly
    idx = np.tile(np.array([5, 3, 9, 1], np.int32), (4, 1))
    mass = np.full((4, 4), 0.125, np.float32)
    for tp in [0.5, 0.74, 0.76, 1.0]:
        n_sel, sel, survive, gate_rr, err = coreset_gpu(d, 1, [tp], idx, mass)
        cs = oracle.coreset_select(idx, mass, tp, 4)
        assert err == ms.OK and list(sel[0, :n_sel[0]]) == cs.sel[0]
        np.testing.assert_array_equal(survive, cs.survive)
    # all-zero and subnormal masses
    for m in [np.zeros((4, 4), np.float32), np.full((4, 4), 1e-40, np.float32)]:
        n_sel, sel, survive, gate_rr, err = coreset_gpu(d, 1, [0.5], idx, m)
        cs = oracle.coreset_select(idx, m, 0.5, 4)
        assert list(sel[0, :n_sel[0]]) == cs.sel[0]
        np.testing.assert_array_equal(gate_rr, cs.gate_rr)


def test_coreset_near_ties_rank_exactly():
    """Aggregates that differ only far below 2^-22 (the same high word of the 2^-54
    fixed point) and exact ties: the ranking still follows the exact sums, then ids."""
    d = ms.ModelDims(H=2048, E=32, k=4, I=512, Is=512, V=1024, P=2, dtype=ms.BF16)
    q = 2.0 ** -25                                   # one ulp of 0.25 in fp32
    idx = np.array([[3, 7, 1, 2], [9, 4, 11, 12]], np.int32)
    mass = np.array([[0.25, 0.25 + q, 0.2, 0.1], [0.1, 0.1, 0.2 + 2 * q, 0.2]], np.float32)
    for tp in [0.2, 0.5, 1.0]:
        n_sel, sel, survive, gate_rr, err = coreset_gpu(d, 1, [tp], idx, mass)
        cs = oracle.coreset_select(idx, mass, tp, 2)
        assert err == ms.OK and list(sel[0, :n_sel[0]]) == cs.sel[0]
        np.testing.assert_array_equal(survive, cs.survive)
    assert cs.sel[0][:4] == [7, 3, 11, 1]           # exact order, not id order


def test_coreset_flags_bad_input():
    d = ms.ModelDims(H=2048, E=32, k=4, I=512, Is=512, V=1024, P=4, dtype=ms.BF16)
    idx = np.tile(np.array([5, 3, 99, 1], np.int32), (4, 1))   # 99 >= E
    _, _, _, _, err = coreset_gpu(d, 1, [0.9], idx, np.full((4, 4), 0.1, np.float32))
    assert err == ms.EDEVINPUT
    idx[:, 2] = 9
    _, _, _, _, err = coreset_gpu(d, 1, [float("nan")], idx, np.full((4, 4), 0.1, np.float32))
    assert err == ms.EDEVINPUT


@pytest.mark.parametrize("tp", [1.0, 0.9, 0.7])
def test_route_then_coreset_c2(tp):
    """Full route + coreset on the Clover-shaped layer (computed logits, margins checked)."""
    cfg = W.LAYER
    d = dims_of(cfg)
    lay = W.device_layer(cfg, 0)
    xa = W.host_activations(cfg, "x_layer", 32)
    idx, mass, gate, logits = route_gpu(d, W.to_device(xa, "bf16"), lay["Wr"])
    n_sel, sel, survive, gate_rr, err = coreset_gpu(d, 1, [tp], idx, mass)
    xo, Wr = synth.as_f64(xa, "bf16"), W.HostLayer(cfg, 0).Wr
    oi, om, _, oz = oracle.route(xo, Wr, cfg.k)
    eps = dot_error_bound(xo, Wr, "tc")
    assert topk_margin_ok(oz, eps, cfg.k).all()
    perm = match_topk(idx, oi, oz, cfg.k, eps)
    cs = oracle.coreset_select(oi, om, tp, 32)
    assert coreset_margin(cs) > 1e-5
    assert list(sel[0, :n_sel[0]]) == cs.sel[0]
    np.testing.assert_array_equal(aligned(survive, perm), cs.survive)
    if tp == 1.0:
        assert n_sel[0] == len(np.unique(oi))
