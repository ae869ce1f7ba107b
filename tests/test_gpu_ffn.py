"""GPU parity of the routed + shared expert FFN (route -> coreset -> experts) against
the fp64 oracle, through the C ABI.  Routing and coreset decisions are first
checked to be identical (inputs with safe margins), then the fp32 FFN output is
compared element by element: max relative error <= 1e-4 (fp32 configuration)
or <= 2e-2 (bf16 weights, fp32 accumulation)."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import moe_expert_step_gb300 as ms
import oracle
import synth
from synth import workloads as W
from tests.helpers import (BF16_TOL, F32_TOL, aligned, coreset_margin, dot_error_bound, match_topk, max_rel, np_,
                           oracle_layer, router_kind, t, topk_margin_ok)

pytestmark = pytest.mark.gpu


def dims_of(cfg):
    return ms.ModelDims(H=cfg.H, E=cfg.E, k=cfg.k, I=cfg.I, Is=cfg.Is, V=cfg.V, P=cfg.P,
                        dtype=ms.BF16 if cfg.dtype == "bf16" else ms.F32)


def gpu_moe(cfg, R, x, lay, top_p):
    """route -> coreset -> ffn on one workspace; returns (idx, mass, n_sel, sel, survive, gate_rr, out)."""
    d = dims_of(cfg)
    T = R * cfg.P
    ws = ms.workspace(d, R)
    idx = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
    mass = torch.empty((T, cfg.k), dtype=torch.float32, device="cuda")
    gate = torch.empty_like(mass)
    n_sel = torch.empty(R, dtype=torch.int32, device="cuda")
    sel = torch.empty((R, cfg.E), dtype=torch.int32, device="cuda")
    survive = torch.empty((T, cfg.k), dtype=torch.uint8, device="cuda")
    gate_rr = torch.empty_like(mass)
    out = torch.empty((T, cfg.H), dtype=torch.float32, device="cuda")
    ms.moe_block_route(d, x, lay["Wr"], idx, mass, gate, ws)
    tp = t(np.full(R, top_p, np.float32))
    ms.coreset_select(d, R, tp, idx, mass, n_sel, sel, survive, gate_rr, ws)
    L = ms.layer(lay["Wr"], lay["Wgu"], lay["Wd"], lay["Wsgu"] if cfg.Is else None, lay["Wsd"] if cfg.Is else None)
    ms.moe_block_ffn(d, R, x, L, gate_rr, out, ws)
    torch.cuda.synchronize()
    assert ms.read_device_error(ws) == ms.OK
    return np_(idx), np_(mass), np_(n_sel), np_(sel), np_(survive).astype(bool), np_(gate_rr), np_(out)


def check_against_oracle(cfg, R, top_p, tol, tag="x_ffn"):
    T = R * cfg.P
    lay = W.device_layer(cfg, 0)
    xa = W.host_activations(cfg, tag, T)
    idx, mass, n_sel, sel, survive, gate_rr, out = gpu_moe(cfg, R, W.to_device(xa, cfg.dtype), lay, top_p)
    ol = oracle_layer(cfg, 0)
    x = synth.as_f64(xa, cfg.dtype)
    oi, om, _, oz = oracle.route(x, ol.Wr, cfg.k)
    eps = dot_error_bound(x, ol.Wr, router_kind(cfg.H, cfg.E, cfg.dtype))
    assert topk_margin_ok(oz, eps, cfg.k).all(), "test input too close to a top-k tie"
    perm = match_topk(idx, oi, oz, cfg.k, eps)
    cs = oracle.coreset_select(oi, om, top_p, cfg.P)
    assert coreset_margin(cs) > 1e-5, "test input too close to the coreset cut"
    np.testing.assert_array_equal(n_sel, cs.n_sel)
    for r in range(R):
        assert list(sel[r, :n_sel[r]]) == cs.sel[r]
    np.testing.assert_array_equal(aligned(survive, perm), cs.survive)
    np.testing.assert_allclose(aligned(gate_rr, perm), cs.gate_rr, rtol=1e-5, atol=1e-7)
    ref = oracle.moe_ffn(x, ol, oi, cs.gate_rr)
    err = max_rel(out, ref)
    assert err <= tol, err
    return err


@pytest.mark.parametrize("top_p", [1.0, 0.9, 0.5])
def test_tiny_fp32(top_p):
    check_against_oracle(W.TINY, 1, top_p, F32_TOL)


@pytest.mark.parametrize("top_p", [1.0, 0.9, 0.7])
def test_clover_layer_bf16(top_p):
    check_against_oracle(W.LAYER, 1, top_p, BF16_TOL)


RAGGED = replace(W.LAYER, name="ragged", family="ragged", H=256, E=64, k=6, I=128, Is=128, V=1024, P=7)
NOSHARED = replace(W.LAYER, name="noshared", family="noshared", H=384, E=48, k=4, I=192, Is=0, V=1024, P=16)
WIDE = replace(W.LAYER, name="wide", family="wide", H=512, E=32, k=8, I=256, Is=384, V=1024, P=32)


@pytest.mark.parametrize("cfg,R,top_p", [(RAGGED, 3, 0.9), (RAGGED, 1, 1.0), (NOSHARED, 2, 0.8), (WIDE, 2, 0.95),
                                         (replace(W.TINY, P=5), 3, 0.9)])
def test_shapes(cfg, R, top_p):
    tol = F32_TOL if cfg.dtype == "f32" else BF16_TOL
    check_against_oracle(cfg, R, top_p, tol)


@pytest.mark.parametrize("R", [4, 16])
def test_clover_layer_batched(R):
    """Several requests: per-request coresets, experts grouped over the union (N up to 256,
    the shared expert split into several token chunks at R = 16)."""
    check_against_oracle(W.LAYER, R, 0.9, BF16_TOL, tag="x_batched")


def test_ffn_is_deterministic():
    cfg = W.LAYER
    lay = W.device_layer(cfg, 0)
    x = W.to_device(W.host_activations(cfg, "x_ffn", 32), "bf16")
    a = gpu_moe(cfg, 1, x, lay, 0.9)[-1]
    b = gpu_moe(cfg, 1, x, lay, 0.9)[-1]
    np.testing.assert_array_equal(a, b)
