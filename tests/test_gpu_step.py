"""Whole-step GPU parity (block_decode_step through the C ABI) against the fp64 oracle.

* tiny fp32 model (embed -> MoE -> LM head): the full LowConfidence loop resolves
  the 8-position block round by round exactly as the oracle does, for every
  coreset top_p and two logit scales (fallback-only and mixed rounds).
* Clover-shaped layer, bf16: one round of one layer + LM head (V = 152064).
* 40-layer stack, bf16, 64 GB of expert weights (the benchmark's launch
  configuration): sampled layers are run on the GPU from the oracle's own
  residual stream at that depth and compared element by element; the full
  40-layer step is checked against the oracle where the two must agree
  exactly (layer 0 routing and coreset) and by properties elsewhere."""
import numpy as np
import pytest
import torch

import moe_expert_step_gb300 as ms
import oracle
import synth
from synth import workloads as W
from tests.helpers import BF16_TOL, F32_TOL, coreset_margin, match_topk, max_rel, np_, oracle_layer, t, topk_margins

pytestmark = pytest.mark.gpu
THR = 0.95


def dims_of(cfg):
    return ms.ModelDims(H=cfg.H, E=cfg.E, k=cfg.k, I=cfg.I, Is=cfg.Is, V=cfg.V, P=cfg.P,
                        dtype=ms.BF16 if cfg.dtype == "bf16" else ms.F32)


def clayer(lay):
    return ms.layer(lay["Wr"], lay["Wgu"], lay["Wd"], lay["Wsgu"], lay["Wsd"])


class Step:
    """Device buffers for block_decode_step on R requests."""

    def __init__(self, cfg, R, n_layers):
        self.cfg, self.R, self.T = cfg, R, R * cfg.P
        self.d = dims_of(cfg)
        self.ws = ms.workspace(self.d, R)
        T = self.T
        self.choice = torch.zeros(T, dtype=torch.int32, device="cuda")
        self.conf = torch.zeros(T, dtype=torch.float32, device="cuda")
        self.accept = torch.zeros(T, dtype=torch.uint8, device="cuda")
        self.n_comm = torch.zeros(R, dtype=torch.int32, device="cuda")
        self.h_out = torch.zeros((T, cfg.H), dtype=torch.float32, device="cuda")
        self.hidden = torch.zeros((T, cfg.H), dtype=torch.float32, device="cuda")
        self.n_sel = torch.zeros((max(1, n_layers), R), dtype=torch.int32, device="cuda")
        self.idx = torch.zeros((max(1, n_layers), T, cfg.k), dtype=torch.int32, device="cuda")

    def run(self, layers, Wlm, top_p, h_in, tokens, masked, scale=1.0):
        ms.block_decode_step(self.d, self.R, layers, Wlm, t(np.full(self.R, top_p, np.float32)), THR, h_in, tokens,
                             masked, self.choice, self.conf, self.accept, self.n_comm, self.ws, h_out=self.h_out,
                             logit_scale=scale, trace_n_sel=self.n_sel, trace_idx=self.idx,
                             trace_hidden=self.hidden)
        torch.cuda.synchronize()
        assert ms.read_device_error(self.ws) == ms.OK


@pytest.mark.parametrize("top_p", [1.0, 0.9, 0.5])
@pytest.mark.parametrize("scale", [1.0, 24.0])
def test_tiny_model_full_loop(top_p, scale):
    cfg = W.TINY
    lay = W.device_layer(cfg, 0)
    Wlm_d = W.device_lm_head(cfg)
    emb, pos = W.tiny_tables(cfg)
    emb_d, pos_d = W.to_device(emb, "f32"), W.to_device(pos, "f32")
    st = Step(cfg, 1, 1)
    tokens = torch.zeros(cfg.P, dtype=torch.int32, device="cuda")
    masked = torch.ones(cfg.P, dtype=torch.uint8, device="cuda")
    h = torch.zeros((cfg.P, cfg.H), dtype=torch.float32, device="cuda")
    ol = oracle_layer(cfg, 0)
    Wlm = W.host_lm_head(cfg)
    o_tok = np.zeros(cfg.P, np.int32)
    o_msk = np.ones(cfg.P, bool)
    rounds, fallbacks = 0, 0
    while o_msk.any():
        assert rounds < cfg.P
        ms.block_embed(st.d, 1, tokens, masked, emb_d, pos_d, cfg.V - 1, h)
        st.run([clayer(lay)], Wlm_d, top_p, h, tokens, masked, scale=scale)
        L = oracle.tiny_model_logits(o_tok, o_msk, emb, pos, ol, Wlm, top_p, cfg.k, cfg.V - 1, scale)
        oc, och = oracle.confidence_and_choice(L)
        assert np.abs(np_(st.conf) - oc).max() < 1e-4
        gap = -np.diff(-np.sort(L, axis=1)[:, :2], axis=1)[:, 0]
        assert (gap > 1e-4).all() and (np.abs(oc[o_msk] - THR) > 1e-4).all()
        res = oracle.lowconfidence_commit(oc, och, o_tok, o_msk, THR, cfg.P)
        o_tok, o_msk = res.tokens, res.masked
        np.testing.assert_array_equal(np_(st.accept).astype(bool), res.accept)
        np.testing.assert_array_equal(np_(tokens), o_tok)
        np.testing.assert_array_equal(np_(masked).astype(bool), o_msk)
        fallbacks += int(res.fallback[0])
        rounds += 1
    if scale == 1.0:
        assert rounds == cfg.P and fallbacks == cfg.P     # confidence ~1/V: one commit per round
    else:
        assert rounds < cfg.P                              # the threshold branch fires


@pytest.fixture(params=[ms.SEPARATE_HEAD, ms.CLUSTER_HEAD, ms.FUSED_COMBINE_HEAD],
                ids=["separate", "cluster", "combine-in-router"])
def fusion(request):
    """Every single-request path of block_decode_step between expert launches: separate
    launches, one cluster launch, the combine inside the router launch."""
    prev = ms.route_fusion()
    ms.set_route_fusion(request.param)
    yield request.param
    ms.set_route_fusion(prev)


@pytest.mark.parametrize("corr", [0.0, 0.9])
def test_clover_layer_step(fusion, corr):
    """corr = 0.9: the block's tokens share a hidden component, so they route alike (fewer
    experts, up to 32 tokens per expert chunk)."""
    cfg = W.LAYER
    lay = W.device_layer(cfg, 0)
    Wlm_d = W.device_lm_head(cfg)
    h0 = W.host_h0(cfg, 1, correlation=corr)
    masked0 = W.masked_subset(cfg, 1)
    tokens = t(np.zeros(cfg.P, np.int32))
    masked = t(masked0.astype(np.uint8))
    st = Step(cfg, 1, 1)
    st.run([clayer(lay)], Wlm_d, 0.9, t(h0), tokens, masked)
    trace = []
    h, hidden, L, oc, och, res = oracle.block_decode_step(
        h0.astype(np.float64), [oracle_layer(cfg, 0)], W.host_lm_head(cfg), 0.9, cfg.k, cfg.P, THR,
        np.zeros(cfg.P, np.int32), masked0, bf16=True, trace=trace)
    tr = trace[0]
    assert (topk_margins(tr["z"], cfg.k) > 1e-4).all() and coreset_margin(tr["coreset"]) > 1e-5
    match_topk(np_(st.idx)[0], tr["idx"], tr["z"], cfg.k)
    assert np_(st.n_sel)[0, 0] == tr["coreset"].n_sel[0]
    assert max_rel(np_(st.h_out), h) <= BF16_TOL
    assert max_rel(np_(st.h_out) - h0, h - h0) <= BF16_TOL       # the MoE update itself
    assert max_rel(np_(st.hidden), hidden) <= BF16_TOL
    assert np.abs(np_(st.conf) - oc).max() < 1e-2


@pytest.fixture(scope="module")
def stack():
    cfg = W.STACK
    layers = [W.device_layer(cfg, l) for l in range(cfg.n_layers)]
    return cfg, layers, W.device_lm_head(cfg), W.host_lm_head(cfg)


@pytest.mark.parametrize("depth", [0, 13, 39])
def test_stack_layer_from_oracle_state(stack, depth, fusion):
    """Layer `depth` of the 40-layer stack, fed the oracle's residual stream at that depth."""
    cfg, layers, Wlm_d, Wlm = stack
    h = W.host_h0(cfg, 1).astype(np.float64)
    for l in range(depth):                          # oracle alone walks down to `depth`
        x = oracle.round_bf16(oracle.rmsnorm(h))
        ol = oracle_layer(cfg, l)
        idx, mass, _, _ = oracle.route(x, ol.Wr, cfg.k)
        h = h + oracle.moe_ffn(x, ol, idx, oracle.coreset_select(idx, mass, 0.9, cfg.P).gate_rr)
    h_in = h.astype(np.float32)
    masked0 = W.masked_subset(cfg, 1)
    st = Step(cfg, 1, 1)
    st.run([clayer(layers[depth])], Wlm_d, 0.9, t(h_in), t(np.zeros(cfg.P, np.int32)), t(masked0.astype(np.uint8)))
    trace = []
    h_ref, hidden, L, oc, och, res = oracle.block_decode_step(
        h_in.astype(np.float64), [oracle_layer(cfg, depth)], Wlm, 0.9, cfg.k, cfg.P, THR,
        np.zeros(cfg.P, np.int32), masked0, bf16=True, trace=trace)
    tr = trace[0]
    ok = topk_margins(tr["z"], cfg.k) > 1e-4
    assert ok.all() and coreset_margin(tr["coreset"]) > 1e-5
    match_topk(np_(st.idx)[0], tr["idx"], tr["z"], cfg.k)
    assert np_(st.n_sel)[0, 0] == tr["coreset"].n_sel[0]
    assert max_rel(np_(st.h_out) - h_in, h_ref - h_in) <= BF16_TOL
    assert max_rel(np_(st.h_out), h_ref) <= BF16_TOL


def test_stack_full_step(stack, fusion):
    """All 40 layers in one call, as timed by the benchmark."""
    cfg, layers, Wlm_d, Wlm = stack
    h0 = W.host_h0(cfg, 1)
    masked0 = W.masked_subset(cfg, 1)
    tokens = t(np.zeros(cfg.P, np.int32))
    masked = t(masked0.astype(np.uint8))
    st = Step(cfg, 1, cfg.n_layers)
    st.run([clayer(l) for l in layers], Wlm_d, 0.9, t(h0), tokens, masked)
    n_sel = np_(st.n_sel)[:, 0]
    idx = np_(st.idx)
    # layer 0 sees identical input on both sides: decisions must agree exactly
    x0 = oracle.round_bf16(oracle.rmsnorm(h0.astype(np.float64)))
    ol = oracle_layer(cfg, 0)
    oi, om, _, oz = oracle.route(x0, ol.Wr, cfg.k)
    assert (topk_margins(oz, cfg.k) > 1e-4).all()
    match_topk(idx[0], oi, oz, cfg.k)
    assert n_sel[0] == oracle.coreset_select(oi, om, 0.9, cfg.P).n_sel[0]
    # properties at every depth: each coreset keeps a prefix covering 90% of its own routing
    for l in range(cfg.n_layers):
        assert 8 <= n_sel[l] <= len(np.unique(idx[l]))
        assert all(len(set(row)) == cfg.k for row in idx[l])
    # commit invariants on the round
    acc = np_(st.accept).astype(bool)
    msk = np_(masked).astype(bool)
    assert acc.sum() == np_(st.n_comm)[0] >= 1
    assert not (acc & ~masked0).any() and not (msk & acc).any()
    hid = np_(st.hidden)
    np.testing.assert_allclose(np.sqrt((hid ** 2).mean(1)), 1.0, rtol=2e-2)


def run_stack_modes(stack, modes):
    cfg, layers, Wlm_d, Wlm = stack
    h0 = W.host_h0(cfg, 1)
    masked0 = W.masked_subset(cfg, 1)
    out = []
    prev = ms.route_fusion()
    try:
        for mode in modes:
            ms.set_route_fusion(mode)
            st = Step(cfg, 1, cfg.n_layers)
            tok = t(np.zeros(cfg.P, np.int32))
            st.run([clayer(l) for l in layers], Wlm_d, 0.9, t(h0), tok, t(masked0.astype(np.uint8)))
            out.append((np_(st.idx), np_(st.n_sel), np_(st.h_out), np_(st.hidden), np_(tok), np_(st.conf)))
    finally:
        ms.set_route_fusion(prev)
    return h0, out


def test_route_fusion_matches_separate_launches(stack):
    """The one-launch router/coreset/gather of a single request and the separate
    launches take the same decisions on every layer of the stack; the residual
    stream they produce differs only by the router's summation order."""
    cfg = stack[0]
    h0, ((i1, n1, h1, x1, _, _), (i2, n2, h2, x2, _, _)) = run_stack_modes(stack, [ms.CLUSTER_HEAD, ms.SEPARATE_HEAD])
    # layer 0: identical inputs; both match the oracle's picks (order inside near-tied
    # runs of logits is a rounding decision of each kernel's summation order)
    x0 = oracle.round_bf16(oracle.rmsnorm(h0.astype(np.float64)))
    oi, om, _, oz = oracle.route(x0, oracle_layer(cfg, 0).Wr, cfg.k)
    assert (topk_margins(oz, cfg.k) > 1e-4).all()
    match_topk(i1[0], oi, oz, cfg.k)
    match_topk(i2[0], oi, oz, cfg.k)
    assert n1[0, 0] == n2[0, 0] == oracle.coreset_select(oi, om, 0.9, cfg.P).n_sel[0]
    agree = [(np.sort(i1[l], 1) == np.sort(i2[l], 1)).all() and n1[l, 0] == n2[l, 0] for l in range(cfg.n_layers)]
    if all(agree):
        assert max_rel(h1, h2) <= BF16_TOL and max_rel(x1, x2) <= BF16_TOL
    else:   # a near-tie flipped deep in the stack: the layers before it still agree
        assert agree[: agree.index(False)] == [True] * agree.index(False)


def test_combine_in_router_is_bit_identical(stack):
    """The combine fused into the router's cluster launch does the separate combine and
    router kernels' arithmetic in the same order: all 40 layers' routing, the residual
    stream, the LM-head input and the commit are bit for bit the same."""
    _, (a, b) = run_stack_modes(stack, [ms.FUSED_COMBINE_HEAD, ms.SEPARATE_HEAD])
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)
