"""Whole-step GPU parity (block_decode_step through the C ABI) against the fp64 oracle.

* tiny fp32 model (embed -> MoE -> LM head): the full LowConfidence loop resolves
  the 8-position block round by round exactly as the oracle does, for every
  coreset top_p and two logit scales (fallback-only and mixed rounds).
* Clover-shaped layer, bf16: one round of one layer + LM head (V = 152064).
* 40-layer stack, bf16, 64 GB of expert weights (the benchmark's launch
  configuration), teacher-forced: the step records every layer's input x_l (the
  bf16 bits its router and experts read) and residual h_l; the oracle takes the
  GPU's x_l and must reproduce layer l's routing, coreset and MoE update
  h_{l+1} - h_l, and from the GPU's final hidden state the LM head's choice and
  the commit.  One request on every 4th layer and the last; 4, 8 and 16
  requests (one coreset per request, experts grouped over the union) on the
  first and last layers.
* Both layer-head paths (separate launches; the combine inside the router's
  cluster launch) give bit-identical steps at 1, 4 and 8 requests."""
import numpy as np
import pytest
import torch

import moe_expert_step_gb300 as ms
import oracle
from synth import workloads as W
from tests.helpers import (BF16_TOL, F32_TOL, aligned, assert_ranked_equal, coreset_margin, max_rel, np_,
                           oracle_layer, oracle_routing, router_kind, t)

pytestmark = pytest.mark.gpu
THR = 0.95


def dims_of(cfg):
    return ms.ModelDims(H=cfg.H, E=cfg.E, k=cfg.k, I=cfg.I, Is=cfg.Is, V=cfg.V, P=cfg.P,
                        dtype={"bf16": ms.BF16, "fp8": ms.FP8}.get(cfg.dtype, ms.F32))


def clayer(lay):
    return ms.layer(lay["Wr"], lay["Wgu"], lay["Wd"], lay["Wsgu"], lay["Wsd"])


class Step:
    """Device buffers for block_decode_step on R requests, with the per-layer trace."""

    def __init__(self, cfg, R, n_layers, trace_xh=False):
        self.cfg, self.R, self.T = cfg, R, R * cfg.P
        self.d = dims_of(cfg)
        self.ws = ms.workspace(self.d, R)
        T, L = self.T, max(1, n_layers)
        self.choice = torch.zeros(T, dtype=torch.int32, device="cuda")
        self.conf = torch.zeros(T, dtype=torch.float32, device="cuda")
        self.accept = torch.zeros(T, dtype=torch.uint8, device="cuda")
        self.n_comm = torch.zeros(R, dtype=torch.int32, device="cuda")
        self.h_out = torch.zeros((T, cfg.H), dtype=torch.float32, device="cuda")
        self.hidden = torch.zeros((T, cfg.H), dtype=torch.float32, device="cuda")
        self.n_sel = torch.zeros((L, R), dtype=torch.int32, device="cuda")
        self.sel = torch.zeros((L, R, cfg.E), dtype=torch.int32, device="cuda")
        self.idx = torch.zeros((L, T, cfg.k), dtype=torch.int32, device="cuda")
        xdt = torch.bfloat16 if cfg.act_dtype == "bf16" else torch.float32
        self.x = torch.zeros((L, T, cfg.H), dtype=xdt, device="cuda") if trace_xh else None
        self.h = torch.zeros((L, T, cfg.H), dtype=torch.float32, device="cuda") if trace_xh else None

    def run(self, layers, Wlm, top_p, h_in, tokens, masked, scale=1.0):
        ms.block_decode_step(self.d, self.R, layers, Wlm, t(np.full(self.R, top_p, np.float32)), THR, h_in, tokens,
                             masked, self.choice, self.conf, self.accept, self.n_comm, self.ws, h_out=self.h_out,
                             logit_scale=scale, trace_n_sel=self.n_sel, trace_idx=self.idx, trace_hidden=self.hidden,
                             trace_sel=self.sel, trace_x=self.x, trace_h=self.h)
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


@pytest.fixture(params=[ms.SEPARATE_HEAD, ms.FUSED_COMBINE_HEAD], ids=["separate", "combine-in-router"])
def fusion(request):
    """Both paths of block_decode_step between expert launches: separate combine / router /
    coreset / gather launches, and the combine inside the router launch."""
    prev = ms.route_fusion()
    ms.set_route_fusion(request.param)
    yield request.param
    ms.set_route_fusion(prev)


def check_routing(cfg, l, st, top_p, Wr=None):
    """Router and coreset of layer l of a traced step against the oracle fed the GPU's own
    input x_l: exact top-k sets (order within the fp32 error window); the coreset's kept
    experts per request exactly where the cut is decided beyond the masses' fp32 error, in
    the oracle's ranking order except among experts whose aggregated masses are within that
    error of each other.
    Returns (x_l, oracle top-k, coreset, tokens whose k-th/(k+1)-th logits were within the
    error bound, taken as the kernel decided)."""
    R, P = st.R, cfg.P
    x = np_(st.x[l]).astype(np.float64)
    Wr = W.HostLayer(cfg, l).Wr if Wr is None else Wr
    idx, mass, z, perm, amb = oracle_routing(x, Wr, cfg.k, router_kind(cfg.H, cfg.E, cfg.dtype), np_(st.idx[l]))
    cs = oracle.coreset_select(idx, mass, top_p, P)
    n_sel, sel = np_(st.n_sel[l]), np_(st.sel[l])
    for r in range(R):
        sub = oracle.CoresetResult(cs.n_sel[r:r + 1], cs.sel[r:r + 1], None, None, cs.ranking[r:r + 1],
                                   cs.agg[r:r + 1], cs.target[r:r + 1])
        if coreset_margin(sub) > 1e-5:
            assert n_sel[r] == cs.n_sel[r], (l, r)
            assert_ranked_equal(sel[r, :n_sel[r]], cs, r, where=(l, r))
    return x, idx, cs, amb


def check_layer(cfg, l, st, top_p, last_h=None, ol=None):
    """Layer l of a traced step against the oracle fed the GPU's own input x_l: routing and
    coreset as in check_routing, and the MoE update h_{l+1} - h_l within the bf16
    tolerance.  Returns the number of tokens taken as the kernel decided (check_routing)."""
    h_l = np_(st.h[l]).astype(np.float64)
    h_next = last_h if last_h is not None else np_(st.h[l + 1]).astype(np.float64)
    ol = ol or oracle_layer(cfg, l)
    x, idx, cs, amb = check_routing(cfg, l, st, top_p, ol.Wr)
    out = oracle.moe_ffn(x, ol, idx, cs.gate_rr)
    err = max_rel(h_next - h_l, out)
    assert err <= BF16_TOL, (l, err)
    return amb


def check_commit(cfg, st, Wlm, tokens_gpu, masked_gpu, masked0):
    """LM head + commit from the GPU's final hidden state (bf16 bits, LM-head input).
    Choice where the top-2 logits are decided beyond the bf16 head's fp32 error; the
    LowConfidence commit where every decision it takes is decided likewise."""
    hid = np_(st.hidden).astype(np.float64)
    L = oracle.lm_logits(hid, Wlm)
    oc, och = oracle.confidence_and_choice(L)
    top2 = -np.sort(-L, axis=1)[:, :2]
    clear = top2[:, 0] - top2[:, 1] > 2e-3
    choice = np_(st.choice)
    np.testing.assert_array_equal(choice[clear], och[clear])
    assert max_rel(np_(st.conf), oc) < 1e-2
    tok0 = np.zeros(st.T, np.int32)
    res = oracle.lowconfidence_commit(oc, och, tok0, masked0, THR, cfg.P)
    for r in range(st.R):
        sl = slice(r * cfg.P, (r + 1) * cfg.P)
        m = masked0[sl]
        c = np.sort(oc[sl][m])[::-1]
        decided = (np.abs(oc[sl][m] - THR) > 1e-3).all() and (len(c) < 2 or c[0] - c[1] > 1e-3 * c[0]) \
            and clear[sl][m].all()
        if decided:
            np.testing.assert_array_equal(np_(st.accept)[sl].astype(bool), res.accept[sl])
            np.testing.assert_array_equal(tokens_gpu[sl], res.tokens[sl])
            np.testing.assert_array_equal(masked_gpu[sl].astype(bool), res.masked[sl])
    acc = np_(st.accept).astype(bool)
    for r in range(st.R):    # invariants everywhere
        sl = slice(r * cfg.P, (r + 1) * cfg.P)
        assert acc[sl].sum() == np_(st.n_comm)[r] >= 1
        assert not (acc[sl] & ~masked0[sl]).any()


@pytest.mark.parametrize("corr", [0.0, 0.9])
def test_clover_layer_step(fusion, corr):
    """One layer + LM head.  corr = 0.9: the block's tokens share a hidden component, so
    they route alike (fewer experts, up to 32 tokens per expert chunk)."""
    cfg = W.LAYER
    lay = W.device_layer(cfg, 0)
    Wlm_d = W.device_lm_head(cfg)
    h0 = W.host_h0(cfg, 1, correlation=corr)
    masked0 = W.masked_subset(cfg, 1)
    tokens = t(np.zeros(cfg.P, np.int32))
    masked = t(masked0.astype(np.uint8))
    st = Step(cfg, 1, 1, trace_xh=True)
    st.run([clayer(lay)], Wlm_d, 0.9, t(h0), tokens, masked)
    np.testing.assert_array_equal(np_(st.h[0]), h0)                 # h_0 is the input
    check_layer(cfg, 0, st, 0.9, last_h=np_(st.h_out).astype(np.float64))
    # the free-running oracle from the same h0 (the GPU's x_0 may differ from it by a bf16 ulp)
    h, hidden, L, oc, och, res = oracle.block_decode_step(
        h0.astype(np.float64), [oracle_layer(cfg, 0)], W.host_lm_head(cfg), 0.9, cfg.k, cfg.P, THR,
        np.zeros(cfg.P, np.int32), masked0, bf16=True)
    assert max_rel(np_(st.h_out) - h0, h - h0) <= BF16_TOL
    assert max_rel(np_(st.hidden), hidden) <= BF16_TOL
    assert np.abs(np_(st.conf) - oc).max() < 1e-2


@pytest.fixture(scope="module")
def stack():
    cfg = W.STACK
    layers = [W.device_layer(cfg, l) for l in range(cfg.n_layers)]
    return cfg, [clayer(l) for l in layers], W.device_lm_head(cfg), W.host_lm_head(cfg)


def run_stack(stack, R, trace_xh=True):
    cfg, layers, Wlm_d, _ = stack
    h0 = W.host_h0(cfg, R)
    masked0 = W.masked_subset(cfg, R)
    tokens = t(np.zeros(R * cfg.P, np.int32))
    masked = t(masked0.astype(np.uint8))
    st = Step(cfg, R, cfg.n_layers, trace_xh=trace_xh)
    st.run(layers, Wlm_d, 0.9, t(h0), tokens, masked)
    return st, h0, masked0, np_(tokens), np_(masked)


def test_stack_full_step_teacher_forced(stack):
    """All 40 layers in one call, as timed by the benchmark, against the oracle fed the
    GPU's own layer input: every layer's routing and coreset; the MoE update of every 4th
    layer and the last (each needs its kept experts' weights generated in fp64); LM head
    and commit from the GPU's final hidden state."""
    cfg, _, _, Wlm = stack
    st, h0, masked0, tok, msk = run_stack(stack, 1)
    np.testing.assert_array_equal(np_(st.h[0]), h0)
    ambiguous = 0
    full = set(range(0, cfg.n_layers - 1, 4)) | {cfg.n_layers - 1}
    for l in range(cfg.n_layers):
        last = np_(st.h_out).astype(np.float64) if l == cfg.n_layers - 1 else None
        ambiguous += check_layer(cfg, l, st, 0.9, last_h=last) if l in full else check_routing(cfg, l, st, 0.9)[3]
    assert ambiguous <= 2          # near-ties at the top-k boundary are rare (about 1e-4 per token)
    # the LM head reads bf16(RMSNorm(h_L))
    hl = np_(st.h_out).astype(np.float64)
    assert max_rel(np_(st.hidden), oracle.round_bf16(oracle.rmsnorm(hl))) <= 2 ** -8
    check_commit(cfg, st, Wlm, tok, msk, masked0)


@pytest.mark.parametrize("R", [4, 8, 16])
def test_stack_batched_teacher_forced(stack, fusion, R):
    """R requests through the 40-layer step (one coreset per request, experts grouped over
    the union of the requests' kept experts) against the oracle fed the GPU's layer inputs:
    every layer's routing and per-request coresets, the first and last layers' MoE updates,
    the commit of every request.  At R = 16 (512 tokens) both modes take the separate
    launches."""
    if R == 16 and fusion == ms.FUSED_COMBINE_HEAD:
        pytest.skip("512 block tokens: the combine-in-router path does not apply (same launches as 'separate')")
    cfg, _, _, Wlm = stack
    st, h0, masked0, tok, msk = run_stack(stack, R)
    np.testing.assert_array_equal(np_(st.h[0]), h0)
    ambiguous = check_layer(cfg, 0, st, 0.9)
    for l in range(1, cfg.n_layers - 1):
        ambiguous += check_routing(cfg, l, st, 0.9)[3]
    ambiguous += check_layer(cfg, cfg.n_layers - 1, st, 0.9, last_h=np_(st.h_out).astype(np.float64))
    # near-ties at the top-k boundary: about 1e-4 per token and layer
    assert ambiguous <= 2 + R * cfg.P * cfg.n_layers // 2000, ambiguous
    n_sel = np_(st.n_sel)
    for r in range(R):               # each request's coreset keeps a covering prefix of its own candidates
        for l in range(cfg.n_layers):
            cand = np.unique(np_(st.idx[l])[r * cfg.P:(r + 1) * cfg.P])
            assert 8 <= n_sel[l, r] <= len(cand)
            assert set(np_(st.sel[l, r, :n_sel[l, r]])) <= set(cand)
    check_commit(cfg, st, Wlm, tok, msk, masked0)


@pytest.mark.parametrize("R", [1, 4, 8])
def test_combine_in_router_is_bit_identical(stack, R):
    """The combine fused into the router's cluster launch does the separate combine and
    router kernels' arithmetic in the same order: all 40 layers' routing and coresets, the
    residual stream, the LM-head input and the commit are bit for bit the same, at one
    request (one 8-token-tile cluster row per tile: 4 tiles) and at 4 and 8 requests
    (16 and 32 tiles of clusters, one coreset per request)."""
    prev = ms.route_fusion()
    outs = []
    try:
        for mode in (ms.FUSED_COMBINE_HEAD, ms.SEPARATE_HEAD):
            ms.set_route_fusion(mode)
            st, _, _, tok, msk = run_stack(stack, R, trace_xh=False)
            outs.append((np_(st.idx), np_(st.n_sel), np_(st.sel), np_(st.h_out), np_(st.hidden), tok, msk,
                         np_(st.conf)))
    finally:
        ms.set_route_fusion(prev)
    for u, v in zip(*outs):
        np.testing.assert_array_equal(u, v)
