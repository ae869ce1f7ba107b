"""Pins for the oracle's composed functions: the LM head (lm_logits), the whole
denoising round of the MoE stack (block_decode_step) and the tiny
embed -> MoE -> LM-head model that drives the round loop (tiny_model_logits).

These compose primitives pinned elsewhere (router, coreset, SwiGLU, RMSNorm,
commit).  What is checked here is the composition itself, each time against
arithmetic written out independently in plain Python loops (math.exp /
math.sqrt, bf16 rounding through torch's own float32 -> bfloat16 cast) or
against special cases whose result is fixed by the definition:

* lm_logits is the explicit triple sum times the scale, and a unit hidden
  vector picks out one column of the head times the scale;
* with zero expert weights every layer adds nothing, so the final residual is
  the input and the LM-head input is bf16(RMSNorm(h_0));
* a stack of one-token blocks at top_p = 1 is the textbook pre-norm residual
  top-k MoE (softmax over the k largest logits as gates, shared expert added),
  layer after layer, with the bf16 hand-over points of the loop body
  ([AIT] section 三: logits = model(block) -> softmax -> conf / choice ->
  accept / fallback);
* requests are independent: a two-request round equals each request's round
  on its own;
* the tiny model with every position masked feeds emb[MASK] + pos[p]; at
  top_p = 1 a position's logits depend on its own input only.

A plausible composition mistake (norm on the wrong tensor, a lost residual,
bf16 rounding at the wrong point or missing, the logit scale applied twice,
the final norm skipped, a coreset taken over the wrong block) fails one of
these.
"""
import math

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")


# ---------------------------------------------------------------------------------- independent helpers
def bf16_torch(v):
    """Nearest-even bfloat16 of float64 values via torch's float32 -> bfloat16 cast."""
    t = torch.tensor(np.asarray(v, np.float64), dtype=torch.float64).to(torch.float32).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


def rms_loops(row, eps=1e-6):
    ms = sum(v * v for v in row) / len(row)
    d = math.sqrt(ms + eps)
    return [v / d for v in row]


def swiglu_loops(x, Wg, Wu, Wd):
    I, H = len(Wg), len(x)
    act = []
    for i in range(I):
        g = sum(Wg[i][h] * x[h] for h in range(H))
        u = sum(Wu[i][h] * x[h] for h in range(H))
        act.append(g / (1.0 + math.exp(-g)) * u)
    return [sum(Wd[h][i] * act[i] for i in range(I)) for h in range(H)]


def topk_moe_token_loops(x, Wr, experts, shared, k):
    """Ordinary top-k MoE of one token: gates = softmax over the k largest router logits
    (ties to the lower expert id), plus the shared expert with weight 1."""
    E, H = len(Wr), len(x)
    z = [sum(Wr[e][h] * x[h] for h in range(H)) for e in range(E)]
    top = sorted(range(E), key=lambda e: (-z[e], e))[:k]
    zmax = max(z[e] for e in top)
    w = [math.exp(z[e] - zmax) for e in top]
    s = sum(w)
    out = [0.0] * H
    for wj, e in zip(w, top):
        y = swiglu_loops(x, *experts[e])
        for h in range(H):
            out[h] += wj / s * y[h]
    ys = swiglu_loops(x, *shared)
    return [out[h] + ys[h] for h in range(H)]


def make_stack(rng, n_layers, H, E, I, Is, std=0.4):
    layers, raw = [], []
    for _ in range(n_layers):
        Wr = rng.normal(scale=std, size=(E, H))
        ex = [tuple(rng.normal(scale=std, size=s) for s in ((I, H), (I, H), (H, I))) for _ in range(E)]
        sh = tuple(rng.normal(scale=std, size=s) for s in ((Is, H), (Is, H), (H, Is)))
        layers.append(oracle.MoELayer(Wr=Wr, expert=lambda e, ex=ex: ex[e], shared=lambda sh=sh: sh))
        raw.append((Wr, ex, sh))
    return layers, raw


def zero_stack(layers):
    z = []
    for l in layers:
        ex = lambda e, l=l: tuple(np.zeros_like(w) for w in l.expert(e))
        sh = tuple(np.zeros_like(w) for w in l.shared())
        z.append(oracle.MoELayer(Wr=l.Wr, expert=ex, shared=lambda sh=sh: sh))
    return z


# ---------------------------------------------------------------------------------- lm_logits
def test_lm_logits_triple_loop_and_scale():
    rng = np.random.default_rng(0)
    P, H, V = 3, 5, 7
    hid, W = rng.normal(size=(P, H)), rng.normal(size=(V, H))
    for scale in (1.0, 2.5, -0.75):
        L = oracle.lm_logits(hid, W, scale)
        for p in range(P):
            for v in range(V):
                ref = scale * sum(hid[p, h] * W[v, h] for h in range(H))
                assert L[p, v] == pytest.approx(ref, rel=1e-13, abs=1e-13)


def test_lm_logits_unit_hidden_selects_a_column():
    rng = np.random.default_rng(1)
    H, V = 6, 9
    W = rng.normal(size=(V, H))
    hid = np.eye(H)[[2, 5]]
    L = oracle.lm_logits(hid, W, 3.0)
    np.testing.assert_array_equal(L[0], 3.0 * W[:, 2])
    np.testing.assert_array_equal(L[1], 3.0 * W[:, 5])


# ---------------------------------------------------------------------------------- block_decode_step
@pytest.mark.parametrize("bf16", [False, True])
def test_step_with_zero_experts_is_norm_and_head(bf16):
    """Zero routed and shared weights: every layer adds 0, so h_L = h_0 exactly and the
    LM head reads bf16(RMSNorm(h_0)) (bf16 configurations) or RMSNorm(h_0)."""
    rng = np.random.default_rng(2)
    H, E, k, I, Is, P, V = 8, 6, 2, 4, 3, 4, 11
    layers, _ = make_stack(rng, 3, H, E, I, Is)
    zl = zero_stack(layers)
    h0 = rng.normal(size=(P, H)) * 3.0
    Wlm = rng.normal(size=(V, H))
    masked = np.array([True, False, True, True])
    tokens = np.array([0, 7, 0, 0], np.int32)
    h, hidden, L, conf, choice, res = oracle.block_decode_step(h0, zl, Wlm, 0.8, k, P, 0.95, tokens, masked,
                                                               bf16=bf16, logit_scale=2.0)
    np.testing.assert_array_equal(h, h0)
    want = np.array([rms_loops(list(r)) for r in h0])
    if bf16:
        want = bf16_torch(want)
        np.testing.assert_array_equal(hidden, want)
    else:
        np.testing.assert_allclose(hidden, want, rtol=1e-14, atol=0)
    for p in range(P):
        for v in range(V):
            assert L[p, v] == pytest.approx(2.0 * sum(hidden[p, j] * Wlm[v, j] for j in range(H)), rel=1e-12, abs=1e-12)
    # the commit is the LowConfidence round on those logits: position 1 was committed already
    assert res.tokens[1] == 7 and not res.accept[1]
    assert res.n_committed[0] == res.accept.sum() >= 1


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("seed", [0, 1])
def test_stack_of_one_token_blocks_is_plain_residual_topk_moe(bf16, seed):
    """One-token blocks at top_p = 1: the coreset keeps the token's own k experts, so each
    layer is an ordinary top-k MoE; the stack is h_{l+1} = h_l + MoE_l(q(RMSNorm(h_l))),
    hidden = q(RMSNorm(h_L)), logits = scale * hidden Wlm^T (q = bf16 rounding or identity)."""
    rng = np.random.default_rng(10 + seed)
    H, E, k, I, Is, T, V, n_layers = 6, 5, 2, 3, 3, 3, 8, 2
    layers, raw = make_stack(rng, n_layers, H, E, I, Is)
    h0 = rng.normal(size=(T, H)) * 2.0
    Wlm = rng.normal(size=(V, H))
    q = bf16_torch if bf16 else (lambda v: np.asarray(v, np.float64))
    h_ref = [list(r) for r in h0]
    for Wr, ex, sh in raw:
        for t in range(T):
            x = list(q(rms_loops(h_ref[t])))
            out = topk_moe_token_loops(x, Wr.tolist(), [tuple(w.tolist() for w in e) for e in ex],
                                       tuple(w.tolist() for w in sh), k)
            h_ref[t] = [h_ref[t][j] + out[j] for j in range(H)]
    hid_ref = q([rms_loops(r) for r in h_ref])
    scale = 1.5
    masked = np.ones(T, bool)
    h, hidden, L, conf, choice, res = oracle.block_decode_step(h0, layers, Wlm, 1.0, k, 1, 0.95,
                                                               np.zeros(T, np.int32), masked, bf16=bf16,
                                                               logit_scale=scale)
    np.testing.assert_allclose(h, np.array(h_ref), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(hidden, hid_ref, rtol=1e-11, atol=1e-11)
    L_ref = np.array([[scale * sum(hid_ref[t][j] * Wlm[v, j] for j in range(H)) for v in range(V)] for t in range(T)])
    np.testing.assert_allclose(L, L_ref, rtol=1e-11, atol=1e-11)
    # every position is its own one-token block: each commits exactly once
    assert res.accept.all() and (res.n_committed == 1).all()
    np.testing.assert_array_equal(res.tokens, np.argmax(L_ref, axis=1))


def test_step_bf16_rounding_points_matter():
    """The bf16 hand-over points are exercised: the bf16 and float64 rounds differ."""
    rng = np.random.default_rng(3)
    H, E, k, I, Is, T, V = 6, 5, 2, 3, 3, 2, 8
    layers, _ = make_stack(rng, 2, H, E, I, Is)
    h0 = rng.normal(size=(T, H))
    Wlm = rng.normal(size=(V, H))
    args = (h0, layers, Wlm, 1.0, k, 1, 0.95, np.zeros(T, np.int32), np.ones(T, bool))
    a = oracle.block_decode_step(*args, bf16=True)
    b = oracle.block_decode_step(*args, bf16=False)
    assert not np.array_equal(a[0], b[0]) and not np.array_equal(a[1], b[1])


@pytest.mark.parametrize("top_p", [1.0, 0.6])
def test_step_requests_are_independent(top_p):
    """Two requests in one round give what each gives alone (decisions exactly, floats up to
    the summation order of the library matmul): the coreset, the commit and everything else
    act within a request's own block."""
    rng = np.random.default_rng(4)
    H, E, k, I, Is, P, V = 8, 7, 3, 4, 4, 3, 10
    layers, _ = make_stack(rng, 2, H, E, I, Is)
    h0 = rng.normal(size=(2 * P, H))
    Wlm = rng.normal(size=(V, H))
    masked = np.array([True, True, False, True, False, True])
    tokens = np.array([0, 0, 4, 0, 2, 0], np.int32)
    both = oracle.block_decode_step(h0, layers, Wlm, [top_p, top_p], k, P, 0.5, tokens, masked, bf16=True)
    for r in range(2):
        sl = slice(r * P, (r + 1) * P)
        one = oracle.block_decode_step(h0[sl], layers, Wlm, top_p, k, P, 0.5, tokens[sl], masked[sl], bf16=True)
        for a, b in zip(both[:5], one[:5]):     # BLAS may order a product's sums by shape
            np.testing.assert_allclose(a[sl], b, rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(both[5].tokens[sl], one[5].tokens)
        np.testing.assert_array_equal(both[5].accept[sl], one[5].accept)
        assert both[5].n_committed[r] == one[5].n_committed[0]


def test_step_trace_is_the_layer_by_layer_composition():
    """The trace's per-layer records chain: layer l's input is bf16(RMSNorm(h_l)) with
    h_{l+1} = h_l + out_l, and the routing/coreset recorded are those of that input."""
    rng = np.random.default_rng(5)
    H, E, k, I, Is, P, V = 8, 6, 2, 4, 3, 4, 9
    layers, _ = make_stack(rng, 3, H, E, I, Is)
    h0 = rng.normal(size=(P, H))
    tr = []
    h, hidden, *_ = oracle.block_decode_step(h0, layers, rng.normal(size=(V, H)), 0.7, k, P, 0.95,
                                             np.zeros(P, np.int32), np.ones(P, bool), bf16=True, trace=tr)
    assert len(tr) == 3
    hr = h0.copy()
    for l, rec in enumerate(tr):
        np.testing.assert_array_equal(rec["x"], bf16_torch([rms_loops(list(r)) for r in hr]))
        idx, mass, _, _ = oracle.route(rec["x"], layers[l].Wr, k)
        np.testing.assert_array_equal(rec["idx"], idx)
        cs = oracle.coreset_select(idx, mass, 0.7, P)
        np.testing.assert_array_equal(rec["coreset"].survive, cs.survive)
        hr = hr + rec["out"]
    np.testing.assert_array_equal(h, hr)
    np.testing.assert_array_equal(hidden, bf16_torch([rms_loops(list(r)) for r in hr]))


# ---------------------------------------------------------------------------------- tiny model
def tiny_setup(seed=6):
    rng = np.random.default_rng(seed)
    H, E, k, I, Is, P, V = 6, 5, 2, 3, 3, 4, 9
    (layer,), raw = make_stack(rng, 1, H, E, I, Is)
    emb = rng.normal(size=(V, H))
    pos = rng.normal(size=(P, H))
    Wlm = rng.normal(size=(V, H))
    return dict(H=H, E=E, k=k, P=P, V=V, layer=layer, raw=raw[0], emb=emb, pos=pos, Wlm=Wlm)


def tiny_logits_loops(s, ids, scale):
    """emb[id] + pos[p] -> h + MoE(RMSNorm(h)) (one-token top-k MoE, top_p = 1) -> scale * RMSNorm(.) Wlm^T."""
    Wr, ex, sh = s["raw"]
    out = []
    for p, i in enumerate(ids):
        h = [s["emb"][i][j] + s["pos"][p][j] for j in range(s["H"])]
        y = topk_moe_token_loops(rms_loops(h), Wr.tolist(), [tuple(w.tolist() for w in e) for e in ex],
                                 tuple(w.tolist() for w in sh), s["k"])
        hn = rms_loops([h[j] + y[j] for j in range(s["H"])])
        out.append([scale * sum(hn[j] * s["Wlm"][v][j] for j in range(s["H"])) for v in range(s["V"])])
    return np.array(out)


def test_tiny_model_all_masked_feeds_mask_embedding():
    """Every position masked: input p is emb[MASK] + pos[p]; whatever the token ids hold is
    ignored.  At top_p = 1 each position is the plain top-k MoE of its own input."""
    s = tiny_setup()
    mask_id = s["V"] - 1
    masked = np.ones(s["P"], bool)
    L1 = oracle.tiny_model_logits(np.zeros(s["P"], np.int32), masked, s["emb"], s["pos"], s["layer"], s["Wlm"], 1.0,
                                  s["k"], mask_id, 4.0)
    L2 = oracle.tiny_model_logits(np.array([3, 1, 4, 1], np.int32), masked, s["emb"], s["pos"], s["layer"],
                                  s["Wlm"], 1.0, s["k"], mask_id, 4.0)
    np.testing.assert_array_equal(L1, L2)
    np.testing.assert_allclose(L1, tiny_logits_loops(s, [mask_id] * s["P"], 4.0), rtol=1e-11, atol=1e-11)


def test_tiny_model_committed_positions_read_their_tokens():
    """A committed position feeds emb[token] + pos[p]; at top_p = 1 only its own row changes."""
    s = tiny_setup(7)
    mask_id = s["V"] - 1
    tokens = np.array([0, 2, 0, 5], np.int32)
    masked = np.array([True, False, True, False])
    L = oracle.tiny_model_logits(tokens, masked, s["emb"], s["pos"], s["layer"], s["Wlm"], 1.0, s["k"], mask_id, 1.0)
    ids = [mask_id, 2, mask_id, 5]
    np.testing.assert_allclose(L, tiny_logits_loops(s, ids, 1.0), rtol=1e-11, atol=1e-11)
    L_all = oracle.tiny_model_logits(tokens, np.ones(4, bool), s["emb"], s["pos"], s["layer"], s["Wlm"], 1.0,
                                     s["k"], mask_id, 1.0)
    np.testing.assert_array_equal(L[[0, 2]], L_all[[0, 2]])
    assert not np.allclose(L[[1, 3]], L_all[[1, 3]])


def test_tiny_model_zero_experts_and_scale():
    """Zero expert weights: logits = scale * RMSNorm(emb[id] + pos[p]) Wlm^T (one final norm,
    the scale once)."""
    s = tiny_setup(8)
    zl = zero_stack([s["layer"]])[0]
    mask_id = s["V"] - 1
    L = oracle.tiny_model_logits(np.zeros(s["P"], np.int32), np.ones(s["P"], bool), s["emb"], s["pos"], zl, s["Wlm"],
                                 0.5, s["k"], mask_id, 3.0)
    for p in range(s["P"]):
        hn = rms_loops([s["emb"][mask_id][j] + s["pos"][p][j] for j in range(s["H"])])
        for v in range(s["V"]):
            assert L[p, v] == pytest.approx(3.0 * sum(hn[j] * s["Wlm"][v][j] for j in range(s["H"])), rel=1e-12,
                                            abs=1e-12)


@pytest.mark.parametrize("seed,top_p", [(9, 0.6), (12, 0.5), (14, 0.4)])
def test_tiny_model_coreset_spans_the_block(seed, top_p):
    """At top_p < 1 the coreset is one decision for the whole block: the logits equal the
    composition route -> coreset over all P positions -> experts with the re-routed gates."""
    s = tiny_setup(seed)
    mask_id = s["V"] - 1
    masked = np.ones(s["P"], bool)
    L = oracle.tiny_model_logits(np.zeros(s["P"], np.int32), masked, s["emb"], s["pos"], s["layer"], s["Wlm"], top_p,
                                 s["k"], mask_id, 1.0)
    h0 = np.array([[s["emb"][mask_id][j] + s["pos"][p][j] for j in range(s["H"])] for p in range(s["P"])])
    x = np.array([rms_loops(list(r)) for r in h0])
    idx, mass, _, _ = oracle.route(x, s["layer"].Wr, s["k"])
    cs = oracle.coreset_select(idx, mass, top_p, s["P"])
    assert not cs.survive.all()                      # the cut removes candidates here ...
    # ... and differently from a coreset taken per position
    assert not np.array_equal(cs.survive, oracle.coreset_select(idx, mass, top_p, 1).survive)
    Wr, ex, sh = s["raw"]
    ref = []
    for p in range(s["P"]):
        y = swiglu_loops(list(x[p]), *(w.tolist() for w in sh))
        for j in range(s["k"]):
            if cs.survive[p, j]:
                ye = swiglu_loops(list(x[p]), *(w.tolist() for w in ex[idx[p, j]]))
                y = [y[i] + cs.gate_rr[p, j] * ye[i] for i in range(s["H"])]
        hn = rms_loops([h0[p][i] + y[i] for i in range(s["H"])])
        ref.append([sum(hn[i] * s["Wlm"][v][i] for i in range(s["H"])) for v in range(s["V"])])
    np.testing.assert_allclose(L, np.array(ref), rtol=1e-11, atol=1e-11)
