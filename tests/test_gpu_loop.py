"""The device-resident LowConfidence loop (block_decode_loop: a CUDA-graph while node
over rounds of block_embed + block_decode_step, condition set on the device).

* tiny fp32 model: the final tokens and the number of rounds equal the fp64
  oracle's loop (the decision margins of every oracle round are checked);
* Clover-shaped bf16 model (2 layers, V = 152064): bit-identical to the same
  rounds driven from the host, call by call, and the cached graph reproduces
  it on a second call;
* the round cap, a block with nothing masked, and max_rounds = 0."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import moe_expert_step_gb300 as ms
import oracle
from synth import workloads as W
from tests.helpers import np_, oracle_layer, t

pytestmark = pytest.mark.gpu
THR = 0.95


def dims_of(cfg):
    return ms.ModelDims(H=cfg.H, E=cfg.E, k=cfg.k, I=cfg.I, Is=cfg.Is, V=cfg.V, P=cfg.P,
                        dtype=ms.BF16 if cfg.dtype == "bf16" else ms.F32)


def clayer(lay):
    return ms.layer(lay["Wr"], lay["Wgu"], lay["Wd"], lay["Wsgu"], lay["Wsd"])


@pytest.fixture(scope="module")
def tiny():
    cfg = W.TINY
    lay = W.device_layer(cfg, 0)
    emb, pos = W.tiny_tables(cfg)
    return cfg, lay, W.device_lm_head(cfg), W.host_lm_head(cfg), emb, pos


def run_loop(cfg, layers, Wlm_d, emb_d, pos_d, top_p, tokens0, masked0, scale=1.0, max_rounds=None, R=1, ws=None):
    d = dims_of(cfg)
    ws = ms.workspace(d, R) if ws is None else ws
    tokens = t(tokens0.astype(np.int32))
    masked = t(masked0.astype(np.uint8))
    rounds = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ms.block_decode_loop(d, R, layers, Wlm_d, emb_d, pos_d, cfg.V - 1, t(np.full(R, top_p, np.float32)), THR,
                         tokens, masked, rounds, ws, max_rounds=max_rounds, logit_scale=scale)
    torch.cuda.synchronize()
    assert ms.read_device_error(ws) == ms.OK
    return np_(tokens), np_(masked).astype(bool), int(np_(rounds)[0])


@pytest.mark.parametrize("top_p", [1.0, 0.9, 0.5])
@pytest.mark.parametrize("scale", [1.0, 24.0])
def test_tiny_loop_matches_oracle(tiny, top_p, scale):
    cfg, lay, Wlm_d, Wlm, emb, pos = tiny
    ol = oracle_layer(cfg, 0)

    def logits_fn(tok, msk, rnd):
        L = oracle.tiny_model_logits(tok, msk, emb, pos, ol, Wlm, top_p, cfg.k, cfg.V - 1, scale)
        conf, _ = oracle.confidence_and_choice(L)
        gap = -np.diff(-np.sort(L, axis=1)[:, :2], axis=1)[:, 0]
        assert (gap > 1e-4).all() and (np.abs(conf[msk] - THR) > 1e-4).all()   # robust decisions
        return L

    o_tok, o_rounds, _ = oracle.lowconfidence_loop(logits_fn, cfg.P, cfg.P, THR)
    tok, msk, rounds = run_loop(cfg, [clayer(lay)], Wlm_d, W.to_device(emb, "f32"), W.to_device(pos, "f32"), top_p,
                                np.zeros(cfg.P), np.ones(cfg.P, bool), scale)
    assert rounds == o_rounds and not msk.any()
    np.testing.assert_array_equal(tok, o_tok)
    if scale == 1.0:
        assert rounds == cfg.P          # fallback only: one commit per round


def test_tiny_loop_cap_and_degenerate(tiny):
    cfg, lay, Wlm_d, Wlm, emb, pos = tiny
    emb_d, pos_d = W.to_device(emb, "f32"), W.to_device(pos, "f32")
    layers = [clayer(lay)]
    # fallback-only model, capped at 3 rounds: exactly 3 positions committed
    tok, msk, rounds = run_loop(cfg, layers, Wlm_d, emb_d, pos_d, 1.0, np.zeros(cfg.P), np.ones(cfg.P, bool),
                                max_rounds=3)
    assert rounds == 3 and msk.sum() == cfg.P - 3
    # nothing masked: no round runs and nothing changes
    tok0 = np.arange(cfg.P)
    tok, msk, rounds = run_loop(cfg, layers, Wlm_d, emb_d, pos_d, 1.0, tok0, np.zeros(cfg.P, bool))
    assert rounds == 0 and not msk.any()
    np.testing.assert_array_equal(tok, tok0)
    # max_rounds = 0 runs nothing either
    tok, msk, rounds = run_loop(cfg, layers, Wlm_d, emb_d, pos_d, 1.0, np.zeros(cfg.P), np.ones(cfg.P, bool),
                                max_rounds=0)
    assert rounds == 0 and msk.all()


def host_rounds(cfg, layers, Wlm_d, emb_d, pos_d, top_p, tokens0, masked0, R=1, scale=1.0):
    """The same rounds driven from the host: block_embed + block_decode_step until nothing is masked."""
    d = dims_of(cfg)
    ws = ms.workspace(d, R)
    T = R * cfg.P
    tokens = t(tokens0.astype(np.int32))
    masked = t(masked0.astype(np.uint8))
    h = torch.empty((T, cfg.H), dtype=torch.float32, device="cuda")
    choice = torch.empty(T, dtype=torch.int32, device="cuda")
    conf = torch.empty(T, dtype=torch.float32, device="cuda")
    accept = torch.empty(T, dtype=torch.uint8, device="cuda")
    ncomm = torch.empty(R, dtype=torch.int32, device="cuda")
    tp = t(np.full(R, top_p, np.float32))
    rounds = 0
    while np_(masked).any():
        ms.block_embed(d, R, tokens, masked, emb_d, pos_d, cfg.V - 1, h)
        ms.block_decode_step(d, R, layers, Wlm_d, tp, THR, h, tokens, masked, choice, conf, accept, ncomm, ws,
                             logit_scale=scale)
        rounds += 1
        assert rounds <= cfg.P
    torch.cuda.synchronize()
    return np_(tokens), rounds


@pytest.mark.parametrize("R", [1, 4])
def test_clover_loop_equals_host_driven_rounds(R):
    """R = 4: four blocks decoded together, each with its own coreset and its own rounds
    (the loop runs until every request's block is resolved)."""
    cfg = replace(W.LAYER, name="clover_2layer", n_layers=2)
    layers = [clayer(W.device_layer(cfg, l)) for l in range(cfg.n_layers)]
    Wlm_d = W.device_lm_head(cfg)
    # synthetic embedding: N(0, 1) bf16 tables from the generator
    emb_d = W.to_device(W.host_activations(cfg, "emb", cfg.V), "bf16")
    pos_d = W.to_device(W.host_activations(cfg, "pos", cfg.P), "bf16")
    masked0 = W.masked_subset(cfg, R)
    tokens0 = np.where(masked0, 0, np.arange(R * cfg.P) % cfg.P + 7)
    h_tok, h_rounds = host_rounds(cfg, layers, Wlm_d, emb_d, pos_d, 0.9, tokens0, masked0, R=R, scale=24.0)
    ws = ms.workspace(dims_of(cfg), R)
    for _ in range(2):                       # the second call reuses the cached graph
        tok, msk, rounds = run_loop(cfg, layers, Wlm_d, emb_d, pos_d, 0.9, tokens0, masked0, scale=24.0, R=R,
                                    ws=ws)
        assert rounds == h_rounds and not msk.any()
        np.testing.assert_array_equal(tok, h_tok)
    np.testing.assert_array_equal(tok[~masked0], tokens0[~masked0])     # committed tokens never change
