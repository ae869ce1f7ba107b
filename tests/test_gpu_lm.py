"""GPU parity of the LM head, the confidence/argmax reduction and the LowConfidence
commit against the fp64 oracle.

* Fed logits (identical on both sides): choice, accept, fallback, tokens and masked
  are bit-exact; conf within 1e-5 relative.
* Vocabulary 152064, hidden 2048, bf16 (tcgen05 LM head): logits within 1e-5 of
  the largest logit, choice exact wherever the oracle's top-2 gap exceeds 1e-2,
  conf within 5e-4, accept/fallback exact (inputs keep conf >= 1e-3 away from 0.95).
* A full block loop over a fixed sequence of per-round hidden states resolves
  every position identically to the oracle, with at least one commit per round."""
import numpy as np
import pytest
import torch

import moe_expert_step_gb300 as ms
import oracle
import synth
from synth import workloads as W
from tests.helpers import max_rel, np_, t
from tests.lm_inputs import hidden_with_confidences, top2_gap

pytestmark = pytest.mark.gpu

THR = 0.95


def outputs(n):
    z = lambda dt: torch.zeros(n, dtype=dt, device="cuda")
    return z(torch.int32), z(torch.float32), z(torch.uint8)


def fed_logits(T, V, key):
    L = synth.host_normal(key, 0, T * V, 1.0, "f32").reshape(T, V)
    rng_u = synth.np_uniform01(key ^ 7, 0, 2 * T).reshape(T, 2)
    for p in range(T):
        top = int(rng_u[p, 0] * V)
        L[p, top] += np.float32(6.0 + 14.0 * rng_u[p, 1])   # spread confidences over (0, 1)
    L[0, 5] = L[0, 9] = L[0].max() + 2.0                  # exact argmax tie: lowest id wins
    return L


@pytest.mark.parametrize("R,P,V", [(1, 32, 152064), (3, 8, 1024), (2, 5, 3000), (1, 1, 77)])
def test_commit_from_fed_logits_exact(R, P, V):
    d = ms.ModelDims(H=2048, E=256, k=8, I=512, Is=512, V=V, P=P, dtype=ms.BF16)
    T = R * P
    L = fed_logits(T, V, synth.tensor_key(0, "fed_lm", R, P, V))
    masked = W.masked_subset(W.LAYER, R, tag=f"fed_mask_{P}")[:T] if P == 32 else \
        (synth.np_uniform01(synth.tensor_key(0, "m", R, P), 0, T) < 0.7)
    masked[0] = True
    tokens = (np.arange(T) * 7 % V).astype(np.int32)
    ws = ms.workspace(d, R)
    tok, msk = t(tokens), t(masked.astype(np.uint8))
    choice, conf, accept = outputs(T)
    n_comm = torch.zeros(R, dtype=torch.int32, device="cuda")
    ms.lm_commit_from_logits(d, R, t(L), THR, tok, msk, choice, conf, accept, n_comm, ws)
    torch.cuda.synchronize()
    oc, och = oracle.confidence_and_choice(L.astype(np.float64))
    res = oracle.lowconfidence_commit(oc, och, tokens, masked, THR, P)
    np.testing.assert_array_equal(np_(choice), och)
    assert max_rel(np_(conf), oc) < 1e-5
    band = np.abs(oc - THR) < 1e-5
    assert not band[masked].any()
    np.testing.assert_array_equal(np_(accept).astype(bool), res.accept)
    np.testing.assert_array_equal(np_(tok), res.tokens)
    np.testing.assert_array_equal(np_(msk).astype(bool), res.masked)
    np.testing.assert_array_equal(np_(n_comm), res.n_committed)


@pytest.fixture(scope="module")
def lm_head():
    cfg = W.LMHEAD
    return cfg, W.device_lm_head(cfg), W.host_lm_head(cfg)


def run_lm(cfg, Wlm_dev, hidden_bits, tokens, masked, R=1, want_logits=False):
    d = ms.ModelDims(H=cfg.H, E=cfg.E, k=cfg.k, I=cfg.I, Is=cfg.Is, V=cfg.V, P=cfg.P, dtype=ms.BF16)
    T = R * cfg.P
    ws = ms.workspace(d, R)
    choice, conf, accept = outputs(T)
    n_comm = torch.zeros(R, dtype=torch.int32, device="cuda")
    logits = torch.empty((T, cfg.V), dtype=torch.float32, device="cuda") if want_logits else None
    ms.lm_head_commit(d, R, W.to_device(hidden_bits, "bf16"), Wlm_dev, THR, tokens, masked, choice, conf, accept,
                      n_comm, ws, logits=logits)
    torch.cuda.synchronize()
    assert ms.read_device_error(ws) == ms.OK
    return np_(choice), np_(conf), np_(accept).astype(bool), np_(n_comm), (np_(logits) if want_logits else None)


def test_lm_head_one_round(lm_head):
    cfg, Wlm_dev, Wlm = lm_head
    bits, hid = hidden_with_confidences(cfg, Wlm, cfg.P, "round0")
    masked0 = W.masked_subset(cfg, 1)
    tokens0 = np.full(cfg.P, 3, np.int32)
    tok, msk = t(tokens0), t(masked0.astype(np.uint8))
    choice, conf, accept, n_comm, logits = run_lm(cfg, Wlm_dev, bits, tok, msk, want_logits=True)
    L = oracle.lm_logits(hid, Wlm)
    assert np.abs(logits - L).max() <= 1e-5 * np.abs(L).max()
    oc, och = oracle.confidence_and_choice(L)
    ok = top2_gap(L) > 1e-2
    assert ok.all()
    np.testing.assert_array_equal(choice, och)
    assert np.abs(conf - oc).max() < 5e-4
    res = oracle.lowconfidence_commit(oc, och, tokens0, masked0, THR, cfg.P)
    np.testing.assert_array_equal(accept, res.accept)
    np.testing.assert_array_equal(np_(msk).astype(bool), res.masked)
    np.testing.assert_array_equal(np_(tok)[ok], res.tokens[ok])
    high = oc[masked0] >= THR
    assert 0 < high.sum() < masked0.sum()          # both confidence classes present


def test_lm_head_batched_requests(lm_head):
    cfg, Wlm_dev, Wlm = lm_head
    R = 3
    bits, hid = hidden_with_confidences(cfg, Wlm, R * cfg.P, "batched")
    masked0 = W.masked_subset(cfg, R, tag="masked_b")
    tokens0 = np.zeros(R * cfg.P, np.int32)
    tok, msk = t(tokens0), t(masked0.astype(np.uint8))
    choice, conf, accept, n_comm, _ = run_lm(cfg, Wlm_dev, bits, tok, msk, R=R)
    L = oracle.lm_logits(hid, Wlm)
    oc, och = oracle.confidence_and_choice(L)
    res = oracle.lowconfidence_commit(oc, och, tokens0, masked0, THR, cfg.P)
    np.testing.assert_array_equal(accept, res.accept)
    np.testing.assert_array_equal(n_comm, res.n_committed)


def test_block_loop_to_resolution(lm_head):
    """Full round loop over a fixed synthetic logit sequence (one hidden state set per round)."""
    cfg, Wlm_dev, Wlm = lm_head
    tokens = np.zeros(cfg.P, np.int32)
    masked = np.ones(cfg.P, bool)
    tok, msk = t(tokens), t(masked.astype(np.uint8))
    rounds = 0
    while masked.any():
        assert rounds < cfg.P
        bits, hid = hidden_with_confidences(cfg, Wlm, cfg.P, f"loop{rounds}", frac_high=0.15)
        choice, conf, accept, n_comm, _ = run_lm(cfg, Wlm_dev, bits, tok, msk)
        oc, och = oracle.confidence_and_choice(oracle.lm_logits(hid, Wlm))
        res = oracle.lowconfidence_commit(oc, och, tokens, masked, THR, cfg.P)
        np.testing.assert_array_equal(accept, res.accept)
        assert n_comm[0] >= 1
        tokens, masked = res.tokens, res.masked
        np.testing.assert_array_equal(np_(msk).astype(bool), masked)
        np.testing.assert_array_equal(np_(tok), tokens)
        rounds += 1
    assert 1 <= rounds <= cfg.P
