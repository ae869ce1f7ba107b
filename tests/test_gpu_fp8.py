"""FP8 E4M3 expert weights (one fp32 scale per weight row) on the GPU against the fp64
oracle fed the dequantised weights (code value x row scale, exact in fp64).

The expert launch converts each weight tile to f16 in tensor memory (exact for
E4M3), multiplies by f16 token rows (the bf16 layer input converted; exact but
for values below f16's normal range) with fp32 accumulation and scales each
accumulator row; the SwiGLU output is rounded to f16 (2^-11 relative, finer
than the bf16 path's 2^-8).  The bound used is FP8_TOL = 4 * 2^-11 ~ 2e-3 max
relative error (two f16-rounded operands per product chain, with margin for
fp32 accumulation); measured errors are ~2e-4 and are printed.  Values that
pass through the bf16 parts (router input, LM-head input) keep the bf16 bound.

Routing and coreset decisions are checked exactly first (inputs with safe
margins), as in the bf16 tests; the generator's device copy of the codes and
scales is checked bit for bit against the host copy."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import moe_expert_step_gb300 as ms
import oracle
import synth
from synth import workloads as W
from tests.helpers import (BF16_TOL, aligned, coreset_margin, dot_error_bound, match_topk, max_rel, np_, oracle_layer,
                           oracle_routing, router_kind, t, topk_margin_ok)

pytestmark = pytest.mark.gpu
FP8_TOL = 4 * 2.0 ** -11


def dims_of(cfg):
    return ms.ModelDims(H=cfg.H, E=cfg.E, k=cfg.k, I=cfg.I, Is=cfg.Is, V=cfg.V, P=cfg.P, dtype=ms.FP8)


def clayer(lay, cfg):
    sh = cfg.Is > 0
    return ms.layer(lay["Wr"], lay["Wgu"], lay["Wd"], lay["Wsgu"] if sh else None, lay["Wsd"] if sh else None,
                    lay["Sgu"], lay["Sd"], lay["Ssgu"] if sh else None, lay["Ssd"] if sh else None)


def test_fp8_generator_device_equals_host():
    cfg = W.LAYER_FP8
    lay = W.device_layer(cfg, 2)
    for name in ("Wgu", "Wd", "Wsgu", "Wsd"):
        n = min(lay[name].numel(), 1 << 20)
        want = synth.host_normal(W.key(cfg, 2, name), 0, n, W.FP8_CODE_STD, "e4m3")
        np.testing.assert_array_equal(np_(lay[name].reshape(-1)[:n]), want)
    for name in ("Sgu", "Sd", "Ssgu", "Ssd"):
        want = synth.host_row_scales(W.key(cfg, 2, name), 0, lay[name].numel())
        np.testing.assert_array_equal(np_(lay[name].reshape(-1)), want)


def gpu_ffn(cfg, R, x, lay, top_p):
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
    ms.coreset_select(d, R, t(np.full(R, top_p, np.float32)), idx, mass, n_sel, sel, survive, gate_rr, ws)
    ms.moe_block_ffn(d, R, x, clayer(lay, cfg), gate_rr, out, ws)
    torch.cuda.synchronize()
    assert ms.read_device_error(ws) == ms.OK
    return np_(idx), np_(n_sel), np_(sel), np_(survive).astype(bool), np_(out)


def check_ffn(cfg, R, top_p, tag="x_ffn"):
    T = R * cfg.P
    lay = W.device_layer(cfg, 0)
    xa = W.host_activations(cfg, tag, T)
    idx, n_sel, sel, survive, out = gpu_ffn(cfg, R, W.to_device(xa, "bf16"), lay, top_p)
    ol = oracle_layer(cfg, 0)
    x = synth.as_f64(xa, "bf16")
    oi, om, _, oz = oracle.route(x, ol.Wr, cfg.k)
    eps = dot_error_bound(x, ol.Wr, router_kind(cfg.H, cfg.E, cfg.dtype))
    assert topk_margin_ok(oz, eps, cfg.k).all(), "test input too close to a top-k tie"
    perm = match_topk(idx, oi, oz, cfg.k, eps)
    cs = oracle.coreset_select(oi, om, top_p, cfg.P)
    assert coreset_margin(cs) > 1e-5, "test input too close to the coreset cut"
    np.testing.assert_array_equal(n_sel, cs.n_sel)
    np.testing.assert_array_equal(aligned(survive, perm), cs.survive)
    ref = oracle.moe_ffn(x, ol, oi, cs.gate_rr)
    err = max_rel(out, ref)
    print(f"{cfg.name} R={R} top_p={top_p}: max rel err {err:.3e}")
    assert err <= FP8_TOL, err
    return err


@pytest.mark.parametrize("top_p", [1.0, 0.9])
def test_fp8_clover_layer_ffn(top_p):
    check_ffn(W.LAYER_FP8, 1, top_p)


RAGGED8 = replace(W.LAYER_FP8, name="ragged_fp8", family="ragged8", H=256, E=64, k=6, I=128, Is=128, V=1024, P=7)
NOSHARED8 = replace(W.LAYER_FP8, name="noshared_fp8", family="noshared8", H=384, E=48, k=4, I=256, Is=0, V=1024,
                    P=16)


@pytest.mark.parametrize("cfg,R,top_p", [(RAGGED8, 3, 0.9), (NOSHARED8, 2, 0.8)])
def test_fp8_shapes(cfg, R, top_p):
    check_ffn(cfg, R, top_p)


def test_fp8_batched():
    """16 requests: token chunks of 64 (the wider instantiation) and the shared expert in several chunks."""
    check_ffn(W.LAYER_FP8, 16, 0.9, tag="x_batched")


@pytest.mark.parametrize("corr", [0.0, 0.9])
def test_fp8_layer_step(corr):
    """One FP8 layer + LM head through block_decode_step (bf16 router, norm and LM head).
    corr = 0.9: the block's tokens share a hidden component, so routed experts get up to 32
    tokens (token-row entries of one and two 16-token granules mixed in the launch's ring)."""
    cfg = W.LAYER_FP8
    lay = W.device_layer(cfg, 0)
    Wlm_d = W.device_lm_head(cfg)
    h0 = W.host_h0(cfg, 1, correlation=corr)
    masked0 = W.masked_subset(cfg, 1)
    d = dims_of(cfg)
    ws = ms.workspace(d, 1)
    T = cfg.P
    tokens = t(np.zeros(T, np.int32))
    masked = t(masked0.astype(np.uint8))
    choice = torch.zeros(T, dtype=torch.int32, device="cuda")
    conf = torch.zeros(T, dtype=torch.float32, device="cuda")
    accept = torch.zeros(T, dtype=torch.uint8, device="cuda")
    ncomm = torch.zeros(1, dtype=torch.int32, device="cuda")
    h_out = torch.zeros((T, cfg.H), dtype=torch.float32, device="cuda")
    hidden = torch.zeros((T, cfg.H), dtype=torch.float32, device="cuda")
    idx = torch.zeros((1, T, cfg.k), dtype=torch.int32, device="cuda")
    xl = torch.zeros((1, T, cfg.H), dtype=torch.bfloat16, device="cuda")
    ms.block_decode_step(d, 1, [clayer(lay, cfg)], Wlm_d, t(np.array([0.9], np.float32)), 0.95, t(h0), tokens,
                         masked, choice, conf, accept, ncomm, ws, h_out=h_out, trace_idx=idx, trace_hidden=hidden,
                         trace_x=xl)
    torch.cuda.synchronize()
    assert ms.read_device_error(ws) == ms.OK
    trace = []
    h, hid, L, oc, och, res = oracle.block_decode_step(
        h0.astype(np.float64), [oracle_layer(cfg, 0)], W.host_lm_head(cfg), 0.9, cfg.k, cfg.P, 0.95,
        np.zeros(cfg.P, np.int32), masked0, bf16=True, trace=trace)
    # routing of the layer input the GPU computed (bf16 bits as its router read them)
    _, _, _, _, amb = oracle_routing(np_(xl)[0].astype(np.float64), oracle_layer(cfg, 0).Wr, cfg.k,
                                     router_kind(cfg.H, cfg.E, cfg.dtype), np_(idx)[0])
    assert amb == 0
    err = max_rel(np_(h_out) - h0, h - h0)
    print(f"fp8 layer step (corr {corr}): MoE update max rel err {err:.3e}")
    assert err <= FP8_TOL
    assert max_rel(np_(hidden), hid) <= BF16_TOL
    assert np.abs(np_(conf) - oc).max() < 1e-2


@pytest.mark.parametrize("kind", ["subnormal", "mixed"])
def test_fp8_codes_convert_exactly(kind):
    """Hand-made layer (zero router: every token takes all 8 experts with mass 1/8): weights
    whose E4M3 codes are all subnormal (m * 2^-9, which the kernel's conversion maps onto
    f16 subnormals) or a mix of every code class (subnormal, normal, +-448, zero), each
    row scaled by 256 so the activations stay in f16's normal range.  A flushed subnormal
    would zero the 'subnormal' output entirely."""
    H, E, k, I, Is, P = 128, 8, 8, 128, 128, 4
    cfg = replace(W.LAYER_FP8, name=f"codes_{kind}", family=f"codes_{kind}", H=H, E=E, k=k, I=I, Is=Is, V=1024,
                  P=P)
    d = dims_of(cfg)
    rng = np.random.default_rng(11 if kind == "subnormal" else 12)

    def codes(shape):
        if kind == "subnormal":
            c = rng.integers(1, 8, size=shape)
        else:
            c = rng.choice(np.array([0, 1, 3, 7, 8, 0x20, 0x38, 0x5A, 0x7E]), size=shape)
        return (c | (rng.integers(0, 2, size=shape) << 7)).astype(np.uint8)

    host = {"Wgu": codes((E, I, 2, H)), "Wd": codes((E, H, I)), "Wsgu": codes((Is, 2, H)), "Wsd": codes((H, Is))}
    scale = 1.0 / 64 if kind == "mixed" else 256.0
    dev = {n: torch.from_numpy(a).cuda() for n, a in host.items()}
    dev["Wr"] = torch.zeros((E, H), dtype=torch.bfloat16, device="cuda")
    for n, rows in (("Sgu", (E, 2 * I)), ("Sd", (E, H)), ("Ssgu", (2 * Is,)), ("Ssd", (H,))):
        dev[n] = torch.full(rows, scale, dtype=torch.float32, device="cuda")
    deq = {n: synth.e4m3_to_f32(a).astype(np.float64) * scale for n, a in host.items()}
    xa = W.host_activations(cfg, "x_codes", P)
    idx, n_sel, sel, survive, out = gpu_ffn(cfg, 1, W.to_device(xa, "bf16"), dev, 1.0)
    assert (idx == np.arange(E)[None, :]).all() and n_sel[0] == E
    ol = oracle.MoELayer(Wr=np.zeros((E, H)),
                         expert=lambda e: (deq["Wgu"][e][:, 0, :], deq["Wgu"][e][:, 1, :], deq["Wd"][e]),
                         shared=lambda: (deq["Wsgu"][:, 0, :], deq["Wsgu"][:, 1, :], deq["Wsd"]))
    x = synth.as_f64(xa, "bf16")
    ref = oracle.moe_ffn(x, ol, idx, np.full((P, E), 1.0 / E))
    assert np.abs(ref).max() > 0
    err = max_rel(out, ref)
    print(f"{kind} codes: max rel err {err:.3e}")
    assert err <= FP8_TOL, err


@pytest.fixture(scope="module")
def stack8():
    cfg = W.STACK_FP8
    layers = [clayer(W.device_layer(cfg, l), cfg) for l in range(cfg.n_layers)]
    return cfg, layers, W.device_lm_head(cfg), W.host_lm_head(cfg)


def test_fp8_stack_full_step_teacher_forced(stack8):
    """All 40 FP8 layers in one call, the FP8 benchmark's configuration, against the oracle
    fed the GPU's own layer input: every layer's routing and coreset; the MoE update (with
    the dequantised weights) of every 8th layer and the last; the LM head and commit from
    the GPU's final hidden state.  The update bound is the bf16 one (the FP8 path rounds its
    SwiGLU rows to f16, finer)."""
    from tests.test_gpu_step import Step, check_commit, check_layer, check_routing
    cfg, layers, Wlm_d, Wlm = stack8
    h0 = W.host_h0(cfg, 1)
    masked0 = W.masked_subset(cfg, 1)
    tokens = t(np.zeros(cfg.P, np.int32))
    masked = t(masked0.astype(np.uint8))
    st = Step(cfg, 1, cfg.n_layers, trace_xh=True)
    st.run(layers, Wlm_d, 0.9, t(h0), tokens, masked)
    np.testing.assert_array_equal(np_(st.h[0]), h0)
    ambiguous = 0
    full = set(range(0, cfg.n_layers - 1, 8)) | {cfg.n_layers - 1}
    for l in range(cfg.n_layers):
        last = np_(st.h_out).astype(np.float64) if l == cfg.n_layers - 1 else None
        ambiguous += check_layer(cfg, l, st, 0.9, last_h=last) if l in full else check_routing(cfg, l, st, 0.9)[3]
    assert ambiguous <= 2
    check_commit(cfg, st, Wlm, np_(tokens), np_(masked), masked0)
