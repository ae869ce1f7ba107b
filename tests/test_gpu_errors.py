"""Failure detection on the GPU without a fault: a bounded wait inside the tensor-core
kernel is made to run out (limit set to zero), the kernel drains what it issued,
frees its tensor memory and reports MOESTEP_ETIMEOUT through the workspace error
word; the context stays usable and the next call (normal limit) is correct."""
import numpy as np
import pytest
import torch

import moe_expert_step_gb300 as ms
from synth import workloads as W
from tests.helpers import np_, t

pytestmark = pytest.mark.gpu


def run_ffn(cfg, lay, x, ws):
    d = ms.ModelDims(H=cfg.H, E=cfg.E, k=cfg.k, I=cfg.I, Is=cfg.Is, V=cfg.V, P=cfg.P, dtype=ms.BF16)
    T = cfg.P
    idx = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
    mass = torch.empty((T, cfg.k), dtype=torch.float32, device="cuda")
    gate = torch.empty_like(mass)
    n_sel = torch.empty(1, dtype=torch.int32, device="cuda")
    sel = torch.empty((1, cfg.E), dtype=torch.int32, device="cuda")
    survive = torch.empty((T, cfg.k), dtype=torch.uint8, device="cuda")
    gate_rr = torch.empty_like(mass)
    out = torch.empty((T, cfg.H), dtype=torch.float32, device="cuda")
    ms.moe_block_route(d, x, lay["Wr"], idx, mass, gate, ws)
    ms.coreset_select(d, 1, t(np.array([0.9], np.float32)), idx, mass, n_sel, sel, survive, gate_rr, ws)
    ms.moe_block_ffn(d, 1, x, ms.layer(lay["Wr"], lay["Wgu"], lay["Wd"], lay["Wsgu"], lay["Wsd"]), gate_rr, out, ws)
    torch.cuda.synchronize()
    return np_(out)


def test_wait_timeout_is_reported_and_recovered():
    cfg = W.LAYER
    lay = W.device_layer(cfg, 0)
    x = W.to_device(W.host_activations(cfg, "x_ffn", 32), "bf16")
    d = ms.ModelDims(H=cfg.H, E=cfg.E, k=cfg.k, I=cfg.I, Is=cfg.Is, V=cfg.V, P=cfg.P, dtype=ms.BF16)
    ws = ms.workspace(d, 1)
    good = run_ffn(cfg, lay, x, ws)
    assert ms.read_device_error(ws) == ms.OK
    try:
        ms.set_wait_timeout_ns(0)
        run_ffn(cfg, lay, x, ws)
        assert ms.read_device_error(ws) == ms.ETIMEOUT
    finally:
        ms.set_wait_timeout_ns(2_000_000_000)
    again = run_ffn(cfg, lay, x, ws)
    assert ms.read_device_error(ws) == ms.OK
    np.testing.assert_array_equal(again, good)
