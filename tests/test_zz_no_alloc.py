"""The router entry point that allocates nothing (moe_block_route_noalloc).

It exists for callers that cannot allocate device memory themselves (a plugin
whose host application owns every device allocation, a runtime with a fixed
device-memory budget): instead of a caller-provided workspace it keeps its
scratch in one fixed array inside the library.  These tests check, through the
C ABI, that two calls in a row give the same result as the workspace-based
moe_block_route on the same inputs, and that calls beyond the fixed scratch are
refused.  The file is collected last so that a failure here cannot hide the
results of the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import moe_expert_step_gb300 as ms
import synth
from synth import workloads as W


def _dims(cfg):
    return ms.ModelDims(H=cfg.H, E=cfg.E, k=cfg.k, I=cfg.I, Is=cfg.Is, V=cfg.V, P=cfg.P,
                        dtype=ms.BF16 if cfg.dtype == "bf16" else ms.F32)


def _router_weights(cfg):
    Wr = torch.empty((cfg.E, cfg.H), dtype=torch.bfloat16 if cfg.dtype == "bf16" else torch.float32, device="cuda")
    synth.dev_fill_normal(Wr.data_ptr(), W.key(cfg, 0, "Wr"), 0, Wr.numel(), cfg.wr_std, cfg.dtype,
                          torch.cuda.current_stream().cuda_stream)
    return Wr


def _outputs(T, k):
    return (torch.full((T, k), -1, dtype=torch.int32, device="cuda"),
            torch.full((T, k), -1.0, dtype=torch.float32, device="cuda"),
            torch.full((T, k), -1.0, dtype=torch.float32, device="cuda"))


@pytest.mark.gpu
@pytest.mark.parametrize("cfg,T", [(W.LAYER, 32), (W.LAYER, 512), (W.TINY, 8)])
def test_noalloc_router_matches_workspace_router(cfg, T):
    d = _dims(cfg)
    Wr = _router_weights(cfg)
    for call, tag in enumerate(["x_noalloc_a", "x_noalloc_b"]):    # two calls in a row, different inputs
        x = W.to_device(W.host_activations(cfg, tag, T), cfg.dtype)
        ws = ms.workspace(d, -(-T // cfg.P))
        ref = _outputs(T, cfg.k)
        ms.moe_block_route(d, x, Wr, *ref, ws)
        got = _outputs(T, cfg.k)
        c0 = ms.launch_count()
        ms.moe_block_route_noalloc(d, x, Wr, *got)
        assert ms.launch_count() == c0 + 1    # counted like the workspace router's launch
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got[0].cpu().numpy(), ref[0].cpu().numpy())
        for g, r in zip(got[1:], ref[1:]):
            np.testing.assert_allclose(g.cpu().numpy(), r.cpu().numpy(), rtol=1e-5, atol=0)


def test_noalloc_router_refuses_calls_beyond_its_scratch():
    d = ms.ModelDims(H=2048, E=256, k=8, I=512, Is=512, V=152064, P=32, dtype=ms.BF16)
    fake = 1 << 20
    # 513 tokens x 256 experts of logits exceed the fixed 131072-entry scratch; refused before any CUDA call
    rc = ms.lib().moe_block_route_noalloc(ctypes.byref(d.c()), 513, fake, fake, fake, fake, fake, None, None)
    assert rc == ms.EUNSUPPORTED
    rc = ms.lib().moe_block_route_noalloc(ctypes.byref(d.c()), 0, fake, fake, fake, fake, fake, None, None)
    assert rc == ms.EINVAL
