"""Shared test utilities: oracle layers built from the synthetic workloads, error metrics,
decision margins (how far an integer decision is from flipping), and device helpers."""
from __future__ import annotations

import math

import numpy as np

import oracle
from synth import workloads as W

BF16_TOL = 2e-2   # max relative error, bf16 weights / fp32 accumulation
F32_TOL = 1e-4    # max relative error, fp32 configuration


def max_rel(a, b) -> float:
    """max |a - b| / max |b| over the whole tensor."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.abs(b).max()
    return float(np.abs(a - b).max() / (den if den > 0 else 1.0))


def oracle_layer(cfg, layer: int) -> oracle.MoELayer:
    hl = W.HostLayer(cfg, layer)
    return oracle.MoELayer(Wr=hl.Wr, expert=hl.expert, shared=hl.shared)


def topk_margins(z: np.ndarray, k: int) -> np.ndarray:
    """Per row: gap between the k-th and (k+1)-th largest logit."""
    s = -np.sort(-np.asarray(z, np.float64), axis=1)
    if s.shape[1] <= k:
        return np.full(s.shape[0], np.inf)
    return s[:, k - 1] - s[:, k]


def coreset_margin(cs: oracle.CoresetResult) -> float:
    """Smallest relative distance between a request's target and the cumulative sums
    around its cut (how much the masses may move before the kept set changes)."""
    best = math.inf
    for r, target in enumerate(cs.target):
        if target is None:
            continue
        agg = cs.agg[r]
        total = sum(agg.values())
        cum = 0
        for e in cs.ranking[r]:
            cum += agg[e]
            best = min(best, abs(cum - target) / total)
    return best


def torch_dev():
    import torch
    return torch.device("cuda:0")


def t(a, dtype=None):
    """numpy -> cuda tensor."""
    import torch
    x = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        x = x.to(dtype)
    return x.cuda()


def np_(x) -> np.ndarray:
    """cuda tensor -> numpy (bf16 widened to float32)."""
    import torch
    if x.dtype == torch.bfloat16:
        x = x.float()
    return x.detach().cpu().numpy()
