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


def match_topk(idx, oi, z, k: int, eps: float = 1e-4) -> np.ndarray:
    """Check a kernel's top-k lists `idx` [T][k] against the oracle's `oi` and return
    the column permutation that aligns them (perm[t, j] = column of idx[t] holding
    oi[t, j]).

    The order of the k picks is a floating-point decision like the k-th/(k+1)-th
    boundary (callers check that one with topk_margins): the kernel accumulates
    logits in fp32 in its own order, so two picks whose fp64 logits lie within
    `eps` of each other may come out in either order.  Such runs of neighbours
    must hold the same experts on both sides; everywhere else the order is
    exact."""
    idx = np.asarray(idx)
    oi = np.asarray(oi)
    assert idx.shape == oi.shape
    zs = np.take_along_axis(np.asarray(z, np.float64), oi.astype(np.int64), axis=1)
    perm = np.empty(oi.shape, np.int64)
    for t in range(oi.shape[0]):
        j = 0
        while j < k:
            e = j + 1
            while e < k and zs[t, e - 1] - zs[t, e] <= eps:
                e += 1
            got = [int(v) for v in idx[t, j:e]]
            assert sorted(got) == sorted(int(v) for v in oi[t, j:e]), (t, j, idx[t], oi[t])
            for u in range(j, e):
                perm[t, u] = j + got.index(int(oi[t, u]))
            j = e
    return perm


def aligned(a, perm) -> np.ndarray:
    """Columns of a per-pick array [T][k] reordered by match_topk's permutation."""
    return np.take_along_axis(np.asarray(a), perm, axis=1)


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
