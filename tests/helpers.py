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


# ------------------------------------------------------------------------------ fp32 router error bound
U32 = 2.0 ** -24   # unit roundoff of binary32


def router_kind(H: int, E: int, dtype: str) -> str:
    """Which router kernel the library runs for a shape: the tensor-core router for bf16
    layers with E % 32 == 0 and H % 512 == 0, the CUDA-core (FFMA) router otherwise."""
    return "tc" if dtype in ("bf16", "fp8") and E % 32 == 0 and H % 512 == 0 else "ffma"


def _tc_order(H: int) -> np.ndarray:
    """K order of the tensor-core routers: eight contiguous K ranges (one per warp pair);
    within a range, 64-wide steps of four m16n8k16 MMAs, MMA jj holding the positions
    h0 + 16 tig + 4 jj + i (tig, i < 4)."""
    span = H // 8
    order = []
    for q in range(8):
        for h0 in range(q * span, (q + 1) * span, 64):
            for jj in range(4):
                order += [h0 + 16 * tig + 4 * jj + i for tig in range(4) for i in range(4)]
    return np.array(order)


def dot_error_bound(x, W, kind: str, block: int = 8) -> np.ndarray:
    """eps[t, e]: a first-order bound on |fl32(x_t . W_e) - x_t . W_e| for the summation order
    of the library's router kernels, from the actual partial sums of the data.

    Model: every fp32 accumulation step (an FMA, an addition, or one m16n8k16 MMA adding 16
    products to its accumulator) errs by at most 2u times the magnitude it handles (u = 2^-24;
    2u also covers truncating adders): for an MMA, 2u (|accumulator| + sum |products|), for an
    addition or FMA, 2u |result|.  Products of bf16 operands are exact in fp32; FMAs round once.
    * "tc": eight K ranges (see _tc_order), MMAs accumulated in order inside a range, the eight
      range totals then added in K order;
    * "ffma": lane l of a warp accumulates with FMAs the elements 256 c + 8 l + j (c, then j in
      order), then a butterfly over the 32 lanes.
    Summing these per-step bounds bounds the total error to first order (the u^2 terms are
    covered by a 1 % margin)."""
    x = np.asarray(x, np.float64)
    W = np.asarray(W, np.float64)
    T, H = x.shape
    E = W.shape[0]
    out = np.empty((T, E))
    if kind == "tc":
        order = _tc_order(H)
        Wo = W[:, order].reshape(E, 8, H // 128, 16)
        for t0 in range(0, T, block):
            xo = x[t0:t0 + block][:, order].reshape(-1, 1, 8, H // 128, 16)
            p = xo * Wo[None]                                   # [tb, E, 8, chunks, 16]
            chunk = p.sum(-1)
            run = np.cumsum(chunk, axis=-1)                     # accumulator after each MMA
            acc_in = np.abs(run[..., :-1]).sum(-1).sum(-1)      # accumulator entering each MMA
            bound = np.abs(p).sum((-1, -2, -3)) + acc_in
            Z = np.cumsum(run[..., -1], axis=-1)                # running total over the K ranges
            bound += np.abs(Z[..., 1:]).sum(-1)
            out[t0:t0 + block] = bound
    elif kind == "ffma":
        passes = -(-H // 256)
        for t0 in range(0, T, block):
            xb = x[t0:t0 + block]
            p = xb[:, None, :] * W[None]                        # [tb, E, H]
            lanes = np.zeros(p.shape[:2] + (32,))
            lane_bound = np.zeros_like(lanes)
            for c in range(passes):
                for j in range(8):
                    hs = c * 256 + 8 * np.arange(32) + j
                    ok = hs < H
                    step = np.zeros(p.shape[:2] + (32,))
                    step[..., ok] = p[..., hs[ok]]
                    lanes = lanes + step
                    lane_bound += np.abs(lanes)
            bound = lane_bound.sum(-1)
            v = lanes
            while v.shape[-1] > 1:                              # butterfly: a binary tree of additions
                v = v[..., : v.shape[-1] // 2] + v[..., v.shape[-1] // 2:]
                bound += np.abs(v).sum(-1)
            out[t0:t0 + block] = bound
    else:
        raise ValueError(kind)
    return 2.0 * U32 * 1.01 * out


def topk_window(x, W, k: int, kind: str) -> np.ndarray:
    """Per-logit error bounds for the router's picks (see dot_error_bound)."""
    return dot_error_bound(x, W, kind)


def topk_margin_ok(z, eps, k: int) -> np.ndarray:
    """Per row: whether the k-th / (k+1)-th boundary is decided beyond the fp32 error bound
    (gap larger than the two logits' bounds added)."""
    z = np.asarray(z, np.float64)
    if z.shape[1] <= k:
        return np.ones(z.shape[0], bool)
    o = np.argsort(-z, axis=1, kind="stable")
    a, b = o[:, k - 1], o[:, k]
    r = np.arange(z.shape[0])
    return z[r, a] - z[r, b] > eps[r, a] + eps[r, b]


SWAP_LOG = []   # (gap, window) of every pick pair that match_topk saw in either order


def match_topk(idx, oi, z, k: int, eps) -> np.ndarray:
    """Check a kernel's top-k lists `idx` [T][k] against the oracle's `oi` and return
    the column permutation that aligns them (perm[t, j] = column of idx[t] holding
    oi[t, j]).

    The order of the k picks is a floating-point decision like the k-th/(k+1)-th
    boundary (callers check that one with topk_margin_ok): the kernel accumulates
    logits in fp32 in its own order, so two neighbouring picks a, b may come out in
    either order only if their fp64 logits differ by at most eps[t, a] + eps[t, b]
    (eps: per-logit bounds from dot_error_bound, or a scalar per logit).  Such runs
    of neighbours must hold the same experts on both sides; everywhere else the
    order is exact.  Pairs seen swapped are recorded in SWAP_LOG."""
    idx = np.asarray(idx)
    oi = np.asarray(oi)
    assert idx.shape == oi.shape
    z = np.asarray(z, np.float64)
    eps = np.broadcast_to(np.asarray(eps, np.float64), z.shape)
    oi64 = oi.astype(np.int64)
    zs = np.take_along_axis(z, oi64, axis=1)
    es = np.take_along_axis(eps, oi64, axis=1)
    perm = np.empty(oi.shape, np.int64)
    for t in range(oi.shape[0]):
        j = 0
        while j < k:
            e = j + 1
            while e < k and zs[t, e - 1] - zs[t, e] <= es[t, e - 1] + es[t, e]:
                e += 1
            got = [int(v) for v in idx[t, j:e]]
            assert sorted(got) == sorted(int(v) for v in oi[t, j:e]), (t, j, idx[t], oi[t])
            for u in range(j, e):
                perm[t, u] = j + got.index(int(oi[t, u]))
            for u in range(j, e - 1):
                if perm[t, u] > perm[t, u + 1]:
                    SWAP_LOG.append((zs[t, u] - zs[t, u + 1], es[t, u] + es[t, u + 1]))
            j = e
    return perm


def oracle_routing(x, Wr, k: int, kind: str, idx_gpu):
    """The oracle's routing of router input x (the bits the kernel read), checked against the
    kernel's top-k `idx_gpu` and returned for the rest of the comparison.

    Where a token's k-th / (k+1)-th logits lie within the fp32 error bound of each other the
    choice is legitimately either way: there the kernel's k experts must be a valid top-k
    within the bound, and the returned routing takes them (the masses are the oracle's
    softmax at those experts), so downstream comparisons stay exact.  Elsewhere the sets
    must agree and the order within the window (match_topk).
    Returns (idx, mass, z, perm, n_ambiguous): idx/mass in the oracle's order, perm aligning
    the kernel's per-pick arrays with it."""
    x = np.asarray(x, np.float64)
    oi, om, _, oz = oracle.route(x, Wr, k)
    eps = dot_error_bound(x, Wr, kind)
    ok = topk_margin_ok(oz, eps, k)
    idx_gpu = np.asarray(idx_gpu)
    idx = oi.copy()
    perm = np.tile(np.arange(k), (x.shape[0], 1))
    if ok.any():
        perm[ok] = match_topk(idx_gpu[ok], oi[ok], oz[ok], k, eps[ok])
    p = oracle.softmax(oz)
    for t in np.flatnonzero(~ok):
        g = [int(e) for e in idx_gpu[t]]
        assert len(set(g)) == k
        kth = np.sort(oz[t])[::-1][k - 1]
        for e in g:    # every pick is within the bound of the k-th largest logit or above it
            assert oz[t, e] >= kth - 2 * eps[t].max(), (t, e)
        idx[t] = sorted(g, key=lambda e: (-oz[t, e], e))
        perm[t] = [g.index(e) for e in idx[t]]
    mass = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    return idx, mass, oz, perm, int((~ok).sum())


def aligned(a, perm) -> np.ndarray:
    """Columns of a per-pick array [T][k] reordered by match_topk's permutation."""
    return np.take_along_axis(np.asarray(a), perm, axis=1)


def assert_ranked_equal(got, cs: oracle.CoresetResult, r: int, tol: float = 1e-5, where=None):
    """The kept experts of request r in ranking order against the oracle's: the same set, and
    the same order except within runs of experts whose aggregated masses lie within
    tol * total of each other (their order is an fp32 decision on computed masses)."""
    want = list(cs.sel[r])
    got = [int(e) for e in got]
    assert sorted(got) == sorted(want), (where, "kept set")
    agg = cs.agg[r]
    total = sum(agg.values()) or 1
    i = 0
    while i < len(want):        # one run of near-equal aggregates at a time
        j = i + 1
        while j < len(want) and abs(agg[want[j - 1]] - agg[want[j]]) <= tol * total:
            j += 1
        assert sorted(got[i:j]) == sorted(want[i:j]), (where, i, got[i:j], want[i:j])
        i = j


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
