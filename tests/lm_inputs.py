"""LM-head test inputs with chosen confidences (test-side; uses the oracle's arithmetic
only through numpy on its fp64 weights, so it lives in tests/).

Recipe: per position j a target confidence c_j is drawn (a fraction `frac_high`
in [0.95 + guard, 0.999], the rest in [0.30, 0.95 - guard]); with n_j ~ N(0, 1)
the fp64 base logits L0_j = Wlm n_j are computed once, and s_j is found by
bisection so that max softmax(s_j L0_j) = c_j (max-softmax grows monotonically
with s >= 0).  The device input is bf16(s_j n_j).  Positions whose rounded input
lands within `guard` of the threshold, or whose top-2 logit gap is below
`min_gap`, are redrawn from a new n_j."""
from __future__ import annotations

import numpy as np

import synth
from synth import workloads as W


def conf_rows(L: np.ndarray) -> np.ndarray:
    m = L.max(axis=-1, keepdims=True)
    return 1.0 / np.exp(L - m).sum(axis=-1)


def scale_for_conf(L0: np.ndarray, target: float) -> float:
    lo, hi = 0.0, 1.0
    while conf_rows(hi * L0) < target and hi < 1e6:
        hi *= 2.0
    for _ in range(50):
        mid = 0.5 * (lo + hi)
        if conf_rows(mid * L0) < target:
            lo = mid
        else:
            hi = mid
    return hi


def top2_gap(L: np.ndarray) -> np.ndarray:
    s = -np.partition(-L, 1, axis=1)[:, :2]
    return np.abs(s[:, 0] - s[:, 1])


def hidden_with_confidences(cfg, Wlm: np.ndarray, rows: int, tag: str, guard: float = 1e-3,
                            frac_high: float = 0.3, threshold: float = 0.95, min_gap: float = 2e-2):
    """bf16 bits [rows][H] and their fp64 values."""
    u = synth.np_uniform01(W.key(cfg, tag, "targets"), 0, 2 * rows).reshape(rows, 2)
    target = np.where(u[:, 0] < frac_high, threshold + guard + (0.999 - threshold - guard) * u[:, 1],
                      0.30 + (threshold - guard - 0.30) * u[:, 1])
    bits = np.zeros((rows, cfg.H), np.uint16)
    todo = np.arange(rows)
    for attempt in range(8):
        if todo.size == 0:
            break
        n = np.stack([synth.host_normal(W.key(cfg, tag, "n", int(j), attempt), 0, cfg.H, 1.0, "f32")
                      for j in todo]).astype(np.float64)
        L0 = n @ Wlm.T
        for row, j in enumerate(todo):
            s = scale_for_conf(L0[row], target[j])
            bits[j] = synth.f32_to_bf16_bits((s * n[row]).astype(np.float32))
        h = synth.bf16_bits_to_f32(bits[todo]).astype(np.float64)
        L = h @ Wlm.T
        bad = (np.abs(conf_rows(L) - threshold) <= guard) | (top2_gap(L) < min_gap)
        todo = todo[bad]
    if todo.size:
        raise RuntimeError("could not place every position outside the guard bands")
    return bits, synth.bf16_bits_to_f32(bits).astype(np.float64)
