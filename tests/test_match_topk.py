"""The top-k comparison used by the GPU parity tests and the fp32 error bound it uses.

Order may differ only inside runs of logits whose gaps lie within the two logits'
fp32 error bounds; the returned permutation aligns per-pick arrays.  The bound
(dot_error_bound) is checked here against fp32 evaluations of the same sums in the
router kernels' orders, written with numpy float32 arithmetic (round to nearest
even), on Clover-shaped router data and on the tiny fp32 configuration."""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads as W
from tests.helpers import (SWAP_LOG, _tc_order, aligned, assert_ranked_equal, dot_error_bound, match_topk, router_kind,
                           topk_margin_ok)


def test_exact_order_is_identity():
    z = np.array([[5.0, 1.0, 4.0, 3.0, 2.0]])
    oi = np.array([[0, 2, 3]])
    np.testing.assert_array_equal(match_topk(oi, oi, z, 3, 1e-6), [[0, 1, 2]])


def test_swap_inside_near_tie_is_aligned():
    z = np.array([[5.0, 4.00005, 4.0, 1.0]])
    oi = np.array([[0, 1, 2]])
    got = np.array([[0, 2, 1]])
    eps = np.full(z.shape, 3e-5)                 # 5e-5 gap within 3e-5 + 3e-5
    n0 = len(SWAP_LOG)
    perm = match_topk(got, oi, z, 3, eps)
    assert len(SWAP_LOG) == n0 + 1
    del SWAP_LOG[n0:]                            # the log reports what the GPU tests see
    np.testing.assert_array_equal(aligned(got, perm), oi)
    mass = np.array([[0.5, 0.2, 0.3]])          # per-pick values in the kernel's order
    np.testing.assert_array_equal(aligned(mass, perm), [[0.5, 0.3, 0.2]])
    with pytest.raises(AssertionError):          # the same swap outside the window is a mismatch
        match_topk(got, oi, z, 3, np.full(z.shape, 2e-5))


@pytest.mark.parametrize("got", [[[1, 0, 2]], [[0, 2, 3]], [[0, 1, 1]]])
def test_rejects_real_differences(got):
    z = np.array([[5.0, 4.0, 3.0, 2.0]])         # gaps of 1: every order is decided
    with pytest.raises(AssertionError):
        match_topk(np.array(got), np.array([[0, 1, 2]]), z, 3, 1e-5)


def test_margin_check_uses_both_bounds():
    z = np.array([[3.0, 2.0, 1.00002, 1.0], [3.0, 2.0, 1.5, 1.0]])
    eps = np.full(z.shape, 1.5e-5)
    np.testing.assert_array_equal(topk_margin_ok(z, eps, 3), [False, True])


def fp32_tc(x, w):
    """x . w in binary32, in the tensor-core routers' order (sum of each MMA's 16 products
    rounded once, added to the accumulator; eight range totals added in K order)."""
    order = _tc_order(len(x))
    p = (x[order] * w[order]).reshape(8, -1, 16)       # exact: bf16 x bf16 fits in binary64
    tot = np.float32(0)
    for q in range(8):
        acc = np.float32(0)
        for c in range(p.shape[1]):
            acc = np.float32(acc + np.float32(p[q, c].sum()))
        tot = np.float32(tot + acc)
    return float(tot)


def fp32_ffma(x, w):
    """x . w in binary32 in the CUDA-core router's order (per-lane FMA chains, then a
    butterfly over 32 lanes)."""
    H = len(x)
    lanes = np.zeros(32, np.float32)
    for c in range(-(-H // 256)):
        for j in range(8):
            for l in range(32):
                h = c * 256 + 8 * l + j
                if h < H:   # one rounding per FMA: the exact product plus the lane's sum
                    lanes[l] = np.float32(np.float64(lanes[l]) + x[h] * w[h])
    v = lanes
    while len(v) > 1:
        v = (v[: len(v) // 2] + v[len(v) // 2:]).astype(np.float32)
    return float(v[0])


@pytest.mark.parametrize("cfg,kind,n", [(W.LAYER, "tc", 24), (W.LAYER, "ffma", 6), (W.TINY, "ffma", 24)])
def test_error_bound_covers_fp32_sums(cfg, kind, n):
    """|fp32 sum - exact| <= bound for router logits of the configurations' data, and the
    bound is far inside the top-k margins the tests rely on (below 1e-4 per logit)."""
    x = synth.as_f64(W.host_activations(cfg, "x_bound", 4), cfg.act_dtype)
    Wr = W.HostLayer(cfg, 0).Wr
    eps = dot_error_bound(x, Wr, kind)
    z = oracle.router_logits(x, Wr)
    rng = np.random.default_rng(0)
    f = fp32_tc if kind == "tc" else fp32_ffma
    worst = 0.0
    for _ in range(n):
        t, e = int(rng.integers(x.shape[0])), int(rng.integers(Wr.shape[0]))
        err = abs(f(x[t], Wr[e]) - z[t, e])
        assert err <= eps[t, e], (t, e, err, eps[t, e])
        worst = max(worst, err / eps[t, e])
    assert worst > 1e-3                        # the bound is not vacuous
    assert eps.max() < 1e-4


def test_router_kind_mirrors_the_dispatch_rule():
    assert router_kind(2048, 256, "bf16") == "tc"
    assert router_kind(256, 16, "f32") == "ffma"
    assert router_kind(256, 64, "bf16") == "ffma"      # H % 512 != 0
    assert router_kind(512, 48, "bf16") == "ffma"      # E % 32 != 0


def _cs(sel, agg):
    return oracle.CoresetResult(np.array([len(sel)]), [sel], None, None, [sel], [agg], [None])


def test_ranked_equal_allows_swaps_only_within_near_ties():
    agg = {3: 1000, 5: 600, 7: 599, 9: 100}          # 5 and 7 within 1e-3 of the total (2299)
    cs = _cs([3, 5, 7, 9], agg)
    assert_ranked_equal([3, 5, 7, 9], cs, 0, tol=1e-3)
    assert_ranked_equal([3, 7, 5, 9], cs, 0, tol=1e-3)
    with pytest.raises(AssertionError):                 # the same swap with a tighter window
        assert_ranked_equal([3, 7, 5, 9], cs, 0, tol=1e-4)
    with pytest.raises(AssertionError):                 # a decided order swapped
        assert_ranked_equal([5, 3, 7, 9], cs, 0, tol=1e-3)
    with pytest.raises(AssertionError):                 # a different kept set
        assert_ranked_equal([3, 5, 7, 11], cs, 0, tol=1e-3)
