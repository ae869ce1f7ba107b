"""The top-k comparison used by the GPU parity tests: order may differ only inside runs
of near-equal logits, and the returned permutation aligns per-pick arrays."""
import numpy as np
import pytest

from tests.helpers import aligned, match_topk


def test_exact_order_is_identity():
    z = np.array([[5.0, 1.0, 4.0, 3.0, 2.0]])
    oi = np.array([[0, 2, 3]])
    np.testing.assert_array_equal(match_topk(oi, oi, z, 3), [[0, 1, 2]])


def test_swap_inside_near_tie_is_aligned():
    z = np.array([[5.0, 4.00005, 4.0, 1.0]])
    oi = np.array([[0, 1, 2]])
    got = np.array([[0, 2, 1]])
    perm = match_topk(got, oi, z, 3)
    np.testing.assert_array_equal(aligned(got, perm), oi)
    mass = np.array([[0.5, 0.2, 0.3]])          # per-pick values in the kernel's order
    np.testing.assert_array_equal(aligned(mass, perm), [[0.5, 0.3, 0.2]])


@pytest.mark.parametrize("got", [[[1, 0, 2]], [[0, 2, 3]], [[0, 1, 1]]])
def test_rejects_real_differences(got):
    z = np.array([[5.0, 4.0, 3.0, 2.0]])         # gaps of 1: every order is decided
    with pytest.raises(AssertionError):
        match_topk(np.array(got), np.array([[0, 1, 2]]), z, 3)
