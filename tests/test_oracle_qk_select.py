"""Pins of the QK selection step's oracle (CPU only): a hand-worked case,
the empty and full masks, overflow past Tc, and properties of random masks."""
import numpy as np

from oracle import qk_select


def test_hand_worked():
    keep = np.array([[0, 1, 1, 0, 1], [0, 0, 0, 0, 0]], dtype=np.uint8)
    idx, count = qk_select.select_positions(keep, 4, -1)
    np.testing.assert_array_equal(idx, [[1, 2, 4, -1], [-1, -1, -1, -1]])
    np.testing.assert_array_equal(count, [3, 0])


def test_full_mask_and_overflow():
    keep = np.ones((1, 7), dtype=np.uint8)
    idx, count = qk_select.select_positions(keep, 7, 2**31 - 1)
    np.testing.assert_array_equal(idx, [np.arange(7)])
    idx, count = qk_select.select_positions(keep, 3, -1)
    np.testing.assert_array_equal(idx, [[0, 1, 2]])
    assert count[0] == 7


def test_random_properties():
    rng = np.random.default_rng(5)
    keep = (rng.random((3, 4, 300)) < 0.6).astype(np.uint8)
    idx, count = qk_select.select_positions(keep, 300, -1)
    for b in range(3):
        for h in range(4):
            n = count[b, h]
            assert n == keep[b, h].sum()
            kept = idx[b, h, :n]
            assert np.all(np.diff(kept) > 0) and np.all(keep[b, h, kept] == 1)
            assert np.all(idx[b, h, n:] == -1)
