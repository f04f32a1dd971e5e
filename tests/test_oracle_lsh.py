"""Pins of the LSH bucket id and the stable bucket sort (CPU only).

Pins: a hand-worked fixture, the one-column special case (sign hash), exact
rational arithmetic on random and crafted near-tie inputs, invariance under
power-of-two scaling, and brute-force stable sorting.
"""
import numpy as np
import pytest
import torch

from conftest import load_golden
from oracle import lsh


def test_golden_identity_rotation():
    g = load_golden("lsh_identity_d2.json")
    h = lsh.lsh_hash(np.array(g["x"], dtype=np.float64), np.array(g["R"]))
    np.testing.assert_array_equal(h, g["h"])
    h_exact = lsh.lsh_hash(np.array(g["x"], dtype=np.float64), np.array(g["R"]), exact_all=True)
    np.testing.assert_array_equal(h_exact, g["h"])


def test_one_column_is_sign_hash():
    # m = 1: candidates [s, -s] -> 0 when s >= 0 (tie at 0 -> 0), 1 when s < 0
    rng = np.random.default_rng(20)
    x = rng.integers(-3, 4, size=(500, 6)).astype(np.float64)
    R = rng.integers(-2, 3, size=(6, 1)).astype(np.float64)
    s = (x.astype(np.int64) @ R.astype(np.int64))[:, 0]  # exact integer dot products
    np.testing.assert_array_equal(lsh.lsh_hash(x, R), (s < 0).astype(np.int32))


def _bf16(a):
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


@pytest.mark.parametrize("m", [2, 8])
def test_certified_equals_exact_random(m):
    rng = np.random.default_rng(21 + m)
    x = _bf16(rng.standard_normal((300, 64)))
    R = _bf16(rng.standard_normal((64, m)))
    np.testing.assert_array_equal(lsh.lsh_hash(x, R), lsh.lsh_hash(x, R, exact_all=True))


def test_exact_ties_take_smallest_index():
    rng = np.random.default_rng(22)
    c0 = _bf16(rng.standard_normal(16))
    R = np.stack([c0, c0, -c0], axis=1)        # columns 0 and 1 equal, column 2 opposite
    x = _bf16(rng.standard_normal((200, 16)))
    h = lsh.lsh_hash(x, R)
    s = x @ c0
    # s > 0: candidates [s, s, -s, -s, -s, s] -> 0 ; s < 0: [s, s, -s, -s, -s, s] -> 2
    np.testing.assert_array_equal(h, np.where(s > 0, 0, 2))
    assert lsh.lsh_hash(np.zeros((1, 16)), R)[0] == 0


def test_cancellation_beyond_float64_uses_exact_path():
    # bf16 holds 2^60 and 1 exactly; s0 = 2^60 + 1 - 2^60 = 1 exactly while a
    # float64 left-to-right sum gives 0
    R = np.array([[1.0, 1.0], [1.0, 0.0], [1.0, 1.0]])
    big = 2.0**60
    x = np.array([[big, 1.0, -big], [big, -1.0, -big]])
    # row 0: s = [1, 0] -> candidates [1, 0, -1, 0] -> 0
    # row 1: s = [-1, 0] -> candidates [-1, 0, 1, 0] -> 2
    np.testing.assert_array_equal(lsh.lsh_hash(x, R), [0, 2])


def test_power_of_two_scaling_invariance():
    # normalisation is a positive scaling: it cannot change the exact argmax
    rng = np.random.default_rng(23)
    x = _bf16(rng.standard_normal((200, 32)))
    R = _bf16(rng.standard_normal((32, 4)))
    h = lsh.lsh_hash(x, R)
    for e in (-20, -3, 5, 40):
        np.testing.assert_array_equal(lsh.lsh_hash(x * 2.0**e, R), h)


def test_bucket_sort_brute_force():
    rng = np.random.default_rng(24)
    for T, nb in ((1, 2), (37, 4), (300, 16), (513, 64)):
        h = rng.integers(0, nb, T)
        perm, hs, off = lsh.bucket_sort(h, nb)
        expect = sorted(range(T), key=lambda p: (h[p], p))
        np.testing.assert_array_equal(perm, expect)
        np.testing.assert_array_equal(hs, [h[p] for p in expect])
        np.testing.assert_array_equal(off, [sum(1 for t in h if t < c) for c in range(nb + 1)])


def test_gather_unsort_round_trip():
    rng = np.random.default_rng(25)
    x = rng.standard_normal((64, 8))
    perm = rng.permutation(64)
    xs = lsh.gather_rows(x, perm)
    for s in range(64):
        np.testing.assert_array_equal(xs[s], x[perm[s]])
    np.testing.assert_array_equal(lsh.unsort_rows(xs, perm), x)


def test_tile_aligned_hand_worked():
    # ids [1, 0, 1, 1, 0], two buckets, tile height 2, 8 rows:
    # plain order perm [1, 4, 0, 2, 3], offsets [0, 2, 5]; bucket 0 keeps rows
    # 0-1, bucket 1 starts at row 2 and its 3 tokens round up to 4 rows (2-5),
    # rows 6-7 follow the last bucket
    perm, hs, off = lsh.bucket_sort(np.array([1, 0, 1, 1, 0]), 2)
    np.testing.assert_array_equal(perm, [1, 4, 0, 2, 3])
    pt, ht, start = lsh.tile_aligned(perm, off, 8, 2, -1)
    np.testing.assert_array_equal(pt, [1, 4, 0, 2, 3, -1, -1, -1])
    np.testing.assert_array_equal(ht, [0, 0, 1, 1, 1, 1, 1, 1])
    np.testing.assert_array_equal(start, [0, 2, 6])


@pytest.mark.parametrize("T,nb,tile", [(1, 4, 128), (300, 64, 128), (1000, 8, 128), (5000, 512, 128), (97, 6, 5)])
def test_tile_aligned_properties(T, nb, tile):
    rng = np.random.default_rng(T + nb)
    h = rng.integers(0, nb, size=T)
    h[: T // 3] = rng.integers(0, max(1, nb // 4), size=T // 3)  # uneven, some buckets empty
    perm, hs, off = lsh.bucket_sort(h, nb)
    nonempty = int((np.diff(off) > 0).sum())
    n_rows = -(-(T + nonempty * (tile - 1)) // tile) * tile  # the bound the product allocates
    pt, ht, start = lsh.tile_aligned(perm, off, n_rows, tile, 2**31 - 1)
    real = pt != 2**31 - 1
    # every token appears once, in the plain sorted order
    np.testing.assert_array_equal(pt[real], perm)
    # bucket ids are non-decreasing, each bucket starts on a tile boundary and
    # holds exactly its tokens followed by padding
    assert np.all(np.diff(ht) >= 0)
    for b in range(nb):
        assert start[b] % tile == 0
        rows = np.nonzero(ht == b)[0]
        n_b = off[b + 1] - off[b]
        if n_b:
            assert rows[0] == start[b] and np.all(real[start[b]:start[b] + n_b])
            assert not np.any(real[start[b] + n_b:start[b + 1]])
            np.testing.assert_array_equal(h[pt[start[b]:start[b] + n_b]], b)
    # no tile holds two buckets
    for t0 in range(0, n_rows, tile):
        assert len(set(ht[t0:t0 + tile].tolist())) == 1
    assert not np.any(real[start[nb]:])
