"""Pins of the coverage oracle: brute force on tiny inputs, the page's 100%
coverage of the live tiles, and the limits of the chunked count."""
import itertools

import numpy as np

from oracle import attention, coverage, lsh, tiles


def brute_chunked(qh, kh, qp, kp, chunk):
    n = 0
    for s, t in itertools.product(range(len(qp)), range(len(kp))):
        if s // chunk - t // chunk in (0, 1) and qh[s] == kh[t] and qp[s] >= kp[t]:
            n += 1
    return n


def sorted_view(rng, T, nb):
    qh = rng.integers(0, nb, T)
    kh = rng.integers(0, nb, T)
    pq, qs, _ = lsh.bucket_sort(qh, nb)
    pk, ks, _ = lsh.bucket_sort(kh, nb)
    return qs, ks, pq, pk


def test_chunked_pairs_brute_force():
    rng = np.random.default_rng(70)
    for T, nb, chunk in [(7, 2, 2), (12, 3, 3), (10, 1, 4), (9, 4, 1)]:
        qs, ks, pq, pk = sorted_view(rng, T, nb)
        assert coverage.chunked_pairs(qs, ks, pq, pk, chunk) == brute_chunked(qs, ks, pq, pk, chunk)


def test_chunked_pairs_limits():
    rng = np.random.default_rng(71)
    qs, ks, pq, pk = sorted_view(rng, 300, 4)
    total = attention.admissible_pairs(attention.mask_hash(qs, ks, q_pos=pq, k_pos=pk))
    assert coverage.chunked_pairs(qs, ks, pq, pk, 300) == total          # one chunk sees everything
    small = coverage.chunked_pairs(qs, ks, pq, pk, 16)
    assert 0 < small < total                                             # short chunks miss collisions
    # the count never drops as chunks grow by whole multiples
    assert coverage.chunked_pairs(qs, ks, pq, pk, 32) >= small


def test_live_tiles_cover_every_admissible_pair():
    rng = np.random.default_rng(72)
    # hash mode on sorted rows
    qs, ks, pq, pk = sorted_view(rng, 700, 8)
    mask = attention.mask_hash(qs, ks, q_pos=pq, k_pos=pk)
    live, _ = tiles.head_tiles("hash", 700, 700, pq, pk, qs, ks)
    assert coverage.pairs_in_live_tiles(mask, live) == attention.admissible_pairs(mask)
    # dropping one live tile that holds pairs loses exactly its pairs
    i, j = [(a, b) for a, b in zip(*np.nonzero(live)) if mask[a * 128:(a + 1) * 128, b * 128:(b + 1) * 128].any()][0]
    cut = live.copy()
    cut[i, j] = False
    lost = int(np.count_nonzero(mask[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]))
    assert coverage.pairs_in_live_tiles(mask, cut) == attention.admissible_pairs(mask) - lost
    # QK mode with sentinel padding, and dense
    qi = np.sort(rng.choice(2000, 500, replace=False)).astype(np.int64)
    ki = np.sort(rng.choice(2000, 450, replace=False)).astype(np.int64)
    qi = np.concatenate([qi, -np.ones(30, np.int64)])
    ki = np.concatenate([ki, np.full(80, 2**31 - 1, np.int64)])
    m2 = attention.mask_qk(qi, ki)
    live2, _ = tiles.head_tiles("qk", 530, 530, qi, ki)
    assert coverage.pairs_in_live_tiles(m2, live2) == attention.admissible_pairs(m2)
    live3, _ = tiles.head_tiles("dense", 300, 300)
    assert coverage.pairs_in_live_tiles(attention.mask_dense(300), live3) == 300 * 301 // 2
