"""Pins of the live-tile specification (CPU only).

Pins: hand-worked fixtures, brute force over the element mask (a tile is
live in QK mode exactly when it holds an admissible pair; FULL exactly when
all 128 x 128 pairs are admissible), coverage of every admissible pair in hash
mode, the closed form of the dense causal tile pattern, and CSR / CSC / work
order against Python's own sort.
"""
import numpy as np
import pytest

from conftest import load_golden
from oracle import attention, lsh, tiles
from synth import K_SENTINEL, Q_SENTINEL


def test_golden_qk_2x2():
    g = load_golden("tiles_qk_2x2.json")
    q_idx = 2 * np.arange(256)
    k_idx = 2 * np.arange(256) + 1
    live, full = tiles.head_tiles("qk", 256, 256, q_idx, k_idx)
    np.testing.assert_array_equal(live, np.array(g["live"], bool))
    np.testing.assert_array_equal(full, np.array(g["full"], bool))
    L = tiles.live_list("qk", 1, 1, 256, 256, q_idx[None, None], k_idx[None, None])
    for key in ("row_ptr", "cols", "fflags", "csc_ptr", "csc_rows", "cflags", "work_fwd", "work_bwd"):
        np.testing.assert_array_equal(L[key], g[key], err_msg=key)


def _runs(runs, T):
    h = np.empty(T, dtype=np.int64)
    for a, b, c in runs:
        h[a:b] = c
    return h


def test_golden_hash_3x3():
    g = load_golden("tiles_hash_3x3.json")
    T = g["T"]
    qh, kh = _runs(g["q_hash_runs"], T), _runs(g["k_hash_runs"], T)
    pos = np.arange(T)
    live, full = tiles.head_tiles("hash", T, T, pos, pos, qh, kh)
    np.testing.assert_array_equal(live, np.array(g["live"], bool))
    np.testing.assert_array_equal(full, np.array(g["full"], bool))
    L = tiles.live_list("hash", 1, 1, T, T, pos[None, None], pos[None, None], qh[None, None], kh[None, None])
    for key in ("row_ptr", "cols", "csc_ptr", "csc_rows", "work_fwd", "work_bwd"):
        np.testing.assert_array_equal(L[key], g[key], err_msg=key)


def _tile_truth(mask, Tq, Tk):
    nQt, nKt = -(-Tq // 128), -(-Tk // 128)
    anyp = np.zeros((nQt, nKt), bool)
    allp = np.zeros((nQt, nKt), bool)
    for i in range(nQt):
        for j in range(nKt):
            blk = mask[128 * i:128 * (i + 1), 128 * j:128 * (j + 1)]
            anyp[i, j] = blk.any()
            allp[i, j] = blk.shape == (128, 128) and blk.all()
    return anyp, allp


@pytest.mark.parametrize("seed,Tq,Tk,keep", [(30, 300, 260, 0.7), (31, 129, 1000, 0.3), (32, 384, 384, 1.0), (33, 5, 700, 0.5)])
def test_qk_live_is_exists_admissible(seed, Tq, Tk, keep):
    rng = np.random.default_rng(seed)
    T = max(Tq, Tk) * 2
    qpos = np.sort(rng.choice(T, size=int(Tq * keep) or 1, replace=False))
    kpos = np.sort(rng.choice(T, size=int(Tk * keep) or 1, replace=False))
    q_idx = np.full(Tq, Q_SENTINEL, np.int64)
    k_idx = np.full(Tk, K_SENTINEL, np.int64)
    q_idx[:len(qpos)] = qpos
    k_idx[:len(kpos)] = kpos
    live, full = tiles.head_tiles("qk", Tq, Tk, q_idx, k_idx)
    anyp, allp = _tile_truth(attention.mask_qk(q_idx, k_idx), Tq, Tk)
    np.testing.assert_array_equal(live, anyp)
    np.testing.assert_array_equal(full, allp)


@pytest.mark.parametrize("seed,T,nb", [(40, 700, 4), (41, 1000, 16), (42, 257, 2), (43, 640, 1)])
def test_hash_coverage_and_full(seed, T, nb):
    rng = np.random.default_rng(seed)
    qh, kh = rng.integers(0, nb, T), rng.integers(0, nb, T)
    pq, qhs, _ = lsh.bucket_sort(qh, nb)
    pk, khs, _ = lsh.bucket_sort(kh, nb)
    live, full = tiles.head_tiles("hash", T, T, pq, pk, qhs, khs)
    mask_sorted = attention.mask_hash(qhs, khs, q_pos=pq, k_pos=pk)
    anyp, allp = _tile_truth(mask_sorted, T, T)
    # every admissible pair lies in a live tile: 100% coverage of in-bucket causal pairs
    assert np.all(live[anyp])
    np.testing.assert_array_equal(full, allp)
    if nb == 1:
        qk_live, _ = tiles.head_tiles("qk", T, T, pq, pk)
        np.testing.assert_array_equal(live, qk_live)


@pytest.mark.parametrize("T", [1, 127, 128, 129, 1000])
def test_dense_is_lower_triangular_tiles(T):
    live, full = tiles.head_tiles("dense", T, T)
    n = -(-T // 128)
    i, j = np.indices((n, n))
    np.testing.assert_array_equal(live, i >= j)
    complete = np.arange(n) < T // 128
    np.testing.assert_array_equal(full, (i > j) & complete[:, None] & complete[None, :])


def test_csr_csc_work_order_consistency():
    rng = np.random.default_rng(50)
    B, H, T, nb = 2, 3, 900, 8
    qh = rng.integers(0, nb, (B, H, T))
    kh = rng.integers(0, nb, (B, H, T))
    pq = np.empty((B, H, T), np.int32); pk = np.empty_like(pq); qs = np.empty_like(pq); ks = np.empty_like(pq)
    for b in range(B):
        for h in range(H):
            pq[b, h], qs[b, h], _ = lsh.bucket_sort(qh[b, h], nb)
            pk[b, h], ks[b, h], _ = lsh.bucket_sort(kh[b, h], nb)
    L = tiles.live_list("hash", B, H, T, T, pq, pk, qs, ks)
    nQt, nKt = L["nQt"], L["nKt"]
    pairs_csr = set()
    for g in range(B * H * nQt):
        cs = L["cols"][L["row_ptr"][g]:L["row_ptr"][g + 1]]
        assert list(cs) == sorted(cs)
        for c, f in zip(cs, L["fflags"][L["row_ptr"][g]:L["row_ptr"][g + 1]]):
            pairs_csr.add((g // nQt, g % nQt, int(c), int(f)))
    pairs_csc = set()
    for g in range(B * H * nKt):
        rs = L["csc_rows"][L["csc_ptr"][g]:L["csc_ptr"][g + 1]]
        assert list(rs) == sorted(rs)
        for r, f in zip(rs, L["cflags"][L["csc_ptr"][g]:L["csc_ptr"][g + 1]]):
            pairs_csc.add((g // nKt, int(r), g % nKt, int(f)))
    assert pairs_csr == pairs_csc
    cnt = np.diff(L["row_ptr"])
    assert sorted(L["work_fwd"].tolist()) == list(range(B * H * nQt))
    keys = [(-cnt[t], t) for t in L["work_fwd"]]
    assert keys == sorted(keys)


def test_work_order_rule():
    # hand-worked: largest count first, ties by id, zero counts last
    assert tiles.work_order([1, 3, 0, 3, 2]) == [1, 3, 4, 0, 2]
    assert tiles.work_order([]) == []
    assert tiles.work_order([0, 0, 0]) == [0, 1, 2]
    # any list: a permutation whose counts never increase and whose ties keep id order
    rng = np.random.default_rng(51)
    counts = rng.integers(0, 6, 500)
    order = tiles.work_order(counts)
    assert sorted(order) == list(range(500))
    for a, b in zip(order, order[1:]):
        assert counts[a] > counts[b] or (counts[a] == counts[b] and a < b)
