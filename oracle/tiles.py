"""Tile metadata and the live-tile work list (exact integer specification).

Test infrastructure only (see the package docstring).

Page: "Faster Causal Attention Over Large Sequences Through Sparse Flash
Attention" (deep-paper.org), "SCFA 解决方案":
  * part 1 (QK-Sparse), tile pruning: tile T_ij (query block Q_i against key
    block K_j) is skipped when max(q_idx_i) < min(k_idx_j);
  * part 2 (Hash-Sparse): keep only tiles whose query-block and key-block
    bucket ids match, and skip bucket tiles that violate causal order.

Readings (the page gives no tile size or encoding):
  * Tiles are 128 x 128. Query tile i covers rows [128 i, min(128 i + 128, Tq)),
    key tile j likewise; only those valid rows enter the min / max.
  * QK and dense modes: live(i, j) = max q_idx(i) >= min k_idx(j), the page's
    skip test negated. Dense mode uses q_idx = k_idx = position.
  * Hash mode: a tile may span several buckets, so "bucket ids match" is read
    as overlapping bucket ranges: live(i, j) = [qh_min(i) <= kh_max(j) and
    kh_min(j) <= qh_max(i)] and max q_idx(i) >= min k_idx(j).
  * FULL(i, j): every one of the 128 x 128 pairs is admissible, so no element
    mask is needed: both tiles complete (128 valid rows), min q_idx(i) >=
    max k_idx(j), and in hash mode qh_min = qh_max = kh_min = kh_max.
  * Encoding: CSR over all (b, h, i) with k-tile columns ascending, CSC over
    all (b, h, j) with q-tile rows ascending, a flag byte per entry (bit 0 =
    FULL). Work order: every query tile (forward) / key tile (backward) id,
    sorted by live count descending, then by id ascending.
"""
from __future__ import annotations

import numpy as np

BM = 128
BN = 128
FLAG_FULL = 1


def tile_stats(vals, T: int, tile: int = BM):
    """Per-tile (min, max) of vals[:T] over valid rows, and the valid-row counts."""
    vals = np.asarray(vals, dtype=np.int64)[:T]
    n = (T + tile - 1) // tile
    mins = np.empty(n, dtype=np.int64)
    maxs = np.empty(n, dtype=np.int64)
    rows = np.empty(n, dtype=np.int64)
    for t in range(n):
        seg = vals[t * tile:min(T, (t + 1) * tile)]
        mins[t] = seg.min()
        maxs[t] = seg.max()
        rows[t] = len(seg)
    return mins, maxs, rows


def head_tiles(mode: str, Tq: int, Tk: int, q_idx=None, k_idx=None, q_hash=None, k_hash=None):
    """Live and FULL matrices [nQt, nKt] of one head."""
    if mode == "dense":
        q_idx = np.arange(Tq)
        k_idx = np.arange(Tk)
    qmin, qmax, qrows = tile_stats(q_idx, Tq, BM)
    kmin, kmax, krows = tile_stats(k_idx, Tk, BN)
    live = qmax[:, None] >= kmin[None, :]
    full = (qrows[:, None] == BM) & (krows[None, :] == BN) & (qmin[:, None] >= kmax[None, :])
    if mode == "hash":
        qhmin, qhmax, _ = tile_stats(q_hash, Tq, BM)
        khmin, khmax, _ = tile_stats(k_hash, Tk, BN)
        overlap = (qhmin[:, None] <= khmax[None, :]) & (khmin[None, :] <= qhmax[:, None])
        live = live & overlap
        one_bucket = (qhmin[:, None] == qhmax[:, None]) & (khmin[None, :] == khmax[None, :]) \
            & (qhmin[:, None] == khmin[None, :])
        full = full & one_bucket
    full = full & live
    return live, full


def work_order(counts):
    """Work order of a tile list: tile ids sorted by live count descending,
    then by id ascending (every id appears, zero counts last)."""
    counts = [max(int(c), 0) for c in counts]
    return sorted(range(len(counts)), key=lambda t: (-counts[t], t))


def live_list(mode: str, B: int, H: int, Tq: int, Tk: int,
              q_idx=None, k_idx=None, q_hash=None, k_hash=None):
    """The whole work list over all heads.

    q_idx/k_idx/q_hash/k_hash: arrays [B, H, T*] (None where the mode has none).
    Returns a dict of int32 / uint8 numpy arrays: row_ptr, cols, fflags,
    csc_ptr, csc_rows, cflags, work_fwd, work_bwd, plus nQt, nKt.
    """
    nQt = (Tq + BM - 1) // BM
    nKt = (Tk + BN - 1) // BN
    row_ptr = [0]
    cols, fflags = [], []
    csc_ptr = [0]
    csc_rows, cflags = [], []
    qcount = np.zeros(B * H * nQt, dtype=np.int64)
    kcount = np.zeros(B * H * nKt, dtype=np.int64)
    for b in range(B):
        for h in range(H):
            args = {}
            if mode in ("qk", "hash"):
                args["q_idx"] = np.asarray(q_idx[b, h])
                args["k_idx"] = np.asarray(k_idx[b, h])
            if mode == "hash":
                args["q_hash"] = np.asarray(q_hash[b, h])
                args["k_hash"] = np.asarray(k_hash[b, h])
            live, full = head_tiles(mode, Tq, Tk, **args)
            g = (b * H + h)
            for i in range(nQt):
                js = np.nonzero(live[i])[0]
                cols.extend(js.tolist())
                fflags.extend([FLAG_FULL if full[i, j] else 0 for j in js])
                row_ptr.append(row_ptr[-1] + len(js))
                qcount[g * nQt + i] = len(js)
            for j in range(nKt):
                is_ = np.nonzero(live[:, j])[0]
                csc_rows.extend(is_.tolist())
                cflags.extend([FLAG_FULL if full[i, j] else 0 for i in is_])
                csc_ptr.append(csc_ptr[-1] + len(is_))
                kcount[g * nKt + j] = len(is_)
    work_fwd = work_order(qcount)
    work_bwd = work_order(kcount)
    i32 = lambda a: np.asarray(a, dtype=np.int32)
    return {
        "nQt": nQt, "nKt": nKt,
        "row_ptr": i32(row_ptr), "cols": i32(cols), "fflags": np.asarray(fflags, dtype=np.uint8),
        "csc_ptr": i32(csc_ptr), "csc_rows": i32(csc_rows), "cflags": np.asarray(cflags, dtype=np.uint8),
        "work_fwd": i32(work_fwd), "work_bwd": i32(work_bwd),
    }
