"""LSH bucket id, stable bucket sort, row gather and unsort (float64 / exact).

Test infrastructure only (see the package docstring).

Page: "Faster Causal Attention Over Large Sequences Through Sparse Flash
Attention" (deep-paper.org), "动态稀疏性为何会破坏它" item 2 and "SCFA
解决方案" part 2: similar tokens are grouped into buckets with LSH (as in
Reformer) and reordered by bucket, which breaks causal order; the results are
put back in the original order. The page gives no LSH construction; the one
used here is the random-rotation argmax of the workload statement:
h(x) = argmax_j v_j with v = [x R, -x R] (2m candidates), R a Gaussian [D, m].

Readings:
  * The argmax is taken over the EXACT real values of v (bfloat16 inputs are
    exact rationals); ties go to the smallest index j. The L2 normalisation of
    x is a positive scaling, which leaves the exact argmax unchanged, so it is
    not applied. A zero vector gets bucket 0.
  * The sort is stable: key (bucket, original position).
  * Tile-aligned layout (tile_aligned): the same sorted order with each
    bucket starting on a multiple of the attention tile height, the gaps
    filled with padding rows that name no token. The page sorts by bucket
    but leaves the row layout open; padding keeps every tile inside one
    bucket, so no tile pair straddles two buckets.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

_U64 = 2.0**-53


def _exact_bucket(x_row: np.ndarray, R: np.ndarray) -> int:
    """argmax over [xR, -xR] in exact rational arithmetic, smallest index on ties."""
    D, m = R.shape
    xs = [Fraction(float(a)) for a in x_row]
    s = []
    for c in range(m):
        acc = Fraction(0)
        for d in range(D):
            acc += xs[d] * Fraction(float(R[d, c]))
        s.append(acc)
    vals = s + [-a for a in s]
    best = 0
    for j in range(1, 2 * m):
        if vals[j] > vals[best]:
            best = j
    return best


def lsh_hash(x, R, exact_all: bool = False) -> np.ndarray:
    """Bucket ids for the rows of x.

    x: [..., D] (bfloat16 values held in any float dtype), R: [D, m].
    Returns int32 [...] in [0, 2m).

    float64 evaluation with a certified error bound: each float64 dot product
    of D exact products has |error| <= gamma_D * sum_d |x_d R_dc|
    (gamma_D = D u / (1 - D u), u = 2^-53). A row whose computed top candidate
    beats every other candidate by more than twice the sum of both bounds has
    the same exact argmax; every other row (and every row when exact_all) is
    recomputed in exact rational arithmetic.
    """
    x = np.asarray(x, dtype=np.float64)
    R = np.asarray(R, dtype=np.float64)
    D, m = R.shape
    shape = x.shape[:-1]
    X = x.reshape(-1, D)
    out = np.empty(X.shape[0], dtype=np.int32)
    if exact_all:
        for n in range(X.shape[0]):
            out[n] = _exact_bucket(X[n], R)
        return out.reshape(shape)
    gamma = D * _U64 / (1.0 - D * _U64)
    absR = np.abs(R)
    for r0 in range(0, X.shape[0], 65536):  # row blocks only bound memory
        Xb = X[r0:r0 + 65536]
        s = Xb @ R
        A = np.abs(Xb) @ absR
        err = gamma * A * (1.0 + 1e-10)
        v = np.concatenate([s, -s], axis=1)
        e = np.concatenate([err, err], axis=1)
        top = np.argmax(v, axis=1)
        rows = np.arange(Xb.shape[0])
        margin = v[rows, top][:, None] - v
        need = 2.0 * (e[rows, top][:, None] + e)
        ok = (margin > need)
        ok[rows, top] = True
        certified = ok.all(axis=1)
        out[r0:r0 + Xb.shape[0]] = top
        for n in np.nonzero(~certified)[0]:
            out[r0 + n] = _exact_bucket(Xb[n], R)
    return out.reshape(shape)


def bucket_sort(h, n_buckets: int):
    """Stable counting sort of one row of bucket ids.

    Returns (perm, h_sorted, bucket_off): perm[s] = original position of the
    token in sorted slot s (ties by position ascending), h_sorted = h[perm],
    bucket_off[c] = number of tokens with bucket < c (length n_buckets + 1).
    """
    h = np.asarray(h, dtype=np.int64)
    perm = np.argsort(h, kind="stable").astype(np.int32)
    counts = np.bincount(h, minlength=n_buckets)
    off = np.zeros(n_buckets + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    return perm, h[perm].astype(np.int32), off


def tile_aligned(perm, bucket_off, n_rows: int, tile: int, pad: int):
    """One head's sorted order re-laid so that every bucket starts on a
    multiple of `tile` rows.

    Bucket b (n_b = bucket_off[b+1] - bucket_off[b] tokens, in their sorted
    order) occupies rows start[b] .. start[b] + n_b - 1, where start[0] = 0 and
    start[b+1] = start[b] + n_b rounded up to a multiple of tile. Every other
    row up to n_rows is padding: position `pad`, and the bucket id of the
    rows around it (bucket n_buckets - 1 after the last bucket). Returns
    (perm_t, h_t, start) with start of length n_buckets + 1.
    """
    off = np.asarray(bucket_off, dtype=np.int64)
    nb = len(off) - 1
    start = np.zeros(nb + 1, dtype=np.int64)
    for b in range(nb):
        n_b = off[b + 1] - off[b]
        start[b + 1] = start[b] + -(-n_b // tile) * tile
    assert start[nb] <= n_rows
    perm_t = np.full(n_rows, pad, dtype=np.int64)
    h_t = np.full(n_rows, nb - 1, dtype=np.int64)
    for b in range(nb):
        n_b = off[b + 1] - off[b]
        h_t[start[b]:start[b + 1]] = b
        perm_t[start[b]:start[b] + n_b] = np.asarray(perm)[off[b]:off[b + 1]]
    return perm_t.astype(np.int32), h_t.astype(np.int32), start.astype(np.int32)


def gather_rows(x, perm):
    """x_sorted[s] = x[perm[s]] (row copy)."""
    return np.asarray(x)[np.asarray(perm, dtype=np.int64)]


def gather_rows_padded(x, perm):
    """x_sorted[s] = x[perm[s]], a zero row where perm[s] names no row."""
    x = np.asarray(x)
    perm = np.asarray(perm, dtype=np.int64)
    inside = (perm >= 0) & (perm < x.shape[0])
    out = np.zeros((perm.shape[0],) + x.shape[1:], dtype=x.dtype)
    out[inside] = x[perm[inside]]
    return out


def unsort_rows(y_sorted, perm):
    """y[perm[s]] = y_sorted[s] (inverse of gather_rows)."""
    y_sorted = np.asarray(y_sorted)
    y = np.empty_like(y_sorted)
    y[np.asarray(perm, dtype=np.int64)] = y_sorted
    return y
