"""The three attention problems end to end, in float64, head by head.

Test infrastructure only (see the package docstring).

Page: "Faster Causal Attention Over Large Sequences Through Sparse Flash
Attention" (deep-paper.org), "SCFA 解决方案". Hash mode is evaluated in the
ORIGINAL token order with the explicit mask (causal AND same bucket), with no
sort at all; the sorted view (perm, sorted hashes, bucket offsets) is
returned separately so that bit-exact index checks can use it.
"""
from __future__ import annotations

import numpy as np

from . import attention, lsh


def _f64(t):
    """bfloat16 torch tensor / array -> float64 numpy (exact)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


def _heads(B, H, heads):
    return [(b, h) for b in range(B) for h in range(H)] if heads is None else list(heads)


def run_dense(q, k, v, do, scale, heads=None, backward=True):
    """Dense causal attention per head. Returns dict of per-head results."""
    q, k, v, do = map(_f64, (q, k, v, do))
    B, H, T, _ = q.shape
    mask = attention.mask_dense(T)
    out = {}
    for b, h in _heads(B, H, heads):
        if backward:
            O, lse, dq, dk, dv = attention.backward(q[b, h], k[b, h], v[b, h], do[b, h], mask, scale)
            out[(b, h)] = dict(o=O, lse=lse, dq=dq, dk=dk, dv=dv, pairs=attention.admissible_pairs(mask))
        else:
            O, lse, _ = attention.forward(q[b, h], k[b, h], v[b, h], mask, scale)
            out[(b, h)] = dict(o=O, lse=lse, pairs=attention.admissible_pairs(mask))
    return out


def run_qk(q, k, v, do, q_idx, k_idx, scale, heads=None, backward=True):
    """QK-sparse attention on compacted rows with original positions."""
    q, k, v, do = map(_f64, (q, k, v, do))
    q_idx = np.asarray(q_idx)
    k_idx = np.asarray(k_idx)
    B, H = q.shape[:2]
    out = {}
    for b, h in _heads(B, H, heads):
        mask = attention.mask_qk(q_idx[b, h], k_idx[b, h])
        if backward:
            O, lse, dq, dk, dv = attention.backward(q[b, h], k[b, h], v[b, h], do[b, h], mask, scale)
            out[(b, h)] = dict(o=O, lse=lse, dq=dq, dk=dk, dv=dv, pairs=attention.admissible_pairs(mask))
        else:
            O, lse, _ = attention.forward(q[b, h], k[b, h], v[b, h], mask, scale)
            out[(b, h)] = dict(o=O, lse=lse, pairs=attention.admissible_pairs(mask))
    return out


def hash_sort_view(x_hash, n_buckets):
    """Per-head stable sort of bucket ids: perm, sorted ids, bucket offsets."""
    x_hash = np.asarray(x_hash)
    B, H, T = x_hash.shape
    perm = np.empty((B, H, T), dtype=np.int32)
    hs = np.empty((B, H, T), dtype=np.int32)
    off = np.empty((B, H, n_buckets + 1), dtype=np.int32)
    for b in range(B):
        for h in range(H):
            perm[b, h], hs[b, h], off[b, h] = lsh.bucket_sort(x_hash[b, h], n_buckets)
    return perm, hs, off


def run_hash(q, k, v, do, R, scale, heads=None, backward=True, q_hash=None, k_hash=None):
    """Hash-sparse attention in original order.

    Returns (results per head, q_hash, k_hash) where the hashes are [B, H, T]
    in original order (computed here unless given).
    """
    q, k, v, do, R = map(_f64, (q, k, v, do, R))
    B, H, T, _ = q.shape
    if q_hash is None:
        q_hash = lsh.lsh_hash(q, R)
    if k_hash is None:
        k_hash = lsh.lsh_hash(k, R)
    out = {}
    for b, h in _heads(B, H, heads):
        mask = attention.mask_hash(q_hash[b, h], k_hash[b, h])
        if backward:
            O, lse, dq, dk, dv = attention.backward(q[b, h], k[b, h], v[b, h], do[b, h], mask, scale)
            out[(b, h)] = dict(o=O, lse=lse, dq=dq, dk=dk, dv=dv, pairs=attention.admissible_pairs(mask))
        else:
            O, lse, _ = attention.forward(q[b, h], k[b, h], v[b, h], mask, scale)
            out[(b, h)] = dict(o=O, lse=lse, pairs=attention.admissible_pairs(mask))
    return out, q_hash, k_hash


def useful_flops(pairs: int, D: int, backward: bool = True) -> float:
    """4 D flops per admissible pair forward, 10 D backward (S recomputed)."""
    return float(pairs) * D * (14.0 if backward else 4.0)


def run_hash_buckets(q, k, v, do, scale, q_hash, k_hash, buckets):
    """Hash-sparse attention of ONE head, evaluated bucket by bucket.

    q, k, v, do: [T, D]; q_hash, k_hash: [T] bucket ids in original order.
    The hash mask (same bucket AND causal) never pairs tokens of different
    buckets, so restricting the explicit-mask problem to the queries and keys
    of one bucket c gives exactly the rows of those queries (O, LSE, dQ) and
    keys (dK, dV) in the whole problem. This is how sequences too long for a
    T x T mask are checked. Returns {c: dict(q_pos, k_pos, o, lse, dq, dk, dv)}.
    """
    q_hash = np.asarray(q_hash)
    k_hash = np.asarray(k_hash)
    out = {}
    for c in buckets:
        qp = np.nonzero(q_hash == c)[0]
        kp = np.nonzero(k_hash == c)[0]
        mask = attention.mask_hash(q_hash[qp], k_hash[kp], q_pos=qp, k_pos=kp)
        O, lse, dq, dk, dv = attention.backward(_f64(q)[qp], _f64(k)[kp], _f64(v)[kp], _f64(do)[qp], mask, scale)
        out[int(c)] = dict(q_pos=qp, k_pos=kp, o=O, lse=lse, dq=dq, dk=dk, dv=dv,
                           pairs=attention.admissible_pairs(mask))
    return out
