"""Explicit-mask float64 attention: masks, forward and backward.

Test infrastructure only (see the package docstring).

Page: "Faster Causal Attention Over Large Sequences Through Sparse Flash
Attention" (deep-paper.org summary of arXiv 2306.01160).
  * "二次方问题": every query scores every key, a T x T matrix.
  * "FlashAttention 的兴起": tiling keeps the attention maths exact; causal
    attention lets a token see only earlier tokens (lower-triangular mask).
  * "SCFA 解决方案", part 1: in QK-sparse mode the element mask compares
    original positions q_idx / k_idx.
  * "SCFA 解决方案", part 2: in hash-sparse mode the element mask requires
    causality and equal bucket ids.
Readings where the page is silent: a query may attend to its own position
(q_idx >= k_idx); a query with no admissible key outputs 0 with LSE = -inf
and passes no gradient; LSE is the natural log of the softmax denominator.
"""
from __future__ import annotations

import numpy as np


def mask_dense(Tq: int, Tk: int | None = None) -> np.ndarray:
    """Causal mask on positions: query p sees key r iff p >= r."""
    Tk = Tq if Tk is None else Tk
    return np.arange(Tq)[:, None] >= np.arange(Tk)[None, :]


def mask_qk(q_idx, k_idx) -> np.ndarray:
    """QK-sparse element mask on compacted rows: q_idx[r] >= k_idx[c]."""
    qi = np.asarray(q_idx, dtype=np.int64)
    ki = np.asarray(k_idx, dtype=np.int64)
    return qi[:, None] >= ki[None, :]


def mask_hash(q_hash, k_hash, q_pos=None, k_pos=None) -> np.ndarray:
    """Hash-sparse element mask: causal on positions AND same bucket id.

    With q_pos/k_pos omitted the rows are in original order (position = row).
    """
    qh = np.asarray(q_hash, dtype=np.int64)
    kh = np.asarray(k_hash, dtype=np.int64)
    qp = np.arange(len(qh)) if q_pos is None else np.asarray(q_pos, dtype=np.int64)
    kp = np.arange(len(kh)) if k_pos is None else np.asarray(k_pos, dtype=np.int64)
    return (qh[:, None] == kh[None, :]) & (qp[:, None] >= kp[None, :])


def forward(q, k, v, mask, scale):
    """Masked softmax attention for one head.

    q: [Tq, D], k, v: [Tk, D], mask: bool [Tq, Tk]. Returns (O [Tq, D],
    LSE [Tq], P [Tq, Tk]) in float64. Rows without an admissible key give
    O = 0, LSE = -inf, P = 0.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    mask = np.asarray(mask, dtype=bool)
    S = scale * (q @ k.T)
    S = np.where(mask, S, -np.inf)
    live = mask.any(axis=1)
    m = np.where(live, S.max(axis=1, initial=-np.inf), 0.0)
    E = np.where(mask, np.exp(S - m[:, None]), 0.0)
    l = E.sum(axis=1)
    l_safe = np.where(live, l, 1.0)
    P = E / l_safe[:, None]
    O = P @ v
    lse = np.where(live, m + np.log(l_safe), -np.inf)
    return O, lse, P


def backward(q, k, v, do, mask, scale):
    """Gradients of L = sum(O * dO) for one head.

    Returns (O, LSE, dQ, dK, dV) in float64, with
    dV = P^T dO, dP = dO V^T, Drow = rowsum(dO * O), dS = P * (dP - Drow),
    dQ = scale * dS K, dK = scale * dS^T Q.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    O, lse, P = forward(q, k, v, mask, scale)
    dv = P.T @ do
    dP = do @ v.T
    Drow = np.sum(do * O, axis=1)
    dS = P * (dP - Drow[:, None])
    dq = scale * (dS @ k)
    dk = scale * (dS.T @ q)
    return O, lse, dq, dk, dv


def admissible_pairs(mask) -> int:
    """Number of unmasked (query, key) pairs: the useful-FLOP count basis."""
    return int(np.count_nonzero(mask))
