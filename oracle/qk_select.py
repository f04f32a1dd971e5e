"""The QK-sparse selection step (float-free, exact).

Test infrastructure only (see the package docstring).

Page: "Faster Causal Attention Over Large Sequences Through Sparse Flash
Attention" (deep-paper.org), "SCFA 解决方案" part 1 "QK-Sparse": queries and
keys dropped by an upstream step leave compacted Q/K/V together with the
original positions of the kept rows (q_idx / k_idx), which the attention
uses for its causal mask.

Reading: which tokens are kept is the caller's policy (a per-head keep
mask); the step turns the mask into the kept positions in ascending order,
padded to a fixed length with a sentinel that names no token.
"""
from __future__ import annotations

import numpy as np


def select_positions(keep, Tc: int, sentinel: int):
    """keep [..., T] (nonzero = kept) -> (idx [..., Tc], count [...]): the
    kept positions of each row in ascending order, then `sentinel`; a row
    keeping more than Tc tokens lists its first Tc and reports its full
    count."""
    keep = np.asarray(keep)
    lead = keep.shape[:-1]
    flat = keep.reshape(-1, keep.shape[-1])
    idx = np.full((flat.shape[0], Tc), sentinel, dtype=np.int64)
    count = np.zeros(flat.shape[0], dtype=np.int64)
    for r in range(flat.shape[0]):
        pos = [t for t in range(flat.shape[1]) if flat[r, t] != 0]
        count[r] = len(pos)
        idx[r, :min(len(pos), Tc)] = pos[:Tc]
    return idx.reshape(lead + (Tc,)).astype(np.int32), count.reshape(lead).astype(np.int32)
