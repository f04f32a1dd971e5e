"""Pair coverage: admissible pairs inside the live tiles, and inside
Reformer-style chunks of the bucket-sorted sequence.

Test infrastructure only (see the package docstring).

Page: "Faster Causal Attention Over Large Sequences Through Sparse Flash
Attention" (deep-paper.org), section "实验与结果": SCFA hash-sparse attention
covers 100% of the bucket collisions, while the coverage of Reformer's
attention drops (Fig. 4). Reading (the page does not describe Reformer's
scheme): after the bucket sort, the sorted rows are cut into chunks of
`chunk` slots and a query sees the keys of its own chunk and of the chunk
before it; coverage is the share of the admissible pairs (same bucket,
causal) that such chunks contain.
"""
from __future__ import annotations

import numpy as np

from . import attention, tiles


def pairs_in_live_tiles(mask, live) -> int:
    """Sum of the explicit element mask over the live 128 x 128 tiles.

    mask: bool [Tq, Tk]; live: bool [nQt, nKt] (tiles.head_tiles).
    """
    mask = np.asarray(mask, dtype=bool)
    total = 0
    for i, j in zip(*np.nonzero(live)):
        total += int(np.count_nonzero(mask[i * tiles.BM:(i + 1) * tiles.BM, j * tiles.BN:(j + 1) * tiles.BN]))
    return total


def chunk_mask(T: int, chunk: int) -> np.ndarray:
    """Sorted slot s may see sorted slot s' iff chunk(s') is chunk(s) or the one before."""
    c = np.arange(T) // chunk
    d = c[:, None] - c[None, :]
    return (d == 0) | (d == 1)


def chunked_pairs(q_hash_sorted, k_hash_sorted, q_pos, k_pos, chunk: int) -> int:
    """Admissible hash-mode pairs (same bucket, q_pos >= k_pos) of one head that
    lie inside a query's chunk or the chunk before it, on sorted rows."""
    mask = attention.mask_hash(q_hash_sorted, k_hash_sorted, q_pos=q_pos, k_pos=k_pos)
    return int(np.count_nonzero(mask & chunk_mask(len(q_pos), chunk)))
