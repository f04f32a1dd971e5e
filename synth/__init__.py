"""Seeded synthetic inputs for sparse causal flash attention workloads.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests. It holds none of the attention, hashing, sorting or tiling
arithmetic: it only draws random numbers, Bernoulli keep masks and the
position-order compaction a caller performs before calling the QK-sparse
kernels (query/key dropping produces smaller, compacted Q/K/V plus the
original positions: "Faster Causal Attention Over Large Sequences Through
Sparse Flash Attention", section "SCFA 解决方案", part 1 "QK-Sparse").

Random streams: numpy's counter-based Philox bit generator, keyed by
(seed, tensor id); float32 standard normals are rounded to bfloat16 with
round-to-nearest-even (torch's conversion). Every tensor is produced on the
host, so the oracle and the GPU see identical bytes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

# Sentinels that pad compacted QK-sparse tensors to a common length per head.
# A padded query sits "before every key" and a padded key "after every query",
# so neither forms an admissible pair with anything.
Q_SENTINEL = -1
K_SENTINEL = 2**31 - 1

# tensor ids of the seeded streams
TID_Q, TID_K, TID_V, TID_DO, TID_R, TID_KEEP_Q, TID_KEEP_K = 1, 2, 3, 4, 5, 6, 7


def _rng(seed: int, tensor_id: int) -> np.random.Generator:
    key = np.array([seed & (2**64 - 1), tensor_id], dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key))


def normal_bf16(seed: int, tensor_id: int, shape) -> torch.Tensor:
    """i.i.d. N(0,1) bfloat16 tensor (CPU), deterministic in (seed, tensor_id)."""
    x = _rng(seed, tensor_id).standard_normal(size=tuple(shape), dtype=np.float32)
    return torch.from_numpy(x).to(torch.bfloat16)


def rotation_bf16(seed: int, D: int, m: int) -> torch.Tensor:
    """Gaussian random-rotation matrix R of shape [D, m] in bfloat16."""
    return normal_bf16(seed, TID_R, (D, m))


def keep_mask(seed: int, tensor_id: int, B: int, H: int, T: int, p_keep: float) -> np.ndarray:
    """Bernoulli(p_keep) keep decision per (batch, head, position)."""
    u = _rng(seed, tensor_id).random(size=(B, H, T))
    return u < p_keep


def compact(x: torch.Tensor, keep: np.ndarray, sentinel: int):
    """Keep the rows selected by `keep` in position order, per (b, h).

    x: [B, H, T, D]; keep: bool [B, H, T]. Returns (xc [B, H, Tc, D], idx
    [B, H, Tc] int32) where Tc is the largest kept count over (b, h); rows past
    a head's own count are zero with idx = sentinel.
    """
    B, H, T, D = x.shape
    counts = keep.sum(axis=2)
    Tc = max(int(counts.max()), 1)
    xc = torch.zeros((B, H, Tc, D), dtype=x.dtype)
    idx = np.full((B, H, Tc), sentinel, dtype=np.int32)
    for b in range(B):
        for h in range(H):
            pos = np.nonzero(keep[b, h])[0]
            n = len(pos)
            idx[b, h, :n] = pos
            if n:
                xc[b, h, :n] = x[b, h, torch.from_numpy(pos.astype(np.int64))]
    return xc, torch.from_numpy(idx)


@dataclass
class Workload:
    """One synthetic workload shaped like the pages' attention benchmarks."""
    name: str
    mode: str            # "dense", "qk" or "hash"
    B: int
    H: int
    T: int
    D: int
    seed: int
    p_keep: float = 1.0  # qk mode: Bernoulli keep probability for queries and keys
    n_buckets: int = 0   # hash mode: number of LSH buckets (R has n_buckets // 2 columns)
    notes: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


WORKLOADS = {
    # small hash case the oracle finishes in seconds
    "hash_b1h2_t512_d64_nb4": Workload("hash_b1h2_t512_d64_nb4", "hash", 1, 2, 512, 64, 1001, n_buckets=4),
    # 122M-LM-shaped attention at 8k tokens, 30% QK drop
    "qk_b4h12_t8192_d64_keep0.7": Workload("qk_b4h12_t8192_d64_keep0.7", "qk", 4, 12, 8192, 64, 1002, p_keep=0.7),
    "hash_b4h12_t8192_d64_nb16": Workload("hash_b4h12_t8192_d64_nb16", "hash", 4, 12, 8192, 64, 1003, n_buckets=16),
    "hash_b2h12_t16384_d64_nb32": Workload("hash_b2h12_t16384_d64_nb32", "hash", 2, 12, 16384, 64, 1004, n_buckets=32),
    "qk_b2h12_t16384_d64_keep0.8": Workload("qk_b2h12_t16384_d64_keep0.8", "qk", 2, 12, 16384, 64, 1004, p_keep=0.8),
    "qk_b2h12_t16384_d64_keep0.7": Workload("qk_b2h12_t16384_d64_keep0.7", "qk", 2, 12, 16384, 64, 1004, p_keep=0.7),
    "qk_b2h12_t16384_d64_keep0.5": Workload("qk_b2h12_t16384_d64_keep0.5", "qk", 2, 12, 16384, 64, 1004, p_keep=0.5),
    "qk_b2h12_t16384_d64_keep0.3": Workload("qk_b2h12_t16384_d64_keep0.3", "qk", 2, 12, 16384, 64, 1004, p_keep=0.3),
    "hash_b1h8_t1048576_d128_nb512": Workload("hash_b1h8_t1048576_d128_nb512", "hash", 1, 8, 1 << 20, 128, 1005, n_buckets=512),
    "dense_b4h12_t8192_d64": Workload("dense_b4h12_t8192_d64", "dense", 4, 12, 8192, 64, 1002),
}


@dataclass
class Problem:
    """Host tensors of one workload instance (all on CPU)."""
    wl: Workload
    q: torch.Tensor        # [B,H,Tq,D] bf16 (compacted in qk mode)
    k: torch.Tensor
    v: torch.Tensor
    do: torch.Tensor       # upstream gradient of O, same layout as q
    q_idx: torch.Tensor | None = None   # qk mode: int32 [B,H,Tq]
    k_idx: torch.Tensor | None = None
    R: torch.Tensor | None = None       # hash mode: [D, m] bf16
    extra: dict = field(default_factory=dict)


def make_problem(wl: Workload, B: int | None = None, H: int | None = None, T: int | None = None) -> Problem:
    """Draw the inputs of `wl` (optionally with smaller B/H/T for quick cases)."""
    B = wl.B if B is None else B
    H = wl.H if H is None else H
    T = wl.T if T is None else T
    D = wl.D
    q = normal_bf16(wl.seed, TID_Q, (B, H, T, D))
    k = normal_bf16(wl.seed, TID_K, (B, H, T, D))
    v = normal_bf16(wl.seed, TID_V, (B, H, T, D))
    do = normal_bf16(wl.seed, TID_DO, (B, H, T, D))
    if wl.mode == "qk":
        kq = keep_mask(wl.seed, TID_KEEP_Q, B, H, T, wl.p_keep)
        kk = keep_mask(wl.seed, TID_KEEP_K, B, H, T, wl.p_keep)
        qc, q_idx = compact(q, kq, Q_SENTINEL)
        doc, _ = compact(do, kq, Q_SENTINEL)
        kc, k_idx = compact(k, kk, K_SENTINEL)
        vc, _ = compact(v, kk, K_SENTINEL)
        return Problem(wl, qc, kc, vc, doc, q_idx, k_idx)
    if wl.mode == "hash":
        R = rotation_bf16(wl.seed, D, wl.n_buckets // 2)
        return Problem(wl, q, k, v, do, R=R)
    return Problem(wl, q, k, v, do)
