"""The seeded input generators: determinism and the compacted QK layout."""
import numpy as np
import torch

import synth


def test_streams_are_deterministic_and_distinct():
    a = synth.normal_bf16(7, synth.TID_Q, (3, 5))
    b = synth.normal_bf16(7, synth.TID_Q, (3, 5))
    c = synth.normal_bf16(7, synth.TID_K, (3, 5))
    assert a.dtype == torch.bfloat16
    assert torch.equal(a, b) and not torch.equal(a, c)


def test_compaction_layout():
    wl = synth.Workload("t", "qk", 2, 3, 300, 64, 99, p_keep=0.6)
    p = synth.make_problem(wl)
    B, H, Tq, D = p.q.shape
    assert p.q_idx.shape == (B, H, Tq) and p.k_idx.dtype == torch.int32
    full_q = synth.normal_bf16(wl.seed, synth.TID_Q, (B, H, wl.T, D))
    for b in range(B):
        for h in range(H):
            qi = p.q_idx[b, h].numpy()
            n = int((qi >= 0).sum())
            assert np.all(np.diff(qi[:n]) > 0) and np.all(qi[n:] == synth.Q_SENTINEL)
            assert torch.equal(p.q[b, h, :n], full_q[b, h, torch.from_numpy(qi[:n].astype(np.int64))])
            assert torch.all(p.q[b, h, n:] == 0)
            ki = p.k_idx[b, h].numpy()
            nk = int((ki != synth.K_SENTINEL).sum())
            assert np.all(np.diff(ki[:nk]) > 0) and np.all(ki[nk:] == synth.K_SENTINEL)
    kept = (p.q_idx >= 0).sum().item() / (B * H * wl.T)
    assert 0.5 < kept < 0.7
