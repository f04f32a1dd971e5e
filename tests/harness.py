"""Helpers shared by the GPU parity tests: tolerances and comparisons.

Tolerances follow the workload statement for bf16 inputs with fp32
accumulation: max abs error <= 2e-2 and relative L2 error <= 5e-3 on O, dQ, dK
and dV against the float64 oracle. LSE (fp32) is held to 2e-3 absolute on
finite entries and must match -inf exactly. Index work is bit-exact.
"""
import numpy as np
import torch

ATOL = 2e-2
REL_L2 = 5e-3
LSE_ATOL = 2e-3


def to_np(t):
    return t.detach().to("cpu").to(torch.float64).numpy() if t.dtype.is_floating_point else t.detach().cpu().numpy()


def check_close(name, got, ref, atol=ATOL, rel_l2=REL_L2):
    g = to_np(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    err = float(np.abs(g - r).max()) if g.size else 0.0
    nr = float(np.linalg.norm(r))
    rl2 = float(np.linalg.norm(g - r)) / nr if nr > 0 else float(np.linalg.norm(g))
    assert err <= atol and rl2 <= rel_l2, f"{name}: max abs {err:.3e} (<= {atol}), rel L2 {rl2:.3e} (<= {rel_l2})"
    return err, rl2


def check_lse(name, got, ref):
    g = to_np(got)
    r = np.asarray(ref, np.float64)
    ninf = np.isneginf(r)
    assert np.array_equal(np.isneginf(g), ninf), f"{name}: -inf pattern differs"
    if (~ninf).any():
        err = float(np.abs(g[~ninf] - r[~ninf]).max())
        assert err <= LSE_ATOL, f"{name}: max abs {err:.3e}"
