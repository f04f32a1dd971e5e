"""CPU checks of the comparison helpers used by the GPU parity tests."""
import numpy as np
import torch

from harness import check_close, half_ulp_bf16


def test_half_ulp_bf16_values():
    assert half_ulp_bf16(np.array([1.0]))[0] == 2.0**-8
    assert half_ulp_bf16(np.array([1.99]))[0] == 2.0**-8
    assert half_ulp_bf16(np.array([8.0]))[0] == 2.0**-5
    assert half_ulp_bf16(np.array([-12.0]))[0] == 2.0**-5
    assert half_ulp_bf16(np.array([0.0]))[0] == 0.0


def test_half_ulp_bounds_bf16_rounding():
    # rounding to bf16 (torch, round to nearest even) moves no value by more
    # than the bound, and some values by exactly that much
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 1.0, 10.0, 1e4)])
    r = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    d = np.abs(r - x)
    hu = half_ulp_bf16(x)
    assert np.all(d <= hu * (1 + 1e-12))
    assert np.max(d / hu) > 0.99


def test_check_close_accepts_rounding_above_8_and_rejects_real_errors():
    ref = np.array([8.0 + 2.0**-5 - 1e-9, 0.5, -3.0])          # just below a bf16 rounding midpoint
    got = torch.tensor(ref).to(torch.bfloat16)                     # stored value moves by ~2^-5
    check_close("rounded", got, ref)
    bad = torch.tensor(ref + np.array([0.0, 0.03, 0.0])).to(torch.bfloat16)
    try:
        check_close("bad", bad, ref)
    except AssertionError:
        return
    raise AssertionError("an error of 0.03 at 0.5 passed")
