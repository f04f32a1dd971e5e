"""The allocation-free QK-sparse forward, scfa_qk_fwd_noalloc.

It exists for callers that may not call cudaMalloc where they run attention
(servers with one fixed memory pool, plugins whose host framework forbids
allocation inside its callbacks): it takes no
workspace and uses a scratch array compiled into the library. These tests call
it through the C ABI and compare it with scfa_qk_fwd (caller workspace) on two
calls in a row, check that the second takes no device memory (free bytes
unchanged around it), and check that a shape too large for the array is
refused on the host. Collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from harness import check_close, check_lse, to_np


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_causal_flash_gb300 import build
    build.build()
    import sparse_causal_flash_gb300 as scfa
    scfa.load()
    fn = scfa._lib.scfa_qk_fwd_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [P, P, P, P, P, I, I, I, I, I, ctypes.c_float, P, P, P]
    fn.restype = I
    return scfa, fn


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point(lib):
    scfa, fn = lib
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for seed, (B, H, T, keep) in ((51, (2, 3, 1500, 0.7)), (52, (1, 4, 900, 0.4))):
        p = synth.make_problem(synth.Workload("na", "qk", B, H, T, 64, seed, p_keep=keep))
        q, k, v = p.q.cuda(), p.k.cuda(), p.v.cuda()
        qi, ki = p.q_idx.cuda(), p.k_idx.cuda()
        Tq, Tk = q.shape[2], k.shape[2]
        o_ref = torch.empty_like(q)
        lse_ref = torch.empty((B, H, Tq), dtype=torch.float32, device="cuda")
        ws = scfa.workspace(scfa.attn_workspace_size(scfa.MODE_QK, 0, B, H, Tq, Tk, 64))
        scfa.scfa_qk_fwd(q, k, v, qi, ki, p.wl.scale, o_ref, lse_ref, ws)
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, Tq), float("nan"), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        rc = fn(_p(q), _p(k), _p(v), _p(qi), _p(ki), B, H, Tq, Tk, 64, p.wl.scale, _p(o), _p(lse), stream)
        assert rc == 0, scfa.status_string(rc)
        torch.cuda.synchronize()
        if seed == 52:
            # after a first call (which may load kernel code lazily), a call
            # takes no device memory
            assert torch.cuda.mem_get_info()[0] == free0
        # the device status word of the compiled-in scratch: the call's
        # pipeline and list checks passed
        st_fn = scfa._lib.scfa_qk_fwd_noalloc_status
        st_fn.argtypes = [ctypes.c_void_p]
        st_fn.restype = ctypes.c_int
        assert st_fn(stream) == 0
        torch.cuda.synchronize()
        check_close("O noalloc", o, to_np(o_ref))
        check_lse("LSE noalloc", lse, to_np(lse_ref))


@pytest.mark.gpu
def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    scfa, fn = lib
    # 64 x 16 heads of 32k rows need far more tile metadata than the array holds
    assert scfa.attn_workspace_size(scfa.MODE_QK, 0, 64, 16, 32768, 32768, 64) > (16 << 20)
    fake = ctypes.c_void_p(256)
    rc = fn(fake, fake, fake, fake, fake, 64, 16, 32768, 32768, 64, 0.125, fake, fake, None)
    assert rc == 3  # SCFA_ERR_WORKSPACE, refused on the host before any launch
