"""Device status word: on-device validation of the index contracts
(SCFA_FLAG_VALIDATE) and the pipeline-timeout path (SCFA_FLAG_DEBUG_STALL).

Bad inputs here are made on the host and are still in bounds for every
kernel: they break an ordering contract, not a memory access. The stall
withholds a load so that a wait runs out after its limit (about 1 s); the
test then checks that the status word says so and that a following normal
step on the same device still matches the float64 oracle.
"""
import time

import numpy as np
import pytest
import torch

import synth
from harness import check_close, check_lse
from oracle import pipelines

pytestmark = pytest.mark.gpu

OK, INVALID, TIMEOUT = 0, 1, 5


@pytest.fixture(scope="module")
def scfa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_causal_flash_gb300 import build
    build.build()
    import sparse_causal_flash_gb300 as s
    return s


def qk_case(D=64, seed=120, B=1, H=2, T=900, keep=0.6):
    p = synth.make_problem(synth.Workload("v", "qk", B, H, T, D, seed, p_keep=keep))
    B, H, Tq, _ = p.q.shape
    Tk = p.k.shape[2]
    return p, B, H, Tq, Tk


def qk_forward(scfa, p, q_idx, k_idx, flags):
    B, H, Tq, D = p.q.shape
    Tk = p.k.shape[2]
    o = torch.empty_like(p.q).cuda()
    lse = torch.empty((B, H, Tq), dtype=torch.float32, device="cuda")
    ws = scfa.workspace(scfa.attn_workspace_size(scfa.MODE_QK, 0, B, H, Tq, Tk, D))
    scfa.scfa_qk_fwd(p.q.cuda(), p.k.cuda(), p.v.cuda(), q_idx.cuda(), k_idx.cuda(), p.wl.scale, o, lse, ws, flags)
    return o, lse, scfa.scfa_get_device_status(ws)


def test_validate_accepts_valid_qk_and_changes_nothing(scfa):
    p, *_ = qk_case()
    o0, l0, s0 = qk_forward(scfa, p, p.q_idx, p.k_idx, 0)
    o1, l1, s1 = qk_forward(scfa, p, p.q_idx, p.k_idx, scfa.FLAG_VALIDATE)
    assert s0 == OK and s1 == OK
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_validate_rejects_bad_qk_indices(scfa):
    p, B, H, Tq, Tk = qk_case()
    # positions not ascending in one head
    qi = p.q_idx.clone()
    qi[0, 1, 10], qi[0, 1, 11] = qi[0, 1, 11].item(), qi[0, 1, 10].item()
    assert qk_forward(scfa, p, qi, p.k_idx, scfa.FLAG_VALIDATE)[2] == INVALID
    # a kept key after the padding sentinel
    ki = p.k_idx.clone()
    n = int((ki[0, 0] != synth.K_SENTINEL).sum())
    if n < Tk:
        ki[0, 0, n:] = synth.K_SENTINEL
        ki[0, 0, Tk - 1] = 10**6
        assert qk_forward(scfa, p, p.q_idx, ki, scfa.FLAG_VALIDATE)[2] == INVALID
    # a negative position that is not the query sentinel
    qi = p.q_idx.clone()
    qi[0, 0, 0] = -5
    assert qk_forward(scfa, p, qi, p.k_idx, scfa.FLAG_VALIDATE)[2] == INVALID


def hash_forward(scfa, q_s, k_s, v_s, pq, pk, qh, kh, scale, flags):
    B, H, T, D = q_s.shape
    o = torch.zeros_like(q_s)
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    ws = scfa.workspace(scfa.attn_workspace_size(scfa.MODE_HASH, 0, B, H, T, T, D))
    scfa.scfa_hash_fwd(q_s, k_s, v_s, pq, pk, qh, kh, scale, o, lse, ws, flags)
    return scfa.scfa_get_device_status(ws)


def test_validate_hash_contracts(scfa):
    from sparse_causal_flash_gb300.pipeline import Step
    p = synth.make_problem(synth.Workload("vh", "hash", 1, 2, 700, 64, 121, n_buckets=8))
    st = Step(scfa.MODE_HASH, 1, 2, 700, 700, 64, n_buckets=8, tiled=False)
    st.run(p.q.cuda(), p.k.cuda(), p.v.cuda(), p.do.cuda(), p.wl.scale, R=p.R.cuda())
    torch.cuda.synchronize()
    args = (st.q_s, st.k_s, st.v_s)
    V, OO = scfa.FLAG_VALIDATE, scfa.FLAG_ORIGINAL_ORDER
    assert hash_forward(scfa, *args, st.pq, st.pk, st.qh, st.kh, p.wl.scale, V | OO) == OK
    # bucket ids out of order
    kh = st.kh.clone()
    kh[0, 1, 5] = kh[0, 1, -1] + 1
    assert hash_forward(scfa, *args, st.pq, st.pk, st.qh, kh, p.wl.scale, V) == INVALID
    # the same output row twice under ORIGINAL_ORDER
    pq = st.pq.clone()
    pq[0, 0, 3] = pq[0, 0, 4]
    assert hash_forward(scfa, *args, pq, st.pk, st.qh, st.kh, p.wl.scale, V | OO) == INVALID
    # without ORIGINAL_ORDER repeated positions are allowed
    assert hash_forward(scfa, *args, pq, st.pk, st.qh, st.kh, p.wl.scale, V) == OK


@pytest.mark.parametrize("D", [64, 128])
def test_pipeline_timeout_reports_status_and_device_stays_usable(scfa, D):
    from sparse_causal_flash_gb300.pipeline import Step
    p, B, H, Tq, Tk = qk_case(D=D, seed=130 + D, T=700)
    q, k, v, do = (t.cuda() for t in (p.q, p.k, p.v, p.do))
    qi, ki = p.q_idx.cuda(), p.k_idx.cuda()
    st = Step(scfa.MODE_QK, B, H, Tq, Tk, D)
    ref = pipelines.run_qk(p.q, p.k, p.v, p.do, p.q_idx.numpy(), p.k_idx.numpy(), p.wl.scale)

    def normal_step_matches_oracle():
        st.run(q, k, v, do, p.wl.scale, q_idx=qi, k_idx=ki)
        torch.cuda.synchronize()
        assert scfa.scfa_get_device_status(st.ws_b) == OK
        for (b, h), r in ref.items():
            check_close(f"O[{b},{h}]", st.o[b, h], r["o"])
            check_lse(f"LSE[{b},{h}]", st.lse[b, h], r["lse"])
            check_close(f"dQ[{b},{h}]", st.dq[b, h], r["dq"])
            check_close(f"dK[{b},{h}]", st.dk[b, h], r["dk"])
            check_close(f"dV[{b},{h}]", st.dv[b, h], r["dv"])

    normal_step_matches_oracle()
    # forward whose K / V never arrive: every CTA's wait runs out
    t0 = time.time()
    scfa.scfa_qk_fwd(q, k, v, qi, ki, p.wl.scale, st.o, st.lse, st.ws_b, scfa.FLAG_DEBUG_STALL | scfa.FLAG_KEEP_O32)
    assert scfa.scfa_get_device_status(st.ws_b) == TIMEOUT
    assert time.time() - t0 > 0.5
    normal_step_matches_oracle()
    # backward whose K / V never arrive, after a normal forward
    scfa.scfa_qk_fwd(q, k, v, qi, ki, p.wl.scale, st.o, st.lse, st.ws_b, scfa.FLAG_KEEP_O32)
    scfa.scfa_qk_bwd(q, k, v, st.o, st.lse, do, qi, ki, p.wl.scale, st.dq, st.dk, st.dv, st.ws_b,
                     scfa.FLAG_REUSE_TILES | scfa.FLAG_KEEP_O32 | scfa.FLAG_DEBUG_STALL)
    assert scfa.scfa_get_device_status(st.ws_b) == TIMEOUT
    normal_step_matches_oracle()
