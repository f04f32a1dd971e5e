"""Pins of the float64 attention oracle against facts other than itself.

Every test here runs on the CPU. The pins: hand-worked fixtures, closed forms
(T = 1, the two-key logistic form, a single admissible key), library routines
(torch scaled_dot_product_attention and autograd in float64), central finite
differences, and the invariants of softmax attention.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

from conftest import golden_value, load_golden
from oracle import attention, pipelines


def _arr(rows):
    return np.array([[golden_value(x) for x in r] for r in rows], dtype=np.float64)


def test_golden_dense_t3():
    g = load_golden("attention_dense_t3_d1.json")
    q, k, v, do = _arr(g["q"]), _arr(g["k"]), _arr(g["v"]), _arr(g["do"])
    mask = attention.mask_dense(3)
    O, lse, dq, dk, dv = attention.backward(q, k, v, do, mask, g["scale"])
    np.testing.assert_allclose(O, _arr(g["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, [golden_value(x) for x in g["lse"]], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, _arr(g["dv"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq, _arr(g["dq"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, _arr(g["dk"]), rtol=0, atol=1e-12)


def test_golden_qk_masked():
    g = load_golden("attention_qk_masked.json")
    mask = attention.mask_qk(g["q_idx"], g["k_idx"])
    np.testing.assert_array_equal(mask, np.array(g["mask"], dtype=bool))
    O, lse, _ = attention.forward(_arr(g["q"]), _arr(g["k"]), _arr(g["v"]), mask, g["scale"])
    np.testing.assert_allclose(O, _arr(g["o"]), rtol=0, atol=1e-12)
    exp_lse = [golden_value(x) for x in g["lse"]]
    assert np.isneginf(lse[2]) and np.isneginf(exp_lse[2])
    np.testing.assert_allclose(lse[:2], exp_lse[:2], rtol=0, atol=1e-12)
    # the padding row and the key after every query get no gradient
    rng = np.random.default_rng(0)
    _, _, dq, dk, dv = attention.backward(_arr(g["q"]), _arr(g["k"]), _arr(g["v"]),
                                          rng.standard_normal((3, 1)), mask, g["scale"])
    assert dq[2, 0] == 0.0 and dk[2, 0] == 0.0 and dv[2, 0] == 0.0


def test_t1_closed_form():
    rng = np.random.default_rng(1)
    q, k, v = (rng.standard_normal((1, 16)) for _ in range(3))
    O, lse, P = attention.forward(q, k, v, attention.mask_dense(1), 0.25)
    np.testing.assert_allclose(O, v, rtol=0, atol=0)
    assert lse[0] == pytest.approx(0.25 * float(q[0] @ k[0]), abs=1e-14)
    assert P[0, 0] == 1.0


def test_two_keys_logistic_form():
    # row 1 of a causal T=2 problem: weight on key 1 is the logistic function of
    # the score difference, O1 = v0 + w (v1 - v0)
    rng = np.random.default_rng(2)
    q, k, v = (rng.standard_normal((2, 8)) for _ in range(3))
    s = 0.3
    O, lse, _ = attention.forward(q, k, v, attention.mask_dense(2), s)
    w = scipy.special.expit(s * q[1] @ (k[1] - k[0]))
    np.testing.assert_allclose(O[1], v[0] + w * (v[1] - v[0]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[1], scipy.special.logsumexp([s * q[1] @ k[0], s * q[1] @ k[1]]), atol=1e-14)


def test_single_admissible_key_copies_value():
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal((4, 8)), rng.standard_normal((5, 8)), rng.standard_normal((5, 8))
    mask = np.zeros((4, 5), dtype=bool)
    for r, c in enumerate([4, 0, 2, 1]):
        mask[r, c] = True
    O, lse, _ = attention.forward(q, k, v, mask, 0.5)
    np.testing.assert_array_equal(O, v[[4, 0, 2, 1]])
    np.testing.assert_allclose(lse, 0.5 * np.einsum("rd,rd->r", q, k[[4, 0, 2, 1]]), atol=1e-14)


def _random_mask(rng, Tq, Tk, p=0.5):
    m = rng.random((Tq, Tk)) < p
    m[0, :] = False  # one empty row
    return m


def test_rows_sum_to_one_and_empty_rows():
    rng = np.random.default_rng(4)
    q, k, v = rng.standard_normal((9, 4)), rng.standard_normal((7, 4)), rng.standard_normal((7, 4))
    mask = _random_mask(rng, 9, 7)
    O, lse, P = attention.forward(q, k, v, mask, 0.7)
    live = mask.any(1)
    np.testing.assert_allclose(P[live].sum(1), 1.0, atol=1e-12)
    assert np.all(P[~mask] == 0)
    assert np.all(O[~live] == 0) and np.all(np.isneginf(lse[~live]))


def _sdpa_reference(q, k, v, do, mask, scale):
    """torch float64 scaled_dot_product_attention + autograd, live rows only."""
    live = mask.any(1)
    qt = torch.tensor(q, requires_grad=True)
    kt = torch.tensor(k, requires_grad=True)
    vt = torch.tensor(v, requires_grad=True)
    m = torch.tensor(mask.copy())
    m[~torch.tensor(live)] = True  # keep SDPA finite on empty rows; they are dropped below
    o = torch.nn.functional.scaled_dot_product_attention(qt[None], kt[None], vt[None], attn_mask=m[None], scale=scale)[0]
    lt = torch.tensor(live)
    (o[lt] * torch.tensor(do)[lt]).sum().backward()
    return o.detach().numpy(), qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy(), live


@pytest.mark.parametrize("seed", [5, 6, 7])
def test_matches_torch_sdpa_and_autograd(seed):
    rng = np.random.default_rng(seed)
    Tq, Tk, D = 13, 11, 8
    q, k, v, do = (rng.standard_normal((Tq if i in (0, 3) else Tk, D)) for i in range(4))
    mask = _random_mask(rng, Tq, Tk, 0.6)
    scale = 1 / math.sqrt(D)
    O, lse, dq, dk, dv = attention.backward(q, k, v, do, mask, scale)
    o_ref, dq_ref, dk_ref, dv_ref, live = _sdpa_reference(q, k, v, do, mask, scale)
    np.testing.assert_allclose(O[live], o_ref[live], atol=1e-12)
    np.testing.assert_allclose(dq, dq_ref, atol=1e-12)
    np.testing.assert_allclose(dk, dk_ref, atol=1e-12)
    np.testing.assert_allclose(dv, dv_ref, atol=1e-12)


def test_dense_causal_matches_sdpa_is_causal():
    rng = np.random.default_rng(8)
    T, D = 17, 16
    q, k, v = (rng.standard_normal((T, D)) for _ in range(3))
    O, _, _ = attention.forward(q, k, v, attention.mask_dense(T), 1 / math.sqrt(D))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q)[None], torch.tensor(k)[None], torch.tensor(v)[None], is_causal=True)[0].numpy()
    np.testing.assert_allclose(O, ref, atol=1e-12)


def test_central_finite_differences():
    rng = np.random.default_rng(9)
    Tq, Tk, D = 5, 6, 3
    q, k, v, do = rng.standard_normal((Tq, D)), rng.standard_normal((Tk, D)), rng.standard_normal((Tk, D)), rng.standard_normal((Tq, D))
    mask = attention.mask_qk([3, 7, 1, -1, 9], [0, 2, 3, 6, 8, 20])
    scale = 0.6

    def loss(q_, k_, v_):
        O, _, _ = attention.forward(q_, k_, v_, mask, scale)
        return float(np.sum(O * do))

    _, _, dq, dk, dv = attention.backward(q, k, v, do, mask, scale)
    eps = 1e-6
    for name, X, G in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name], args_m[name] = Xp, Xm
            num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"]) - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * eps)
        np.testing.assert_allclose(G, num, atol=1e-7, err_msg=name)


def test_gradient_invariants():
    # softmax is shift invariant per row, so sum over keys of dK is zero; every
    # live query distributes exactly its dO over the values
    rng = np.random.default_rng(10)
    Tq, Tk, D = 20, 16, 8
    q, do = rng.standard_normal((Tq, D)), rng.standard_normal((Tq, D))
    k, v = rng.standard_normal((Tk, D)), rng.standard_normal((Tk, D))
    mask = _random_mask(rng, Tq, Tk, 0.4)
    _, _, dq, dk, dv = attention.backward(q, k, v, do, mask, 0.35)
    live = mask.any(1)
    np.testing.assert_allclose(dk.sum(0), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(0), do[live].sum(0), atol=1e-12)
    assert np.all(dq[~live] == 0)


def test_modes_reduce_to_dense():
    # no drop -> QK-sparse equals dense causal; one bucket -> hash equals dense
    rng = np.random.default_rng(11)
    T, D = 40, 8
    x = torch.from_numpy(rng.standard_normal((1, 1, T, D))).to(torch.bfloat16)
    q, k, v, do = x, x.roll(3, dims=2), x.flip(2), x.roll(7, dims=2)
    dense = pipelines.run_dense(q, k, v, do, 0.3)[(0, 0)]
    idx = np.arange(T, dtype=np.int32)[None, None]
    qk = pipelines.run_qk(q, k, v, do, idx, idx, 0.3)[(0, 0)]
    same = np.zeros((1, 1, T), dtype=np.int32)
    hs, _, _ = pipelines.run_hash(q, k, v, do, np.ones((D, 1)), 0.3, q_hash=same, k_hash=same)
    for key in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_array_equal(qk[key], dense[key])
        np.testing.assert_array_equal(hs[(0, 0)][key], dense[key])
    assert dense["pairs"] == T * (T + 1) // 2


def test_hash_mask_sorted_view_is_a_permutation():
    # computing on bucket-sorted rows with original positions, then putting the
    # rows back, equals computing in original order
    rng = np.random.default_rng(12)
    T, D, nb = 50, 8, 4
    q, k, v, do = (rng.standard_normal((T, D)) for _ in range(4))
    qh, kh = rng.integers(0, nb, T), rng.integers(0, nb, T)
    O, lse, dq, dk, dv = attention.backward(q, k, v, do, attention.mask_hash(qh, kh), 0.4)
    pq, pk = np.argsort(qh, kind="stable"), np.argsort(kh, kind="stable")
    ms = attention.mask_hash(qh[pq], kh[pk], q_pos=pq, k_pos=pk)
    Os, lses, dqs, dks, dvs = attention.backward(q[pq], k[pk], v[pk], do[pq], ms, 0.4)
    np.testing.assert_allclose(O[pq], Os, atol=1e-12)
    np.testing.assert_allclose(dq[pq], dqs, atol=1e-12)
    np.testing.assert_allclose(dk[pk], dks, atol=1e-12)
    np.testing.assert_allclose(dv[pk], dvs, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse[pq]), np.isneginf(lses))


def test_bucketwise_hash_equals_whole_problem():
    # the block-diagonal structure of the hash mask: per-bucket subproblems
    # reproduce every row of the full explicit-mask problem
    rng = np.random.default_rng(13)
    T, D, nb = 90, 8, 5
    q, k, v, do = (rng.standard_normal((T, D)) for _ in range(4))
    qh, kh = rng.integers(0, nb, T), rng.integers(0, nb, T)
    O, lse, dq, dk, dv = attention.backward(q, k, v, do, attention.mask_hash(qh, kh), 0.4)
    per = pipelines.run_hash_buckets(q, k, v, do, 0.4, qh, kh, range(nb))
    seen_q, seen_k = [], []
    for c, r in per.items():
        np.testing.assert_allclose(r["o"], O[r["q_pos"]], atol=1e-12)
        np.testing.assert_allclose(r["dq"], dq[r["q_pos"]], atol=1e-12)
        np.testing.assert_allclose(r["dk"], dk[r["k_pos"]], atol=1e-12)
        np.testing.assert_allclose(r["dv"], dv[r["k_pos"]], atol=1e-12)
        np.testing.assert_array_equal(np.isneginf(r["lse"]), np.isneginf(lse[r["q_pos"]]))
        seen_q += list(r["q_pos"])
        seen_k += list(r["k_pos"])
    assert sorted(seen_q) == list(range(T)) and sorted(seen_k) == list(range(T))
