"""GPU parity of every step of the hot path against the float64 oracle.

Index work (LSH bucket ids, sort permutation, sorted ids, bucket offsets,
gathered / unsorted rows, live-tile lists) must be bit-exact; O, dQ, dK, dV
within max abs 2e-2 and relative L2 5e-3; LSE within 2e-3 (and -inf exactly).
Sizes span several 128-row tiles with ragged tails; the full-size workloads
are checked on sampled heads.
"""
import math

import numpy as np
import pytest
import torch

import synth
from harness import check_close, check_lse, to_np
from oracle import attention, coverage, lsh, pipelines, tiles

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def scfa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_causal_flash_gb300 import build
    build.build()
    import sparse_causal_flash_gb300 as s
    return s


def cuda(t):
    return t.contiguous().cuda()


Q_PAD, K_PAD = -1, 2**31 - 1  # positions of padding rows in the tile-aligned layout


def sorted_views(x_hash, nb, Ts=None, pad=Q_PAD):
    """The oracle's sorted view of [B,H,T] bucket ids: the plain stable sort,
    or (Ts given) its tile-aligned layout of Ts rows per head."""
    perm, hs, off = pipelines.hash_sort_view(x_hash, nb)
    if Ts is None:
        return perm, hs, off
    B, H, _ = perm.shape
    out = [np.empty((B, H, Ts), np.int32), np.empty((B, H, Ts), np.int32), np.empty((B, H, nb + 1), np.int32)]
    for b in range(B):
        for h in range(H):
            for a, v in zip(out, lsh.tile_aligned(perm[b, h], off[b, h], Ts, 128, pad)):
                a[b, h] = v
    return tuple(out)


def check_lse_sorted(name, got, ref, perm):
    """LSE in sorted order against the oracle's LSE in original order; rows
    whose perm entry names no token (padding) must be -inf."""
    perm = np.asarray(perm)
    inside = (perm >= 0) & (perm < len(ref))
    m = torch.from_numpy(inside).to(got.device)
    check_lse(name, got[m], np.asarray(ref)[perm[inside]])
    assert bool(torch.all(torch.isneginf(got[~m]))), f"{name}: a padding row is not -inf"


# ------------------------------------------------------------------ LSH + sort
@pytest.mark.parametrize("B,H,T,D,nb", [(1, 2, 512, 64, 4), (2, 3, 1000, 64, 16), (1, 2, 700, 128, 64),
                                        (2, 3, 1000, 64, 32)])
def test_lsh_hash_bitexact(scfa, B, H, T, D, nb):
    x = synth.normal_bf16(77, 1, (B, H, T, D))
    R = synth.rotation_bf16(77, D, nb // 2)
    h = torch.empty((B, H, T), dtype=torch.int32, device="cuda")
    scfa.lsh_hash(cuda(x), cuda(R), nb, h)
    ref = lsh.lsh_hash(x.double().numpy(), R.double().numpy())
    np.testing.assert_array_equal(h.cpu().numpy(), ref)


def test_lsh_hash_exact_ties_and_cancellation(scfa):
    D, m = 64, 4
    rng = np.random.default_rng(5)
    c0 = torch.from_numpy(rng.standard_normal(D)).to(torch.bfloat16)
    R = torch.stack([c0, c0, -c0, torch.zeros(D, dtype=torch.bfloat16)], dim=1)  # ties between columns
    rows = [torch.zeros(D, dtype=torch.bfloat16)]                                   # all candidates 0
    rows += [synth.normal_bf16(9, 1, (D,)) for _ in range(60)]
    big = torch.zeros(D, dtype=torch.bfloat16)                                      # 2^60 + 1 - 2^60
    big[0], big[1], big[2] = 2.0**60, 1.0, -(2.0**60)
    rows.append(big)
    x = torch.stack(rows)[None, None]
    R2 = R.clone()
    R2[:, 3] = torch.ones(D, dtype=torch.bfloat16)
    for RR in (R, R2):
        h = torch.empty((1, 1, x.shape[2]), dtype=torch.int32, device="cuda")
        scfa.lsh_hash(cuda(x), cuda(RR), 2 * m, h)
        ref = lsh.lsh_hash(x.double().numpy(), RR.double().numpy())
        np.testing.assert_array_equal(h.cpu().numpy(), ref)


@pytest.mark.parametrize("D,m", [(64, 8), (64, 16), (128, 16), (128, 256)])
def test_lsh_hash_tensor_core_path_ties_and_edges(scfa, D, m):
    # shapes that take the tensor-core first pass (D 64 / 128, m a multiple of
    # 8): exact column ties, all-zero rows, cancellation beyond fp32, a
    # subnormal entry and huge magnitudes must all come out as the oracle says
    rng = np.random.default_rng(6 + D + m)
    c0 = torch.from_numpy(rng.standard_normal(D)).to(torch.bfloat16)
    cols = [c0, c0, -c0, torch.zeros(D, dtype=torch.bfloat16)]
    cols += [torch.from_numpy(rng.standard_normal(D)).to(torch.bfloat16) for _ in range(m - 4)]
    R = torch.stack(cols, dim=1)
    rows = [torch.zeros(D, dtype=torch.bfloat16)]
    rows += [synth.normal_bf16(10 + D, 1, (D,)) for _ in range(300)]
    big = torch.zeros(D, dtype=torch.bfloat16)
    big[0], big[1], big[2] = 2.0**60, 1.0, -(2.0**60)
    rows.append(big)
    tiny = synth.normal_bf16(11, 1, (D,)).clone()
    tiny[3] = torch.tensor(2.0**-130).to(torch.bfloat16)   # subnormal in bf16
    rows.append(tiny)
    huge = synth.normal_bf16(12, 1, (D,)) * 2.0**100
    rows.append(huge.to(torch.bfloat16))
    x = torch.stack(rows)[None, None]
    h = torch.empty((1, 1, x.shape[2]), dtype=torch.int32, device="cuda")
    scfa.lsh_hash(cuda(x), cuda(R), 2 * m, h)
    ref = lsh.lsh_hash(x.double().numpy(), R.double().numpy())
    np.testing.assert_array_equal(h.cpu().numpy(), ref)


def per_head_hash_ref(x, R):
    """Oracle ids with rotation R[h] for head h (lsh.lsh_hash per head)."""
    return np.concatenate([lsh.lsh_hash(x[:, h:h + 1].double().numpy(), R[h].double().numpy())
                           for h in range(x.shape[1])], axis=1)


@pytest.mark.parametrize("B,H,T,D,nb", [(2, 3, 1000, 64, 16), (1, 2, 700, 128, 64), (2, 2, 300, 32, 8),
                                        (1, 3, 5000, 64, 16), (2, 2, 129, 64, 512)])
def test_lsh_hash_heads_bitexact(scfa, B, H, T, D, nb):
    # one rotation per head: tensor-core path (D 64 / 128), CUDA-core path
    # (D 32), heads of several tiles with a ragged last one, m = 256
    x = synth.normal_bf16(93, 1, (B, H, T, D))
    R = synth.normal_bf16(93, 7, (H, D, nb // 2))
    h = torch.empty((B, H, T), dtype=torch.int32, device="cuda")
    scfa.lsh_hash_heads(cuda(x), cuda(R), nb, h)
    np.testing.assert_array_equal(h.cpu().numpy(), per_head_hash_ref(x, R))
    # a rotation per head is not the shared rotation: head 1 differs from
    # hashing it with head 0's rotation
    h0 = lsh.lsh_hash(x[:, 1:2].double().numpy(), R[0].double().numpy())
    assert not np.array_equal(h.cpu().numpy()[:, 1:2], h0)


@pytest.mark.parametrize("tiled", [False, True])
def test_hash_parity_per_head_r(scfa, tiled):
    """The hash step with one rotation per head against the oracle's
    hash-sparse attention on the per-head ids."""
    from sparse_causal_flash_gb300.pipeline import Step
    B, H, T, D, nb = 1, 3, 1100, 64, 8
    p = synth.make_problem(synth.Workload("hr", "hash", B, H, T, D, 94, n_buckets=nb))
    R = synth.normal_bf16(94, 7, (H, D, nb // 2))
    st = Step(scfa.MODE_HASH, B, H, T, T, D, n_buckets=nb, tiled=tiled, per_head_r=True)
    st.run(cuda(p.q), cuda(p.k), cuda(p.v), cuda(p.do), p.wl.scale, R=cuda(R))
    torch.cuda.synchronize()
    assert scfa.scfa_get_device_status(st.ws_b) == 0
    qh = per_head_hash_ref(p.q, R)
    kh = per_head_hash_ref(p.k, R)
    pq, _, _ = sorted_views(qh, nb, st.Ts if tiled else None, Q_PAD)
    np.testing.assert_array_equal(st.pq.cpu().numpy(), pq)
    ref, _, _ = pipelines.run_hash(p.q, p.k, p.v, p.do, p.R, p.wl.scale, q_hash=qh, k_hash=kh)
    compare_heads(st, ref, ref.keys(), lse_perm=pq)


@pytest.mark.parametrize("D,m,T", [(64, 8, 3001), (128, 64, 500)])
def test_lsh_hash_every_row_certified(scfa, D, m, T):
    # every column of R appears twice, once negated: each row's top value is
    # an exact tie, so every row goes through the certified second pass with
    # several candidates; spread over many warps and CTAs
    half = synth.rotation_bf16(91, D, m // 2)
    R = torch.cat([half, -half.flip(1)], dim=1)
    x = synth.normal_bf16(92, 1, (1, 2, T, D))
    h = torch.empty((1, 2, T), dtype=torch.int32, device="cuda")
    scfa.lsh_hash(cuda(x), cuda(R), 2 * m, h)
    ref = lsh.lsh_hash(x.double().numpy(), R.double().numpy())
    np.testing.assert_array_equal(h.cpu().numpy(), ref)


@pytest.mark.parametrize("B,H,T,D,nb", [(1, 2, 512, 64, 4), (2, 3, 1000, 64, 16), (1, 1, 5000, 64, 512),
                                        (1, 2, 20000, 64, 64), (1, 1, 40000, 128, 512)])
def test_bucket_sort_and_gather_bitexact(scfa, B, H, T, D, nb):
    x = synth.normal_bf16(78, 2, (B, H, T, D))
    R = synth.rotation_bf16(78, D, nb // 2)
    dev = dict(dtype=torch.int32, device="cuda")
    hs = torch.empty((B, H, T), **dev)
    perm = torch.empty((B, H, T), **dev)
    off = torch.empty((B, H, nb + 1), **dev)
    xs = torch.empty((B, H, T, D), dtype=torch.bfloat16, device="cuda")
    ws = scfa.workspace(scfa.lsh_workspace_size(B, H, T, nb))
    scfa.lsh_bucket_sort(cuda(x), cuda(R), nb, hs, perm, off, xs, ws)
    href = lsh.lsh_hash(x.double().numpy(), R.double().numpy())
    pr, hr, orf = pipelines.hash_sort_view(href, nb)
    np.testing.assert_array_equal(perm.cpu().numpy(), pr)
    np.testing.assert_array_equal(hs.cpu().numpy(), hr)
    np.testing.assert_array_equal(off.cpu().numpy(), orf)
    xs_ref = torch.stack([torch.stack([x[b, h][torch.from_numpy(pr[b, h]).long()] for h in range(H)]) for b in range(B)])
    assert torch.equal(xs.cpu().view(torch.int16), xs_ref.view(torch.int16))
    # unsort puts every row back, bit for bit
    back = torch.empty_like(xs)
    scfa.lsh_unsort(xs, perm, back)
    assert torch.equal(back.cpu().view(torch.int16), x.view(torch.int16))
    g = torch.empty_like(xs)
    scfa.lsh_gather(cuda(x), perm, g)
    assert torch.equal(g.cpu().view(torch.int16), xs_ref.view(torch.int16))


@pytest.mark.parametrize("B,H,T,D,nb", [(1, 2, 512, 64, 4), (2, 3, 1000, 64, 16), (1, 1, 5000, 64, 512),
                                        (1, 2, 20000, 64, 64), (1, 1, 3000, 128, 32), (1, 1, 130, 64, 256)])
def test_bucket_sort_tiled_bitexact(scfa, B, H, T, D, nb):
    """lsh_bucket_sort_tiled: perm, bucket ids, bucket starts and gathered rows
    bit for bit against the oracle's tile-aligned view of its own sort, for
    queries (padding position -1) and keys (padding position INT32_MAX);
    padding rows are zero, and unsort puts every real row back."""
    x = synth.normal_bf16(79, 2, (B, H, T, D))
    R = synth.rotation_bf16(79, D, nb // 2)
    Ts = scfa.scfa_tiled_rows(T, nb)
    assert Ts % 128 == 0 and Ts >= T
    href = lsh.lsh_hash(x.double().numpy(), R.double().numpy())
    ws = scfa.workspace(scfa.lsh_workspace_size(B, H, T, nb))
    dev = dict(dtype=torch.int32, device="cuda")
    for pad in (Q_PAD, K_PAD):
        hs = torch.empty((B, H, Ts), **dev)
        perm = torch.empty((B, H, Ts), **dev)
        start = torch.empty((B, H, nb + 1), **dev)
        xs = torch.full((B, H, Ts, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        scfa.lsh_bucket_sort_tiled(cuda(x), cuda(R), nb, pad, hs, perm, start, xs, ws)
        pr, hr, sr = sorted_views(href, nb, Ts, pad)
        np.testing.assert_array_equal(perm.cpu().numpy(), pr)
        np.testing.assert_array_equal(hs.cpu().numpy(), hr)
        np.testing.assert_array_equal(start.cpu().numpy(), sr)
        xs_ref = np.stack([np.stack([lsh.gather_rows_padded(x[b, h].view(torch.int16).numpy(), pr[b, h])
                                     for h in range(H)]) for b in range(B)])
        np.testing.assert_array_equal(xs.cpu().view(torch.int16).numpy(), xs_ref)
        back = torch.zeros_like(cuda(x))
        scfa.lsh_unsort(xs, perm, back)
        assert torch.equal(back.cpu().view(torch.int16), x.view(torch.int16))
        g = torch.full_like(xs, float("nan"))
        scfa.lsh_gather(cuda(x), perm, g)
        assert torch.equal(g.view(torch.int16), xs.view(torch.int16))


# ------------------------------------------------------------------ tiles
def read_tiles(scfa, ws, mode, B, H, Tq, Tk, D):
    tv = scfa.scfa_tile_view_get(ws, mode, B, H, Tq, Tk, D)
    base = ws.data_ptr()
    nq, nk = B * H * tv.n_q_tiles, B * H * tv.n_k_tiles

    def arr(ptr, n, dt):
        off = ptr - base
        size = np.dtype(dt).itemsize
        return ws[off:off + n * size].cpu().numpy().view(dt).copy()

    torch.cuda.synchronize()
    row_ptr = arr(tv.row_ptr, nq + 1, np.int32)
    csc_ptr = arr(tv.csc_ptr, nk + 1, np.int32)
    nl = int(row_ptr[-1])
    return {
        "row_ptr": row_ptr, "cols": arr(tv.cols, nl, np.int32), "fflags": arr(tv.fflags, nl, np.uint8),
        "csc_ptr": csc_ptr, "csc_rows": arr(tv.csc_rows, int(csc_ptr[-1]), np.int32),
        "cflags": arr(tv.cflags, int(csc_ptr[-1]), np.uint8),
        "work_fwd": arr(tv.work_fwd, nq, np.int32), "work_bwd": arr(tv.work_bwd, nk, np.int32),
        "pair_count": arr(tv.pair_count, B * H * ((tv.n_q_tiles + 1) // 2), np.int32),
        "pair_list": arr(tv.pair_list, nl, np.int32),
        "work_pairs": arr(tv.work_pairs, B * H * ((tv.n_q_tiles + 1) // 2), np.int32),
        "nQt": tv.n_q_tiles,
    }


def expected_pairs(ref, nQt):
    """Union lists of query-tile pairs (2m, 2m + 1), merged from the oracle's
    CSR rows, with their sizes."""
    row_ptr, cols, ff = ref["row_ptr"], ref["cols"], ref["fflags"]
    BH = (len(row_ptr) - 1) // nQt
    nP = (nQt + 1) // 2
    counts, lists = [], {}
    for bh in range(BH):
        for m in range(nP):
            ent = {}
            for g in range(2):
                i = 2 * m + g
                if i >= nQt:
                    continue
                r = bh * nQt + i
                for c, f in zip(cols[row_ptr[r]:row_ptr[r + 1]], ff[row_ptr[r]:row_ptr[r + 1]]):
                    ent[int(c)] = ent.get(int(c), 0) | ((1 | (2 if f & 1 else 0)) << (2 * g))
            lists[bh * nP + m] = [(c << 4) | b for c, b in sorted(ent.items())]
            counts.append(len(ent))
    return np.array(counts, np.int32), lists


def check_work_order(name, got, counts):
    """A work list hands out every tile id once, either by live count
    descending then id ascending, or in natural id order (include/scfa.h
    documents when each is taken; the order is a scheduling choice, so only
    these properties are checked)."""
    n = len(counts)
    np.testing.assert_array_equal(np.sort(got), np.arange(n), err_msg=f"{name}: not a permutation of the tile ids")
    if not np.array_equal(got, np.arange(n)):
        np.testing.assert_array_equal(got, tiles.work_order(counts), err_msg=name)


def compare_tiles(got, ref):
    for key in ("row_ptr", "cols", "fflags", "csc_ptr", "csc_rows", "cflags"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    check_work_order("work_fwd", got["work_fwd"], np.diff(ref["row_ptr"]))
    check_work_order("work_bwd", got["work_bwd"], np.diff(ref["csc_ptr"]))
    nQt = got["nQt"]
    counts, lists = expected_pairs(ref, nQt)
    np.testing.assert_array_equal(got["pair_count"], counts, err_msg="pair_count")
    check_work_order("work_pairs", got["work_pairs"], counts)
    nP = (nQt + 1) // 2
    for pid, want in lists.items():
        start = ref["row_ptr"][(pid // nP) * nQt + 2 * (pid % nP)]
        np.testing.assert_array_equal(got["pair_list"][start:start + len(want)], want, err_msg=f"pair_list {pid}")


@pytest.mark.parametrize("T,keep", [(1000, 0.7), (3000, 0.3), (8192, 0.7)])
def test_tiles_qk_bitexact(scfa, T, keep):
    wl = synth.Workload("t", "qk", 2, 3, T, 64, 91, p_keep=keep)
    p = synth.make_problem(wl)
    B, H, Tq, _ = p.q.shape
    Tk = p.k.shape[2]
    ws = scfa.workspace(scfa.attn_workspace_size(scfa.MODE_QK, 1, B, H, Tq, Tk, 64))
    scfa.scfa_tiles(scfa.MODE_QK, cuda(p.q_idx), cuda(p.k_idx), None, None, B, H, Tq, Tk, 64, ws)
    got = read_tiles(scfa, ws, scfa.MODE_QK, B, H, Tq, Tk, 64)
    compare_tiles(got, tiles.live_list("qk", B, H, Tq, Tk, p.q_idx.numpy(), p.k_idx.numpy()))


@pytest.mark.parametrize("T,nb", [(512, 4), (1000, 8), (8192, 16)])
def test_tiles_hash_bitexact(scfa, T, nb):
    rng = np.random.default_rng(T + nb)
    B, H = 2, 2
    qh = rng.integers(0, nb, (B, H, T))
    kh = rng.integers(0, nb, (B, H, T))
    pq, qs, _ = pipelines.hash_sort_view(qh, nb)
    pk, ks, _ = pipelines.hash_sort_view(kh, nb)
    ws = scfa.workspace(scfa.attn_workspace_size(scfa.MODE_HASH, 1, B, H, T, T, 64))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    scfa.scfa_tiles(scfa.MODE_HASH, t(pq), t(pk), t(qs), t(ks), B, H, T, T, 64, ws)
    got = read_tiles(scfa, ws, scfa.MODE_HASH, B, H, T, T, 64)
    compare_tiles(got, tiles.live_list("hash", B, H, T, T, pq, pk, qs, ks))


def test_tiles_natural_order(scfa):
    # 4096 key tiles that each see one query tile (buckets of exactly 128
    # rows): the live list is checked bit for bit, and the key-tile work list
    # takes the natural order that include/scfa.h documents for lists whose
    # summed live counts reach 4096 times their largest count
    B, H, T = 1, 4, 131072
    pos = np.broadcast_to(np.arange(T, dtype=np.int32), (B, H, T))
    qs = np.broadcast_to((np.arange(T) // 128).astype(np.int32), (B, H, T))
    ks = np.broadcast_to((np.arange(T) // 128).astype(np.int32), (B, H, T))
    ws = scfa.workspace(scfa.attn_workspace_size(scfa.MODE_HASH, 1, B, H, T, T, 64))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    scfa.scfa_tiles(scfa.MODE_HASH, t(pos), t(pos), t(qs), t(ks), B, H, T, T, 64, ws)
    got = read_tiles(scfa, ws, scfa.MODE_HASH, B, H, T, T, 64)
    ref = tiles.live_list("hash", B, H, T, T, pos, pos, qs, ks)
    compare_tiles(got, ref)
    np.testing.assert_array_equal(got["work_bwd"], np.arange(B * H * (T // 128)))


def test_live_sized_workspace(scfa):
    """Lists sized for the live count (scfa_tiles_count +
    scfa_attn_workspace_size_live) give the same lists and the same results
    as the worst-case workspace; one entry short, every list stays empty and
    the status word says SCFA_ERR_WORKSPACE."""
    B, H, T, D, nb = 1, 3, 3000, 64, 8
    p = synth.make_problem(synth.Workload("ls", "hash", B, H, T, D, 150, n_buckets=nb))
    from sparse_causal_flash_gb300.pipeline import Step
    st = Step(scfa.MODE_HASH, B, H, T, T, D, n_buckets=nb, gather=False)  # sorted copies of all four
    st.run(p.q.cuda(), p.k.cuda(), p.v.cuda(), p.do.cuda(), p.wl.scale, R=p.R.cuda())
    Ts = st.Ts  # rows of the sorted (tile-aligned) tensors
    n_live = torch.zeros(1, dtype=torch.int32, device="cuda")
    wc = scfa.workspace(scfa.attn_workspace_size_live(scfa.MODE_HASH, 0, B, H, Ts, Ts, D, 0))
    scfa.scfa_tiles_count(scfa.MODE_HASH, st.pq, st.pk, st.qh, st.kh, B, H, Ts, Ts, wc, n_live)
    torch.cuda.synchronize()
    nl = int(n_live.item())
    ref = tiles.live_list("hash", B, H, Ts, Ts, st.pq.cpu().numpy(), st.pk.cpu().numpy(), st.qh.cpu().numpy(),
                          st.kh.cpu().numpy())
    assert nl == int(ref["row_ptr"][-1])
    worst = scfa.attn_workspace_size(scfa.MODE_HASH, 1, B, H, Ts, Ts, D)
    live = scfa.attn_workspace_size_live(scfa.MODE_HASH, 1, B, H, Ts, Ts, D, nl)
    assert live < worst
    e = lambda: torch.empty((B, H, T, D), dtype=torch.bfloat16, device="cuda")
    flags = scfa.FLAG_ORIGINAL_ORDER | scfa.FLAG_KEEP_O32
    outs = {}
    # one byte short of the live size holds fewer than nl entries
    assert scfa.attn_workspace_capacity(scfa.MODE_HASH, 1, B, H, Ts, Ts, D, live - 1) < nl
    for name, size in (("worst", worst), ("live", live), ("short", live - 1)):
        ws = scfa.workspace(size)
        o, dq, dk, dv = e(), e(), e(), e()
        lse = torch.empty((B, H, Ts), dtype=torch.float32, device="cuda")
        scfa.scfa_hash_fwd(st.q_s, st.k_s, st.v_s, st.pq, st.pk, st.qh, st.kh, p.wl.scale, o, lse, ws, flags)
        scfa.scfa_hash_bwd(st.q_s, st.k_s, st.v_s, o, lse, st.do_s, st.pq, st.pk, st.qh, st.kh, p.wl.scale,
                           dq, dk, dv, ws, flags | scfa.FLAG_REUSE_TILES)
        torch.cuda.synchronize()
        outs[name] = (scfa.scfa_get_device_status(ws), o, lse, dk, dv, ws)
    assert outs["worst"][0] == 0 and outs["live"][0] == 0
    got = read_tiles(scfa, outs["live"][5], scfa.MODE_HASH, B, H, Ts, Ts, D)
    for key in ("row_ptr", "cols", "fflags", "csc_ptr", "csc_rows", "cflags"):  # (no pair lists at D = 64)
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    for i, name in ((1, "O"), (2, "LSE"), (3, "dK"), (4, "dV")):
        assert torch.equal(outs["worst"][i], outs["live"][i]), name
    assert outs["short"][0] == 3  # SCFA_ERR_WORKSPACE
    tv = read_tiles(scfa, outs["short"][5], scfa.MODE_HASH, B, H, Ts, Ts, D)
    assert not tv["row_ptr"].any() and not tv["csc_ptr"].any()


@pytest.mark.parametrize("T", [1, 130, 1000])
def test_tiles_dense_bitexact(scfa, T):
    ws = scfa.workspace(scfa.attn_workspace_size(scfa.MODE_DENSE, 1, 1, 2, T, T, 64))
    scfa.scfa_tiles(scfa.MODE_DENSE, None, None, None, None, 1, 2, T, T, 64, ws)
    got = read_tiles(scfa, ws, scfa.MODE_DENSE, 1, 2, T, T, 64)
    compare_tiles(got, tiles.live_list("dense", 1, 2, T, T))


# ------------------------------------------------------------------ pair counts
def device_count(scfa, mode, q_idx, k_idx, q_hash, k_hash, B, H, Tq, Tk, ws):
    c = torch.zeros(1, dtype=torch.int64, device="cuda")
    scfa.scfa_count_pairs(mode, q_idx, k_idx, q_hash, k_hash, B, H, Tq, Tk, 64, ws, c)
    torch.cuda.synchronize()
    return int(c.item())


@pytest.mark.parametrize("mode,T,arg", [("qk", 3000, 0.6), ("qk", 1000, 0.2), ("hash", 2000, 8), ("hash", 700, 1),
                                        ("dense", 700, None), ("dense", 1, None)])
def test_count_pairs_equals_all_admissible_pairs(scfa, mode, T, arg):
    """The on-device count of admissible pairs inside the live tiles equals
    the oracle's count over the whole explicit mask (the page's 100%
    coverage), exactly."""
    B, H = 2, 3
    t32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    if mode == "qk":
        p = synth.make_problem(synth.Workload("c", "qk", B, H, T, 64, 80, p_keep=arg))
        qi, ki = p.q_idx.numpy(), p.k_idx.numpy()
        Tq, Tk = qi.shape[2], ki.shape[2]
        args = (scfa.MODE_QK, t32(qi), t32(ki), None, None)
        want = sum(attention.admissible_pairs(attention.mask_qk(qi[b, h], ki[b, h])) for b in range(B) for h in range(H))
    elif mode == "hash":
        rng = np.random.default_rng(T + arg)
        pq, qs, _ = pipelines.hash_sort_view(rng.integers(0, arg, (B, H, T)), arg)
        pk, ks, _ = pipelines.hash_sort_view(rng.integers(0, arg, (B, H, T)), arg)
        Tq = Tk = T
        args = (scfa.MODE_HASH, t32(pq), t32(pk), t32(qs), t32(ks))
        want = sum(attention.admissible_pairs(attention.mask_hash(qs[b, h], ks[b, h], q_pos=pq[b, h], k_pos=pk[b, h]))
                   for b in range(B) for h in range(H))
    else:
        Tq = Tk = T
        args = (scfa.MODE_DENSE, None, None, None, None)
        want = B * H * attention.admissible_pairs(attention.mask_dense(T))
    ws = scfa.workspace(scfa.attn_workspace_size(args[0], 1, B, H, Tq, Tk, 64))
    scfa.scfa_tiles(*args, B, H, Tq, Tk, 64, ws)
    assert device_count(scfa, *args, B, H, Tq, Tk, ws) == want


@pytest.mark.parametrize("chunk", [32, 128, 300, 2048])
def test_count_chunked_pairs_bitexact(scfa, chunk):
    """Reformer-style chunk coverage on the bucket-sorted rows, counted on the
    device, equals the oracle's count for every head."""
    B, H, T, nb = 2, 2, 2000, 8
    rng = np.random.default_rng(90 + chunk)
    pq, qs, _ = pipelines.hash_sort_view(rng.integers(0, nb, (B, H, T)), nb)
    pk, ks, _ = pipelines.hash_sort_view(rng.integers(0, nb, (B, H, T)), nb)
    t32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    c = torch.zeros(1, dtype=torch.int64, device="cuda")
    scfa.scfa_count_chunked_pairs(t32(pq), t32(pk), t32(qs), t32(ks), chunk, c)
    torch.cuda.synchronize()
    want = sum(coverage.chunked_pairs(qs[b, h], ks[b, h], pq[b, h], pk[b, h], chunk) for b in range(B) for h in range(H))
    assert int(c.item()) == want


# ------------------------------------------------------------------ attention
def run_step(scfa, p, mode, flags=0, tiled=False, gather=False, shared_qk=False):
    from sparse_causal_flash_gb300.pipeline import Step
    B, H, Tq, D = p.q.shape
    Tk = p.k.shape[2]
    st = Step(mode, B, H, Tq, Tk, D, n_buckets=p.wl.n_buckets, flags=flags, tiled=tiled, gather=gather,
              shared_qk=shared_qk)
    st.run(cuda(p.q), cuda(p.k), cuda(p.v), cuda(p.do), p.wl.scale,
           q_idx=None if p.q_idx is None else cuda(p.q_idx), k_idx=None if p.k_idx is None else cuda(p.k_idx),
           R=None if p.R is None else cuda(p.R))
    torch.cuda.synchronize()
    assert scfa.STATUS.get(scfa.scfa_get_device_status(st.ws_b)) == "ok"
    return st


def compare_heads(st, ref, heads, lse_perm=None):
    for (b, h) in heads:
        r = ref[(b, h)]
        check_close(f"O[{b},{h}]", st.o[b, h], r["o"])
        if lse_perm is None:
            check_lse(f"LSE[{b},{h}]", st.lse[b, h], r["lse"])
        else:
            check_lse_sorted(f"LSE[{b},{h}]", st.lse[b, h], r["lse"], lse_perm[b, h])
        check_close(f"dQ[{b},{h}]", st.dq[b, h], r["dq"])
        check_close(f"dK[{b},{h}]", st.dk[b, h], r["dk"])
        check_close(f"dV[{b},{h}]", st.dv[b, h], r["dv"])


@pytest.mark.parametrize("B,H,T,D,keep,seed", [(2, 3, 1000, 64, 0.7, 11), (1, 2, 2000, 64, 0.3, 12),
                                               (1, 2, 300, 64, 0.9, 13), (1, 3, 1100, 128, 0.6, 14)])
def test_qk_parity(scfa, B, H, T, D, keep, seed):
    p = synth.make_problem(synth.Workload("qk", "qk", B, H, T, D, seed, p_keep=keep))
    st = run_step(scfa, p, scfa.MODE_QK)
    ref = pipelines.run_qk(p.q, p.k, p.v, p.do, p.q_idx.numpy(), p.k_idx.numpy(), p.wl.scale)
    compare_heads(st, ref, ref.keys())


@pytest.mark.parametrize("B,H,T,D,nb,seed", [(1, 2, 512, 64, 4, 1001), (1, 2, 1000, 64, 8, 21),
                                             (2, 1, 1500, 64, 2, 22), (1, 2, 1300, 128, 8, 23)])
def test_hash_parity(scfa, B, H, T, D, nb, seed):
    p = synth.make_problem(synth.Workload("h", "hash", B, H, T, D, seed, n_buckets=nb))
    st = run_step(scfa, p, scfa.MODE_HASH)
    ref, qh, kh = pipelines.run_hash(p.q, p.k, p.v, p.do, p.R, p.wl.scale)
    pq, _, _ = pipelines.hash_sort_view(qh, nb)
    compare_heads(st, ref, ref.keys(), lse_perm=pq)


@pytest.mark.parametrize("B,H,T,D,nb,seed", [(1, 2, 512, 64, 4, 1001), (1, 2, 1000, 64, 8, 21),
                                             (1, 1, 1000, 64, 64, 24), (1, 2, 1300, 128, 8, 23)])
def test_hash_parity_tiled(scfa, B, H, T, D, nb, seed):
    """The hash step on the tile-aligned sorted layout (padding rows between
    buckets): results in original order within tolerance, LSE in the padded
    sorted order (padding rows -inf), and the live-tile lists of the padded
    index arrays bit for bit."""
    p = synth.make_problem(synth.Workload("ht", "hash", B, H, T, D, seed, n_buckets=nb))
    st = run_step(scfa, p, scfa.MODE_HASH, tiled=True)
    assert st.Ts == scfa.scfa_tiled_rows(T, nb) and st.q_s.shape[2] == st.Ts
    ref, qh, kh = pipelines.run_hash(p.q, p.k, p.v, p.do, p.R, p.wl.scale)
    pq, qs, _ = sorted_views(qh, nb, st.Ts, Q_PAD)
    pk, ks, _ = sorted_views(kh, nb, st.Ts, K_PAD)
    np.testing.assert_array_equal(st.pq.cpu().numpy(), pq)
    np.testing.assert_array_equal(st.pk.cpu().numpy(), pk)
    compare_heads(st, ref, ref.keys(), lse_perm=pq)
    got = read_tiles(scfa, st.ws_b, scfa.MODE_HASH, B, H, st.Ts, st.Ts, D)
    want = tiles.live_list("hash", B, H, st.Ts, st.Ts, pq, pk, qs, ks)
    for key in ("row_ptr", "cols", "fflags", "csc_ptr", "csc_rows", "cflags"):
        np.testing.assert_array_equal(got[key], want[key], err_msg=key)


@pytest.mark.parametrize("tiled,gather", [(False, True), (True, True), (True, "q"), (True, "kv"), (False, "q")])
@pytest.mark.parametrize("B,H,T,D,nb,seed", [(1, 2, 1000, 64, 8, 21), (2, 1, 1500, 64, 2, 22),
                                             (1, 1, 1000, 64, 64, 24), (1, 2, 1300, 128, 8, 23),
                                             (1, 1, 77, 64, 4, 25)])
def test_hash_parity_gather(scfa, B, H, T, D, nb, seed, tiled, gather):
    """Row gathers inside the attention kernels (SCFA_FLAG_GATHER_Q: q, dO;
    SCFA_FLAG_GATHER_KV: k, v; read in original order through the sort's
    permutations): results within tolerance of the oracle, and equal to
    those of the step that materialises the sorted copies (padding rows are
    masked either way)."""
    p = synth.make_problem(synth.Workload("hg", "hash", B, H, T, D, seed, n_buckets=nb))
    st = run_step(scfa, p, scfa.MODE_HASH, tiled=tiled, gather=gather)
    assert (st.q_s is None) == (gather in (True, "q")) and (st.k_s is None) == (gather in (True, "kv"))
    ref, qh, kh = pipelines.run_hash(p.q, p.k, p.v, p.do, p.R, p.wl.scale)
    pq, _, _ = sorted_views(qh, nb, st.Ts if tiled else None, Q_PAD)
    np.testing.assert_array_equal(st.pq.cpu().numpy(), pq)
    compare_heads(st, ref, ref.keys(), lse_perm=pq)
    st0 = run_step(scfa, p, scfa.MODE_HASH, tiled=tiled, gather=False)
    for name in ("o", "lse", "dk", "dv"):
        a, b = getattr(st, name), getattr(st0, name)
        assert torch.equal(a, b), f"{name}: gathered rows differ from the sorted copies"
    # dQ sums the key tiles' contributions with fp32 reduce-adds in schedule order
    check_close("dQ gathered vs copies", st.dq, to_np(st0.dq), atol=1e-2, rel_l2=2e-3)


@pytest.mark.parametrize("D", [64, 128])
def test_hash_shared_qk_gather(scfa, D):
    """Shared-QK hashing with row gathers equals the same step on sorted copies."""
    p = synth.make_problem(synth.Workload("hsg", "hash", 1, 2, 900, D, 26, n_buckets=8))
    st = run_step(scfa, p, scfa.MODE_HASH, tiled=True, gather=True, shared_qk=True)
    st0 = run_step(scfa, p, scfa.MODE_HASH, tiled=True, gather=False, shared_qk=True)
    for name in ("o", "lse", "dk", "dv"):
        assert torch.equal(getattr(st, name), getattr(st0, name)), name
    check_close("dQ gathered vs copies", st.dq, to_np(st0.dq), atol=1e-2, rel_l2=2e-3)


@pytest.mark.parametrize("D", [64, 128])
def test_hash_sorted_order_entry_points(scfa, D):
    """The hash step writes O / dQ / dK / dV in original order from inside the
    kernels; the same entry points without SCFA_FLAG_ORIGINAL_ORDER keep every
    row tensor in sorted order, and lsh_unsort then gives the same results.
    With 8 buckets some dV entries pass 8 in magnitude, where the bf16
    rounding of the stored value is part of the tolerance (tests/harness.py)."""
    nb = 8
    p = synth.make_problem(synth.Workload("hs", "hash", 1, 2, 900, D, 31 + D, n_buckets=nb))
    st = run_step(scfa, p, scfa.MODE_HASH)
    B, H, T, _ = p.q.shape
    e = lambda: torch.empty((B, H, T, D), dtype=torch.bfloat16, device="cuda")
    o_s, dq_s, dk_s, dv_s = e(), e(), e(), e()
    lse_s = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    ws = scfa.workspace(scfa.attn_workspace_size(scfa.MODE_HASH, 1, B, H, T, T, D))
    k32 = scfa.FLAG_KEEP_O32
    scfa.scfa_hash_fwd(st.q_s, st.k_s, st.v_s, st.pq, st.pk, st.qh, st.kh, p.wl.scale, o_s, lse_s, ws, k32)
    scfa.scfa_hash_bwd(st.q_s, st.k_s, st.v_s, o_s, lse_s, st.do_s, st.pq, st.pk, st.qh, st.kh, p.wl.scale,
                       dq_s, dk_s, dv_s, ws, scfa.FLAG_REUSE_TILES | k32)
    back = {}
    for name, y_s, perm in (("o", o_s, st.pq), ("dq", dq_s, st.pq), ("dk", dk_s, st.pk), ("dv", dv_s, st.pk)):
        back[name] = e()
        scfa.lsh_unsort(y_s, perm, back[name])
    torch.cuda.synchronize()
    assert torch.equal(lse_s, st.lse)
    assert torch.equal(back["o"].view(torch.int16), st.o.view(torch.int16))  # the forward is deterministic
    ref, qh, _ = pipelines.run_hash(p.q, p.k, p.v, p.do, p.R, p.wl.scale)
    for (b, h), r in ref.items():
        for key in ("o", "dq", "dk", "dv"):
            check_close(f"sorted-order {key}[{b},{h}]", back[key][b, h], r[key])


@pytest.mark.parametrize("D", [64, 128])
def test_original_order_skips_rows_outside_range(scfa, D):
    """SCFA_FLAG_ORIGINAL_ORDER: a sorted row whose index lies outside [0, T)
    is neither written nor read. Such a query (index -1) sees no key and such
    a key (index T) is seen by no query. Outputs start as NaN: the original
    rows that no sorted row maps to must stay NaN, every other row must match
    the oracle evaluated in sorted order with the same indices."""
    B, H, T, nb = 1, 2, 300, 4
    p = synth.make_problem(synth.Workload("oo", "hash", B, H, T, D, 61 + D, n_buckets=nb))
    st = run_step(scfa, p, scfa.MODE_HASH)  # the sorted views of this problem
    pq, pk = st.pq.cpu().numpy().copy(), st.pk.cpu().numpy().copy()
    rng = np.random.default_rng(D)
    for h in range(H):
        pq[0, h, rng.choice(T, 5, replace=False)] = -1
        pk[0, h, rng.choice(T, 5, replace=False)] = T
    t32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    gpq, gpk = t32(pq), t32(pk)
    nan = lambda: torch.full((B, H, T, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    o, dq, dk, dv = nan(), nan(), nan(), nan()
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    ws = scfa.workspace(scfa.attn_workspace_size(scfa.MODE_HASH, 1, B, H, T, T, D))
    oo = scfa.FLAG_ORIGINAL_ORDER | scfa.FLAG_KEEP_O32
    scfa.scfa_hash_fwd(st.q_s, st.k_s, st.v_s, gpq, gpk, st.qh, st.kh, p.wl.scale, o, lse, ws, oo)
    scfa.scfa_hash_bwd(st.q_s, st.k_s, st.v_s, o, lse, st.do_s, gpq, gpk, st.qh, st.kh, p.wl.scale,
                       dq, dk, dv, ws, oo | scfa.FLAG_REUSE_TILES)
    torch.cuda.synchronize()
    assert scfa.scfa_get_device_status(ws) == 0
    qh, kh = st.qh.cpu().numpy(), st.kh.cpu().numpy()
    f64 = lambda t: t.cpu().double().numpy()
    for h in range(H):
        mask = attention.mask_hash(qh[0, h], kh[0, h], q_pos=pq[0, h], k_pos=pk[0, h])
        O, L, dQ, dK, dV = attention.backward(f64(st.q_s[0, h]), f64(st.k_s[0, h]), f64(st.v_s[0, h]),
                                              f64(st.do_s[0, h]), mask, p.wl.scale)
        check_lse(f"LSE[{h}]", lse[0, h], L)
        for name, got, ref, perm in (("O", o, O, pq), ("dQ", dq, dQ, pq), ("dK", dk, dK, pk), ("dV", dv, dV, pk)):
            g = got[0, h].cpu()
            inr = (perm[0, h] >= 0) & (perm[0, h] < T)
            rows = perm[0, h][inr]
            unmapped = np.setdiff1d(np.arange(T), rows)
            assert len(unmapped) == 5 and torch.all(torch.isnan(g[torch.from_numpy(unmapped)])), f"{name}[{h}]"
            check_close(f"{name}[{h}]", g[torch.from_numpy(rows.astype(np.int64))], ref[inr])


@pytest.mark.parametrize("B,H,T,D", [(1, 2, 700, 64), (2, 1, 128, 64), (1, 1, 1, 64), (1, 2, 900, 128)])
def test_dense_parity(scfa, B, H, T, D):
    p = synth.make_problem(synth.Workload("d", "dense", B, H, T, D, 31))
    st = run_step(scfa, p, scfa.MODE_DENSE)
    ref = pipelines.run_dense(p.q, p.k, p.v, p.do, p.wl.scale)
    compare_heads(st, ref, ref.keys())


def test_no_prune_gives_identical_results(scfa):
    p = synth.make_problem(synth.Workload("qk", "qk", 1, 2, 1500, 64, 41, p_keep=0.6))
    a = run_step(scfa, p, scfa.MODE_QK)
    b = run_step(scfa, p, scfa.MODE_QK, flags=scfa.FLAG_NO_PRUNE)
    for name in ("o", "lse", "dk", "dv"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    check_close("dQ no-prune", b.dq, to_np(a.dq), atol=1e-2, rel_l2=2e-3)


def test_repeat_run_is_bit_identical_forward(scfa):
    p = synth.make_problem(synth.Workload("h", "hash", 1, 2, 1000, 64, 42, n_buckets=8))
    a = run_step(scfa, p, scfa.MODE_HASH)
    o1, l1, dk1, dv1 = a.o.clone(), a.lse.clone(), a.dk.clone(), a.dv.clone()
    b = run_step(scfa, p, scfa.MODE_HASH)
    assert torch.equal(o1, b.o) and torch.equal(l1, b.lse)
    assert torch.equal(dk1, b.dk) and torch.equal(dv1, b.dv)


def test_empty_rows_output_zero(scfa):
    # queries placed before every key: no admissible key -> O = 0, LSE = -inf, dQ = 0
    B, H, Tq, Tk, D = 1, 1, 200, 300, 64
    q_idx = torch.arange(Tq, dtype=torch.int32)[None, None]
    k_idx = (torch.arange(Tk, dtype=torch.int32) + 150)[None, None]
    q = synth.normal_bf16(3, 1, (B, H, Tq, D))
    k = synth.normal_bf16(3, 2, (B, H, Tk, D))
    v = synth.normal_bf16(3, 3, (B, H, Tk, D))
    do = synth.normal_bf16(3, 4, (B, H, Tq, D))
    p = synth.Problem(synth.Workload("e", "qk", B, H, Tq, D, 3), q, k, v, do, q_idx, k_idx)
    st = run_step(scfa, p, scfa.MODE_QK)
    assert torch.all(st.o[0, 0, :150] == 0) and torch.all(torch.isneginf(st.lse[0, 0, :150]))
    assert torch.all(st.dq[0, 0, :150] == 0)
    ref = pipelines.run_qk(q, k, v, do, q_idx.numpy(), k_idx.numpy(), p.wl.scale)
    compare_heads(st, ref, ref.keys())


@pytest.mark.parametrize("D", [64, 128])
def test_query_tiles_without_live_key_tile(scfa, D):
    """Whole query tiles that see no key (every position before the first
    key's) have no backward work item: their dQ rows are written as zero all
    the same, like O = 0 and LSE = -inf. Outputs start as NaN and the call
    goes straight through the C-ABI; a ragged last tile and a second head
    whose every tile is live ride along."""
    B, H, Tq, Tk = 1, 2, 300, 333
    q_idx = torch.arange(Tq, dtype=torch.int32).repeat(B, H, 1).contiguous()
    k_idx = torch.arange(Tk, dtype=torch.int32).repeat(B, H, 1).contiguous()
    k_idx[0, 0] += 260  # head 0: queries 0..259 (query tiles 0 and 1) see no key
    q = synth.normal_bf16(5, 1, (B, H, Tq, D))
    k = synth.normal_bf16(5, 2, (B, H, Tk, D))
    v = synth.normal_bf16(5, 3, (B, H, Tk, D))
    do = synth.normal_bf16(5, 4, (B, H, Tq, D))
    scale = 1.0 / math.sqrt(D)
    nan = lambda t: torch.full(t, float("nan"), dtype=torch.bfloat16, device="cuda")
    o, dq, dk, dv = nan((B, H, Tq, D)), nan((B, H, Tq, D)), nan((B, H, Tk, D)), nan((B, H, Tk, D))
    lse = torch.empty((B, H, Tq), dtype=torch.float32, device="cuda")
    ws = scfa.workspace(scfa.attn_workspace_size(scfa.MODE_QK, 1, B, H, Tq, Tk, D))
    g = [t.cuda() for t in (q, k, v, do, q_idx, k_idx)]
    scfa.scfa_qk_fwd(g[0], g[1], g[2], g[4], g[5], scale, o, lse, ws)
    scfa.scfa_qk_bwd(g[0], g[1], g[2], o, lse, g[3], g[4], g[5], scale, dq, dk, dv, ws, scfa.FLAG_REUSE_TILES)
    torch.cuda.synchronize()
    assert scfa.scfa_get_device_status(ws) == 0
    assert torch.all(o[0, 0, :260] == 0) and torch.all(torch.isneginf(lse[0, 0, :260]))
    assert torch.all(dq[0, 0, :260] == 0)
    ref = pipelines.run_qk(q, k, v, do, q_idx.numpy(), k_idx.numpy(), scale)
    f = lambda t: t.cpu().double().numpy()
    for (b, h), r in ref.items():
        check_lse(f"LSE[{h}]", lse[b, h], r["lse"])
        for key, got in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
            check_close(f"{key}[{h}]", got[b, h], r[key])


def test_sentinel_padded_heads(scfa):
    # heads with very different kept counts; padding rows must stay inert
    p = synth.make_problem(synth.Workload("qk", "qk", 1, 4, 700, 64, 44, p_keep=0.5))
    p.q_idx[0, 1, 100:] = synth.Q_SENTINEL
    p.q[0, 1, 100:] = 0
    p.k_idx[0, 2, 50:] = synth.K_SENTINEL
    p.k[0, 2, 50:] = 0
    st = run_step(scfa, p, scfa.MODE_QK)
    ref = pipelines.run_qk(p.q, p.k, p.v, p.do, p.q_idx.numpy(), p.k_idx.numpy(), p.wl.scale)
    compare_heads(st, ref, ref.keys())
    assert torch.all(st.o[0, 1, 100:] == 0)
    assert torch.all(st.dk[0, 2, 50:] == 0) and torch.all(st.dv[0, 2, 50:] == 0)


# ------------------------------------------------------------------ full-size workloads, sampled heads
def test_full_qk_8k_sampled_heads(scfa):
    wl = synth.WORKLOADS["qk_b4h12_t8192_d64_keep0.7"]
    p = synth.make_problem(wl)
    st = run_step(scfa, p, scfa.MODE_QK)
    heads = [(0, 0), (3, 11)]
    ref = pipelines.run_qk(p.q, p.k, p.v, p.do, p.q_idx.numpy(), p.k_idx.numpy(), wl.scale, heads=heads)
    compare_heads(st, ref, heads)
    # the bench's unit count: admissible pairs inside the live tiles, on the device
    B, H, Tq, _ = p.q.shape
    qi, ki = p.q_idx.numpy(), p.k_idx.numpy()
    want = sum(attention.admissible_pairs(attention.mask_qk(qi[b, h], ki[b, h])) for b in range(B) for h in range(H))
    assert device_count(scfa, scfa.MODE_QK, cuda(p.q_idx), cuda(p.k_idx), None, None, B, H, Tq, p.k.shape[2],
                        st.ws_b) == want


@pytest.mark.parametrize("tiled,gather", [(False, False), (True, False), (True, True), (True, "kv")])
def test_full_hash_8k_sampled_heads(scfa, tiled, gather):
    wl = synth.WORKLOADS["hash_b4h12_t8192_d64_nb16"]
    p = synth.make_problem(wl)
    st = run_step(scfa, p, scfa.MODE_HASH, tiled=tiled, gather=gather)
    heads = [(0, 0), (1, 5), (2, 9), (3, 11)]
    qh = lsh.lsh_hash(p.q.double().numpy(), p.R.double().numpy())
    kh = lsh.lsh_hash(p.k.double().numpy(), p.R.double().numpy())
    pq, qs, _ = sorted_views(qh, wl.n_buckets, st.Ts if tiled else None, Q_PAD)
    np.testing.assert_array_equal(st.qh.cpu().numpy(), qs)
    np.testing.assert_array_equal(st.pq.cpu().numpy(), pq)
    ref, _, _ = pipelines.run_hash(p.q, p.k, p.v, p.do, p.R, wl.scale, heads=heads, q_hash=qh, k_hash=kh)
    compare_heads(st, ref, heads, lse_perm=pq)
    # the bench's unit count: admissible pairs inside the live tiles (device)
    # against the oracle's hash mask over every head, from the oracle's ids
    want = sum(attention.admissible_pairs(attention.mask_hash(qh[b, h], kh[b, h]))
               for b in range(wl.B) for h in range(wl.H))
    assert device_count(scfa, scfa.MODE_HASH, st.pq, st.pk, st.qh, st.kh, wl.B, wl.H, st.Ts, st.Ts, st.ws_b) == want


@pytest.mark.parametrize("tiled,gather", [(False, False), (True, False), (True, True), (True, "kv")])
def test_full_hash_16k_sampled_heads(scfa, tiled, gather):
    """Hash-sparse B2 H12 T16384 D64 with 32 buckets, in the bench's launch
    configuration: bucket ids and sorted views of every head bit-exact, and
    three whole heads within tolerance (the oracle evaluates each head bucket
    by bucket, exact because the hash mask never pairs two buckets)."""
    wl = synth.WORKLOADS["hash_b2h12_t16384_d64_nb32"]
    p = synth.make_problem(wl)
    st = run_step(scfa, p, scfa.MODE_HASH, tiled=tiled, gather=gather)
    assert scfa.scfa_get_device_status(st.ws_b) == 0
    R = p.R.double().numpy()
    qh = lsh.lsh_hash(p.q.double().numpy(), R)
    kh = lsh.lsh_hash(p.k.double().numpy(), R)
    Ts = st.Ts if tiled else None
    pq, qs, oq = sorted_views(qh, wl.n_buckets, Ts, Q_PAD)
    pk, ks, ok_ = sorted_views(kh, wl.n_buckets, Ts, K_PAD)
    np.testing.assert_array_equal(st.pq.cpu().numpy(), pq)
    np.testing.assert_array_equal(st.qh.cpu().numpy(), qs)
    np.testing.assert_array_equal(st.offq.cpu().numpy(), oq)
    np.testing.assert_array_equal(st.pk.cpu().numpy(), pk)
    np.testing.assert_array_equal(st.kh.cpu().numpy(), ks)
    np.testing.assert_array_equal(st.offk.cpu().numpy(), ok_)
    for (b, h) in [(0, 0), (0, 7), (1, 11)]:
        ref = pipelines.run_hash_buckets(p.q[b, h], p.k[b, h], p.v[b, h], p.do[b, h], wl.scale, qh[b, h], kh[b, h],
                                         range(wl.n_buckets))
        o, dq, dk, dv = (torch.zeros((wl.T, wl.D), dtype=torch.float64) for _ in range(4))
        lse = np.full(wl.T, -np.inf)
        for r in ref.values():
            qp = torch.from_numpy(r["q_pos"].astype(np.int64))
            kp = torch.from_numpy(r["k_pos"].astype(np.int64))
            o[qp], dq[qp], lse[r["q_pos"]] = torch.from_numpy(r["o"]), torch.from_numpy(r["dq"]), r["lse"]
            dk[kp], dv[kp] = torch.from_numpy(r["dk"]), torch.from_numpy(r["dv"])
        check_close(f"O[{b},{h}]", st.o[b, h], o.numpy())
        check_lse_sorted(f"LSE[{b},{h}]", st.lse[b, h], lse, pq[b, h])
        check_close(f"dQ[{b},{h}]", st.dq[b, h], dq.numpy())
        check_close(f"dK[{b},{h}]", st.dk[b, h], dk.numpy())
        check_close(f"dV[{b},{h}]", st.dv[b, h], dv.numpy())


@pytest.mark.parametrize("name", ["qk_b2h12_t16384_d64_keep0.8", "qk_b2h12_t16384_d64_keep0.3"])
def test_full_qk_16k_sampled_heads(scfa, name):
    """QK-sparse B2 H12 T16384 D64 at 20% and 70% drop, in the bench's launch
    configuration, checked on three whole heads against the explicit-mask
    oracle."""
    wl = synth.WORKLOADS[name]
    p = synth.make_problem(wl)
    st = run_step(scfa, p, scfa.MODE_QK)
    assert scfa.scfa_get_device_status(st.ws_b) == 0
    heads = [(0, 0), (0, 6), (1, 11)]
    ref = pipelines.run_qk(p.q, p.k, p.v, p.do, p.q_idx.numpy(), p.k_idx.numpy(), wl.scale, heads=heads)
    compare_heads(st, ref, heads)


def test_full_hash_1m_sampled_buckets(scfa):
    """Million-token hash-sparse workload (B1 H8 T=2^20 D128, 512 buckets), in
    the bench's launch configuration. Checked on one head: its query and key
    bucket ids and sort permutations bit-exact, and every row of three whole
    buckets (the hash mask is block-diagonal by bucket) within tolerance."""
    wl = synth.WORKLOADS["hash_b1h8_t1048576_d128_nb512"]
    p = synth.make_problem(wl)
    st = run_step(scfa, p, scfa.MODE_HASH, tiled=True)
    Ts = st.Ts
    assert scfa.scfa_get_device_status(st.ws_b) == 0
    # the lists are sized for the live tiles, not for every tile pair
    assert st.live_sized
    fixed = scfa.attn_workspace_size_live(scfa.MODE_HASH, 1, wl.B, wl.H, Ts, Ts, wl.D, 0)
    assert st.ws_b.numel() - fixed < 64 << 20
    assert scfa.attn_workspace_size(scfa.MODE_HASH, 1, wl.B, wl.H, Ts, Ts, wl.D) - fixed > 7e9
    h0 = 5
    q, k, v, do = (t[0, h0] for t in (p.q, p.k, p.v, p.do))
    R = p.R.double().numpy()
    qh = lsh.lsh_hash(q.double().numpy(), R)
    kh = lsh.lsh_hash(k.double().numpy(), R)
    pq, qs, oq = lsh.bucket_sort(qh, wl.n_buckets)
    pk, ks, ok_ = lsh.bucket_sort(kh, wl.n_buckets)
    pq, qs, _ = lsh.tile_aligned(pq, oq, Ts, 128, Q_PAD)
    pk, ks, _ = lsh.tile_aligned(pk, ok_, Ts, 128, K_PAD)
    np.testing.assert_array_equal(st.pq[0, h0].cpu().numpy(), pq)
    np.testing.assert_array_equal(st.qh[0, h0].cpu().numpy(), qs)
    np.testing.assert_array_equal(st.pk[0, h0].cpu().numpy(), pk)
    np.testing.assert_array_equal(st.kh[0, h0].cpu().numpy(), ks)
    counts = np.bincount(qh, minlength=wl.n_buckets)
    buckets = sorted({int(np.argmax(counts)), int(qh[-1]), 7})
    ref = pipelines.run_hash_buckets(q, k, v, do, wl.scale, qh, kh, buckets)
    inv_q = np.empty(wl.T, dtype=np.int64)  # sorted row of each query position
    real = pq != Q_PAD
    inv_q[pq[real]] = np.nonzero(real)[0]
    o, dq, dk, dv = (t[0, h0].cpu() for t in (st.o, st.dq, st.dk, st.dv))
    lse_sorted = st.lse[0, h0].cpu().numpy()
    for c, r in ref.items():
        qp = torch.from_numpy(r["q_pos"].astype(np.int64))
        kp = torch.from_numpy(r["k_pos"].astype(np.int64))
        check_close(f"O bucket {c}", o[qp], r["o"])
        check_lse(f"LSE bucket {c}", torch.from_numpy(lse_sorted[inv_q[r["q_pos"]]]), r["lse"])
        check_close(f"dQ bucket {c}", dq[qp], r["dq"])
        check_close(f"dK bucket {c}", dk[kp], r["dk"])
        check_close(f"dV bucket {c}", dv[kp], r["dv"])


# ------------------------------------------------------------------ host pipeline
def test_host_pipeline_overlapped_copies(scfa):
    """Three hash-sparse steps submitted back to back from pinned host memory
    (the third reuses the first device slot while the copies of the others
    are in flight): every step's host results match the oracle."""
    from sparse_causal_flash_gb300.pipeline import HostPipeline
    B, H, T, D, nb = 1, 2, 640, 64, 4
    pipe = HostPipeline(scfa.MODE_HASH, B, H, T, T, D, n_buckets=nb)
    Ts = pipe.steps[0].Ts  # LSE stays in the (tile-aligned) sorted order
    probs, hins, houts = [], [], []
    shapes = [((B, H, T, D), torch.bfloat16), ((B, H, Ts), torch.float32)] + [((B, H, T, D), torch.bfloat16)] * 3
    for i in range(3):
        p = synth.make_problem(synth.Workload("hp", "hash", B, H, T, D, 70 + i, n_buckets=nb))
        hin = {n: getattr(p, n).contiguous().pin_memory() for n in ("q", "k", "v", "do", "R")}
        hout = [torch.empty(s, dtype=dt, pin_memory=True) for s, dt in shapes]
        pipe.submit(hin, hout, p.wl.scale)
        probs.append(p)
        hins.append(hin)
        houts.append(hout)
    pipe.synchronize()
    for i, (p, (o, lse, dq, dk, dv)) in enumerate(zip(probs, houts)):
        ref, qh, _ = pipelines.run_hash(p.q, p.k, p.v, p.do, p.R, p.wl.scale)
        pq, _, _ = sorted_views(qh, nb, Ts, Q_PAD)
        for (b, h), r in ref.items():
            check_close(f"step {i} O[{b},{h}]", o[b, h], r["o"])
            check_lse_sorted(f"step {i} LSE[{b},{h}]", lse[b, h], r["lse"], pq[b, h])
            check_close(f"step {i} dQ[{b},{h}]", dq[b, h], r["dq"])
            check_close(f"step {i} dK[{b},{h}]", dk[b, h], r["dk"])
            check_close(f"step {i} dV[{b},{h}]", dv[b, h], r["dv"])


# ------------------------------------------------------------------ NEXT-3 variants
@pytest.mark.parametrize("B,H,T,p_keep,seed", [(2, 3, 1000, 0.7, 91), (1, 2, 20000, 0.3, 92), (1, 4, 300, 1.0, 93)])
def test_qk_select_and_compaction_bitexact(scfa, B, H, T, p_keep, seed):
    """The selection step on the device: kept positions and counts bit for
    bit against the oracle; the compaction through them (lsh_gather) equals
    the workload's own compacted Q/K/V/dO and positions; lsh_unsort puts the
    kept rows back and leaves the dropped ones alone; an all-dropped head and
    a too-short Tc are reported through the counts."""
    from oracle import qk_select
    D = 64
    wl = synth.Workload("sel", "qk", B, H, T, D, seed, p_keep=p_keep)
    prob = synth.make_problem(wl)
    full = {n: synth.normal_bf16(seed, tid, (B, H, T, D)) for n, tid in
            (("q", synth.TID_Q), ("k", synth.TID_K), ("v", synth.TID_V), ("do", synth.TID_DO))}
    masks = {"q": synth.keep_mask(seed, synth.TID_KEEP_Q, B, H, T, p_keep),
             "k": synth.keep_mask(seed, synth.TID_KEEP_K, B, H, T, p_keep)}
    for side, sent, rows, want_idx in (("q", Q_PAD, ("q", "do"), prob.q_idx), ("k", K_PAD, ("k", "v"), prob.k_idx)):
        Tc = want_idx.shape[2]
        keep = torch.from_numpy(masks[side].astype(np.uint8)).cuda()
        idx = torch.empty((B, H, Tc), dtype=torch.int32, device="cuda")
        cnt = torch.empty((B, H), dtype=torch.int32, device="cuda")
        scfa.scfa_qk_select(keep, sent, idx, cnt)
        ref_idx, ref_cnt = qk_select.select_positions(masks[side], Tc, sent)
        np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
        np.testing.assert_array_equal(cnt.cpu().numpy(), ref_cnt)
        np.testing.assert_array_equal(idx.cpu().numpy(), want_idx.numpy())
        for n in rows:
            xc = torch.full((B, H, Tc, D), float("nan"), dtype=torch.bfloat16, device="cuda")
            scfa.lsh_gather(cuda(full[n]), idx, xc)
            assert torch.equal(xc.cpu().view(torch.int16), getattr(prob, n).view(torch.int16)), n
            back = torch.zeros((B, H, T, D), dtype=torch.bfloat16, device="cuda")
            scfa.lsh_unsort(xc, idx, back)
            kept = torch.from_numpy(masks[side])[..., None]
            want = torch.where(kept, full[n], torch.zeros_like(full[n]))
            assert torch.equal(back.cpu().view(torch.int16), want.view(torch.int16)), n
    # one head keeps nothing, and a Tc shorter than the largest count
    keep = torch.from_numpy(masks["q"].astype(np.uint8)).cuda()
    keep[0, 0] = 0
    Tc = max(1, int(keep.sum(-1).max()) // 2)
    idx = torch.empty((B, H, Tc), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B, H), dtype=torch.int32, device="cuda")
    scfa.scfa_qk_select(keep, Q_PAD, idx, cnt)
    ref_idx, ref_cnt = qk_select.select_positions(keep.cpu().numpy(), Tc, Q_PAD)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_array_equal(cnt.cpu().numpy(), ref_cnt)
    assert int(cnt[0, 0]) == 0 and bool(torch.all(idx[0, 0] == Q_PAD))


def test_lsh_sort_ids_layouts_and_bad_ids(scfa):
    """Sorting given bucket ids (no hashing): the plain layout and the
    tile-aligned one bit for bit against the oracle; an id outside
    [0, n_buckets) is reported in the status word (it takes no slot)."""
    B, H, T, nb = 2, 3, 3000, 37
    rng = np.random.default_rng(95)
    ids = rng.integers(0, nb, (B, H, T)).astype(np.int32)
    ids[0, 1, :900] = 5  # one large bucket
    g = torch.from_numpy(ids).cuda()
    ws = scfa.workspace(scfa.lsh_workspace_size(B, H, T, nb))
    dev = dict(dtype=torch.int32, device="cuda")
    for Ts, pad in ((T, 0), (scfa.scfa_tiled_rows(T, nb), K_PAD)):
        hs, perm = torch.empty((B, H, Ts), **dev), torch.empty((B, H, Ts), **dev)
        start = torch.empty((B, H, nb + 1), **dev)
        scfa.lsh_sort_ids(g, nb, pad, hs, perm, start, ws)
        want = sorted_views(ids, nb, None if Ts == T else Ts, pad)
        for got, ref in zip((perm, hs, start), want):
            np.testing.assert_array_equal(got.cpu().numpy(), ref)
        assert scfa.scfa_get_device_status(ws) == 0
    bad = g.clone()
    bad[1, 2, 17] = nb
    hs, perm = torch.empty((B, H, T), **dev), torch.empty((B, H, T), **dev)
    start = torch.empty((B, H, nb + 1), **dev)
    scfa.lsh_sort_ids(bad, nb, 0, hs, perm, start, ws)
    assert scfa.scfa_get_device_status(ws) == 1  # SCFA_ERR_INVALID


@pytest.mark.parametrize("tiled", [False, True])
def test_shared_qk_hash_parity(scfa, tiled):
    """Shared-QK hashing: one bucket id per token, from its query, used for
    its key too (keys sorted by their queries' ids). Against the oracle's
    hash-sparse attention with k_hash = q_hash."""
    from sparse_causal_flash_gb300.pipeline import Step
    B, H, T, D, nb = 1, 2, 1000, 64, 8
    p = synth.make_problem(synth.Workload("sq", "hash", B, H, T, D, 97, n_buckets=nb))
    st = Step(scfa.MODE_HASH, B, H, T, T, D, n_buckets=nb, tiled=tiled, shared_qk=True)
    st.run(cuda(p.q), cuda(p.k), cuda(p.v), cuda(p.do), p.wl.scale, R=cuda(p.R))
    torch.cuda.synchronize()
    assert scfa.scfa_get_device_status(st.ws_b) == 0
    qh = lsh.lsh_hash(p.q.double().numpy(), p.R.double().numpy())
    Ts = st.Ts if tiled else None
    pq, qs, _ = sorted_views(qh, nb, Ts, Q_PAD)
    pk, ks, _ = sorted_views(qh, nb, Ts, K_PAD)
    np.testing.assert_array_equal(st.pq.cpu().numpy(), pq)
    np.testing.assert_array_equal(st.pk.cpu().numpy(), pk)
    np.testing.assert_array_equal(st.kh.cpu().numpy(), ks)
    ref, _, _ = pipelines.run_hash(p.q, p.k, p.v, p.do, p.R, p.wl.scale, q_hash=qh, k_hash=qh)
    compare_heads(st, ref, ref.keys(), lse_perm=pq)


@pytest.mark.parametrize("mode,tiled", [("qk", None), ("hash", True), ("hash", False)])
def test_graph_replay_matches_eager_step(scfa, mode, tiled):
    """A step captured as one CUDA graph (Step.capture) and replayed gives the
    eager step's O, LSE, dQ, dK, dV bit for bit, and replays repeatably."""
    from sparse_causal_flash_gb300.pipeline import Step
    if mode == "qk":
        p = synth.make_problem(synth.Workload("g", "qk", 1, 3, 900, 64, 88, p_keep=0.6))
    else:
        p = synth.make_problem(synth.Workload("g", "hash", 1, 3, 900, 64, 89, n_buckets=8))
    B, H, Tq, D = p.q.shape
    Tk = p.k.shape[2]
    m = scfa.MODE_QK if mode == "qk" else scfa.MODE_HASH
    st = Step(m, B, H, Tq, Tk, D, n_buckets=p.wl.n_buckets, tiled=tiled)
    ins = (cuda(p.q), cuda(p.k), cuda(p.v), cuda(p.do), p.wl.scale)
    kw = dict(q_idx=None if p.q_idx is None else cuda(p.q_idx), k_idx=None if p.k_idx is None else cuda(p.k_idx),
              R=None if p.R is None else cuda(p.R))
    st.run(*ins, **kw)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (st.o, st.lse, st.dq, st.dk, st.dv)]
    g = st.capture(*ins, **kw)
    for rep in range(2):
        for t in (st.o, st.lse, st.dq, st.dk, st.dv):
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert scfa.scfa_get_device_status(st.ws_b) == 0
        for a, b in zip(eager, (st.o, st.lse, st.dq, st.dk, st.dv)):
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32)), rep
