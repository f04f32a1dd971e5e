"""One fwd+bwd step of each SCFA mode, composed from C-ABI calls.

Call order only (no arithmetic): the hash-sparse step hashes and
bucket-sorts queries and keys, moves into sorted order the rows of q, k, v
and dO that the attention kernels do not gather themselves through the
permutations (by default at head dimension 64: q and dO are moved, k and v
are gathered in the kernels), and runs the sparse attention forward and
backward in sorted order, whose kernels write O, dQ, dK and dV straight back
to original row order
(SCFA_FLAG_ORIGINAL_ORDER; "Faster Causal Attention Over Large Sequences
Through Sparse Flash Attention", deep-paper.org, sections
"动态稀疏性为何会破坏它" and "SCFA 解决方案" part 2). LSE stays in sorted query
order (the backward consumes it there). Buffers are allocated once per shape
and reused. The query side and the key side of the hash step are independent
until the attention, so the key side runs on a second stream, joined by an
event. HostPipeline runs steps on batches held in
pinned host memory with the host/device copies overlapped with the kernels.
"""
from __future__ import annotations

import torch

from . import (FLAG_GATHER_KV, FLAG_GATHER_Q, FLAG_KEEP_O32, FLAG_ORIGINAL_ORDER, FLAG_REUSE_TILES, MODE_DENSE, MODE_HASH, MODE_QK, attn_workspace_size,
               attn_workspace_size_live, lsh_bucket_sort, lsh_bucket_sort_tiled, lsh_gather, lsh_hash, lsh_hash_heads,
               lsh_sort_ids,
               lsh_workspace_size,
               scfa_dense_bwd, scfa_tiled_rows,
               scfa_dense_fwd, scfa_hash_bwd, scfa_hash_fwd, scfa_qk_bwd, scfa_qk_fwd, scfa_tiles_count, workspace)

# Above this many bytes of worst-case live-tile lists (every tile pair), the
# hash step sizes its lists for the live count of each batch instead.
LIVE_SIZED_ABOVE = 256 << 20
# position of the padding rows of the tile-aligned sorted layout: a query that
# sees no key, a key that no query sees
Q_PAD, K_PAD = -1, 2**31 - 1


class Step:
    """Buffers and the launch sequence of one fwd+bwd step for a fixed shape."""

    def __init__(self, mode: int, B: int, H: int, Tq: int, Tk: int, D: int, n_buckets: int = 0,
                 device="cuda", flags: int = 0, tiled=None, shared_qk: bool = False, gather=None,
                 per_head_r: bool = False, keep_o32: bool = False):
        """tiled (hash mode; the default): sort into the tile-aligned layout,
        every bucket starting on a tile boundary (lsh_bucket_sort_tiled); the
        sorted tensors then have Ts = scfa_tiled_rows(T, n_buckets) rows per
        head. tiled=False keeps the plain sorted order (Ts = T).
        shared_qk (hash mode): one hash per token, of its query, for both its
        query and its key (Reformer's shared-QK hashing); keys are sorted by
        those ids (lsh_sort_ids), so every token shares a bucket with itself.
        gather (hash mode): "q" (q and dO), "kv" (k and v), True (all four)
        or False: no sorted copies of those tensors; the attention kernels
        read their rows through the sort's permutations (SCFA_FLAG_GATHER_Q,
        SCFA_FLAG_GATHER_KV). The default, None, is "kv" at D = 64 on the
        tile-aligned layout (the fastest there on GB300: the backward's
        query-tile ring waits on gathered rows, its resident key tile does
        not) and False otherwise (at D = 128 the two-tile forward is slower
        with gathered key tiles).
        per_head_r (hash mode): one rotation per head, R [H, D, n_buckets // 2]
        (lsh_hash_heads); the ids are then sorted with lsh_sort_ids.
        keep_o32: the forward also keeps O in fp32 for the backward's
        rowsum(dO * O) (SCFA_FLAG_KEEP_O32). The default uses the bf16 O, as
        FlashAttention's backward does: 2-4% faster per step on GB300, and
        the gradients stay within the parity tolerance with room to spare."""
        self.mode, self.B, self.H, self.Tq, self.Tk, self.D = mode, B, H, Tq, Tk, D
        self.nb = n_buckets
        self.flags = flags
        self.keep_o32 = bool(keep_o32)
        self.tiled = mode == MODE_HASH and (tiled is None or bool(tiled))
        self.shared_qk = mode == MODE_HASH and bool(shared_qk)
        self.per_head_r = mode == MODE_HASH and bool(per_head_r)
        if gather is None:
            gather = "kv" if (self.tiled and D == 64) else False
        g = "qkv" if gather is True else (gather or "")
        if g not in ("", "q", "kv", "qkv"):
            raise ValueError(f"gather must be False, True, 'q', 'kv' or 'qkv', not {gather!r}")
        self.gq = mode == MODE_HASH and "q" in g
        self.gkv = mode == MODE_HASH and "kv" in g
        # rows per head of the sorted tensors (hash mode) or of q / k
        self.Ts = scfa_tiled_rows(Tq, n_buckets) if self.tiled else Tq
        dev = torch.device(device)
        bf = dict(dtype=torch.bfloat16, device=dev)
        i32 = dict(dtype=torch.int32, device=dev)
        self.o = torch.empty((B, H, Tq, D), **bf)
        # LSE stays in sorted order (with its padding rows in the tiled layout)
        self.lse = torch.empty((B, H, self.Ts), dtype=torch.float32, device=dev)
        self.dq = torch.empty((B, H, Tq, D), **bf)
        self.dk = torch.empty((B, H, Tk, D), **bf)
        self.dv = torch.empty((B, H, Tk, D), **bf)
        # one backward-sized workspace: the forward call builds the live-tile
        # list in it and the backward call reuses that list
        self.device = dev
        Ta, Tb = (self.Ts, self.Ts) if mode == MODE_HASH else (Tq, Tk)  # rows the attention calls see
        self.Ta = Ta
        worst = attn_workspace_size(mode, 1, B, H, Ta, Tb, D)
        fixed = attn_workspace_size_live(mode, 1, B, H, Ta, Tb, D, 0)
        self.live_sized = mode == MODE_HASH and worst - fixed > LIVE_SIZED_ABOVE
        if self.live_sized:
            # lists sized per batch from its live-tile count (scfa_tiles_count)
            self.ws_count = workspace(attn_workspace_size_live(mode, 0, B, H, Ta, Tb, D, 0), dev)
            self.n_live = torch.zeros(1, dtype=torch.int32, device=dev)
            self.list_cap = 0
            self.ws_b = None
        else:
            self.ws_b = workspace(worst, dev)
        self.ws_f = self.ws_b
        if mode == MODE_HASH:
            T, Ts = Tq, self.Ts
            self.ws_l = workspace(lsh_workspace_size(B, H, T, n_buckets), dev)
            self.ws_lk = workspace(lsh_workspace_size(B, H, T, n_buckets), dev)
            self.side = torch.cuda.Stream(device=dev)
            self.ev = [torch.cuda.Event() for _ in range(5)]
            self.qh = torch.empty((B, H, Ts), **i32)
            self.kh = torch.empty((B, H, Ts), **i32)
            self.pq = torch.empty((B, H, Ts), **i32)
            self.pk = torch.empty((B, H, Ts), **i32)
            self.offq = torch.empty((B, H, n_buckets + 1), **i32)
            self.offk = torch.empty((B, H, n_buckets + 1), **i32)
            # sorted copies of the tensors the kernels do not gather themselves
            self.q_s = self.do_s = self.k_s = self.v_s = None
            if not self.gq:
                self.q_s = torch.empty((B, H, Ts, D), **bf)
                self.do_s = torch.empty((B, H, Ts, D), **bf)
            if not self.gkv:
                self.k_s = torch.empty((B, H, Ts, D), **bf)
                self.v_s = torch.empty((B, H, Ts, D), **bf)
            if self.shared_qk or self.per_head_r:
                self.ids = torch.empty((B, H, T), **i32)  # bucket ids in original order
            if self.per_head_r and not self.shared_qk:
                self.kids = torch.empty((B, H, T), **i32)

    def run(self, q, k, v, do, scale, q_idx=None, k_idx=None, R=None, stream=None, mark=None):
        """Forward + backward. Results land in self.o/lse/dq/dk/dv.

        mark(name): if given, every call runs on the one stream and mark is
        called after each named stage (for per-stage timing)."""
        # the backward reuses the forward's live-tile list (and, with
        # keep_o32, its fp32 O in the shared workspace)
        f = self.flags | (FLAG_KEEP_O32 if self.keep_o32 else 0)
        fr = f | FLAG_REUSE_TILES
        tick = mark if mark is not None else (lambda name: None)
        if self.mode == MODE_DENSE:
            scfa_dense_fwd(q, k, v, scale, self.o, self.lse, self.ws_f, f, stream)
            tick("fwd")
            scfa_dense_bwd(q, k, v, self.o, self.lse, do, scale, self.dq, self.dk, self.dv, self.ws_b, fr, stream)
            tick("bwd")
        elif self.mode == MODE_QK:
            scfa_qk_fwd(q, k, v, q_idx, k_idx, scale, self.o, self.lse, self.ws_f, f, stream)
            tick("fwd")
            scfa_qk_bwd(q, k, v, self.o, self.lse, do, q_idx, k_idx, scale, self.dq, self.dk, self.dv, self.ws_b,
                        fr, stream)
            tick("bwd")
        else:
            main = stream if stream is not None else torch.cuda.current_stream()
            # key side (hash, sort, K and V gathers) on the second stream
            side = self.side if mark is None else main
            if self.shared_qk:
                self._shared_qk_sorts(q, k, v, do, R, main, side, tick)
            elif self.per_head_r:
                self._per_head_sorts(q, k, v, do, R, main, side, tick)
            else:
                self._sorts(q, k, v, do, R, main, side, tick)
            main.wait_event(self.ev[1])
            if self.live_sized:
                self._size_lists(main)
            # O, dQ, dK, dV go straight to original row order (pq / pk map
            # sorted rows to original ones); LSE stays in sorted order
            # the kernels gather the rows of q, dO through pq and of k, v
            # through pk where they have no sorted copies
            g = FLAG_ORIGINAL_ORDER | (FLAG_GATHER_Q if self.gq else 0) | (FLAG_GATHER_KV if self.gkv else 0)
            xq, xdo = (q, do) if self.gq else (self.q_s, self.do_s)
            xk, xv = (k, v) if self.gkv else (self.k_s, self.v_s)
            scfa_hash_fwd(xq, xk, xv, self.pq, self.pk, self.qh, self.kh, scale, self.o, self.lse, self.ws_f, f | g,
                          main)
            tick("fwd")
            if not self.gq:
                main.wait_event(self.ev[4])  # dO in sorted order (moved during the forward)
            scfa_hash_bwd(xq, xk, xv, self.o, self.lse, xdo, self.pq, self.pk, self.qh, self.kh, scale, self.dq,
                          self.dk, self.dv, self.ws_b, fr | g, main)
            tick("bwd")
        return self

    def capture(self, q, k, v, do, scale, q_idx=None, k_idx=None, R=None):
        """One whole step (every kernel of run(), both streams joined by
        events) as a CUDA graph on these input tensors, which must stay
        alive and in place: graph.replay() reruns it without per-launch
        overhead. Live-sized steps read the live count back on the host every
        step and cannot be captured."""
        if self.live_sized:
            raise RuntimeError("a live-sized step reads its live count on the host and cannot be captured")
        self.run(q, k, v, do, scale, q_idx=q_idx, k_idx=k_idx, R=R)  # attributes and modules set up
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run(q, k, v, do, scale, q_idx=q_idx, k_idx=k_idx, R=R)
        return g

    def _hash(self, x, R, ids, stream):
        (lsh_hash_heads if self.per_head_r else lsh_hash)(x, R, self.nb, ids, stream)

    def _shared_qk_sorts(self, q, k, v, do, R, main, side, tick):
        nb = self.nb
        self._hash(q, R, self.ids, main)
        tick("hash_q")
        self.ev[0].record(main)
        side.wait_event(self.ev[0])
        lsh_sort_ids(self.ids, nb, K_PAD, self.kh, self.pk, self.offk, self.ws_lk, 0, side)
        if not self.gkv:
            lsh_gather(k, self.pk, self.k_s, side)
            lsh_gather(v, self.pk, self.v_s, side)
        tick("sort_gather_k_v")
        self.ev[1].record(side)
        lsh_sort_ids(self.ids, nb, Q_PAD, self.qh, self.pq, self.offq, self.ws_l, 0, main)
        if not self.gq:
            lsh_gather(q, self.pq, self.q_s, main)
        self._move_do_late(do, main, side)
        tick("sort_gather_q_do")

    def _sorts(self, q, k, v, do, R, main, side, tick):
        nb = self.nb
        self.ev[0].record(main)
        side.wait_event(self.ev[0])

        def sort(x, pad, hs, perm, off, x_sorted, ws, st):
            if self.tiled:
                lsh_bucket_sort_tiled(x, R, nb, pad, hs, perm, off, x_sorted, ws, 0, st)
            else:
                lsh_bucket_sort(x, R, nb, hs, perm, off, x_sorted, ws, 0, st)

        # with query-side gathers alone the query stream has time to spare:
        # it moves V once the key sort is done, the key stream moves K
        split = self.gq and not self.gkv
        sort(k, K_PAD, self.kh, self.pk, self.offk, None if (self.gkv or split) else self.k_s, self.ws_lk, side)
        tick("hash_sort_gather_k")
        if split:
            self.ev[2].record(side)
            lsh_gather(k, self.pk, self.k_s, side)
        elif not self.gkv:
            lsh_gather(v, self.pk, self.v_s, side)
        tick("gather_v")
        self.ev[1].record(side)
        sort(q, Q_PAD, self.qh, self.pq, self.offq, None if self.gq else self.q_s, self.ws_l, main)
        tick("hash_sort_gather_q")
        if split:
            main.wait_event(self.ev[2])
            lsh_gather(v, self.pk, self.v_s, main)
        self._move_do_late(do, main, side)
        tick("gather_do")

    def _per_head_sorts(self, q, k, v, do, R, main, side, tick):
        nb = self.nb
        self.ev[0].record(main)
        side.wait_event(self.ev[0])
        lsh_hash_heads(k, R, nb, self.kids, side)
        lsh_sort_ids(self.kids, nb, K_PAD, self.kh, self.pk, self.offk, self.ws_lk, 0, side)
        if not self.gkv:
            lsh_gather(k, self.pk, self.k_s, side)
            lsh_gather(v, self.pk, self.v_s, side)
        tick("hash_sort_k_v")
        self.ev[1].record(side)
        lsh_hash_heads(q, R, nb, self.ids, main)
        lsh_sort_ids(self.ids, nb, Q_PAD, self.qh, self.pq, self.offq, self.ws_l, 0, main)
        if not self.gq:
            lsh_gather(q, self.pq, self.q_s, main)
        self._move_do_late(do, main, side)
        tick("hash_sort_q_do")

    def _move_do_late(self, do, main, side):
        """dO into sorted order on the second stream once the query sort is
        done: only the backward reads it, so the move runs under the forward
        (run() waits for it before the backward)."""
        if self.gq:
            return
        self.ev[3].record(main)
        side.wait_event(self.ev[3])
        lsh_gather(do, self.pq, self.do_s, side)
        self.ev[4].record(side)

    def _size_lists(self, stream):
        """Count this batch's live tiles (reads one int back) and grow the
        workspace if its lists cannot hold them (with an eighth to spare)."""
        scfa_tiles_count(MODE_HASH, self.pq, self.pk, self.qh, self.kh, self.B, self.H, self.Ts, self.Ts,
                         self.ws_count, self.n_live, stream)
        stream.synchronize()
        need = int(self.n_live.item())
        if self.ws_b is None or need > self.list_cap:
            self.list_cap = need + need // 8 + 1024
            self.ws_b = None
            self.ws_b = workspace(attn_workspace_size_live(MODE_HASH, 1, self.B, self.H, self.Ts, self.Ts, self.D,
                                                           self.list_cap), self.device)
            self.ws_f = self.ws_b


class HostPipeline:
    """Fwd+bwd steps on batches held in pinned host memory, with the copies
    hidden under the kernels.

    Two Steps (two sets of device inputs, outputs and workspaces) alternate:
    while step t runs on the compute stream, a host-to-device stream fills the
    other slot with the inputs of step t+1 and a device-to-host stream drains
    the results of step t-1. Events order the three streams (call order only,
    no arithmetic). Results of each step are copied into the host tensors
    passed with it; `synchronize()` waits for everything submitted.
    """

    INPUTS = ("q", "k", "v", "do", "q_idx", "k_idx", "R")

    def __init__(self, mode: int, B: int, H: int, Tq: int, Tk: int, D: int, n_buckets: int = 0,
                 device="cuda", flags: int = 0, tiled=None, shared_qk: bool = False, gather=None,
                 per_head_r: bool = False, graphs: bool = True):
        self.device = torch.device(device)
        self.steps = [Step(mode, B, H, Tq, Tk, D, n_buckets=n_buckets, device=self.device, flags=flags,
                           tiled=tiled, shared_qk=shared_qk, gather=gather, per_head_r=per_head_r)
                      for _ in range(2)]
        # graphs: from its second use on, a slot's step runs as one CUDA graph
        # captured on the slot's device input buffers (not for live-sized
        # steps, which read their live count back every step)
        self.use_graphs = bool(graphs)
        self.graphs = [None, None]
        self.h2d = torch.cuda.Stream(device=self.device)
        self.d2h = torch.cuda.Stream(device=self.device)
        self.inputs = [None, None]
        self.in_ready = [torch.cuda.Event() for _ in range(2)]
        self.computed = [torch.cuda.Event() for _ in range(2)]
        self.drained = [torch.cuda.Event() for _ in range(2)]
        self.used = [False, False]
        self.n = 0

    def submit(self, host_inputs: dict, host_outputs, scale: float, stream=None, before=None):
        """Queue one step and return at once.

        host_inputs: pinned CPU tensors by name (q, k, v, do, and q_idx / k_idx
        / R where the mode has them; None or absent otherwise). host_outputs:
        pinned CPU tensors for o, lse, dq, dk, dv, in that order. stream: the
        compute stream (default: the current one). before(stream): called on
        the compute stream just before the step's kernels.
        """
        s = self.n & 1
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        if self.inputs[s] is None:
            self.inputs[s] = {n: (torch.empty(t.shape, dtype=t.dtype, device=self.device) if t is not None else None)
                              for n in self.INPUTS for t in [host_inputs.get(n)]}
            # the blocks were allocated on the compute stream, whose earlier
            # kernels may still use that memory: the uploads wait for them
            self.h2d.wait_stream(main)
        dst = self.inputs[s]
        if self.used[s]:
            self.h2d.wait_event(self.computed[s])  # the step two calls back has read this slot
        with torch.cuda.stream(self.h2d):
            for n in self.INPUTS:
                src = host_inputs.get(n)
                if src is not None:
                    dst[n].copy_(src, non_blocking=True)
        self.in_ready[s].record(self.h2d)
        main.wait_event(self.in_ready[s])
        if self.used[s]:
            main.wait_event(self.drained[s])  # this slot's previous results have reached the host
        if before is not None:
            before(main)
        st = self.steps[s]
        ins = (dst["q"], dst["k"], dst["v"], dst["do"], scale)
        kw = dict(q_idx=dst["q_idx"], k_idx=dst["k_idx"], R=dst["R"])
        if self.use_graphs and self.used[s] and hasattr(st, "capture") and not getattr(st, "live_sized", False):
            with torch.cuda.stream(main):
                if self.graphs[s] is None:
                    self.graphs[s] = (st.capture(*ins, **kw), scale)
                g, g_scale = self.graphs[s]
                if g_scale != scale:  # the scale is part of the captured step
                    st.run(*ins, stream=main, **kw)
                else:
                    g.replay()
        else:
            st.run(*ins, stream=main, **kw)
        self.computed[s].record(main)
        self.d2h.wait_event(self.computed[s])
        with torch.cuda.stream(self.d2h):
            for h, o in zip(host_outputs, (st.o, st.lse, st.dq, st.dk, st.dv)):
                h.copy_(o, non_blocking=True)
        self.drained[s].record(self.d2h)
        self.used[s] = True
        self.n += 1
        return st

    def wait_copies(self, stream):
        """Make `stream` wait for every copy submitted so far."""
        stream.wait_stream(self.h2d)
        stream.wait_stream(self.d2h)

    def synchronize(self):
        self.h2d.synchronize()
        self.d2h.synchronize()
        torch.cuda.synchronize(self.device)
