#!/usr/bin/env python
"""Benchmark of sparse causal flash attention (SCFA) forward + backward on GB300.

One step = one pass of the hot path over one batch of synthetic input: the
live-tile metadata, the attention forward, the backward pre-pass, the
attention backward and the dQ finalisation (hash mode adds the LSH hash,
bucket sort, row gathers and unsorts). Default workload: QK-sparse,
B=4, H=12, T=8192, D=64, each head keeping each query and key with
probability 0.7 (30% drop), bf16 N(0,1) inputs.

Reported (one JSON line on rank 0):
  value        useful TFLOP/s of the whole job: 14 * D * (admissible pairs)
               per step (4 D forward + 10 D backward per pair), divided by the
               device time of the step; inputs resident in HBM; L2 flushed
               (256 MiB write) before every timed step, outside its events.
  e2e          the same metric through the library's HostPipeline: every
               step's inputs come from pinned host memory and O, LSE, dQ, dK,
               dV go back to it, all inside one timed span; the copies of
               step t+1 / t-1 overlap the kernels of step t.
  dense        the library's own dense causal kernels at the same (B,H,T,D).
  roofline     the dominant attention kernel (timed alone with CUDA events
               recorded by the library around its launch) against the
               measured bf16 tensor peak.
  cpu_baseline the float64 CPU oracle on a bounded sample of the workload.

--impl reference times that oracle on the host cores as the reference arm.
Multi-GPU (torchrun): every rank runs its own replica of the workload (the
heads are independent problems; no collective on the data path); timing is
the max over ranks and value sums the units of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SCFA fwd+bwd ms and useful TFLOP/s vs own dense causal, % of BF16 TC peak"
DEFAULT_WORKLOAD = "qk_b4h12_t8192_d64_keep0.7"
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-secondary", action="store_true", help="skip the other target workloads")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU oracle sample budget")
    return ap.parse_args()


# ---------------------------------------------------------------------------- units
def host_pairs_qk(prob) -> int:
    """Admissible pairs of a QK-sparse problem from its index lists (host):
    per kept query, the kept keys at or before its position."""
    qi = prob.q_idx.numpy().astype(np.int64)
    ki = prob.k_idx.numpy().astype(np.int64)
    total = 0
    for b in range(qi.shape[0]):
        for h in range(qi.shape[1]):
            q = qi[b, h][qi[b, h] >= 0]
            k = np.sort(ki[b, h][ki[b, h] != 2**31 - 1])
            total += int(np.searchsorted(k, q, side="right").sum())
    return total


def host_pairs_hash(step) -> int:
    """Admissible pairs of a hash-sparse step (host): the (position, bucket)
    of every token, read from the sorted arrays whatever their layout (rows
    that name no token are skipped), then per bucket the keys at or before
    each query's position."""
    T = step.Tq
    pq, qh = step.pq.cpu().numpy().astype(np.int64), step.qh.cpu().numpy().astype(np.int64)
    pk, kh = step.pk.cpu().numpy().astype(np.int64), step.kh.cpu().numpy().astype(np.int64)
    total = 0
    for b in range(pq.shape[0]):
        for h in range(pq.shape[1]):
            qi = (pq[b, h] >= 0) & (pq[b, h] < T)
            ki = (pk[b, h] >= 0) & (pk[b, h] < T)
            assert qi.sum() == T and ki.sum() == T
            qb = np.empty(T, np.int64)
            kb = np.empty(T, np.int64)
            qb[pq[b, h][qi]] = qh[b, h][qi]
            kb[pk[b, h][ki]] = kh[b, h][ki]
            nb = int(max(qb.max(), kb.max())) + 1
            kpos = [np.nonzero(kb == c)[0] for c in range(nb)]
            for c in range(nb):
                qpos = np.nonzero(qb == c)[0]
                if len(qpos) and len(kpos[c]):
                    total += int(np.searchsorted(kpos[c], qpos, side="right").sum())
    return total


def admissible_pairs(scfa, wl, prob, step, dev) -> int:
    """Unit count of a step: admissible pairs inside the live tiles, counted on
    the device from the list the step built (scfa_count_pairs), and checked
    against a host count of the whole mask (the two agree when the live tiles
    cover every admissible pair, which the GPU tests also check against the
    oracle)."""
    import torch
    B, H, Tq, D = step.B, step.H, step.Tq, step.D
    count = torch.zeros(1, dtype=torch.int64, device=dev)
    if wl.mode == "dense":
        scfa.scfa_count_pairs(scfa.MODE_DENSE, None, None, None, None, B, H, Tq, Tq, D, step.ws_b, count)
        host = B * H * Tq * (Tq + 1) // 2
    elif wl.mode == "qk":
        scfa.scfa_count_pairs(scfa.MODE_QK, prob.q_idx.to(dev), prob.k_idx.to(dev), None, None, B, H, Tq, step.Tk, D,
                              step.ws_b, count)
        host = host_pairs_qk(prob)
    else:
        scfa.scfa_count_pairs(scfa.MODE_HASH, step.pq, step.pk, step.qh, step.kh, B, H, step.Ts, step.Ts, D,
                              step.ws_b, count)
        host = host_pairs_hash(step)
    device = int(count.item())
    assert device == host, f"pair count: device {device} != host {host}"
    return device


def kernels_per_step(mode: str, D: int = 64, T: int = 0, n_buckets: int = 0, tiled: bool = True,
                     gather_kv: bool = True) -> int:
    """Library kernels launched per step (the library's own launch sequence).
    gather_kv: the attention kernels read K and V rows through the key
    permutation (the tile-aligned step's default at D = 64), so neither is
    moved."""
    # header init with the tile stats of both sides, count, scans with the
    # work orders, fill (+ pair lists and their order at D = 128)
    tiles = 4 + (2 if D == 128 else 0)
    attn = 1 + 3         # forward; backward pre-pass, backward, dQ finalise
    if mode == "hash":
        m = n_buckets // 2
        lsh = 2 if (D in (64, 128) and m % 8 == 0 and 8 <= m <= 256) else 1  # tensor-core pass + certified pass
        # chunk counts, scan, scatter; bucket starts and spread (heads of up
        # to 16,384 rows get the tile-aligned layout from the sort itself)
        sort = (3 if T > 16384 else 1) + (2 if (tiled and T > 16384) else 0)
        moves = 2 if (tiled and gather_kv and D == 64) else 4  # Q, dO (and K, V) into sorted order
        return tiles + attn + 2 * (lsh + sort) + moves  # per q / k: hash, sort
    return tiles + attn


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(gpu_index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                self.rows.append((time.time(), parts))

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        inside = [p for (t, p) in self.rows if t0 - 0.2 <= t <= t1 + 0.2]
        use = inside if len(inside) >= 3 else [p for (_, p) in self.rows]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[2]) for p in use if num(p[2]) is not None]
        smax = [num(p[3]) for p in use if num(p[3]) is not None]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for p in use:
            for name, val in zip(names, p[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(use), "samples_in_timed_region": len(inside)}


# ---------------------------------------------------------------------------- CPU oracle sample
def oracle_sample(wl, prob, budget_s: float, max_heads: int | None = None):
    """Run the float64 oracle head by head until the budget is spent."""
    from oracle import pipelines
    if wl.mode == "hash" and wl.T > 16384:
        return oracle_sample_buckets(wl, prob, budget_s)
    heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    flops = 0.0
    done = []
    t0 = time.perf_counter()
    for bh in heads:
        if wl.mode == "qk":
            r = pipelines.run_qk(prob.q, prob.k, prob.v, prob.do, prob.q_idx.numpy(), prob.k_idx.numpy(), wl.scale,
                                 heads=[bh])
        elif wl.mode == "hash":
            r, _, _ = pipelines.run_hash(prob.q[bh[0]:bh[0] + 1, bh[1]:bh[1] + 1], prob.k[bh[0]:bh[0] + 1, bh[1]:bh[1] + 1],
                                         prob.v[bh[0]:bh[0] + 1, bh[1]:bh[1] + 1],
                                         prob.do[bh[0]:bh[0] + 1, bh[1]:bh[1] + 1], prob.R, wl.scale)
        else:
            r = pipelines.run_dense(prob.q, prob.k, prob.v, prob.do, wl.scale, heads=[bh])
        pairs = sum(x["pairs"] for x in r.values())
        flops += pipelines.useful_flops(pairs, wl.D)
        done.append(bh)
        if time.perf_counter() - t0 >= budget_s or (max_heads and len(done) >= max_heads):
            break
    el = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(done)} of {wl.B * wl.H} heads, full fwd+bwd each, float64 numpy/OpenBLAS, {el:.1f} s",
            "seconds": el, "heads": len(done)}


def oracle_sample_buckets(wl, prob, budget_s: float):
    """Long hash-sparse sequences: hash one head, then whole buckets (exact rows)."""
    from oracle import lsh, pipelines
    t0 = time.perf_counter()
    q, k, v, do = (t[0, 0] for t in (prob.q, prob.k, prob.v, prob.do))
    R = prob.R.double().numpy()
    qh = lsh.lsh_hash(q.double().numpy(), R)
    kh = lsh.lsh_hash(k.double().numpy(), R)
    flops, nb_done = 0.0, 0
    for c in range(wl.n_buckets):
        r = pipelines.run_hash_buckets(q, k, v, do, wl.scale, qh, kh, [c])
        flops += pipelines.useful_flops(r[c]["pairs"], wl.D)
        nb_done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"head (0,0): LSH ids of all {wl.T} queries and keys, then fwd+bwd of {nb_done} of "
                      f"{wl.n_buckets} buckets (exact rows), float64 numpy/OpenBLAS, {el:.1f} s",
            "seconds": el, "buckets": nb_done}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def load_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    e = rec.get(kernel)
    if not e:
        return None
    src = os.path.join(ROOT, "sparse_causal_flash_gb300", "csrc", e["source"])
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    if digest != e.get("sha256") or e.get("workload") is None:
        return None
    return e


# ---------------------------------------------------------------------------- reference arm
def run_reference(args, wl, rank, world):
    if rank != 0:
        return
    import synth
    prob = synth.make_problem(wl)
    heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    from oracle import pipelines

    long_hash = wl.mode == "hash" and wl.T > 16384
    if long_hash:
        # a T x T mask does not fit: hash head (0, 0) once (set-up, untimed),
        # then each step is one whole bucket of it (exact rows)
        from oracle import lsh
        hq_, hk_ = (prob.q[0, 0], prob.k[0, 0])
        R = prob.R.double().numpy()
        qh0 = lsh.lsh_hash(hq_.double().numpy(), R)
        kh0 = lsh.lsh_hash(hk_.double().numpy(), R)
        heads = list(range(wl.n_buckets))

    def one(bh):
        if long_hash:
            r = pipelines.run_hash_buckets(prob.q[0, 0], prob.k[0, 0], prob.v[0, 0], prob.do[0, 0], wl.scale,
                                           qh0, kh0, [bh])
            return pipelines.useful_flops(r[bh]["pairs"], wl.D)
        if wl.mode == "qk":
            r = pipelines.run_qk(prob.q, prob.k, prob.v, prob.do, prob.q_idx.numpy(), prob.k_idx.numpy(), wl.scale,
                                 heads=[bh])
        elif wl.mode == "hash":
            sl = lambda t: t[bh[0]:bh[0] + 1, bh[1]:bh[1] + 1]
            r, _, _ = pipelines.run_hash(sl(prob.q), sl(prob.k), sl(prob.v), sl(prob.do), prob.R, wl.scale)
        else:
            r = pipelines.run_dense(prob.q, prob.k, prob.v, prob.do, wl.scale, heads=[bh])
        return pipelines.useful_flops(sum(x["pairs"] for x in r.values()), wl.D)

    for i in range(args.warmup):
        one(heads[i % len(heads)])
    flops = 0.0
    t0 = time.perf_counter()
    for i in range(args.steps):
        flops += one(heads[i % len(heads)])
    el = time.perf_counter() - t0
    value = flops / el / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "H": wl.H, "T": wl.T, "D": wl.D,
                   "step": ("one bucket of head (0,0), fwd+bwd (its LSH ids computed once in set-up)" if long_hash
                            else "one (batch, head) problem of the workload, fwd+bwd, cycling over heads")},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": (f"{args.steps} buckets of head (0,0), one per step, float64 fwd+bwd" if long_hash
                                    else f"{args.steps} heads of {wl.B * wl.H}, one per step, float64 fwd+bwd")},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- our arm
# Other target workloads, measured in the same run (hash 8k; hash and QK 16k
# with the drop sweep of the 16k configuration). The million-token workload
# runs with --workload (about 50 ms per step plus a dense comparator of
# seconds).
SECONDARY = ("hash_b4h12_t8192_d64_nb16", "hash_b2h12_t16384_d64_nb32", "qk_b2h12_t16384_d64_keep0.8",
             "qk_b2h12_t16384_d64_keep0.7", "qk_b2h12_t16384_d64_keep0.5", "qk_b2h12_t16384_d64_keep0.3")
REFORMER_CHUNKS = (64, 128, 256, 512)


class Runner:
    """Device-side measurement of one workload at a time (timing, stages,
    naive baseline, dense comparator, coverage)."""

    def __init__(self, scfa, torch, dev, stream, dist, peaks):
        self.scfa, self.torch, self.dev, self.stream, self.dist = scfa, torch, dev, stream, dist
        self.flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.peak_burst, self.peak_sus, self.peak_kind = peaks
        self.dense_cache = {}
        self.graphs = []  # captured steps alive while they are timed

    def timed(self, run, K, kernel_events=False):
        """K steps, each after an L2 flush, CUDA events on the compute stream."""
        torch, scfa, stream = self.torch, self.scfa, self.stream
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        kev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(2)]
               for _ in range(K)] if kernel_events else None
        if kev is not None:  # torch creates the CUDA event on first record; the library re-records it
            for pair in kev:
                for a, b in pair:
                    a.record(stream)
                    b.record(stream)
        if self.dist is not None:
            self.dist.barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        for i in range(K):
            self.flush.zero_()
            if kev is not None:
                scfa.scfa_set_kernel_events(0, *kev[i][0])
                scfa.scfa_set_kernel_events(1, *kev[i][1])
            ev[i][0].record(stream)
            run()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        if self.dist is not None:
            self.dist.barrier()
        t1 = time.time()
        scfa.scfa_set_kernel_events(0)
        scfa.scfa_set_kernel_events(1)
        ms = [a.elapsed_time(b) for a, b in ev]
        kms = None
        if kev is not None:
            kms = ([a.elapsed_time(b) for (a, b) in (x[0] for x in kev)],
                   [a.elapsed_time(b) for (a, b) in (x[1] for x in kev)])
        return ms, kms, t0, t1

    def stages(self, step, args_, kw, scale):
        """One step with every call on the compute stream and an event after
        each stage (ms per stage; the hash step's two streams are serialised)."""
        torch = self.torch
        names, evs = [], []
        start = torch.cuda.Event(enable_timing=True)

        def mark(name):
            e = torch.cuda.Event(enable_timing=True)
            e.record(self.stream)
            names.append(name)
            evs.append(e)

        out = {}
        for rep in range(3):
            names.clear()
            evs.clear()
            self.flush.zero_()
            start.record(self.stream)
            step.run(*args_, scale, mark=mark, **kw)
            torch.cuda.synchronize()
            prev = start
            for n, e in zip(names, evs):
                out.setdefault(n, []).append(prev.elapsed_time(e))
                prev = e
        return {n: statistics.median(v) for n, v in out.items()}

    def graph_run(self, step, args_, kw, scale):
        """The step as one CUDA graph (graph.replay per step), or None when it
        cannot be captured (live-sized lists are read back every step)."""
        if getattr(step, "live_sized", False):
            return None
        g = step.capture(*args_, scale, **kw)
        self.graphs.append(g)
        for _ in range(3):
            g.replay()
        self.torch.cuda.synchronize()
        return g.replay

    def dense_ms(self, wl, K):
        from sparse_causal_flash_gb300.pipeline import Step
        import synth
        key = (wl.B, wl.H, wl.T, wl.D)
        if key not in self.dense_cache:
            torch, dev = self.torch, self.dev
            dstep = Step(self.scfa.MODE_DENSE, wl.B, wl.H, wl.T, wl.T, wl.D, device=dev)
            t = [synth.normal_bf16(wl.seed, tid, (wl.B, wl.H, wl.T, wl.D)).to(dev)
                 for tid in (synth.TID_Q, synth.TID_K, synth.TID_V, synth.TID_DO)]
            run = lambda: dstep.run(*t, wl.scale)
            once = wl.T >= (1 << 20)  # a dense 2^20-token causal step takes seconds: timed once
            for _ in range(0 if once else 3):
                run()
            if not once:
                run = self.graph_run(dstep, t, {}, wl.scale) or run
            n = 1 if once else K
            dms, _, _, _ = self.timed(run, n)
            self.dense_cache[key] = (sum(dms) / n, n)
            self.graphs.clear()
            del dstep, t, run
            torch.cuda.empty_cache()
        return self.dense_cache[key]

    def measure(self, wl, steps, detail=True, e2e_steps=0):
        """Everything about one workload; returns (record, step objects kept for e2e)."""
        import synth
        from sparse_causal_flash_gb300.pipeline import Step
        scfa, torch, dev = self.scfa, self.torch, self.dev
        prob = synth.make_problem(wl)
        mode = {"dense": scfa.MODE_DENSE, "qk": scfa.MODE_QK, "hash": scfa.MODE_HASH}[wl.mode]
        B, H, Tq, D = prob.q.shape
        Tk = prob.k.shape[2]
        step = Step(mode, B, H, Tq, Tk, D, n_buckets=wl.n_buckets, device=dev)
        args_ = [t.to(dev) for t in (prob.q, prob.k, prob.v, prob.do)]
        kw = dict(q_idx=prob.q_idx.to(dev) if prob.q_idx is not None else None,
                  k_idx=prob.k_idx.to(dev) if prob.k_idx is not None else None,
                  R=prob.R.to(dev) if prob.R is not None else None)
        run = lambda: step.run(*args_, wl.scale, **kw)
        for _ in range(3):
            run()
        torch.cuda.synchronize()
        assert scfa.scfa_get_device_status(step.ws_b) == 0, f"{wl.name}: device status not ok after warm-up"
        pairs = admissible_pairs(scfa, wl, prob, step, dev)
        useful = 14.0 * D * pairs
        # kernel times: eager steps with the library's events around the two
        # attention kernels
        ms_eager, kms, t0e, t1e = self.timed(run, steps, kernel_events=True)
        assert scfa.scfa_get_device_status(step.ws_b) == 0, f"{wl.name}: device status not ok after the timed steps"
        fwd_ms, bwd_ms = statistics.mean(kms[0]), statistics.mean(kms[1])
        long_region = (t1e - t0e) > 1.0
        # the step time: the whole step as one CUDA graph replayed per step (no
        # per-launch gaps), eager where the step cannot be captured
        grun = self.graph_run(step, args_, kw, wl.scale)
        graphed = grun is not None
        if graphed:
            ms, _, t0, t1 = self.timed(grun, steps)
            assert scfa.scfa_get_device_status(step.ws_b) == 0, f"{wl.name}: device status not ok after the graph steps"
            self.graphs.clear()
            del grun
        else:
            ms, t0, t1 = ms_eager, t0e, t1e
        peak = self.peak_sus if long_region else self.peak_burst
        if bwd_ms >= fwd_ms:
            dom = "attn_bwd_kernel" if D == 64 else "attn_bwd128_kernel"
            dom_ms, dom_flops = bwd_ms, 10.0 * D * pairs
        else:
            dom = "attn_fwd1_kernel" if D == 64 else "attn_fwd_kernel"
            dom_ms, dom_flops = fwd_ms, 4.0 * D * pairs
        achieved = dom_flops / (dom_ms / 1e3) / 1e12
        rec = {"workload": wl.name, "mode": wl.mode, "B": B, "H": H, "T": wl.T, "Tq": Tq, "Tk": Tk, "D": D,
               "admissible_pairs": pairs, "useful_flop_per_step": useful, "steps": steps,
               "ms_per_step": sum(ms) / steps, "ms_per_step_median": statistics.median(ms),
               "useful_tflops": useful / (sum(ms) / steps / 1e3) / 1e12,
               "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                            "frac": achieved / peak, "kernel_ms": dom_ms,
                            "peak_source": f"{self.peak_kind} bf16 {'sustained' if long_region else 'burst'}",
                            "fwd_kernel_ms": fwd_ms, "bwd_kernel_ms": bwd_ms,
                            "fwd_kernel_tflops": 4.0 * D * pairs / (fwd_ms / 1e3) / 1e12,
                            "bwd_kernel_tflops": 10.0 * D * pairs / (bwd_ms / 1e3) / 1e12},
               "timed_region_s": t1 - t0, "_t0": t0, "_t1": t1,
               "launch": "one CUDA graph per step (graph.replay)" if graphed else "eager",
               "ms_per_step_eager": sum(ms_eager) / steps}
        rec["pct_of_bf16_peak"] = 100.0 * rec["useful_tflops"] / peak
        if wl.mode == "qk":
            rec["p_keep"] = wl.p_keep
        if wl.mode == "hash":
            rec["n_buckets"] = wl.n_buckets
            # which row tensors the attention kernels gather through the
            # sort's permutations instead of reading sorted copies
            rec["row_gathers"] = ("q, dO" if step.gq else "") + (", " if step.gq and step.gkv else "") + \
                ("k, v" if step.gkv else "")
        if detail:
            st = self.stages(step, args_, kw, wl.scale)
            st["fwd_kernel"] = fwd_ms
            st["tiles_in_fwd_call"] = max(st["fwd"] - fwd_ms, 0.0)
            st["bwd_kernel"] = bwd_ms
            st["bwd_pre_and_dq_finalise"] = max(st["bwd"] - bwd_ms, 0.0)
            rec["stages_ms"] = st
            if wl.mode != "dense":
                # the pages' naive baselines ("实验与结果", Fig. 3 and 7): every
                # tile computed with the element mask (hash: the full T x T
                # matrix then the mask; QK: the whole compacted rectangle)
                nstep = Step(mode, B, H, Tq, Tk, D, n_buckets=wl.n_buckets, device=dev, flags=scfa.FLAG_NO_PRUNE,
                             tiled=False)
                nrun = lambda: nstep.run(*args_, wl.scale, **kw)
                nrun()
                nrun = self.graph_run(nstep, args_, kw, wl.scale) or nrun
                nk = max(3, steps // 4)
                nms, _, _, _ = self.timed(nrun, nk)
                rec["naive_no_prune"] = {"ms_per_step": sum(nms) / nk, "steps": nk,
                                         "speedup_scfa_vs_naive": (sum(nms) / nk) / rec["ms_per_step"]}
                self.graphs.clear()
                del nstep, nrun
                torch.cuda.empty_cache()
                d_ms, dn = self.dense_ms(wl, max(3, steps // 4))
                rec["dense"] = {"ms_per_step": d_ms, "steps": dn,
                                "useful_tflops": 14.0 * D * B * H * wl.T * (wl.T + 1) / 2 / (d_ms / 1e3) / 1e12,
                                "speedup_sparse_vs_dense": d_ms / rec["ms_per_step"]}
            if wl.mode == "hash":
                # bucket-collision coverage (Fig. 4): SCFA's live tiles vs a
                # Reformer-style chunked attention over the same sort
                # (Reformer chunks the plain sorted sequence: sorted again here
                # without the tile-aligned padding)
                cnt = torch.zeros(1, dtype=torch.int64, device=dev)
                cov = {"scfa_live_tiles": 1.0}
                i32 = dict(dtype=torch.int32, device=dev)
                plain = {}
                for side, x in (("q", prob.q), ("k", prob.k)):
                    hs, pm = torch.empty((B, H, Tq), **i32), torch.empty((B, H, Tq), **i32)
                    off = torch.empty((B, H, wl.n_buckets + 1), **i32)
                    wsl = scfa.workspace(scfa.lsh_workspace_size(B, H, Tq, wl.n_buckets), dev)
                    scfa.lsh_bucket_sort(x.to(dev), kw["R"], wl.n_buckets, hs, pm, off, None, wsl)
                    plain[side] = (hs, pm)
                for c in REFORMER_CHUNKS:
                    scfa.scfa_count_chunked_pairs(plain["q"][1], plain["k"][1], plain["q"][0], plain["k"][0], c, cnt)
                    cov[f"reformer_chunk{c}"] = int(cnt.item()) / pairs
                rec["coverage"] = cov
        keep = (step, args_, kw, prob) if e2e_steps else None
        if not e2e_steps:
            del step, args_, kw
            torch.cuda.empty_cache()
        return rec, keep


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    import synth
    wl = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl, rank, world)

    prob = synth.make_problem(wl)  # host tensors (also used by the CPU oracle sample)
    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_base = oracle_sample(wl, prob, args.cpu_seconds)  # before the first GPU call
    del prob

    import torch
    import sparse_causal_flash_gb300 as scfa
    from sparse_causal_flash_gb300 import build as scfa_build
    from sparse_causal_flash_gb300.replicas import job_throughput, max_over_ranks
    scfa_build.build()
    scfa.load()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    R = Runner(scfa, torch, dev, stream, dist, load_peaks())

    sampler = ClockSampler(local) if rank == 0 else None
    rec, keep = R.measure(wl, args.steps, detail=not args.no_dense, e2e_steps=0 if args.no_e2e else 1)
    clocks = sampler.stop(rec.pop("_t0"), rec.pop("_t1")) if sampler else None
    total_ms = max_over_ranks(rec["ms_per_step"] * args.steps, dev)
    ms_per_step = total_ms / args.steps
    useful = rec["useful_flop_per_step"]
    value = job_throughput(useful, args.steps, total_ms, world) / 1e12
    roofline = dict(rec["roofline"])
    tr = load_traffic(roofline["kernel"])
    roofline["traffic"] = None if tr is None else tr["bytes_per_launch"]

    e2e = None
    if keep is not None:
        from sparse_causal_flash_gb300.pipeline import HostPipeline
        step, _, _, prob = keep
        B, H, Tq, D = prob.q.shape
        Tk = prob.k.shape[2]
        mode = {"dense": scfa.MODE_DENSE, "qk": scfa.MODE_QK, "hash": scfa.MODE_HASH}[wl.mode]
        pin = lambda t: t.contiguous().pin_memory() if t is not None else None
        hin = {"q": pin(prob.q), "k": pin(prob.k), "v": pin(prob.v), "do": pin(prob.do),
               "q_idx": pin(prob.q_idx), "k_idx": pin(prob.k_idx), "R": pin(prob.R)}
        outs = [step.o, step.lse, step.dq, step.dk, step.dv]
        houts = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
        h2d = sum(t.numel() * t.element_size() for t in hin.values() if t is not None)
        d2h = sum(t.numel() * t.element_size() for t in houts)
        del keep, step
        torch.cuda.empty_cache()
        pipe = HostPipeline(mode, B, H, Tq, Tk, D, n_buckets=wl.n_buckets, device=dev)
        # every step uploads its inputs from the host inside the span; when
        # they are larger than the L2 (129 MiB) that is the real case and no
        # flush is added, otherwise L2 is flushed before every step
        big = h2d > 129 * 2**20
        before = None if big else (lambda s_: R.flush.zero_())
        # warm-up: each of the two slots runs eagerly once, then is captured
        # as a CUDA graph at its second use; all of that before the span
        for _ in range(4):
            pipe.submit(hin, houts, wl.scale, stream=stream, before=before)
        pipe.synchronize()
        K = max(5, args.steps // 2)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        # one span from before the first upload to after the last download:
        # every step's copies are inside it, overlapped with other steps' kernels
        e0.record(stream)
        pipe.h2d.wait_event(e0)
        pipe.d2h.wait_event(e0)
        for _ in range(K):
            pipe.submit(hin, houts, wl.scale, stream=stream, before=before)
        pipe.wait_copies(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        for st_ in pipe.steps:
            assert scfa.scfa_get_device_status(st_.ws_b) == 0, "device status not ok after the e2e steps"
        tot = max_over_ranks(e0.elapsed_time(e1), dev)
        e2e = {"value": job_throughput(useful, K, tot, world) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": tot / K, "steps": K,
               "copies": "overlapped with the kernels of neighbouring steps (two device slots, one copy stream "
                         "each way)",
               "l2": (f"not flushed: each step uploads {h2d / 1e6:.0f} MB of inputs (more than the 129 MiB L2) "
                      "from pinned host memory inside the span") if big else
                     "flushed before every step inside the span (inputs smaller than L2)"}
        del pipe
        torch.cuda.empty_cache()

    secondary = []
    if not args.no_secondary and wl.name == DEFAULT_WORKLOAD:
        for name in SECONDARY:
            r2, _ = R.measure(synth.WORKLOADS[name], max(10, args.steps // 2), detail=True)
            r2.pop("_t0", None)
            r2.pop("_t1", None)
            secondary.append(r2)

    if rank == 0:
        cfg = {"workload": wl.name, "mode": wl.mode, "B": wl.B, "H": wl.H, "T": wl.T, "D": wl.D,
               "Tq": rec["Tq"], "Tk": rec["Tk"], "admissible_pairs": rec["admissible_pairs"],
               "useful_flop_per_step": useful,
               "l2": "flushed before every timed step (256 MiB write), outside the step's events",
               "parallelism": f"replicas x{world}"}
        if wl.mode == "qk":
            cfg["p_keep"] = wl.p_keep
        if wl.mode == "hash":
            cfg["n_buckets"] = wl.n_buckets
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
            "pct_of_bf16_peak": 100.0 * (value / world) / roofline["peak"],
            "launch": rec.get("launch"), "ms_per_step_eager": rec.get("ms_per_step_eager"),
            "dense": rec.get("dense"), "naive_no_prune": rec.get("naive_no_prune"), "stages_ms": rec.get("stages_ms"),
            "roofline": roofline, "cpu_baseline": cpu_base, "e2e": e2e,
            "gpu_launches": kernels_per_step(wl.mode, wl.D, wl.T, getattr(wl, "n_buckets", 0)) * args.steps,
            "clocks": clocks, "secondary": secondary,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
