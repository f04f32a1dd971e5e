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
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU oracle sample budget")
    return ap.parse_args()


# ---------------------------------------------------------------------------- units
def admissible_pairs(wl, prob, step=None) -> int:
    """Exact count of unmasked (query, key) pairs of the whole workload."""
    if wl.mode == "dense":
        return wl.B * wl.H * wl.T * (wl.T + 1) // 2
    if wl.mode == "qk":
        qi = prob.q_idx.numpy().astype(np.int64)
        ki = prob.k_idx.numpy().astype(np.int64)
        total = 0
        for b in range(qi.shape[0]):
            for h in range(qi.shape[1]):
                q = qi[b, h][qi[b, h] >= 0]
                k = np.sort(ki[b, h][ki[b, h] != 2**31 - 1])
                total += int(np.searchsorted(k, q, side="right").sum())
        return total
    # hash: bucket ranges from the library's own (bit-exact) stable sort; inside
    # a bucket both lists are in position order
    pq = step.pq.cpu().numpy().astype(np.int64)
    pk = step.pk.cpu().numpy().astype(np.int64)
    oq = step.offq.cpu().numpy().astype(np.int64)
    ok = step.offk.cpu().numpy().astype(np.int64)
    total = 0
    for b in range(pq.shape[0]):
        for h in range(pq.shape[1]):
            for c in range(oq.shape[2] - 1):
                qpos = pq[b, h, oq[b, h, c]:oq[b, h, c + 1]]
                kpos = pk[b, h, ok[b, h, c]:ok[b, h, c + 1]]
                if len(qpos) and len(kpos):
                    total += int(np.searchsorted(kpos, qpos, side="right").sum())
    return total


def kernels_per_step(mode: str, D: int = 64, T: int = 0, n_buckets: int = 0) -> int:
    """Library kernels launched per step (the library's own launch sequence)."""
    tiles = 6 + (1 if D == 128 else 0)  # tile stats (q, k), count, scan, fill, work order (+ pair lists at D = 128)
    attn = 1 + 3         # forward; backward pre-pass, backward, dQ finalise
    if mode == "hash":
        m = n_buckets // 2
        lsh = 2 if (D in (64, 128) and m % 8 == 0 and 8 <= m <= 256) else 1  # tensor-core pass + certified pass
        sort = 3 if T > 8192 else 1                                          # chunk counts, scan, scatter
        return tiles + attn + 2 * (lsh + sort + 1) + 2   # per q / k: hash, sort, gather; gather V / dO
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

    import torch
    import sparse_causal_flash_gb300 as scfa
    from sparse_causal_flash_gb300 import build as scfa_build
    from sparse_causal_flash_gb300.pipeline import Step
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

    mode = {"dense": scfa.MODE_DENSE, "qk": scfa.MODE_QK, "hash": scfa.MODE_HASH}[wl.mode]
    B, H, Tq, D = prob.q.shape
    Tk = prob.k.shape[2]
    step = Step(mode, B, H, Tq, Tk, D, n_buckets=wl.n_buckets, device=dev)
    q, k, v, do = (t.to(dev) for t in (prob.q, prob.k, prob.v, prob.do))
    q_idx = prob.q_idx.to(dev) if prob.q_idx is not None else None
    k_idx = prob.k_idx.to(dev) if prob.k_idx is not None else None
    R = prob.R.to(dev) if prob.R is not None else None
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def run_once():
        step.run(q, k, v, do, wl.scale, q_idx=q_idx, k_idx=k_idx, R=R)

    for _ in range(max(args.warmup, 3)):
        run_once()
    torch.cuda.synchronize()
    assert scfa.scfa_get_device_status(step.ws_b) == 0, "device status not ok after warm-up"
    pairs = admissible_pairs(wl, prob, step)
    useful = 14.0 * D * pairs

    def timed(run, K, kernel_events=False):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        kev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(2)]
               for _ in range(K)] if kernel_events else None
        if kev is not None:  # torch creates the CUDA event on first record; the library re-records it
            for pair in kev:
                for a, b in pair:
                    a.record(stream)
                    b.record(stream)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        for i in range(K):
            flush.zero_()
            if kev is not None:
                scfa.scfa_set_kernel_events(0, *kev[i][0])
                scfa.scfa_set_kernel_events(1, *kev[i][1])
            ev[i][0].record(stream)
            run()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        t1 = time.time()
        scfa.scfa_set_kernel_events(0)
        scfa.scfa_set_kernel_events(1)
        ms = [a.elapsed_time(b) for a, b in ev]
        kms = None
        if kev is not None:
            kms = ([a.elapsed_time(b) for (a, b) in (x[0] for x in kev)],
                   [a.elapsed_time(b) for (a, b) in (x[1] for x in kev)])
        return ms, kms, t0, t1

    sampler = ClockSampler(local) if rank == 0 else None
    ms, kms, t0, t1 = timed(run_once, args.steps, kernel_events=True)
    clocks = sampler.stop(t0, t1) if sampler else None
    assert scfa.scfa_get_device_status(step.ws_b) == 0, "device status not ok after the timed steps"
    total_ms = max_over_ranks(sum(ms), dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(useful, args.steps, total_ms, world) / 1e12

    # the attention kernels timed alone (events recorded by the library around each launch)
    fwd_ms = statistics.mean(kms[0])
    bwd_ms = statistics.mean(kms[1])
    peak_burst, peak_sus, peak_kind = load_peaks()
    long_region = (t1 - t0) > 1.0
    peak = peak_sus if long_region else peak_burst
    if bwd_ms >= fwd_ms:
        # D = 128 runs the full-D key-tile kernel
        dom = "attn_bwd_kernel" if D == 64 else "attn_bwd128_kernel"
        dom_ms, dom_flops, src = bwd_ms, 10.0 * D * pairs, "attn_bwd.cu"
    else:
        # D = 64 runs the single-query-tile kernel, D = 128 the query-tile-pair kernel
        dom = "attn_fwd1_kernel" if D == 64 else "attn_fwd_kernel"
        dom_ms, dom_flops, src = fwd_ms, 4.0 * D * pairs, "attn_fwd.cu"
    achieved = dom_flops / (dom_ms / 1e3) / 1e12
    tr = load_traffic(dom)
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": None if tr is None else tr["bytes_per_launch"],
                "peak_source": f"{peak_kind} bf16 {'sustained' if long_region else 'burst'}",
                "kernel_ms": dom_ms, "fwd_kernel_ms": fwd_ms, "bwd_kernel_ms": bwd_ms,
                "fwd_kernel_tflops": 4.0 * D * pairs / (fwd_ms / 1e3) / 1e12,
                "bwd_kernel_tflops": 10.0 * D * pairs / (bwd_ms / 1e3) / 1e12}

    dense = None
    if not args.no_dense and wl.mode != "dense":
        dstep = Step(scfa.MODE_DENSE, wl.B, wl.H, wl.T, wl.T, D, device=dev)
        dq_ = synth.normal_bf16(wl.seed, synth.TID_Q, (wl.B, wl.H, wl.T, D)).to(dev)
        dk_ = synth.normal_bf16(wl.seed, synth.TID_K, (wl.B, wl.H, wl.T, D)).to(dev)
        dv_ = synth.normal_bf16(wl.seed, synth.TID_V, (wl.B, wl.H, wl.T, D)).to(dev)
        ddo = synth.normal_bf16(wl.seed, synth.TID_DO, (wl.B, wl.H, wl.T, D)).to(dev)
        run_dense = lambda: dstep.run(dq_, dk_, dv_, ddo, wl.scale)
        once = wl.T >= (1 << 20)  # a dense 2^20-token causal step takes seconds: timed once
        for _ in range(0 if once else 3):
            run_dense()
        dK = 1 if once else max(5, args.steps // 4)
        dms, _, _, _ = timed(run_dense, dK)
        d_ms = sum(dms) / dK
        d_useful = 14.0 * D * wl.B * wl.H * wl.T * (wl.T + 1) / 2
        dense = {"ms_per_step": d_ms, "useful_tflops": d_useful / (d_ms / 1e3) / 1e12, "steps": dK,
                 "speedup_sparse_vs_dense": d_ms / ms_per_step}
        del dstep, dq_, dk_, dv_, ddo

    e2e = None
    if not args.no_e2e:
        from sparse_causal_flash_gb300.pipeline import HostPipeline
        pin = lambda t: t.contiguous().pin_memory() if t is not None else None
        hin = {"q": pin(prob.q), "k": pin(prob.k), "v": pin(prob.v), "do": pin(prob.do),
               "q_idx": pin(prob.q_idx), "k_idx": pin(prob.k_idx), "R": pin(prob.R)}
        outs = [step.o, step.lse, step.dq, step.dk, step.dv]
        houts = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
        h2d = sum(t.numel() * t.element_size() for t in hin.values() if t is not None)
        d2h = sum(t.numel() * t.element_size() for t in houts)
        pipe = HostPipeline(mode, B, H, Tq, Tk, D, n_buckets=wl.n_buckets, device=dev)
        flush_before = lambda s: flush.zero_()

        for _ in range(3):
            pipe.submit(hin, houts, wl.scale, stream=stream, before=flush_before)
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
            pipe.submit(hin, houts, wl.scale, stream=stream, before=flush_before)
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
                         "each way); L2 flushed before every step inside the span"}
        del pipe

    if rank == 0:
        cfg = {"workload": wl.name, "mode": wl.mode, "B": wl.B, "H": wl.H, "T": wl.T, "D": wl.D,
               "Tq": Tq, "Tk": Tk, "admissible_pairs": pairs, "useful_flop_per_step": useful,
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
            "pct_of_bf16_peak": 100.0 * (value / world) / peak,
            "dense": dense, "roofline": roofline, "cpu_baseline": cpu_base, "e2e": e2e,
            "gpu_launches": kernels_per_step(wl.mode, wl.D, wl.T, getattr(wl, "n_buckets", 0)) * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
