"""The N > 1 path of the benchmark on CPU: two gloo ranks (no GPU needed).

Each rank runs its own replica; only timings are combined: the job time is
the max over ranks and the job throughput counts every rank's units. Also: the
reference arm prints from rank 0 only, and concurrent builds are serialised.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from sparse_causal_flash_gb300.replicas import job_throughput, max_over_ranks
    my_ms = [40.0, 55.0][rank]                 # per-rank device time of 10 steps
    job_ms = max_over_ranks(my_ms)
    q.put((rank, job_ms, job_throughput(1e12, 10, job_ms, world)))
    dist.destroy_process_group()


def test_two_gloo_ranks_combine_timings():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=5) for _ in range(2))
    for rank, job_ms, thr in out:
        assert job_ms == 55.0                      # the slowest rank
        assert thr == pytest.approx(2 * 1e12 * 10 / 0.055)


def test_single_process_is_identity():
    from sparse_causal_flash_gb300.replicas import job_throughput, max_over_ranks
    assert max_over_ranks(3.5) == 3.5
    assert job_throughput(2.0, 5, 1000.0, 1) == 10.0


def test_reference_arm_prints_from_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--workload", "hash_b1h2_t512_d64_nb4"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
