"""The C-ABI library builds, loads and exports every declared entry point,
and rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import numpy as np

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def scfa():
    from sparse_causal_flash_gb300 import build
    build.build()
    import sparse_causal_flash_gb300 as s
    return s


def declared_functions():
    src = open(os.path.join(ROOT, "include", "scfa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?(?:long\s+)?[A-Za-z_][A-Za-z0-9_]*\*?\s+\*?([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("scfa_qk_fwd", "scfa_qk_bwd", "scfa_hash_fwd", "scfa_hash_bwd", "scfa_dense_fwd",
                 "scfa_dense_bwd", "lsh_bucket_sort", "lsh_unsort", "lsh_gather", "lsh_hash", "scfa_tiles"):
        assert must in names


def test_library_exports_every_declared_symbol(scfa):
    lib = ctypes.CDLL(scfa.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", scfa.LIB_PATH], capture_output=True, text=True).stdout
    for name in declared_functions():
        assert re.search(rf"\bT {name}$", out, flags=re.M), name
    assert set(scfa.EXPORTED) <= set(declared_functions())


def test_host_validation_without_gpu(scfa):
    lib = scfa._lib
    # null pointers -> invalid, before any CUDA call
    assert lib.scfa_qk_fwd(None, None, None, None, None, 1, 1, 128, 128, 64, 0.125, None, None, None, 0, 0, None) == 1
    # unsupported head dimension
    fake = ctypes.c_void_p(256)
    assert lib.scfa_dense_fwd(fake, fake, fake, 1, 1, 128, 96, 0.1, fake, fake, fake, 1 << 30, 0, None) == 2
    # misaligned pointer
    bad = ctypes.c_void_p(258)
    assert lib.scfa_dense_fwd(bad, fake, fake, 1, 1, 128, 64, 0.1, fake, fake, fake, 1 << 30, 0, None) == 1
    # workspace too small
    assert lib.scfa_dense_fwd(fake, fake, fake, 1, 1, 128, 64, 0.1, fake, fake, fake, 16, 0, None) == 3
    # rows in original order exist only for hash mode
    assert lib.scfa_dense_fwd(fake, fake, fake, 1, 1, 128, 64, 0.1, fake, fake, fake, 1 << 30, 16, None) == 1
    # an fp32 copy of O needs the backward-sized workspace, even in the forward
    fwd_ws = scfa.attn_workspace_size(scfa.MODE_DENSE, 0, 1, 1, 128, 128, 64)
    assert lib.scfa_dense_fwd(fake, fake, fake, 1, 1, 128, 64, 0.1, fake, fake, fake, fwd_ws, 32, None) == 3
    # odd bucket count
    assert lib.lsh_hash(fake, fake, 1, 1, 16, 64, 5, fake, None) == 1
    assert scfa.status_string(5) == "device pipeline wait timed out"


def test_workspace_sizes_grow_with_shape(scfa):
    a = scfa.attn_workspace_size(scfa.MODE_QK, 0, 1, 1, 1000, 1000, 64)
    b = scfa.attn_workspace_size(scfa.MODE_QK, 1, 1, 1, 1000, 1000, 64)
    c = scfa.attn_workspace_size(scfa.MODE_QK, 1, 2, 1, 1000, 1000, 64)
    assert 0 < a < b < c
    assert b - a >= 1000 * 64 * 4  # the fp32 dQ accumulator
    assert scfa.attn_workspace_size(scfa.MODE_QK, 0, 0, 1, 10, 10, 64) == 0


@pytest.mark.parametrize("mode,B,H,T,D", [(0, 1, 2, 1000, 64), (1, 2, 3, 3000, 64), (2, 1, 3, 3000, 128),
                                          (2, 1, 8, 1 << 16, 64), (1, 1, 1, 1 << 19, 64)])
def test_workspace_capacity_is_exact_and_the_same_for_every_call(scfa, mode, B, H, T, D):
    """Host arithmetic only. A workspace of scfa_attn_workspace_size_live(n)
    bytes holds at least n list entries and one byte less holds fewer; the
    layout depends on the size alone, so a forward and a backward on the
    same workspace see the same lists; the worst-case sizes hold every tile
    pair."""
    n_t = (T + 127) // 128
    max_live = B * H * n_t * n_t
    cap = lambda kind, nbytes: scfa.attn_workspace_capacity(mode, kind, B, H, T, T, D, nbytes)
    for kind in (0, 1):
        worst = scfa.attn_workspace_size(mode, kind, B, H, T, T, D)
        assert cap(kind, worst) == max_live
        fixed = scfa.attn_workspace_size_live(mode, kind, B, H, T, T, D, 0)
        assert cap(kind, fixed) >= 0 and cap(kind, fixed - 1) == -1
        for n in sorted({x for x in (0, 1, 35, 36, 100, 326, 4095, 4096, max_live // 3, max_live - 1, max_live)
                         if 0 <= x <= max_live}):
            size = scfa.attn_workspace_size_live(mode, kind, B, H, T, T, D, n)
            assert cap(kind, size) >= n, (kind, n)
            if n > 0:
                assert cap(kind, size - 1) < n, (kind, n)
            for nbytes in (size - 1, size, size + 1000):
                if cap(1, nbytes) >= 0:
                    assert cap(0, nbytes) == cap(1, nbytes), (n, nbytes)
        # more bytes never hold fewer entries, except where a forward-only
        # workspace grows past the backward's fixed part and takes its layout
        t1 = scfa.attn_workspace_size_live(mode, 1, B, H, T, T, D, 0)
        for lo, hi in ((fixed, t1 - 1), (t1, worst + 4096)):
            if hi <= lo:
                continue
            caps = [cap(kind, int(x)) for x in np.linspace(lo, hi, 257).astype(np.int64)]
            assert all(a <= b for a, b in zip(caps, caps[1:]))
    # a forward-only workspace never holds fewer lists than its size promises,
    # also where it is large enough to take the backward's layout
    assert scfa.attn_workspace_size(mode, 0, B, H, T, T, D) <= scfa.attn_workspace_size(mode, 1, B, H, T, T, D)
