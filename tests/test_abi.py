"""The C-ABI library builds, loads and exports every declared entry point,
and rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re
import subprocess

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
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\*?\s+\*?([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
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
