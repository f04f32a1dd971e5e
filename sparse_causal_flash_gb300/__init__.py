"""Python binding of libscfa.so (sparse causal flash attention on GB300).

Argument marshalling only: every function hands device pointers of torch
tensors to the C ABI declared in include/scfa.h, which launches the CUDA
kernels. Nothing here computes any part of the attention, hashing, sorting
or tiling. PyTorch provides device memory and streams.

The shared library is loaded on first use; if it is missing or lacks a
declared entry point, that first call raises ImportError: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libscfa.so")

MODE_DENSE, MODE_QK, MODE_HASH = 0, 1, 2
FLAG_NO_PRUNE, FLAG_VALIDATE, FLAG_DEBUG_SYNC, FLAG_REUSE_TILES, FLAG_ORIGINAL_ORDER = 1, 2, 4, 8, 16
FLAG_KEEP_O32, FLAG_DEBUG_STALL, FLAG_GATHER_Q, FLAG_GATHER_KV = 32, 64, 128, 256
TILE = 128
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace", 4: "CUDA error", 5: "device timeout"}


class ScfaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({code})")
        self.code = code


_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_S = ctypes.c_size_t
_U = ctypes.c_uint

_SIGS = {
    "scfa_status_string": ([_I], ctypes.c_char_p),
    "scfa_attn_workspace_size": ([_I, _I, _I, _I, _I, _I, _I], _S),
    "scfa_attn_workspace_size_live": ([_I, _I, _I, _I, _I, _I, _I, ctypes.c_longlong], _S),
    "scfa_attn_workspace_capacity": ([_I, _I, _I, _I, _I, _I, _I, _S], ctypes.c_longlong),
    "scfa_tiles_count": ([_I, _P, _P, _P, _P, _I, _I, _I, _I, _P, _S, _P, _P], _I),
    "scfa_dense_fwd": ([_P, _P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _S, _U, _P], _I),
    "scfa_dense_bwd": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _P, _S, _U, _P], _I),
    "scfa_qk_fwd": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _S, _U, _P], _I),
    "scfa_qk_bwd": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _S, _U, _P], _I),
    "scfa_hash_fwd": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _S, _U, _P], _I),
    "scfa_hash_bwd": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _S, _U, _P],
                      _I),
    "lsh_workspace_size": ([_I, _I, _I, _I], _S),
    "lsh_hash": ([_P, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "lsh_hash_heads": ([_P, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "lsh_bucket_sort": ([_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _S, _U, _P], _I),
    "scfa_tiled_rows": ([_I, _I], _I),
    "lsh_bucket_sort_tiled": ([_P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_int32, _P, _P, _P, _P, _P, _S, _U, _P], _I),
    "lsh_sort_ids": ([_P, _I, _I, _I, _I, _I, ctypes.c_int32, _P, _P, _P, _P, _S, _U, _P], _I),
    "scfa_qk_select": ([_P, _I, _I, _I, _I, ctypes.c_int32, _P, _P, _P], _I),
    "lsh_gather": ([_P, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "lsh_unsort": ([_P, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "scfa_tiles": ([_I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _S, _U, _P], _I),
    "scfa_tile_view_get": ([_P, _I, _I, _I, _I, _I, _I, _P], _I),
    "scfa_get_device_status": ([_P, _P], _I),
    "scfa_count_pairs": ([_I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _S, _P, _P], _I),
    "scfa_count_chunked_pairs": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _P], _I),
    "scfa_set_kernel_events": ([_I, _P, _P], _I),
}
EXPORTED = tuple(_SIGS)


class _Lib:
    """libscfa.so with typed entry points, opened on first attribute access."""

    def __init__(self):
        self._dll = None

    def _open(self):
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with `python -m sparse_causal_flash_gb300.build`")
        dll = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            try:
                fn = getattr(dll, name)
            except AttributeError as e:
                raise ImportError(f"{LIB_PATH} lacks {name}: rebuild it") from e
            fn.argtypes = args
            fn.restype = res
        self._dll = dll

    def __getattr__(self, name):
        if self._dll is None:
            self._open()
        return getattr(self._dll, name)


_lib = _Lib()


def load() -> None:
    """Open libscfa.so now (raises ImportError if it is missing)."""
    _lib.scfa_status_string


class TileView(ctypes.Structure):
    _fields_ = [("row_ptr", _P), ("cols", _P), ("fflags", _P), ("csc_ptr", _P), ("csc_rows", _P),
                ("cflags", _P), ("work_fwd", _P), ("work_bwd", _P), ("pair_count", _P), ("pair_list", _P),
                ("work_pairs", _P), ("n_q_tiles", _I), ("n_k_tiles", _I)]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, code: int):
    if code != 0:
        raise ScfaError(fn, code)


def _need(t, dtype, name):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA tensor of {dtype}, got {t.dtype} on {t.device}")


def attn_workspace_size(mode, backward, B, H, Tq, Tk, D) -> int:
    return int(_lib.scfa_attn_workspace_size(mode, int(backward), B, H, Tq, Tk, D))


def attn_workspace_size_live(mode, backward, B, H, Tq, Tk, D, n_live) -> int:
    """Bytes of a workspace whose live-tile lists hold n_live entries."""
    return int(_lib.scfa_attn_workspace_size_live(mode, int(backward), B, H, Tq, Tk, D, int(n_live)))


def attn_workspace_capacity(mode, backward, B, H, Tq, Tk, D, ws_bytes) -> int:
    """Live-tile list entries a workspace of ws_bytes holds (-1: too small)."""
    return int(_lib.scfa_attn_workspace_capacity(mode, int(backward), B, H, Tq, Tk, D, int(ws_bytes)))


def scfa_tiles_count(mode, q_idx, k_idx, q_hash, k_hash, B, H, Tq, Tk, ws, n_live, stream=None):
    """Live-tile count of a problem into the int32 CUDA tensor n_live (asynchronous)."""
    _need(n_live, torch.int32, "n_live")
    _check("scfa_tiles_count", _lib.scfa_tiles_count(mode, _ptr(q_idx), _ptr(k_idx), _ptr(q_hash), _ptr(k_hash), B, H,
                                                     Tq, Tk, _ptr(ws), ws.numel(), _ptr(n_live), _stream(stream)))


def lsh_workspace_size(B, H, T, n_buckets) -> int:
    return int(_lib.lsh_workspace_size(B, H, T, n_buckets))


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Caller-owned workspace (torch allocations are 256-byte aligned)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------- attention
def scfa_dense_fwd(q, k, v, scale, o, lse, ws, flags=0, stream=None):
    B, H, T, D = q.shape
    _check("scfa_dense_fwd", _lib.scfa_dense_fwd(_ptr(q), _ptr(k), _ptr(v), B, H, T, D, scale, _ptr(o), _ptr(lse),
                                                 _ptr(ws), ws.numel(), flags, _stream(stream)))


def scfa_dense_bwd(q, k, v, o, lse, do, scale, dq, dk, dv, ws, flags=0, stream=None):
    B, H, T, D = q.shape
    _check("scfa_dense_bwd", _lib.scfa_dense_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), B, H, T, D,
                                                 scale, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), flags,
                                                 _stream(stream)))


def scfa_qk_fwd(q, k, v, q_idx, k_idx, scale, o, lse, ws, flags=0, stream=None):
    B, H, Tq, D = q.shape
    Tk = k.shape[2]
    _check("scfa_qk_fwd", _lib.scfa_qk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(q_idx), _ptr(k_idx), B, H, Tq, Tk, D,
                                           scale, _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), flags, _stream(stream)))


def scfa_qk_bwd(q, k, v, o, lse, do, q_idx, k_idx, scale, dq, dk, dv, ws, flags=0, stream=None):
    B, H, Tq, D = q.shape
    Tk = k.shape[2]
    _check("scfa_qk_bwd", _lib.scfa_qk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(q_idx),
                                           _ptr(k_idx), B, H, Tq, Tk, D, scale, _ptr(dq), _ptr(dk), _ptr(dv),
                                           _ptr(ws), ws.numel(), flags, _stream(stream)))


def scfa_hash_fwd(q_s, k_s, v_s, q_idx, k_idx, q_hash, k_hash, scale, o_s, lse_s, ws, flags=0, stream=None):
    """o_s: [B,H,T,D] in sorted order, or [B,H,T_orig,D] in original order
    with FLAG_ORIGINAL_ORDER (its row count is passed as T_orig); with
    FLAG_GATHER_Q q_s, with FLAG_GATHER_KV k_s and v_s are the original-order
    [B,H,T_orig,D] tensors. T is the sorted row count, from q_idx [B,H,T]."""
    B, H, T = q_idx.shape
    D = q_s.shape[3]
    _check("scfa_hash_fwd", _lib.scfa_hash_fwd(_ptr(q_s), _ptr(k_s), _ptr(v_s), _ptr(q_idx), _ptr(k_idx),
                                               _ptr(q_hash), _ptr(k_hash), B, H, T, o_s.shape[2], D, scale,
                                               _ptr(o_s), _ptr(lse_s), _ptr(ws), ws.numel(), flags,
                                               _stream(stream)))


def scfa_hash_bwd(q_s, k_s, v_s, o_s, lse_s, do_s, q_idx, k_idx, q_hash, k_hash, scale, dq_s, dk_s, dv_s, ws,
                  flags=0, stream=None):
    B, H, T = q_idx.shape
    D = q_s.shape[3]
    _check("scfa_hash_bwd", _lib.scfa_hash_bwd(_ptr(q_s), _ptr(k_s), _ptr(v_s), _ptr(o_s), _ptr(lse_s), _ptr(do_s),
                                               _ptr(q_idx), _ptr(k_idx), _ptr(q_hash), _ptr(k_hash), B, H, T,
                                               dq_s.shape[2], D, scale, _ptr(dq_s), _ptr(dk_s), _ptr(dv_s),
                                               _ptr(ws), ws.numel(), flags, _stream(stream)))


# ---------------------------------------------------------------- LSH / sort / gather
def lsh_hash(x, R, n_buckets, hash_out, stream=None):
    B, H, T, D = x.shape
    _check("lsh_hash", _lib.lsh_hash(_ptr(x), _ptr(R), B, H, T, D, n_buckets, _ptr(hash_out), _stream(stream)))


def lsh_hash_heads(x, R, n_buckets, hash_out, stream=None):
    """One rotation per head: R [H, D, n_buckets // 2]; hash_out [B,H,T]."""
    B, H, T, D = x.shape
    if R.dim() != 3 or R.shape[0] != H or R.shape[1] != D:
        raise ValueError(f"lsh_hash_heads: R must be [H={H}, D={D}, m], got {tuple(R.shape)}")
    _check("lsh_hash_heads", _lib.lsh_hash_heads(_ptr(x), _ptr(R), B, H, T, D, n_buckets, _ptr(hash_out),
                                                 _stream(stream)))


def lsh_bucket_sort(x, R, n_buckets, hash_sorted, perm, bucket_off, x_sorted, ws, flags=0, stream=None):
    B, H, T, D = x.shape
    _check("lsh_bucket_sort", _lib.lsh_bucket_sort(_ptr(x), _ptr(R), B, H, T, D, n_buckets, _ptr(hash_sorted),
                                                   _ptr(perm), _ptr(bucket_off), _ptr(x_sorted), _ptr(ws),
                                                   ws.numel(), flags, _stream(stream)))


def scfa_tiled_rows(T, n_buckets) -> int:
    """Rows per head of the tile-aligned sorted layout (lsh_bucket_sort_tiled)."""
    return int(_lib.scfa_tiled_rows(int(T), int(n_buckets)))


def lsh_bucket_sort_tiled(x, R, n_buckets, pad, hash_sorted, perm, bucket_start, x_sorted, ws, flags=0,
                          stream=None):
    """Bucket sort with every bucket starting on a 128-row boundary; perm,
    hash_sorted [B,H,T_sorted], bucket_start [B,H,n_buckets+1], x_sorted
    [B,H,T_sorted,D] or None. pad: the perm value of padding rows (-1 for
    queries, 2**31 - 1 for keys)."""
    B, H, T, D = x.shape
    _check("lsh_bucket_sort_tiled", _lib.lsh_bucket_sort_tiled(
        _ptr(x), _ptr(R), B, H, T, D, n_buckets, perm.shape[2], int(pad), _ptr(hash_sorted), _ptr(perm),
        _ptr(bucket_start), _ptr(x_sorted), _ptr(ws), ws.numel(), flags, _stream(stream)))


def lsh_sort_ids(hash_, n_buckets, pad, hash_sorted, perm, bucket_start, ws, flags=0, stream=None):
    """Stable sort of given bucket ids [B,H,T]: plain layout when perm has T
    rows per head, tile-aligned when it has scfa_tiled_rows(T, n_buckets)."""
    B, H, T = hash_.shape
    _check("lsh_sort_ids", _lib.lsh_sort_ids(_ptr(hash_), B, H, T, n_buckets, perm.shape[2], int(pad),
                                             _ptr(hash_sorted), _ptr(perm), _ptr(bucket_start), _ptr(ws),
                                             ws.numel(), flags, _stream(stream)))


def scfa_qk_select(keep, sentinel, idx, count, stream=None):
    """Positions of the kept tokens of each head (ascending), then the
    sentinel: keep [B,H,T] uint8 -> idx [B,H,Tc] int32, count [B,H] int32."""
    B, H, T = keep.shape
    _check("scfa_qk_select", _lib.scfa_qk_select(_ptr(keep), B, H, T, idx.shape[2], int(sentinel), _ptr(idx),
                                                 _ptr(count), _stream(stream)))


def lsh_gather(x, perm, x_sorted, stream=None):
    """x_sorted[b,h,s] = x[b,h,perm[b,h,s]] (a zero row where perm is outside [0, T))."""
    B, H, T, D = x.shape
    _check("lsh_gather", _lib.lsh_gather(_ptr(x), _ptr(perm), B, H, T, x_sorted.shape[2], D, _ptr(x_sorted),
                                         _stream(stream)))


def lsh_unsort(y_sorted, perm, y, stream=None):
    B, H, T, D = y.shape
    _check("lsh_unsort", _lib.lsh_unsort(_ptr(y_sorted), _ptr(perm), B, H, T, y_sorted.shape[2], D, _ptr(y),
                                         _stream(stream)))


# ---------------------------------------------------------------- tiles
def scfa_tiles(mode, q_idx, k_idx, q_hash, k_hash, B, H, Tq, Tk, D, ws, flags=0, stream=None):
    _check("scfa_tiles", _lib.scfa_tiles(mode, _ptr(q_idx), _ptr(k_idx), _ptr(q_hash), _ptr(k_hash), B, H, Tq, Tk,
                                         D, _ptr(ws), ws.numel(), flags, _stream(stream)))


def scfa_tile_view_get(ws, mode, B, H, Tq, Tk, D) -> TileView:
    tv = TileView()
    _check("scfa_tile_view_get", _lib.scfa_tile_view_get(_ptr(ws), mode, B, H, Tq, Tk, D, ctypes.byref(tv)))
    return tv


def scfa_count_pairs(mode, q_idx, k_idx, q_hash, k_hash, B, H, Tq, Tk, D, ws, count, stream=None):
    """Admissible pairs inside the live tiles held by `ws`, into the int64 CUDA tensor `count`."""
    _need(count, torch.int64, "count")
    _check("scfa_count_pairs", _lib.scfa_count_pairs(mode, _ptr(q_idx), _ptr(k_idx), _ptr(q_hash), _ptr(k_hash), B, H,
                                                     Tq, Tk, D, _ptr(ws), ws.numel(), _ptr(count), _stream(stream)))


def scfa_count_chunked_pairs(q_idx, k_idx, q_hash, k_hash, chunk, count, stream=None):
    """Admissible hash-mode pairs within a query's chunk or the chunk before, into `count`."""
    _need(count, torch.int64, "count")
    B, H, T = q_idx.shape
    _check("scfa_count_chunked_pairs", _lib.scfa_count_chunked_pairs(_ptr(q_idx), _ptr(k_idx), _ptr(q_hash),
                                                                     _ptr(k_hash), B, H, T, chunk, _ptr(count),
                                                                     _stream(stream)))


def scfa_get_device_status(ws, stream=None) -> int:
    return int(_lib.scfa_get_device_status(_ptr(ws), _stream(stream)))


def scfa_set_kernel_events(which: int, start=None, stop=None):
    """Record torch.cuda.Event `start` / `stop` around the fwd (0) / bwd (1) attention kernel."""
    sp = None if start is None else ctypes.c_void_p(start.cuda_event)
    ep = None if stop is None else ctypes.c_void_p(stop.cuda_event)
    _check("scfa_set_kernel_events", _lib.scfa_set_kernel_events(which, sp, ep))


def status_string(code: int) -> str:
    return _lib.scfa_status_string(code).decode()
