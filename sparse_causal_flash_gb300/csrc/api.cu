// The C ABI of libscfa.so: argument validation, workspace layout, tensor-map
// creation and the launch sequence of every entry point declared in scfa.h.
#include <cudaTypedefs.h>

#include <climits>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace scfa {

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 3-D map over a [BH][T][D] bf16 tensor; box = 64 columns x 128 rows x 1 head,
// 128-byte swizzle; rows past T read as zero.
bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, int D, long long T, long long BH) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(T) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kTile), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_bf16_rows(CUtensorMap* map, const void* base, int D, long long rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over a [BH][T][D] fp32 tensor; box = 32 columns x 128 rows x 1
// head, 128-byte swizzle (used by TMA reduce-add; rows past T are skipped).
bool make_tmap_f32_3d(CUtensorMap* map, void* base, int D, long long T, long long BH) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4, static_cast<cuuint64_t>(T) * D * 4};
  cuuint32_t box[3] = {32, static_cast<cuuint32_t>(kTile), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool attn_ws_layout(int mode, int backward, int B, int H, int Tq, int Tk, int D, AttnWs* L, long long cap) {
  if (mode < SCFA_MODE_DENSE || mode > SCFA_MODE_HASH) return false;
  if (B < 1 || H < 1 || Tq < 1 || Tk < 1 || D < 1) return false;
  AttnWs w;
  w.nQt = (Tq + kTile - 1) / kTile;
  w.nKt = (Tk + kTile - 1) / kTile;
  const long long BH = static_cast<long long>(B) * H;
  w.n_qtiles = BH * w.nQt;
  w.n_ktiles = BH * w.nKt;
  w.nPairs = (w.nQt + 1) / 2;
  w.n_pairs = BH * w.nPairs;
  w.max_live = w.n_qtiles * w.nKt;
  if (w.max_live >= INT_MAX || w.n_qtiles >= INT_MAX / 2 || w.n_ktiles >= INT_MAX / 2) return false;
  w.cap = (cap < 0 || cap > w.max_live) ? w.max_live : cap;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  w.header = take(sizeof(WsHeader));
  w.qstat = take(sizeof(int4) * w.n_qtiles);
  w.kstat = take(sizeof(int4) * w.n_ktiles);
  w.qcount = take(sizeof(int32_t) * w.n_qtiles);
  w.kcount = take(sizeof(int32_t) * w.n_ktiles);
  w.row_ptr = take(sizeof(int32_t) * (w.n_qtiles + 1));
  w.csc_ptr = take(sizeof(int32_t) * (w.n_ktiles + 1));
  w.work_fwd = take(sizeof(int32_t) * w.n_qtiles);
  w.work_bwd = take(sizeof(int32_t) * w.n_ktiles);
  w.cursor = take(sizeof(int32_t) * (w.nQt + 2 * w.nKt + 3));
  w.pcount = take(sizeof(int32_t) * w.n_pairs);
  w.work_pairs = take(sizeof(int32_t) * w.n_pairs);
  w.vbits_bytes = sizeof(uint32_t) * static_cast<size_t>(BH) * ((Tq + 31) / 32 + (Tk + 31) / 32);
  w.vbits = take(w.vbits_bytes);
  if (backward) {
    w.dq_acc = take(sizeof(float) * static_cast<size_t>(BH) * Tq * D);
    w.qmeta = take(4 * sizeof(float) * static_cast<size_t>(BH) * w.nQt * kTile);
  }
  w.cols = take(sizeof(int32_t) * w.cap);
  w.csc_rows = take(sizeof(int32_t) * w.cap);
  w.ulist = take(sizeof(int32_t) * w.cap);
  w.fflags = take(w.cap);
  w.cflags = take(w.cap);
  w.total = off;
  *L = w;
  return true;
}

// The layout of a `ws_bytes` workspace depends on its size alone, not on the
// call: a workspace that holds the backward's fixed part always lays out the
// backward's arrays, so a forward and a SCFA_FLAG_REUSE_TILES backward on it
// agree on where the lists are. The lists take the largest entry count that
// fits after that (at most every tile pair).
bool attn_ws_fit(int mode, int backward, int B, int H, int Tq, int Tk, int D, size_t ws_bytes, AttnWs* L) {
  AttnWs w;
  if (!attn_ws_layout(mode, 1, B, H, Tq, Tk, D, &w, 0)) return false;
  const int kind = ws_bytes >= w.total ? 1 : 0;
  if (backward && kind == 0) return false;
  if (!attn_ws_layout(mode, kind, B, H, Tq, Tk, D, &w, 0) || ws_bytes < w.total) return false;
  // largest cap in [0, max_live] whose layout fits (total grows with cap)
  long long lo = 0, hi = w.max_live;
  while (lo < hi) {
    const long long mid = lo + (hi - lo + 1) / 2;
    AttnWs t;
    if (attn_ws_layout(mode, kind, B, H, Tq, Tk, D, &t, mid) && t.total <= ws_bytes) lo = mid;
    else hi = mid - 1;
  }
  if (!attn_ws_layout(mode, kind, B, H, Tq, Tk, D, &w, lo)) return false;
  *L = w;
  return true;
}

// Bytes of a workspace whose lists hold `cap` entries for a call of the given
// kind: a forward-only layout that would reach past the backward's fixed part
// takes the backward's layout instead (see attn_ws_fit).
size_t attn_ws_bytes(int mode, int backward, int B, int H, int Tq, int Tk, int D, long long cap) {
  AttnWs w, f1;
  if (!attn_ws_layout(mode, backward, B, H, Tq, Tk, D, &w, cap)) return 0;
  if (backward || !attn_ws_layout(mode, 1, B, H, Tq, Tk, D, &f1, 0) || w.total < f1.total) return w.total;
  return attn_ws_layout(mode, 1, B, H, Tq, Tk, D, &w, cap) ? w.total : 0;
}

static cudaEvent_t g_events[2][2] = {{nullptr, nullptr}, {nullptr, nullptr}};

void record_kernel_event(int which, bool start, cudaStream_t st) {
  cudaEvent_t e = g_events[which][start ? 0 : 1];
  if (e) cudaEventRecord(e, st);
}

bool lsh_ws_layout(int B, int H, int T, int n_buckets, LshWs* L) {
  if (B < 1 || H < 1 || T < 1 || n_buckets < 2) return false;
  LshWs w;
  size_t off = 0;
  w.header = off;
  off = align_up(off + sizeof(WsHeader), 256);
  w.hash = off;
  off = align_up(off + sizeof(int32_t) * static_cast<size_t>(B) * H * T, 256);
  w.chunk = off;
  if (T > kSortChunk) {
    const size_t chunks = (static_cast<size_t>(T) + kSortChunk - 1) / kSortChunk;
    off = align_up(off + sizeof(int32_t) * static_cast<size_t>(B) * H * chunks * n_buckets, 256);
  }
  w.perm_u = off;
  off = align_up(off + sizeof(int32_t) * static_cast<size_t>(B) * H * T, 256);
  w.hs_u = off;
  off = align_up(off + sizeof(int32_t) * static_cast<size_t>(B) * H * T, 256);
  w.off_u = off;
  off = align_up(off + sizeof(int32_t) * static_cast<size_t>(B) * H * (n_buckets + 1), 256);
  w.total = off;
  *L = w;
  return true;
}

}  // namespace scfa

using namespace scfa;

namespace {

constexpr int kMaxBuckets = 32768;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

inline scfa_status finish(cudaError_t e, unsigned flags, cudaStream_t st) {
  if (e != cudaSuccess) return SCFA_ERR_CUDA;
  if (flags & SCFA_FLAG_DEBUG_SYNC) {
    if (cudaStreamSynchronize(st) != cudaSuccess) return SCFA_ERR_CUDA;
  }
  return SCFA_OK;
}

// Shared validation + launch sequence of the six attention entry points.
scfa_status run_attention(int mode, bool backward, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const uint16_t* o_in, const float* lse_in, const uint16_t* do_,
                          const int32_t* q_idx, const int32_t* k_idx, const int32_t* q_hash, const int32_t* k_hash,
                          int B, int H, int Tq, int Tk, int To, int D, float scale,
                          uint16_t* o, float* lse, uint16_t* dq, uint16_t* dk, uint16_t* dv,
                          void* ws, size_t ws_bytes, unsigned flags, void* stream) {
  if (!q || !k || !v || !ws) return SCFA_ERR_INVALID;
  if (B < 1 || H < 1 || Tq < 1 || Tk < 1) return SCFA_ERR_INVALID;
  if (!(scale == scale) || scale <= 0.f) return SCFA_ERR_INVALID;
  if (D != 64 && D != 128) return SCFA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return SCFA_ERR_INVALID;
  if (mode != SCFA_MODE_DENSE && (!q_idx || !k_idx)) return SCFA_ERR_INVALID;
  if (mode == SCFA_MODE_HASH && (!q_hash || !k_hash)) return SCFA_ERR_INVALID;
  if ((flags & SCFA_FLAG_ORIGINAL_ORDER) && (mode != SCFA_MODE_HASH || Tq != Tk)) return SCFA_ERR_INVALID;
  // original-order tensors have To rows per head (at most the sorted count);
  // without a row map they are the sorted tensors themselves
  if ((flags & SCFA_FLAG_ORIGINAL_ORDER) ? (To < 1 || To > Tq) : To != Tq) return SCFA_ERR_INVALID;
  // row gathers read original-order inputs through the row maps (the gather
  // coordinates are 32-bit row numbers)
  const bool gather_q = (flags & SCFA_FLAG_GATHER_Q) != 0, gather_kv = (flags & SCFA_FLAG_GATHER_KV) != 0;
  if ((gather_q || gather_kv) &&
      (!(flags & SCFA_FLAG_ORIGINAL_ORDER) || static_cast<long long>(B) * H * To >= (1ll << 31)))
    return SCFA_ERR_INVALID;
  if (!backward) {
    if (!o || !lse || !aligned16(o)) return SCFA_ERR_INVALID;
  } else {
    if (!o_in || !lse_in || !do_ || !dq || !dk || !dv) return SCFA_ERR_INVALID;
    if (!aligned16(o_in) || !aligned16(do_) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
      return SCFA_ERR_INVALID;
  }
  // with SCFA_FLAG_KEEP_O32 the forward also needs the backward's workspace
  // (its fp32 copy of O lives where the backward keeps the dQ accumulator)
  const bool keep_o32 = (flags & SCFA_FLAG_KEEP_O32) != 0;
  const int kind = (backward || keep_o32) ? 1 : 0;
  AttnWs L;
  if (!attn_ws_layout(mode, kind, B, H, Tq, Tk, D, &L, 0)) return SCFA_ERR_UNSUPPORTED;
  // the live-tile lists get whatever the workspace holds past its fixed part
  // (a list that does not fit is reported on the device, see scfa.h)
  if (!aligned256(ws) || !attn_ws_fit(mode, kind, B, H, Tq, Tk, D, ws_bytes, &L)) return SCFA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  cudaError_t e = cudaSuccess;
  if (!(flags & SCFA_FLAG_REUSE_TILES)) {
    // (clears the status word first)
    e = launch_tiles(mode, q_idx, k_idx, q_hash, k_hash, B, H, Tq, Tk, flags, w, L, st, D == 128);
    if (e != cudaSuccess) return SCFA_ERR_CUDA;
  }
  if (flags & SCFA_FLAG_VALIDATE) {
    e = launch_validate(mode, (flags & SCFA_FLAG_ORIGINAL_ORDER) != 0, q_idx, k_idx, q_hash, k_hash, B, H, Tq, Tk, To, w,
                        L, st);
    if (e != cudaSuccess) return SCFA_ERR_CUDA;
  }
  AttnArgs a;
  a.mode = mode;
  a.B = B;
  a.H = H;
  a.Tq = Tq;
  a.Tk = Tk;
  a.D = D;
  a.scale = scale;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o_in;
  a.do_ = do_;
  a.lse_in = lse_in;
  a.q_idx = q_idx;
  a.k_idx = k_idx;
  a.q_hash = q_hash;
  a.k_hash = k_hash;
  a.o_out = o;
  a.lse_out = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  const bool original = (flags & SCFA_FLAG_ORIGINAL_ORDER) != 0;
  a.q_rows = original ? q_idx : nullptr;
  a.k_rows = original ? k_idx : nullptr;
  a.To = To;
  a.o32 = keep_o32 ? reinterpret_cast<float*>(w + L.dq_acc) : nullptr;
  a.stall = (flags & SCFA_FLAG_DEBUG_STALL) ? 1 : 0;
  a.gather_q = gather_q ? 1 : 0;
  a.gather_kv = gather_kv ? 1 : 0;
  a.ws = w;
  a.L = &L;
  e = backward ? launch_attn_bwd(a, st) : launch_attn_fwd(a, st);
  return finish(e, flags, st);
}

}  // namespace

extern "C" {

const char* scfa_status_string(scfa_status s) {
  switch (s) {
    case SCFA_OK: return "ok";
    case SCFA_ERR_INVALID: return "invalid argument";
    case SCFA_ERR_UNSUPPORTED: return "unsupported size or head dimension";
    case SCFA_ERR_WORKSPACE: return "workspace too small or misaligned";
    case SCFA_ERR_CUDA: return "CUDA error";
    case SCFA_ERR_TIMEOUT: return "device pipeline wait timed out";
    default: return "unknown status";
  }
}

size_t scfa_attn_workspace_size(int mode, int backward, int B, int H, int Tq, int Tk, int D) {
  return attn_ws_bytes(mode, backward, B, H, Tq, Tk, D, -1);
}

size_t scfa_attn_workspace_size_live(int mode, int backward, int B, int H, int Tq, int Tk, int D, long long n_live) {
  if (n_live < 0) return 0;
  return attn_ws_bytes(mode, backward, B, H, Tq, Tk, D, n_live);
}

long long scfa_attn_workspace_capacity(int mode, int backward, int B, int H, int Tq, int Tk, int D,
                                       size_t ws_bytes) {
  AttnWs L;
  if (!attn_ws_fit(mode, backward, B, H, Tq, Tk, D, ws_bytes, &L)) return -1;
  return L.cap;
}

scfa_status scfa_dense_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int H, int T, int D,
                           float scale, uint16_t* o, float* lse, void* ws, size_t ws_bytes, unsigned flags,
                           void* stream) {
  return run_attention(SCFA_MODE_DENSE, false, q, k, v, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                       nullptr, B, H, T, T, T, D, scale, o, lse, nullptr, nullptr, nullptr, ws, ws_bytes, flags,
                       stream);
}

scfa_status scfa_dense_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* o,
                           const float* lse, const uint16_t* do_, int B, int H, int T, int D, float scale,
                           uint16_t* dq, uint16_t* dk, uint16_t* dv, void* ws, size_t ws_bytes, unsigned flags,
                           void* stream) {
  return run_attention(SCFA_MODE_DENSE, true, q, k, v, o, lse, do_, nullptr, nullptr, nullptr, nullptr, B, H, T,
                       T, T, D, scale, nullptr, nullptr, dq, dk, dv, ws, ws_bytes, flags, stream);
}

scfa_status scfa_qk_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* q_idx,
                        const int32_t* k_idx, int B, int H, int Tq, int Tk, int D, float scale, uint16_t* o,
                        float* lse, void* ws, size_t ws_bytes, unsigned flags, void* stream) {
  return run_attention(SCFA_MODE_QK, false, q, k, v, nullptr, nullptr, nullptr, q_idx, k_idx, nullptr, nullptr, B,
                       H, Tq, Tk, Tq, D, scale, o, lse, nullptr, nullptr, nullptr, ws, ws_bytes, flags, stream);
}

scfa_status scfa_qk_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* o,
                        const float* lse, const uint16_t* do_, const int32_t* q_idx, const int32_t* k_idx, int B,
                        int H, int Tq, int Tk, int D, float scale, uint16_t* dq, uint16_t* dk, uint16_t* dv,
                        void* ws, size_t ws_bytes, unsigned flags, void* stream) {
  return run_attention(SCFA_MODE_QK, true, q, k, v, o, lse, do_, q_idx, k_idx, nullptr, nullptr, B, H, Tq, Tk, Tq,
                       D, scale, nullptr, nullptr, dq, dk, dv, ws, ws_bytes, flags, stream);
}

scfa_status scfa_hash_fwd(const uint16_t* q_s, const uint16_t* k_s, const uint16_t* v_s, const int32_t* q_idx,
                          const int32_t* k_idx, const int32_t* q_hash, const int32_t* k_hash, int B, int H, int T,
                          int T_orig, int D, float scale, uint16_t* o_s, float* lse_s, void* ws, size_t ws_bytes,
                          unsigned flags, void* stream) {
  return run_attention(SCFA_MODE_HASH, false, q_s, k_s, v_s, nullptr, nullptr, nullptr, q_idx, k_idx, q_hash,
                       k_hash, B, H, T, T, T_orig, D, scale, o_s, lse_s, nullptr, nullptr, nullptr, ws, ws_bytes,
                       flags, stream);
}

scfa_status scfa_hash_bwd(const uint16_t* q_s, const uint16_t* k_s, const uint16_t* v_s, const uint16_t* o_s,
                          const float* lse_s, const uint16_t* do_s, const int32_t* q_idx, const int32_t* k_idx,
                          const int32_t* q_hash, const int32_t* k_hash, int B, int H, int T, int T_orig, int D,
                          float scale, uint16_t* dq_s, uint16_t* dk_s, uint16_t* dv_s, void* ws, size_t ws_bytes,
                          unsigned flags, void* stream) {
  return run_attention(SCFA_MODE_HASH, true, q_s, k_s, v_s, o_s, lse_s, do_s, q_idx, k_idx, q_hash, k_hash, B, H,
                       T, T, T_orig, D, scale, nullptr, nullptr, dq_s, dk_s, dv_s, ws, ws_bytes, flags, stream);
}

size_t lsh_workspace_size(int B, int H, int T, int n_buckets) {
  LshWs L;
  if (!lsh_ws_layout(B, H, T, n_buckets, &L)) return 0;
  return L.total;
}

static scfa_status check_lsh_args(const uint16_t* x, const uint16_t* R, int B, int H, int T, int D, int nb) {
  if (!x || !R) return SCFA_ERR_INVALID;
  if (B < 1 || H < 1 || T < 1) return SCFA_ERR_INVALID;
  if (D < 8 || D > 256 || (D % 8) != 0) return SCFA_ERR_UNSUPPORTED;
  if (nb < 2 || nb > kMaxBuckets || (nb % 2) != 0) return SCFA_ERR_INVALID;
  if (!aligned16(x)) return SCFA_ERR_INVALID;
  return SCFA_OK;
}

scfa_status lsh_hash(const uint16_t* x, const uint16_t* R, int B, int H, int T, int D, int n_buckets,
                     int32_t* hash, void* stream) {
  scfa_status s = check_lsh_args(x, R, B, H, T, D, n_buckets);
  if (s != SCFA_OK) return s;
  if (!hash) return SCFA_ERR_INVALID;
  if ((static_cast<size_t>(D) * ((n_buckets / 2 + 3) & ~3) + 256u * (D / 2 + 1)) * sizeof(float) > 200 * 1024)
    return SCFA_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(B) * H * T;
  // no workspace here: a pipeline timeout lands in a library-owned status word
  return finish(launch_lsh_hash(x, R, rows, D, n_buckets / 2, hash, lsh_scratch_status(),
                                static_cast<cudaStream_t>(stream)),
                0, nullptr);
}

scfa_status lsh_hash_heads(const uint16_t* x, const uint16_t* R, int B, int H, int T, int D, int n_buckets,
                           int32_t* hash, void* stream) {
  scfa_status s = check_lsh_args(x, R, B, H, T, D, n_buckets);
  if (s != SCFA_OK) return s;
  if (!hash) return SCFA_ERR_INVALID;
  if ((static_cast<size_t>(D) * ((n_buckets / 2 + 3) & ~3) + 256u * (D / 2 + 1)) * sizeof(float) > 200 * 1024)
    return SCFA_ERR_UNSUPPORTED;
  return finish(launch_lsh_hash_heads(x, R, B, H, T, D, n_buckets / 2, hash, lsh_scratch_status(),
                                      static_cast<cudaStream_t>(stream)),
                0, nullptr);
}

scfa_status lsh_bucket_sort(const uint16_t* x, const uint16_t* R, int B, int H, int T, int D, int n_buckets,
                            int32_t* hash_sorted, int32_t* perm, int32_t* bucket_off, uint16_t* x_sorted, void* ws,
                            size_t ws_bytes, unsigned flags, void* stream) {
  scfa_status s = check_lsh_args(x, R, B, H, T, D, n_buckets);
  if (s != SCFA_OK) return s;
  if (!hash_sorted || !perm || !bucket_off || !ws) return SCFA_ERR_INVALID;
  if (x_sorted && !aligned16(x_sorted)) return SCFA_ERR_INVALID;
  if ((static_cast<size_t>(D) * ((n_buckets / 2 + 3) & ~3) + 256u * (D / 2 + 1)) * sizeof(float) > 200 * 1024)
    return SCFA_ERR_UNSUPPORTED;
  LshWs L;
  if (!lsh_ws_layout(B, H, T, n_buckets, &L)) return SCFA_ERR_INVALID;
  if (!aligned256(ws) || ws_bytes < L.total) return SCFA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* hash = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + L.hash);
  const long long rows = static_cast<long long>(B) * H * T;
  cudaError_t e = launch_lsh_hash(x, R, rows, D, n_buckets / 2, hash,
                                  reinterpret_cast<int*>(static_cast<char*>(ws) + L.header), st);
  if (e == cudaSuccess)
    e = launch_bucket_sort(hash, B * H, T, n_buckets, perm, hash_sorted, bucket_off,
                           reinterpret_cast<int32_t*>(static_cast<char*>(ws) + L.chunk), st);
  if (e == cudaSuccess && x_sorted) e = launch_gather(x, perm, B * H, T, T, D, x_sorted, false, st);
  return finish(e, flags, st);
}

int scfa_tiled_rows(int T, int n_buckets) {
  if (T < 1 || n_buckets < 1) return -1;
  // every non-empty bucket rounds up by less than one tile
  const long long nb = n_buckets < T ? n_buckets : T;
  const long long rows = (static_cast<long long>(T) + nb * (kTile - 1) + kTile - 1) / kTile * kTile;
  return rows > INT_MAX ? -1 : static_cast<int>(rows);
}

// The tile-aligned layout straight from the sort kernel, or from the plain
// sort plus the layout pass: the former needs heads of one CTA and room for
// three shared histograms' worth of buckets.
static cudaError_t sort_tiled(const int32_t* hash, int BH, int T, int nb, int T_sorted, int32_t pad, int32_t* perm,
                              int32_t* hash_sorted, int32_t* bucket_start, char* w, const LshWs& L, cudaStream_t st) {
  if (T <= kSortChunk && static_cast<size_t>(nb) * 3 * sizeof(int32_t) <= 160 * 1024)
    return launch_bucket_sort(hash, BH, T, nb, perm, hash_sorted, bucket_start, nullptr, st, T_sorted, pad);
  int32_t* perm_u = reinterpret_cast<int32_t*>(w + L.perm_u);
  int32_t* off_u = reinterpret_cast<int32_t*>(w + L.off_u);
  cudaError_t e = launch_bucket_sort(hash, BH, T, nb, perm_u, reinterpret_cast<int32_t*>(w + L.hs_u), off_u,
                                     reinterpret_cast<int32_t*>(w + L.chunk), st);
  if (e == cudaSuccess) e = launch_tiled_layout(perm_u, off_u, BH, T, T_sorted, nb, pad, perm, hash_sorted, bucket_start, st);
  return e;
}

scfa_status lsh_bucket_sort_tiled(const uint16_t* x, const uint16_t* R, int B, int H, int T, int D, int n_buckets,
                                  int T_sorted, int32_t pad, int32_t* hash_sorted, int32_t* perm,
                                  int32_t* bucket_start, uint16_t* x_sorted, void* ws, size_t ws_bytes,
                                  unsigned flags, void* stream) {
  scfa_status s = check_lsh_args(x, R, B, H, T, D, n_buckets);
  if (s != SCFA_OK) return s;
  if (!hash_sorted || !perm || !bucket_start || !ws) return SCFA_ERR_INVALID;
  if (x_sorted && !aligned16(x_sorted)) return SCFA_ERR_INVALID;
  const int need = scfa_tiled_rows(T, n_buckets);
  if (need < 0 || T_sorted < need) return SCFA_ERR_INVALID;
  if (pad >= 0 && pad < T) return SCFA_ERR_INVALID;  // a padding row must not name a real row
  if ((static_cast<size_t>(D) * ((n_buckets / 2 + 3) & ~3) + 256u * (D / 2 + 1)) * sizeof(float) > 200 * 1024)
    return SCFA_ERR_UNSUPPORTED;
  LshWs L;
  if (!lsh_ws_layout(B, H, T, n_buckets, &L)) return SCFA_ERR_INVALID;
  if (!aligned256(ws) || ws_bytes < L.total) return SCFA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  int32_t* hash = reinterpret_cast<int32_t*>(w + L.hash);
  const long long rows = static_cast<long long>(B) * H * T;
  cudaError_t e = launch_lsh_hash(x, R, rows, D, n_buckets / 2, hash, reinterpret_cast<int*>(w + L.header), st);
  if (e == cudaSuccess)
    e = sort_tiled(hash, B * H, T, n_buckets, T_sorted, pad, perm, hash_sorted, bucket_start, w, L, st);
  if (e == cudaSuccess && x_sorted) e = launch_gather(x, perm, B * H, T_sorted, T, D, x_sorted, false, st);
  return finish(e, flags, st);
}

scfa_status lsh_sort_ids(const int32_t* hash, int B, int H, int T, int n_buckets, int T_sorted, int32_t pad,
                         int32_t* hash_sorted, int32_t* perm, int32_t* bucket_start, void* ws, size_t ws_bytes,
                         unsigned flags, void* stream) {
  if (!hash || !hash_sorted || !perm || !bucket_start || !ws || B < 1 || H < 1 || T < 1) return SCFA_ERR_INVALID;
  if (n_buckets < 1 || n_buckets > kMaxBuckets) return SCFA_ERR_INVALID;
  const bool tiled = T_sorted != T;
  if (tiled) {
    const int need = scfa_tiled_rows(T, n_buckets);
    if (need < 0 || T_sorted < need || (pad >= 0 && pad < T)) return SCFA_ERR_INVALID;
  }
  LshWs L;
  if (!lsh_ws_layout(B, H, T, n_buckets, &L)) return SCFA_ERR_INVALID;
  if (!aligned256(ws) || ws_bytes < L.total) return SCFA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  int* status = reinterpret_cast<int*>(w + L.header);
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), st);
  if (e == cudaSuccess) e = launch_ids_check(hash, static_cast<long long>(B) * H * T, n_buckets, status, st);
  int32_t* chunk = reinterpret_cast<int32_t*>(w + L.chunk);
  if (e == cudaSuccess && !tiled) e = launch_bucket_sort(hash, B * H, T, n_buckets, perm, hash_sorted, bucket_start,
                                                         chunk, st);
  if (e == cudaSuccess && tiled)
    e = sort_tiled(hash, B * H, T, n_buckets, T_sorted, pad, perm, hash_sorted, bucket_start, w, L, st);
  return finish(e, flags, st);
}

scfa_status lsh_gather(const uint16_t* x, const int32_t* perm, int B, int H, int T, int T_sorted, int D,
                       uint16_t* x_sorted, void* stream) {
  if (!x || !perm || !x_sorted || B < 1 || H < 1 || T < 1 || T_sorted < 1) return SCFA_ERR_INVALID;
  if (D < 8 || (D % 8) != 0) return SCFA_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(x_sorted)) return SCFA_ERR_INVALID;
  return finish(launch_gather(x, perm, B * H, T_sorted, T, D, x_sorted, false, static_cast<cudaStream_t>(stream)),
                0, nullptr);
}

scfa_status lsh_unsort(const uint16_t* y_sorted, const int32_t* perm, int B, int H, int T, int T_sorted, int D,
                       uint16_t* y, void* stream) {
  if (!y_sorted || !perm || !y || B < 1 || H < 1 || T < 1 || T_sorted < 1) return SCFA_ERR_INVALID;
  if (D < 8 || (D % 8) != 0) return SCFA_ERR_UNSUPPORTED;
  if (!aligned16(y_sorted) || !aligned16(y)) return SCFA_ERR_INVALID;
  return finish(launch_gather(y_sorted, perm, B * H, T_sorted, T, D, y, true, static_cast<cudaStream_t>(stream)), 0,
                nullptr);
}

scfa_status scfa_tiles(int mode, const int32_t* q_idx, const int32_t* k_idx, const int32_t* q_hash,
                       const int32_t* k_hash, int B, int H, int Tq, int Tk, int D, void* ws, size_t ws_bytes,
                       unsigned flags, void* stream) {
  if (!ws || B < 1 || H < 1 || Tq < 1 || Tk < 1) return SCFA_ERR_INVALID;
  if (mode != SCFA_MODE_DENSE && (!q_idx || !k_idx)) return SCFA_ERR_INVALID;
  if (mode == SCFA_MODE_HASH && (!q_hash || !k_hash)) return SCFA_ERR_INVALID;
  AttnWs L;
  if (!attn_ws_layout(mode, 0, B, H, Tq, Tk, D, &L, 0)) return SCFA_ERR_INVALID;
  if (!aligned256(ws) || !attn_ws_fit(mode, 0, B, H, Tq, Tk, D, ws_bytes, &L)) return SCFA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return finish(launch_tiles(mode, q_idx, k_idx, q_hash, k_hash, B, H, Tq, Tk, flags, static_cast<char*>(ws), L, st),
                flags, st);
}

scfa_status scfa_tiles_count(int mode, const int32_t* q_idx, const int32_t* k_idx, const int32_t* q_hash,
                             const int32_t* k_hash, int B, int H, int Tq, int Tk, void* ws, size_t ws_bytes,
                             int32_t* n_live, void* stream) {
  if (!ws || !n_live || B < 1 || H < 1 || Tq < 1 || Tk < 1) return SCFA_ERR_INVALID;
  if (mode != SCFA_MODE_DENSE && (!q_idx || !k_idx)) return SCFA_ERR_INVALID;
  if (mode == SCFA_MODE_HASH && (!q_hash || !k_hash)) return SCFA_ERR_INVALID;
  AttnWs L;
  if (!attn_ws_layout(mode, 0, B, H, Tq, Tk, 64, &L, 0)) return SCFA_ERR_INVALID;
  if (!aligned256(ws) || ws_bytes < L.total) return SCFA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  cudaError_t e = launch_tiles(mode, q_idx, k_idx, q_hash, k_hash, B, H, Tq, Tk, 0, w, L, st, false, true);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(n_live, &reinterpret_cast<WsHeader*>(w + L.header)->n_live, sizeof(int32_t),
                        cudaMemcpyDeviceToDevice, st);
  return e == cudaSuccess ? SCFA_OK : SCFA_ERR_CUDA;
}

scfa_status scfa_tile_view_get(const void* ws, int mode, int B, int H, int Tq, int Tk, int D, scfa_tile_view* out) {
  if (!ws || !out) return SCFA_ERR_INVALID;
  AttnWs L;
  if (!attn_ws_layout(mode, 1, B, H, Tq, Tk, D, &L, 0)) return SCFA_ERR_INVALID;
  // the lists are where the call that built them recorded them
  WsHeader h;
  if (cudaMemcpy(&h, ws, sizeof(WsHeader), cudaMemcpyDeviceToHost) != cudaSuccess) return SCFA_ERR_CUDA;
  const char* w = static_cast<const char*>(ws);
  out->row_ptr = reinterpret_cast<const int32_t*>(w + L.row_ptr);
  out->cols = reinterpret_cast<const int32_t*>(w + h.list_off[kListCols]);
  out->fflags = reinterpret_cast<const uint8_t*>(w + h.list_off[kListFflags]);
  out->csc_ptr = reinterpret_cast<const int32_t*>(w + L.csc_ptr);
  out->csc_rows = reinterpret_cast<const int32_t*>(w + h.list_off[kListCscRows]);
  out->cflags = reinterpret_cast<const uint8_t*>(w + h.list_off[kListCflags]);
  out->work_fwd = reinterpret_cast<const int32_t*>(w + L.work_fwd);
  out->work_bwd = reinterpret_cast<const int32_t*>(w + L.work_bwd);
  out->pair_count = reinterpret_cast<const int32_t*>(w + L.pcount);
  out->pair_list = reinterpret_cast<const int32_t*>(w + h.list_off[kListPairs]);
  out->work_pairs = reinterpret_cast<const int32_t*>(w + L.work_pairs);
  out->n_q_tiles = L.nQt;
  out->n_k_tiles = L.nKt;
  return SCFA_OK;
}

scfa_status scfa_set_kernel_events(int which, void* start_event, void* stop_event) {
  if (which < 0 || which > 1) return SCFA_ERR_INVALID;
  g_events[which][0] = static_cast<cudaEvent_t>(start_event);
  g_events[which][1] = static_cast<cudaEvent_t>(stop_event);
  return SCFA_OK;
}

scfa_status scfa_get_device_status(const void* ws, void* stream) {
  if (!ws) return SCFA_ERR_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return SCFA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SCFA_ERR_CUDA;
  return v;
}

}  // extern "C"
