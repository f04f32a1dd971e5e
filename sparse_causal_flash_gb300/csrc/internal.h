// Host-side internals shared by the translation units of libscfa.so:
// workspace layouts and the launchers of each kernel family.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/scfa.h"

namespace scfa {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Byte offsets of the arrays an attention call keeps in its workspace.
struct AttnWs {
  int nQt = 0, nKt = 0;
  long long n_qtiles = 0, n_ktiles = 0;  // over all heads
  long long max_live = 0;                // every (query tile, key tile) pair
  long long cap = 0;                     // entries the live lists hold (<= max_live)
  size_t header = 0;
  size_t qstat = 0, kstat = 0;           // int4 per tile: min idx, max idx, min hash, max hash
  size_t qcount = 0, kcount = 0;         // live count per q tile / k tile
  size_t row_ptr = 0, csc_ptr = 0;
  size_t cols = 0, csc_rows = 0;
  size_t fflags = 0, cflags = 0;
  size_t work_fwd = 0, work_bwd = 0;
  size_t cursor = 0;                     // scratch of the work-order sort
  // forward scheduling unit: a pair of adjacent query tiles (2m, 2m + 1) of
  // one head that share K / V loads over the union of their live lists
  int nPairs = 0;                        // per head
  long long n_pairs = 0;                 // over all heads
  size_t pcount = 0;                     // union size per pair
  size_t ulist = 0;                      // union list of pair m of head bh at row_ptr[bh * nQt + 2m]:
                                         // (key tile << 4) | bits (1 live for 2m, 2 FULL for 2m,
                                         // 4 live for 2m + 1, 8 FULL for 2m + 1), key tiles ascending
  size_t work_pairs = 0;                 // pair ids by union size descending
  size_t dq_acc = 0;                     // backward: fp32 dQ accumulator [B,H,Tq,D]
  size_t vbits = 0, vbits_bytes = 0;     // SCFA_FLAG_VALIDATE: one bit per row of q and of k
  size_t qmeta = 0;                      // backward: per-query metadata padded to whole tiles, four
                                         // [B*H][nQt*128] arrays: -LSE*log2(e) and -rowsum(dO*O)*scale
                                         // (fp32), position and bucket id (int32)
  size_t total = 0;
};

// Layout with lists of `cap` entries (cap < 0: every tile pair); returns false
// if the sizes are out of range. The live-tile lists come last, after the
// backward's arrays.
bool attn_ws_layout(int mode, int backward, int B, int H, int Tq, int Tk, int D, AttnWs* L, long long cap = -1);
// The layout of a `ws_bytes` workspace, the same for every call on it: the
// backward's arrays whenever it holds them, then lists as long as fit (at most
// every tile pair). False if the fixed part the call needs does not fit.
bool attn_ws_fit(int mode, int backward, int B, int H, int Tq, int Tk, int D, size_t ws_bytes, AttnWs* L);
// Workspace bytes for lists of `cap` entries (cap < 0: every tile pair).
size_t attn_ws_bytes(int mode, int backward, int B, int H, int Tq, int Tk, int D, long long cap);

struct LshWs {
  size_t header = 0;
  size_t hash = 0;    // int32 [B,H,T], original order
  size_t chunk = 0;   // int32 [B*H][chunks][n_buckets]: per-chunk counts, then scatter bases (long rows)
  size_t perm_u = 0, hs_u = 0;  // int32 [B,H,T]: the plain sorted order (tile-aligned sort)
  size_t off_u = 0;             // int32 [B,H,n_buckets+1]
  size_t total = 0;
};
constexpr int kSortChunk = 16384;  // rows longer than this are sorted by several CTAs
bool lsh_ws_layout(int B, int H, int T, int n_buckets, LshWs* L);

int num_sms();

// tiles.cu
// with_pairs: also build the union lists and order of query-tile pairs (the
// head-dimension-128 forward walks those)
// count_only: per-tile statistics, live counts and their scan only (the
// header's n_live then holds the total; no lists are written)
cudaError_t launch_tiles(int mode, const int32_t* q_idx, const int32_t* k_idx,
                         const int32_t* q_hash, const int32_t* k_hash,
                         int B, int H, int Tq, int Tk, unsigned flags,
                         char* ws, const AttnWs& L, cudaStream_t st, bool with_pairs = true,
                         bool count_only = false);

// SCFA_FLAG_VALIDATE: contract checks of the index inputs into the status word
cudaError_t launch_validate(int mode, bool original, const int32_t* q_idx, const int32_t* k_idx,
                            const int32_t* q_hash, const int32_t* k_hash, int B, int H, int Tq, int Tk, int To,
                            char* ws, const AttnWs& L, cudaStream_t st);

// lsh.cu
// status: a device int the tensor-core path may raise a timeout in (NULL keeps
// the CUDA-core kernel)
cudaError_t launch_lsh_hash(const uint16_t* x, const uint16_t* R, long long rows, int D, int m,
                            int32_t* hash, int* status, cudaStream_t st);
// one rotation per head: R is [H][D][m], head h of x ([B,H,T,D]) uses R[h]
cudaError_t launch_lsh_hash_heads(const uint16_t* x, const uint16_t* R, int B, int H, int T, int D, int m,
                                  int32_t* hash, int* status, cudaStream_t st);
int* lsh_scratch_status();  // device status word of the workspace-free lsh_hash call
cudaError_t launch_lsh_hash_cuda(const uint16_t* x, const uint16_t* R, long long rows, int D, int m,
                                 int32_t* hash, cudaStream_t st);
// chunk_ws: the workspace's chunk array (used when T > kSortChunk)
cudaError_t launch_bucket_sort(const int32_t* hash, int BH, int T, int n_buckets,
                               int32_t* perm, int32_t* hash_sorted, int32_t* bucket_off,
                               int32_t* chunk_ws, cudaStream_t st, int Ts = 0, int pad = 0);
// Ts rows per head in the sorted tensor, To in the original-order one
cudaError_t launch_gather(const uint16_t* x, const int32_t* perm, int BH, int Ts, int To, int D,
                          uint16_t* out, bool unsort, cudaStream_t st);
// bucket ids outside [0, nb) -> SCFA_ERR_INVALID in *status
cudaError_t launch_ids_check(const int32_t* ids, long long n, int nb, int* status, cudaStream_t st);
// plain sorted order (perm_u, off_u) -> tile-aligned order of Ts rows per head
cudaError_t launch_tiled_layout(const int32_t* perm_u, const int32_t* off_u, int BH, int T, int Ts, int nb, int pad,
                                int32_t* perm, int32_t* hash_sorted, int32_t* start, cudaStream_t st);

// attn_fwd.cu / attn_bwd.cu
struct AttnArgs {
  int mode;
  int B, H, Tq, Tk, D;
  float scale;
  const uint16_t *q, *k, *v, *o, *do_;
  const float* lse_in;
  const int32_t *q_idx, *k_idx, *q_hash, *k_hash;
  uint16_t* o_out;
  float* lse_out;
  uint16_t *dq, *dk, *dv;
  // hash mode with SCFA_FLAG_ORIGINAL_ORDER: destination row (within the
  // head) of each sorted query / key row; null = rows stay in place
  const int32_t *q_rows, *k_rows;
  int To;  // rows per head of the original-order tensors (= Tq without a row map)
  // SCFA_FLAG_KEEP_O32: the fp32 copy of O in the workspace (the forward
  // writes it, the backward pre-pass reads it); null otherwise
  float* o32;
  int stall;  // SCFA_FLAG_DEBUG_STALL
  // SCFA_FLAG_GATHER_Q: q and do, SCFA_FLAG_GATHER_KV: k and v are
  // original-order [B,H,To,D] tensors whose rows the kernels gather through
  // q_idx / k_idx
  int gather_q, gather_kv;
  char* ws;
  const AttnWs* L;
};
// 2-D map over `rows` rows of a bf16 [rows][D] tensor; box = 64 columns x 1
// row (for tile::gather4), 128-byte swizzle
bool make_tmap_bf16_rows(CUtensorMap* map, const void* base, int D, long long rows);
cudaError_t launch_attn_fwd(const AttnArgs& a, cudaStream_t st);

// profiling hook: events recorded around the main fwd (0) / bwd (1) kernel
void record_kernel_event(int which, bool start, cudaStream_t st);
cudaError_t launch_attn_bwd(const AttnArgs& a, cudaStream_t st);

}  // namespace scfa
