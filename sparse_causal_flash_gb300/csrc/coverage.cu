// Pair counts: how many admissible (query, key) pairs the live tiles cover,
// and how many a Reformer-style chunked attention would cover.
//
// Page: "Faster Causal Attention Over Large Sequences Through Sparse Flash
// Attention" (deep-paper.org), section "实验与结果": against Reformer, SCFA
// hash-sparse attention covers 100% of the bucket collisions while Reformer's
// coverage drops (Fig. 4). A pair (query r, key c) is admissible when the
// element mask of the mode keeps it: q_idx >= k_idx (QK), r >= c (dense), and
// in hash mode also q_hash == k_hash.
//
// scfa_count_pairs walks the live-tile list held in a workspace (CSR by query
// tile) and counts the admissible pairs inside each live tile: one warp per
// query tile, lane u holding query rows u, u + 32, u + 64, u + 96, the key
// tile's metadata staged in shared memory. 100% coverage means this count
// equals the admissible pairs of the whole problem.
//
// scfa_count_chunked_pairs counts, in hash mode on bucket-sorted rows, the
// admissible pairs whose key lies in the query's chunk of `chunk` sorted rows
// or in the chunk before it (the chunking of Reformer's LSH attention): one
// thread per query.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace scfa {
namespace {

constexpr int kCountWarps = 8;

__global__ void __launch_bounds__(kCountWarps * 32)
count_live_pairs_kernel(int mode, const int32_t* __restrict__ q_idx, const int32_t* __restrict__ k_idx,
                        const int32_t* __restrict__ q_hash, const int32_t* __restrict__ k_hash,
                        int Tq, int Tk, int nQt, long long n_qtiles, const int32_t* __restrict__ row_ptr,
                        const int* ws_header, unsigned long long* __restrict__ count) {
  const int32_t* const cols = ws_list<int32_t>(ws_header, kListCols);
  __shared__ int32_t kid[kCountWarps][kTile];
  __shared__ int32_t khs[kCountWarps][kTile];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  unsigned long long total = 0;
  for (long long g = static_cast<long long>(blockIdx.x) * kCountWarps + w; g < n_qtiles;
       g += static_cast<long long>(gridDim.x) * kCountWarps) {
    const long long bh = g / nQt;
    const int i = static_cast<int>(g % nQt);
    int qi[4], qh[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = i * kTile + lane + 32 * u;
      const bool v = r < Tq;
      const long long gr = bh * Tq + r;
      qi[u] = !v ? INT_MIN : (mode == SCFA_MODE_DENSE ? r : q_idx[gr]);
      qh[u] = (v && mode == SCFA_MODE_HASH) ? q_hash[gr] : 0;
    }
    for (int e = row_ptr[g]; e < row_ptr[g + 1]; ++e) {
      const int j = cols[e];
      __syncwarp();
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = j * kTile + lane + 32 * u;
        const bool v = c < Tk;
        const long long gc = bh * Tk + c;
        kid[w][lane + 32 * u] = !v ? INT_MAX : (mode == SCFA_MODE_DENSE ? c : k_idx[gc]);
        khs[w][lane + 32 * u] = (v && mode == SCFA_MODE_HASH) ? k_hash[gc] : INT_MIN;
      }
      __syncwarp();
      unsigned n = 0;
      for (int c = 0; c < kTile; ++c) {
        const int kc = kid[w][c];
        const int hc = khs[w][c];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          bool adm = qi[u] >= kc && kc != INT_MAX;
          if (mode == SCFA_MODE_HASH) adm = adm && qh[u] == hc;
          n += adm ? 1u : 0u;
        }
      }
      total += n;
    }
  }
  for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
  if (lane == 0 && total) atomicAdd(count, total);
}

__global__ void count_chunked_pairs_kernel(const int32_t* __restrict__ q_idx, const int32_t* __restrict__ k_idx,
                                           const int32_t* __restrict__ q_hash, const int32_t* __restrict__ k_hash,
                                           long long rows, int T, int chunk, unsigned long long* __restrict__ count) {
  unsigned long long total = 0;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < rows;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long bh = t / T;
    const int s = static_cast<int>(t - bh * T);
    const int qi = q_idx[t], qh = q_hash[t];
    const int c = s / chunk;
    const int lo = c > 0 ? (c - 1) * chunk : 0;
    const int hi = min(T, (c + 1) * chunk);
    const int32_t* ki = k_idx + bh * T;
    const int32_t* kh = k_hash + bh * T;
    for (int k = lo; k < hi; ++k) total += (kh[k] == qh && qi >= ki[k]) ? 1u : 0u;
  }
  for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
  if ((threadIdx.x & 31) == 0 && total) atomicAdd(count, total);
}

}  // namespace
}  // namespace scfa

using namespace scfa;

extern "C" scfa_status scfa_count_pairs(int mode, const int32_t* q_idx, const int32_t* k_idx, const int32_t* q_hash,
                                        const int32_t* k_hash, int B, int H, int Tq, int Tk, int D, const void* ws,
                                        size_t ws_bytes, unsigned long long* count, void* stream) {
  if (!ws || !count || B < 1 || H < 1 || Tq < 1 || Tk < 1) return SCFA_ERR_INVALID;
  if (mode != SCFA_MODE_DENSE && (!q_idx || !k_idx)) return SCFA_ERR_INVALID;
  if (mode == SCFA_MODE_HASH && (!q_hash || !k_hash)) return SCFA_ERR_INVALID;
  AttnWs L;  // row pointers at their fixed place; the lists where the builder recorded them
  if (!attn_ws_layout(mode, 0, B, H, Tq, Tk, D, &L, 0)) return SCFA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < L.total) return SCFA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const char* w = static_cast<const char*>(ws);
  if (cudaMemsetAsync(count, 0, sizeof(unsigned long long), st) != cudaSuccess) return SCFA_ERR_CUDA;
  long long blocks = (L.n_qtiles + kCountWarps - 1) / kCountWarps;
  if (blocks > 16LL * num_sms()) blocks = 16LL * num_sms();
  count_live_pairs_kernel<<<static_cast<int>(blocks), kCountWarps * 32, 0, st>>>(
      mode, q_idx, k_idx, q_hash, k_hash, Tq, Tk, L.nQt, L.n_qtiles, reinterpret_cast<const int32_t*>(w + L.row_ptr),
      reinterpret_cast<const int*>(w + L.header), count);
  return cudaGetLastError() == cudaSuccess ? SCFA_OK : SCFA_ERR_CUDA;
}

extern "C" scfa_status scfa_count_chunked_pairs(const int32_t* q_idx, const int32_t* k_idx, const int32_t* q_hash,
                                                const int32_t* k_hash, int B, int H, int T, int chunk,
                                                unsigned long long* count, void* stream) {
  if (!q_idx || !k_idx || !q_hash || !k_hash || !count || B < 1 || H < 1 || T < 1 || chunk < 1)
    return SCFA_ERR_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(count, 0, sizeof(unsigned long long), st) != cudaSuccess) return SCFA_ERR_CUDA;
  const long long rows = static_cast<long long>(B) * H * T;
  long long blocks = (rows + 255) / 256;
  if (blocks > 16LL * num_sms()) blocks = 16LL * num_sms();
  count_chunked_pairs_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(q_idx, k_idx, q_hash, k_hash, rows, T, chunk,
                                                                      count);
  return cudaGetLastError() == cudaSuccess ? SCFA_OK : SCFA_ERR_CUDA;
}
