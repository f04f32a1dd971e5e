// The QK-sparse selection step: the page's QK-sparse mode ("SCFA 解决方案",
// part 1 "QK-Sparse") takes queries and keys that an upstream step dropped,
// compacted into Q/K/V with their original positions q_idx / k_idx. Given a
// per-head keep mask (the policy that sets it is the caller's), this writes
// the positions of the kept tokens in ascending order, padded with a
// sentinel, and the kept count; the rows themselves then move with
// lsh_gather (compaction, zero rows at the sentinels) and lsh_unsort
// (gradients back to full length).
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace scfa {
namespace {

constexpr int kSelectThreads = 512;

// One CTA per (b,h): thread t owns a contiguous slice of the mask; a block
// scan of the slice counts gives each thread its first output slot.
__global__ void __launch_bounds__(kSelectThreads) qk_select_kernel(const uint8_t* __restrict__ keep, int T, int Tc,
                                                                  int32_t sentinel, int32_t* __restrict__ idx,
                                                                  int32_t* __restrict__ count) {
  __shared__ int wsum[kSelectThreads / 32];
  __shared__ int s_total;
  const long long bh = blockIdx.x;
  const uint8_t* k = keep + bh * T;
  int32_t* out = idx + bh * Tc;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int per = (T + kSelectThreads - 1) / kSelectThreads;
  const int b0 = min(T, tid * per), b1 = min(T, b0 + per);
  int c = 0;
  for (int i = b0; i < b1; ++i) c += k[i] != 0;
  int x = c;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = lane < kSelectThreads / 32 ? wsum[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kSelectThreads / 32) wsum[lane] = s;
    if (lane == 31) s_total = s;
  }
  __syncthreads();
  int run = x - c + (w > 0 ? wsum[w - 1] : 0);
  for (int i = b0; i < b1; ++i) {
    if (k[i] != 0) {
      if (run < Tc) out[run] = i;
      ++run;
    }
  }
  const int total = s_total;
  for (int s = min(total, Tc) + tid; s < Tc; s += kSelectThreads) out[s] = sentinel;
  if (tid == 0) count[bh] = total;
}

}  // namespace
}  // namespace scfa

using namespace scfa;

extern "C" scfa_status scfa_qk_select(const uint8_t* keep, int B, int H, int T, int Tc, int32_t sentinel,
                                      int32_t* idx, int32_t* count, void* stream) {
  if (!keep || !idx || !count || B < 1 || H < 1 || T < 1 || Tc < 1) return SCFA_ERR_INVALID;
  if (sentinel >= 0 && sentinel < T) return SCFA_ERR_INVALID;  // a sentinel must name no token
  const long long BH = static_cast<long long>(B) * H;
  if (BH > INT_MAX) return SCFA_ERR_INVALID;
  qk_select_kernel<<<static_cast<int>(BH), kSelectThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      keep, T, Tc, sentinel, idx, count);
  return cudaGetLastError() == cudaSuccess ? SCFA_OK : SCFA_ERR_CUDA;
}
