// LSH bucket ids, stable bucket sort, row gather and unsort.
//
// Page: "Faster Causal Attention Over Large Sequences Through Sparse Flash
// Attention" (deep-paper.org), section "动态稀疏性为何会破坏它", item 2 (LSH
// groups similar tokens into buckets, as in Reformer) and section "SCFA
// 解决方案" part 2 (queries and keys carry bucket ids and original indices;
// reordering by bucket breaks the causal order). The construction is the
// random-rotation argmax h(x) = argmax_j [x R, -x R]_j, R a [D, m] Gaussian.
//
// Bucket ids are defined on EXACT values (ties -> smallest j). The fast path
// evaluates x R in fp32: every bf16 x bf16 product is exact inside an FMA, so
// each dot product is off by at most gamma_D * sum_d |x_d R_dc| plus one
// half-ulp of the smallest subnormal per step. A row whose top candidate
// leads every other candidate by more than the sum of both bounds (doubled
// for slack) keeps its fp32 argmax. Other rows are recomputed exactly: each
// product is an integer (8-bit x 8-bit significands) times a power of two in
// [2^-266, 2^240], so a 576-bit two's-complement fixed-point accumulator with
// its least significant bit at 2^-266 holds every sum of up to 256 products
// exactly.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace scfa {
namespace {

constexpr int kLimbs = 18;        // 18 x 32 = 576 bits
constexpr int kFixLsbExp = -266;  // exponent of the accumulator's lowest bit

struct Fix576 {
  uint32_t w[kLimbs];
};

__device__ __forceinline__ void fix_zero(Fix576& a) {
#pragma unroll
  for (int i = 0; i < kLimbs; ++i) a.w[i] = 0;
}

// bf16 bits -> (negative, integer significand, exponent): value = +-M * 2^E
__device__ __forceinline__ void bf16_parts(uint16_t b, bool* neg, uint32_t* M, int* E) {
  *neg = (b >> 15) != 0;
  const int e = (b >> 7) & 0xFF;
  const uint32_t mant = b & 0x7Fu;
  if (e == 0) {
    *M = mant;
    *E = -133;
  } else {
    *M = mant | 0x80u;
    *E = e - 134;
  }
}

// a += (neg ? -1 : 1) * mag * 2^(shift + kFixLsbExp), 0 <= shift <= 506, mag < 2^16
__device__ void fix_add(Fix576& a, uint32_t mag, int shift, bool neg) {
  if (mag == 0) return;
  const int L = shift >> 5;
  const uint64_t v = static_cast<uint64_t>(mag) << (shift & 31);
  const uint32_t part[2] = {static_cast<uint32_t>(v), static_cast<uint32_t>(v >> 32)};
  if (!neg) {
    uint64_t carry = 0;
    for (int i = L; i < kLimbs; ++i) {
      const uint64_t add = (i - L < 2 ? part[i - L] : 0u);
      const uint64_t s = static_cast<uint64_t>(a.w[i]) + add + carry;
      a.w[i] = static_cast<uint32_t>(s);
      carry = s >> 32;
      if (i - L >= 1 && carry == 0) break;
    }
  } else {
    uint64_t borrow = 0;
    for (int i = L; i < kLimbs; ++i) {
      const uint64_t sub = (i - L < 2 ? part[i - L] : 0u) + borrow;
      const uint64_t cur = a.w[i];
      a.w[i] = static_cast<uint32_t>(cur - sub);
      borrow = (cur < sub) ? 1u : 0u;
      if (i - L >= 1 && borrow == 0) break;
    }
  }
}

__device__ void fix_negate(Fix576& a) {
  uint64_t carry = 1;
  for (int i = 0; i < kLimbs; ++i) {
    const uint64_t s = static_cast<uint64_t>(~a.w[i]) + carry;
    a.w[i] = static_cast<uint32_t>(s);
    carry = s >> 32;
  }
}

// signed compare: returns true iff a > b
__device__ bool fix_greater(const Fix576& a, const Fix576& b) {
  const int ta = static_cast<int>(a.w[kLimbs - 1]), tb = static_cast<int>(b.w[kLimbs - 1]);
  if (ta != tb) return ta > tb;
  for (int i = kLimbs - 2; i >= 0; --i)
    if (a.w[i] != b.w[i]) return a.w[i] > b.w[i];
  return false;
}

__device__ void fix_dot(const uint16_t* __restrict__ x, const uint16_t* __restrict__ R, int D, int m, int c,
                        Fix576& acc) {
  fix_zero(acc);
  for (int d = 0; d < D; ++d) {
    bool nx, nr;
    uint32_t Mx, Mr;
    int Ex, Er;
    bf16_parts(x[d], &nx, &Mx, &Ex);
    bf16_parts(R[d * m + c], &nr, &Mr, &Er);
    fix_add(acc, Mx * Mr, Ex + Er - kFixLsbExp, nx != nr);
  }
}

// Exact argmax over [x R, -x R] with the smallest index on ties.
__device__ int exact_bucket(const uint16_t* __restrict__ x, const uint16_t* __restrict__ R, int D, int m) {
  Fix576 best, cur;
  int best_j = 0;
  fix_dot(x, R, D, m, 0, best);
  for (int j = 1; j < 2 * m; ++j) {
    fix_dot(x, R, D, m, j % m, cur);
    if (j >= m) fix_negate(cur);
    if (fix_greater(cur, best)) {
      best = cur;
      best_j = j;
    }
  }
  return best_j;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// One thread per row; R staged in shared memory as fp32 [D][m].
__global__ void lsh_hash_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ R,
                                long long rows, int D, int m, int32_t* __restrict__ hash) {
  extern __shared__ float sR[];
  for (int i = threadIdx.x; i < D * m; i += blockDim.x) sR[i] = bf16_to_f32(R[i]);
  __syncthreads();
  // fp32 rounding bound of one dot product, doubled: 2 * gamma_D with gamma_D < (D+1) 2^-24
  const float rel = static_cast<float>(D + 1) * 0x1p-23f;
  const float absb = static_cast<float>(D) * 0x1p-148f;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long r = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; r < rows; r += stride) {
    const uint16_t* xr = x + r * D;
    float xv[256];
    for (int d8 = 0; d8 < D; d8 += 8) {
      const uint4 u = *reinterpret_cast<const uint4*>(xr + d8);
      const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        xv[d8 + 2 * t] = __uint_as_float(ws[t] << 16);
        xv[d8 + 2 * t + 1] = __uint_as_float(ws[t] & 0xFFFF0000u);
      }
    }
    float top = -INFINITY, second = -INFINITY, emax = 0.f;
    int top_j = 0;
    for (int c = 0; c < m; ++c) {
      float s = 0.f, a = 0.f;
      for (int d = 0; d < D; ++d) {
        const float rv = sR[d * m + c];
        s = fmaf(xv[d], rv, s);
        a = fmaf(fabsf(xv[d]), fabsf(rv), a);
      }
      emax = fmaxf(emax, a * rel + absb);
      // candidate c (+s) and candidate m + c (-s)
      const float cand[2] = {s, -s};
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const float v = cand[t];
        if (v > top) {
          second = top;
          top = v;
          top_j = c + t * m;
        } else if (v > second) {
          second = v;
        }
      }
    }
    // certified when the lead beats twice the largest per-candidate bound
    int h = top_j;
    if (!(top - second > 2.f * emax * 1.0001f)) h = exact_bucket(xr, R, D, m);
    hash[r] = h;
  }
}

// Stable counting sort of one (b,h) row of bucket ids per CTA. Warp w owns a
// contiguous slice of the row; per-warp histograms give each warp its start
// in every bucket, and the warp then scatters its slice in order, ranking
// equal ids inside each 32-element step with __match_any_sync.
__global__ void bucket_sort_kernel(const int32_t* __restrict__ hash, int T, int nb,
                                   int32_t* __restrict__ perm, int32_t* __restrict__ hash_sorted,
                                   int32_t* __restrict__ bucket_off) {
  extern __shared__ int32_t hist[];  // [nwarps][nb], then [nb] totals
  const int nw = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long bh = blockIdx.x;
  const int32_t* hrow = hash + bh * T;
  int32_t* prow = perm + bh * T;
  int32_t* srow = hash_sorted + bh * T;
  int32_t* orow = bucket_off + bh * (nb + 1);
  int32_t* tot = hist + nw * nb;
  for (int i = threadIdx.x; i < (nw + 1) * nb; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int per = ((T + nw - 1) / nw + 31) / 32 * 32;
  const int b0 = min(T, w * per), b1 = min(T, b0 + per);
  int32_t* my = hist + w * nb;
  for (int base = b0; base < b1; base += 32) {
    const int i = base + lane;
    const int h = i < b1 ? hrow[i] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, h);
    if (h >= 0 && (peers & ((1u << lane) - 1u)) == 0) my[h] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // per bucket: exclusive prefix over warps; totals
  for (int c = threadIdx.x; c < nb; c += blockDim.x) {
    int run = 0;
    for (int ww = 0; ww < nw; ++ww) {
      const int t = hist[ww * nb + c];
      hist[ww * nb + c] = run;
      run += t;
    }
    tot[c] = run;
  }
  __syncthreads();
  // exclusive scan of the totals over buckets (warp 0), written to bucket_off
  if (w == 0) {
    int run = 0;
    for (int base = 0; base < nb; base += 32) {
      const int c = base + lane;
      const int v = c < nb ? tot[c] : 0;
      int x = v;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (c < nb) {
        tot[c] = run + x - v;
        orow[c] = run + x - v;
      }
      run += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) orow[nb] = run;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < nb; c += blockDim.x) {
    const int base = tot[c];
    for (int ww = 0; ww < nw; ++ww) hist[ww * nb + c] += base;
  }
  __syncthreads();
  for (int base = b0; base < b1; base += 32) {
    const int i = base + lane;
    const int h = i < b1 ? hrow[i] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, h);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int start = h >= 0 ? my[h] : 0;
    __syncwarp();
    if (h >= 0) {
      prow[start + rank] = i;
      srow[start + rank] = h;
      if (rank == 0) my[h] = start + __popc(peers);
    }
    __syncwarp();
  }
}

// 16-byte vector row moves. gather: out[s] = x[perm[s]]; unsort: out[perm[s]] = x[s].
__global__ void row_move_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ perm,
                                long long rows, int T, int chunks, uint4* __restrict__ out, int unsort) {
  const long long n = rows * chunks;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < n; g += stride) {
    const long long row = g / chunks;
    const int ch = static_cast<int>(g - row * chunks);
    const long long head0 = row - row % T;
    const int p = perm[row];
    if (p < 0 || p >= T) continue;
    if (unsort) out[(head0 + p) * chunks + ch] = x[g];
    else out[g] = x[(head0 + p) * chunks + ch];
  }
}

}  // namespace

cudaError_t launch_lsh_hash(const uint16_t* x, const uint16_t* R, long long rows, int D, int m,
                            int32_t* hash, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(D) * m * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(lsh_hash_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int block = 128;
  long long g = (rows + block - 1) / block;
  const long long cap = static_cast<long long>(num_sms()) * 16;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  lsh_hash_kernel<<<static_cast<int>(g), block, smem, st>>>(x, R, rows, D, m, hash);
  return cudaGetLastError();
}

cudaError_t launch_bucket_sort(const int32_t* hash, int BH, int T, int nb,
                               int32_t* perm, int32_t* hash_sorted, int32_t* bucket_off, cudaStream_t st) {
  const size_t budget = 160 * 1024;
  int nw = static_cast<int>(budget / (static_cast<size_t>(nb) * sizeof(int32_t))) - 1;
  if (nw > 32) nw = 32;
  if (nw < 1) nw = 1;
  const size_t smem = static_cast<size_t>(nw + 1) * nb * sizeof(int32_t);
  cudaError_t e = cudaFuncSetAttribute(bucket_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  bucket_sort_kernel<<<BH, nw * 32, smem, st>>>(hash, T, nb, perm, hash_sorted, bucket_off);
  return cudaGetLastError();
}

cudaError_t launch_gather(const uint16_t* x, const int32_t* perm, int BH, int T, int D,
                          uint16_t* out, bool unsort, cudaStream_t st) {
  const int chunks = D / 8;
  const long long rows = static_cast<long long>(BH) * T;
  const long long n = rows * chunks;
  const int block = 256;
  long long g = (n + block - 1) / block;
  const long long cap = static_cast<long long>(num_sms()) * 16;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  row_move_kernel<<<static_cast<int>(g), block, 0, st>>>(reinterpret_cast<const uint4*>(x), perm, rows, T, chunks,
                                                         reinterpret_cast<uint4*>(out), unsort ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace scfa
