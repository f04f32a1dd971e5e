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

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// One thread per row. A block stages its rows in shared memory as bf16 pairs
// with a padded stride (thread t reads row t without bank conflicts) and R as
// fp32 [D][m4] (m4 = m rounded up to 4, zero columns appended), so one 16-byte
// load of R feeds four columns. A compiler memory barrier at each column group
// keeps the row loads inside the loop instead of hoisting the whole row into
// registers.
//
// Certification, three levels, all exact in outcome:
//  1. fp32: every candidate's fp32 value is within
//     gamma_D * sum_d |x_d R_dc| <= gamma_D * ||x||_2 * max_c ||R_c||_2
//     (Cauchy-Schwarz; both norms rounded up, plus subnormal slack) of its
//     exact value; emax doubles that. If the top beats the runner-up by more
//     than thr = 2 emax, the top is the exact argmax.
//  2. Otherwise only candidates within thr of the top can win; the pass keeps
//     the four best candidates, and if the fourth is also within thr (so more
//     might be) every column is screened again. Each remaining candidate gets
//     its EXACT value: with every product written as an integer times 2^e,
//     the sum is an exact 128-bit integer once the row's exponent span (of x
//     times that of R) is at most 100 bits, else an exact 576-bit one.
//     Candidates are compared in index order with a strict comparison, which
//     keeps the smallest index among exact ties.
constexpr int kHashRows = 256;

// The rows of x as n_seg x n_heads segments of seg_rows rows, segment (s, h)
// starting at row (s * n_heads + h) * seg_rows: with one rotation per head
// ([B,H,T,D] rows, seg_rows = T, n_seg = B, n_heads = H) the CTAs with
// blockIdx.y = h stage rotation h (R + h * r_stride) and take the chunks of
// head h's segments; with one shared rotation the rows are one segment.
struct LshSegs {
  long long seg_rows;
  int n_seg, n_heads;
  long long r_stride;
};
// chunk u (of n_seg * ceil(seg_rows / chunk)) of head h: first row, row count
__device__ __forceinline__ void seg_chunk(const LshSegs& g, int h, long long u, int chunk, long long* r0, int* nr) {
  const long long nc = (g.seg_rows + chunk - 1) / chunk;
  const long long sgi = u / nc, c = u - sgi * nc;
  *r0 = (sgi * g.n_heads + h) * g.seg_rows + c * chunk;
  const long long left = g.seg_rows - c * chunk;
  *nr = static_cast<int>(left < chunk ? left : chunk);
}
__host__ __device__ __forceinline__ long long seg_units(const LshSegs& g, int chunk) {
  return static_cast<long long>(g.n_seg) * ((g.seg_rows + chunk - 1) / chunk);
}

// R as fp32 [D][m4] in shared memory (zero columns appended), the largest
// column norm ||R_c||_2 rounded up and the exponent range of R's nonzero
// entries; every thread of the block calls it.
__device__ void lsh_prologue(const uint16_t* __restrict__ R, int D, int m, float* sR, float* rnmax_out,
                             int* r_emin_out, int* r_emax_out) {
  const int m4 = (m + 3) & ~3;
  for (int i = threadIdx.x; i < D * m4; i += blockDim.x) {
    const int d = i / m4, c = i % m4;
    sR[i] = c < m ? bf16_to_f32(R[d * m + c]) : 0.f;
  }
  // largest column norm ||R_c||_2 rounded up (squares of bf16 are exact in
  // fp32 unless subnormal: D 2^-148 slack; the sum: (D+2) 2^-22 relative),
  // and the range of the exponents E of the nonzero entries of R (value =
  // M 2^E with an integer M < 256)
  __shared__ float s_rn;
  __shared__ int s_remin, s_remax;
  if (threadIdx.x == 0) {
    s_rn = 0.f;
    s_remin = INT_MAX;
    s_remax = INT_MIN;
  }
  __syncthreads();
  {
    float mx = 0.f;
    for (int c = threadIdx.x; c < m; c += blockDim.x) {
      float ss = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) ss = fmaf(sR[d * m4 + c], sR[d * m4 + c], ss);
      mx = fmaxf(mx, sqrtf(ss * (1.f + static_cast<float>(D + 2) * 0x1p-22f) + static_cast<float>(D) * 0x1p-148f) *
                         1.000001f);
    }
    int emn = INT_MAX, emx = INT_MIN;
    for (int i = threadIdx.x; i < D * m4; i += blockDim.x) {
      bool ng;
      uint32_t M;
      int E;
      bf16_parts(static_cast<uint16_t>(__float_as_uint(sR[i]) >> 16), &ng, &M, &E);
      if (M != 0) {
        emn = min(emn, E);
        emx = max(emx, E);
      }
    }
    for (int o = 16; o; o >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      emn = min(emn, __shfl_xor_sync(0xffffffffu, emn, o));
      emx = max(emx, __shfl_xor_sync(0xffffffffu, emx, o));
    }
    if ((threadIdx.x & 31) == 0) {
      atomicMax(reinterpret_cast<int*>(&s_rn), __float_as_int(mx));
      atomicMin(&s_remin, emn);
      atomicMax(&s_remax, emx);
    }
  }
  __syncthreads();
  *rnmax_out = s_rn;
  *r_emin_out = s_remin;
  *r_emax_out = s_remax;
}

// Exact bucket id of one row: fp32 screening with the certified bound, exact
// re-evaluation of near ties. xrow: the row as bf16 pairs (32-bit words, in
// shared or global memory); xr: the same row in global memory.
__device__ int hash_row(const uint32_t* xrow, const uint16_t* __restrict__ xr, const float* sR,
                        const uint16_t* __restrict__ R, int D, int m, float rnmax, int r_emin, int r_emax) {
  const int m4 = (m + 3) & ~3;
  const float4* sR4 = reinterpret_cast<const float4*>(sR);
  // fp32 rounding bound of one dot product, doubled: 2 * gamma_D with gamma_D < (D+1) 2^-24
  const float rel = static_cast<float>(D + 1) * 0x1p-23f;
  const float absb = static_cast<float>(D) * 0x1p-148f;
    auto xval = [&](int d) -> float {
    const uint32_t w = xrow[d >> 1];
    return __uint_as_float((d & 1) ? (w & 0xFFFF0000u) : (w << 16));
  };
  // ||x||_2 rounded up: squares of bf16 are exact unless subnormal
  // (covered by D 2^-148), the fp32 sum by the (D+2) 2^-22 factor
  float l2sq = 0.f;
  for (int d = 0; d < D; ++d) l2sq = fmaf(xval(d), xval(d), l2sq);
  const float l2 = sqrtf(l2sq * (1.f + static_cast<float>(D + 2) * 0x1p-22f) + static_cast<float>(D) * 0x1p-148f) *
                   1.000001f;
  const float emax = l2 * rnmax * rel * 1.000001f + absb;
  // the four best candidates (values t, candidate indices j)
  float t0 = -INFINITY, t1 = -INFINITY, t2 = -INFINITY, t3 = -INFINITY;
  int j0 = 0, j1 = 0, j2 = 0;
  for (int c0 = 0; c0 < m4; c0 += 4) {
    asm volatile("" ::: "memory");
    float sv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int d2 = 0; d2 < D; d2 += 2) {
      const uint32_t w = xrow[d2 >> 1];
      const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xFFFF0000u);
      const float4 ra = sR4[(d2 * m4 + c0) >> 2];
      const float4 rb = sR4[((d2 + 1) * m4 + c0) >> 2];
      sv[0] = fmaf(x1, rb.x, fmaf(x0, ra.x, sv[0]));
      sv[1] = fmaf(x1, rb.y, fmaf(x0, ra.y, sv[1]));
      sv[2] = fmaf(x1, rb.z, fmaf(x0, ra.z, sv[2]));
      sv[3] = fmaf(x1, rb.w, fmaf(x0, ra.w, sv[3]));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u;
      if (c >= m) break;
      // candidate c (+s) and candidate m + c (-s)
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const float v = t ? -sv[u] : sv[u];
        const int j = c + t * m;
        if (v > t3) {
          if (v > t2) {
            t3 = t2;
            if (v > t1) {
              t2 = t1; j2 = j1;
              if (v > t0) { t1 = t0; j1 = j0; t0 = v; j0 = j; } else { t1 = v; j1 = j; }
            } else { t2 = v; j2 = j; }
          } else { t3 = v; }
        }
      }
    }
  }
  int h = j0;
  const float thr = 2.f * emax * 1.0001f;
  if (!(t0 - t1 > thr)) {
    const bool few = (t0 - t3 > thr);  // every candidate within thr of the top is among the four
    int cj[3];
    int nc = 0;
    if (few) {
      cj[nc++] = j0;
      if (t0 - t1 <= thr) cj[nc++] = j1;
      if (t0 - t2 <= thr) cj[nc++] = j2;
    }
    // exponent span of the row's products
    int xemin = INT_MAX, xemax = INT_MIN;
    for (int d = 0; d < D; ++d) {
      bool ng;
      uint32_t M;
      int E;
      bf16_parts(static_cast<uint16_t>(__float_as_uint(xval(d)) >> 16), &ng, &M, &E);
      if (M != 0) {
        xemin = min(xemin, E);
        xemax = max(xemax, E);
      }
    }
    const bool any_term = xemin != INT_MAX && r_emin != INT_MAX;
    const int ebase = any_term ? xemin + r_emin : 0;
    const bool fits128 = !any_term || (xemax + r_emax) - ebase <= 100;
    // exact sum of column c as an integer times 2^ebase (fits128 only)
    auto exact128 = [&](int c) -> __int128 {
      __int128 acc = 0;
      if (!any_term) return acc;
      for (int d = 0; d < D; ++d) {
        bool nx, nr2;
        uint32_t Mx, Mr;
        int Ex, Er;
        bf16_parts(static_cast<uint16_t>(__float_as_uint(xval(d)) >> 16), &nx, &Mx, &Ex);
        bf16_parts(static_cast<uint16_t>(__float_as_uint(sR[d * m4 + c]) >> 16), &nr2, &Mr, &Er);
        if (Mx == 0 || Mr == 0) continue;
        const __int128 term = static_cast<__int128>(Mx * Mr) << (Ex + Er - ebase);
        acc = (nx != nr2) ? acc - term : acc + term;
      }
      return acc;
    };
    auto is_cand = [&](int j) -> bool {
      if (few) {
        bool in = false;
        for (int k = 0; k < nc; ++k) in = in || (cj[k] == j);
        return in;
      }
      const int c = j < m ? j : j - m;
      float sc = 0.f;
      for (int d = 0; d < D; ++d) sc = fmaf(xval(d), sR[d * m4 + c], sc);
      const float vj = j < m ? sc : -sc;
      return (t0 - vj <= thr) || (vj != vj);
    };
    int best_j = -1;
    if (fits128) {
      __int128 best = 0;
      for (int j = 0; j < 2 * m; ++j) {
        if (!is_cand(j)) continue;
        const __int128 v = (j < m) ? exact128(j) : -exact128(j - m);
        if (best_j < 0 || v > best) {
          best = v;
          best_j = j;
        }
      }
    } else {
      Fix576 best, cur;
      for (int j = 0; j < 2 * m; ++j) {
        if (!is_cand(j)) continue;
        fix_dot(xr, R, D, m, j < m ? j : j - m, cur);
        if (j >= m) fix_negate(cur);
        if (best_j < 0 || fix_greater(cur, best)) {
          best = cur;
          best_j = j;
        }
      }
    }
    h = best_j >= 0 ? best_j : j0;
  }
  return h;
}

__global__ void __launch_bounds__(kHashRows) lsh_hash_kernel(const uint16_t* __restrict__ x,
                                                             const uint16_t* __restrict__ R, LshSegs sg,
                                                             int D, int m, int32_t* __restrict__ hash) {
  const int m4 = (m + 3) & ~3;
  const int xs = D / 2 + 1;  // padded row stride of the staged rows, in 32-bit words
  extern __shared__ float smem[];
  float* sR = smem;                                                  // [D][m4]
  uint32_t* sX = reinterpret_cast<uint32_t*>(smem + D * m4);         // [kHashRows][xs]
  float rnmax;
  int r_emin, r_emax;
  R += blockIdx.y * sg.r_stride;
  lsh_prologue(R, D, m, sR, &rnmax, &r_emin, &r_emax);
  const int wpr = D / 2;  // 32-bit words per row
  const long long n_units = seg_units(sg, kHashRows);
  for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
    long long r0;
    int nr;
    seg_chunk(sg, blockIdx.y, u, kHashRows, &r0, &nr);
    __syncthreads();
    const uint32_t* gx = reinterpret_cast<const uint32_t*>(x + r0 * D);
    for (int i = threadIdx.x; i < nr * wpr; i += blockDim.x) sX[(i / wpr) * xs + (i % wpr)] = gx[i];
    __syncthreads();
    if (threadIdx.x >= nr) continue;
    const long long r = r0 + threadIdx.x;
    hash[r] = hash_row(sX + threadIdx.x * xs, x + r * D, sR, R, D, m, rnmax, r_emin, r_emax);
  }
}

// Certified bucket id of one row, computed by a whole warp (the id is
// returned in every lane). xr: the row in global memory; sR: R as fp32
// [D][m4] in shared memory with rnmax / r_emin / r_emax from lsh_prologue;
// sx: D floats of shared memory for this warp. The lanes share the row,
// screen the columns lane + 32 k in fp32 with the same bound as the
// single-thread path (it holds for any summation order), and evaluate every
// candidate within the threshold of the top exactly in 128-bit integers, one
// candidate at a time split over the lanes; the largest value wins, the
// smallest index on ties. A row whose exponent span needs more than 128 bits
// goes to the single-thread path (576-bit accumulator) on lane 0.
__device__ int fix_row_warp(const uint16_t* __restrict__ xr, const uint16_t* __restrict__ R, const float* sR,
                            float* sx, int D, int m, float rnmax, int r_emin, int r_emax, int lane) {
  const int m4 = (m + 3) & ~3;
  const float rel = static_cast<float>(D + 1) * 0x1p-23f;
  const float absb = static_cast<float>(D) * 0x1p-148f;
  // stage the row; norm and exponent range of its nonzero entries
  float l2sq = 0.f;
  int xemin = INT_MAX, xemax = INT_MIN;
  for (int d = lane; d < D; d += 32) {
    const uint16_t bb = xr[d];
    const float v = bf16_to_f32(bb);
    sx[d] = v;
    l2sq = fmaf(v, v, l2sq);
    bool ng;
    uint32_t M;
    int E;
    bf16_parts(bb, &ng, &M, &E);
    if (M != 0) {
      xemin = min(xemin, E);
      xemax = max(xemax, E);
    }
  }
  for (int o = 16; o; o >>= 1) {
    l2sq += __shfl_xor_sync(0xffffffffu, l2sq, o);
    xemin = min(xemin, __shfl_xor_sync(0xffffffffu, xemin, o));
    xemax = max(xemax, __shfl_xor_sync(0xffffffffu, xemax, o));
  }
  __syncwarp();
  const float l2 = sqrtf(l2sq * (1.f + static_cast<float>(D + 2) * 0x1p-22f) + static_cast<float>(D) * 0x1p-148f) *
                   1.000001f;
  const float emax = l2 * rnmax * rel * 1.000001f + absb;
  const float thr = 2.f * emax * 1.0001f;
  // fp32 values of this lane's columns c = lane + 32 k (m <= 256: k < 8),
  // each summed over d in order; the warp's top value
  float scv[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) scv[k] = 0.f;
#pragma unroll 4
  for (int d = 0; d < D; ++d) {
    const float xv = sx[d];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = lane + 32 * k;
      if (c < m) scv[k] = fmaf(xv, sR[d * m4 + c], scv[k]);
    }
  }
  float best_v = -INFINITY;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if (lane + 32 * k < m) best_v = fmaxf(best_v, fmaxf(scv[k], -scv[k]));
  float t0 = best_v;
  for (int o = 16; o; o >>= 1) t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, o));
  // exact values of the candidates (within thr of the top, or NaN)
  const bool any_term = xemin != INT_MAX && r_emin != INT_MAX;
  const int ebase = any_term ? xemin + r_emin : 0;
  const bool fits128 = !any_term || (xemax + r_emax) - ebase <= 100;
  int h;
  if (fits128) {
    // candidates (column, sign) one at a time, each summed exactly by the
    // whole warp: lane l takes d = l, l + 32, ... (an integer sum, so the
    // order does not matter), then a butterfly of the 128-bit partials
    bool have = false;
    __int128 bv = 0;
    int bj = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = lane + 32 * k;
      const float sc = c < m ? scv[k] : 0.f;
      const bool cp = c < m && ((t0 - sc <= thr) || (sc != sc));
      const bool cn = c < m && ((t0 + sc <= thr) || (sc != sc));
      unsigned todo_c = __ballot_sync(0xffffffffu, cp || cn);
      const unsigned pos_mask = __ballot_sync(0xffffffffu, cp), neg_mask = __ballot_sync(0xffffffffu, cn);
      while (todo_c) {
        const int bit = __ffs(todo_c) - 1;
        todo_c &= todo_c - 1;
        const int cc = bit + 32 * k;
        __int128 acc = 0;
        if (any_term) {
          for (int d = lane; d < D; d += 32) {
            bool nx, nr2;
            uint32_t Mx, Mr;
            int Ex, Er;
            bf16_parts(static_cast<uint16_t>(__float_as_uint(sx[d]) >> 16), &nx, &Mx, &Ex);
            bf16_parts(static_cast<uint16_t>(__float_as_uint(sR[d * m4 + cc]) >> 16), &nr2, &Mr, &Er);
            if (Mx == 0 || Mr == 0) continue;
            const __int128 term = static_cast<__int128>(Mx * Mr) << (Ex + Er - ebase);
            acc = (nx != nr2) ? acc - term : acc + term;
          }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const unsigned long long lo = static_cast<unsigned long long>(acc);
          const long long hi = static_cast<long long>(acc >> 64);
          const unsigned long long olo = __shfl_xor_sync(0xffffffffu, lo, o);
          const long long ohi = __shfl_xor_sync(0xffffffffu, hi, o);
          acc += (static_cast<__int128>(ohi) << 64) | static_cast<__int128>(olo);
        }
        // (+) column cc, then (-) column cc + m: larger value, then smaller index
        if (((pos_mask >> bit) & 1u) && (!have || acc > bv || (acc == bv && cc < bj))) {
          bv = acc;
          bj = cc;
          have = true;
        }
        if (((neg_mask >> bit) & 1u) && (!have || -acc > bv || (-acc == bv && cc + m < bj))) {
          bv = -acc;
          bj = cc + m;
          have = true;
        }
      }
    }
    h = bj;
  } else {
    // exponent span beyond 128 bits: the single-thread path on lane 0
    int hh = 0;
    if (lane == 0) hh = hash_row(reinterpret_cast<const uint32_t*>(xr), xr, sR, R, D, m, rnmax, r_emin, r_emax);
    h = __shfl_sync(0xffffffffu, hh, 0);
  }
  return h;
}

// Second pass after the tensor-core pass: rows it left at -1 (near ties,
// non-finite or subnormal values, huge magnitudes) get the certified
// computation, one warp per row (fix_row_warp). A CTA takes kFixSeg
// consecutive rows at a time: its threads scan the ids, collect the flagged
// rows (a fraction of a percent) in a shared list, and the warps then share
// that list evenly.
constexpr int kFixWarps = 8;
constexpr int kFixSeg = 2048;  // rows per CTA step; the shared list holds up to this many

__global__ void __launch_bounds__(kFixWarps * 32, 2) lsh_fix_kernel(const uint16_t* __restrict__ x,
                                                                 const uint16_t* __restrict__ R, LshSegs sg,
                                                                 int D, int m, int32_t* __restrict__ hash) {
  extern __shared__ float smem[];
  const int m4 = (m + 3) & ~3;
  float* sR = smem;                      // [D][m4]
  float* sxall = smem + D * m4;          // [kFixWarps][D]
  float rnmax;
  int r_emin, r_emax;
  R += blockIdx.y * sg.r_stride;
  lsh_prologue(R, D, m, sR, &rnmax, &r_emin, &r_emax);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* sx = sxall + warp * D;
  __shared__ int s_n;
  __shared__ int s_list[kFixSeg];  // offsets of the flagged rows in the segment
  const long long n_units = seg_units(sg, kFixSeg);
  for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
    long long seg;
    int nseg;
    seg_chunk(sg, blockIdx.y, u, kFixSeg, &seg, &nseg);
    __syncthreads();  // the previous segment's list is consumed
    if (threadIdx.x == 0) s_n = 0;
    __syncthreads();
    // all eight ids of this thread are loaded before any is tested (one
    // memory latency, not eight)
    constexpr int kPer = kFixSeg / (kFixWarps * 32);
    int hv[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = threadIdx.x + j * kFixWarps * 32;
      hv[j] = i < nseg ? hash[seg + i] : 0;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if (hv[j] < 0) s_list[atomicAdd(&s_n, 1)] = threadIdx.x + j * kFixWarps * 32;
    __syncthreads();
    const int n_flag = s_n;
    for (int li = warp; li < n_flag; li += kFixWarps) {
      const long long r = seg + s_list[li];
      const int h = fix_row_warp(x + r * D, R, sR, sx, D, m, rnmax, r_emin, r_emax, lane);
      if (lane == 0) hash[r] = h;
      __syncwarp();
    }
  }
}

// ---------------------------------------------------------------------------
// Tensor-core first pass (D = 64 or 128, m a multiple of 8, m <= 256):
// X R for 128 rows at a time on tcgen05 (bf16 products are exact, fp32
// accumulation in TMEM), then per row the best and second-best candidate of
// [xR, -xR]. The row keeps the best when it leads by more than twice a bound
// on the accumulation error, taken loose (2^-14 ||x||_2 max_c ||R_c||_2: 4x
// D additions each losing 2^-23 of a partial sum at D = 128, 8x at D = 64);
// every other row, and every row with a subnormal, non-finite or huge value,
// is left at -1 for the certified second pass (lsh_fix_kernel).
// Roles: warp 0 TMA producer (x tiles, 4 stages), warp 1 MMA issuer and
// TMEM owner (one accumulator of m_pad columns per epilogue warpgroup), then
// two or four epilogue warpgroups taking the tiles in turn (thread = row =
// TMEM lane). R sits in shared memory for the whole kernel as the MN-major B
// operand ([D][64]-column swizzled sub-tiles).
// ---------------------------------------------------------------------------
constexpr int kTcStages = 4;
constexpr float kTcRel = 0x1p-14f;

template <int D>
struct __align__(1024) LshTcSmem {
  uint8_t x[kTcStages][D / 64][kTile * 128];  // [stage][64-column sub-tile][128 rows x 128 B]
  uint8_t r[4][D * 128];                      // up to 4 sub-tiles of [D rows][64 columns]
  uint64_t x_full[kTcStages], x_empty[kTcStages];
  uint64_t acc_full[4], acc_empty[4], drain;  // one accumulator per epilogue warpgroup
  uint32_t tmem_base;
  int abort_flag;
  int r_bad;  // R holds a subnormal or non-finite value: every row goes to the second pass
  float rnmax;
};

// G epilogue warpgroups take the tiles in turn, each with its own TMEM
// accumulator: four when four accumulators fit in TMEM (m <= 128), else two.
template <int D, int G>
__global__ void __launch_bounds__(64 + 128 * G, 1)
lsh_hash_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const uint16_t* __restrict__ R, LshSegs sg,
                   int m, int m_pad, int32_t* __restrict__ hash, int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  LshTcSmem<D>& sm = *reinterpret_cast<LshTcSmem<D>*>(smem_raw + pad);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // tiles: 128-row chunks of this head's segments (rotation blockIdx.y)
  const long long n_tiles = seg_units(sg, kTile);
  const int hd = blockIdx.y;
  R += hd * sg.r_stride;
  const uint32_t acc_cols = m_pad < 32 ? 32u : static_cast<uint32_t>(m_pad);
  const uint32_t need = acc_cols * G;
  const uint32_t tmem_cols = need <= 32 ? 32u : (need <= 64 ? 64u : (need <= 128 ? 128u : (need <= 256 ? 256u : 512u)));

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&sm.x_full[s], 1);
      mbar_init(&sm.x_empty[s], 1 + 128);  // the MMA commit and the 128 epilogue threads (row norms)
    }
    for (int b = 0; b < G; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], 128);
    }
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    sm.r_bad = 0;
    sm.rnmax = 0.f;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
  }
  __syncthreads();
  // R -> shared memory in the swizzled MN-major layout: sub-tile c / 64, row d,
  // 16-byte chunk (c % 64) / 8; columns past m are zero. Also the largest
  // column norm (rounded up) and a check for subnormal / non-finite entries.
  {
    const int n_sub = (m_pad + 63) / 64;
    for (int idx = threadIdx.x; idx < n_sub * D * 8; idx += blockDim.x) {
      const int st = idx / (D * 8), d = (idx / 8) % D, ch = idx % 8;
      uint32_t w[4];
      for (int u = 0; u < 4; ++u) {
        const int c0 = st * 64 + ch * 8 + 2 * u;
        const uint32_t lo = c0 < m ? R[static_cast<long long>(d) * m + c0] : 0u;
        const uint32_t hi = c0 + 1 < m ? R[static_cast<long long>(d) * m + c0 + 1] : 0u;
        w[u] = lo | (hi << 16);
        for (int k = 0; k < 2; ++k) {
          const uint32_t b = k ? hi : lo;
          const uint32_t e = (b >> 7) & 0xFFu, mant = b & 0x7Fu;
          if ((e == 0 && mant != 0) || e == 0xFFu) sm.r_bad = 1;
        }
      }
      *reinterpret_cast<uint4*>(&sm.r[st][0] + sw128_offset(d, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  {
    // column norms from the staged copy
    float mx = 0.f;
    for (int c = threadIdx.x; c < m; c += blockDim.x) {
      const uint8_t* sub = &sm.r[c >> 6][0];
      const int ch = (c & 63) >> 3, w16 = c & 7;
      float ss = 0.f;
      for (int d = 0; d < D; ++d) {
        const uint16_t b = *reinterpret_cast<const uint16_t*>(sub + sw128_offset(d, ch) + 2 * w16);
        const float v = bf16_to_f32(b);
        ss = fmaf(v, v, ss);
      }
      mx = fmaxf(mx, sqrtf(ss * (1.f + static_cast<float>(D + 2) * 0x1p-22f)) * 1.000001f);
    }
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) atomicMax(reinterpret_cast<int*>(&sm.rnmax), __float_as_int(mx));
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
        const int s = it % kTcStages;
        long long r0;
        int nr;
        seg_chunk(sg, hd, t, kTile, &r0, &nr);
        if (!mbar_wait(&sm.x_empty[s], ((it / kTcStages) & 1) ^ 1, abort_flag, status)) break;
        mbar_arrive_expect_tx(&sm.x_full[s], D * kTile * 2);
        for (int sub = 0; sub < D / 64; ++sub)
          tma_load_3d(sm.x[s][sub], &tm_x, &sm.x_full[s], sub * 64, static_cast<int>(r0), 0);
      }
      for (int d = 1; d <= kTcStages && d <= it; ++d) {
        const int i2 = it - d;
        mbar_wait_drain(&sm.x_full[i2 % kTcStages], (i2 / kTcStages) & 1, status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTile, m_pad, 0, 1);
      const uint64_t xdesc = smem_desc_sw128(smem_u32(sm.x[0][0]), 16, 1024);
      const uint64_t rdesc = smem_desc_sw128(smem_u32(sm.r[0]), D * 128, 1024);
      constexpr uint32_t kStage16 = (D / 64) * kTile * 128 >> 4;
      int it = 0;
      for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
        const int s = it % kTcStages, b = it % G;
        if (!mbar_wait(&sm.acc_empty[b], ((it / G) & 1) ^ 1, abort_flag, status)) break;
        if (!mbar_wait(&sm.x_full[s], (it / kTcStages) & 1, abort_flag, status)) break;
        tc_fence_after();
        const uint64_t a = xdesc + static_cast<uint64_t>(s * kStage16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(tmem + acc_cols * b, a + kstep_off16(kk, kTile * 128), rdesc + static_cast<uint64_t>(kk * 128),
                      idesc, kk > 0);
        tc_commit(&sm.acc_full[b]);
        tc_commit(&sm.x_empty[s]);
      }
      tc_commit(&sm.drain);
      mbar_wait_drain(&sm.drain, 0, status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int eg = (warp - 2) >> 2;      // epilogue warpgroup: tiles it with it % G == eg
    const int rr = quarter * 32 + lane;  // row of the tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float rnmax = sm.rnmax;
    const bool r_bad = sm.r_bad != 0;
    int it = eg;
    for (long long t = blockIdx.x + static_cast<long long>(eg) * gridDim.x; t < n_tiles;
         t += static_cast<long long>(G) * gridDim.x, it += G) {
      const int s = it % kTcStages, b = it % G;
      bool ok = mbar_wait(&sm.acc_full[b], (it / G) & 1, abort_flag, status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      // ||x||_2 of this row from the staged tile (rounded up), and a check
      // for subnormal entries. Both bf16 halves of a word at once: with a
      // the magnitude bits of a half, a + 0x7F80 reaches bit 15 iff the
      // exponent is nonzero, a + 0x7FFF iff a != 0 (neither carries out of
      // the half). A non-finite entry makes l2sq inf or NaN, which the
      // l2 < 2^60 test below turns away.
      float l2sq = 0.f;
      uint32_t sub_bits = 0;
#pragma unroll
      for (int sub = 0; sub < D / 64; ++sub) {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint4 q4 = *reinterpret_cast<const uint4*>(&sm.x[s][sub][0] + sw128_offset(rr, ch));
          const uint32_t wv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float lo = __uint_as_float(wv[u] << 16), hi = __uint_as_float(wv[u] & 0xFFFF0000u);
            l2sq = fmaf(lo, lo, fmaf(hi, hi, l2sq));
            const uint32_t a = wv[u] & 0x7FFF7FFFu;
            sub_bits |= (a + 0x7FFF7FFFu) & ~(a + 0x7F807F80u);
          }
        }
      }
      const bool x_bad = (sub_bits & 0x80008000u) != 0;
      mbar_arrive(&sm.x_empty[s]);
      const float l2 = sqrtf(l2sq * (1.f + static_cast<float>(D + 2) * 0x1p-22f)) * 1.000001f;
      const float emax = l2 * rnmax * kTcRel;
      // best and second best of [s, -s] over the m real columns
      float t0 = -INFINITY, t1 = -INFINITY;
      int j0 = 0;
      const uint32_t col0 = acc_cols * b;
      for (int c0 = 0; c0 < m_pad; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(lane_base + col0 + c0, v);
        tmem_wait_ld();
        tmem_ld_fence(v);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int c = c0 + u;
          if (c < m) {
            const float sv = __uint_as_float(v[u]);
            const float a = fmaxf(sv, -sv);
            const int j = sv >= 0.f ? c : c + m;  // for sv == 0 both tie: the smaller index, c
            const float bmin = fminf(sv, -sv);    // the other sign of the same column
            // the pair (a, bmin) enters the running top two
            if (a > t0) {
              t1 = fmaxf(t0, bmin);
              t0 = a;
              j0 = j;
            } else {
              t1 = fmaxf(t1, a);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.acc_empty[b]);
      long long r0;
      int nr;
      seg_chunk(sg, hd, t, kTile, &r0, &nr);
      const long long row = r0 + rr;
      if (rr < nr) {
        const bool clear = !r_bad && !x_bad && l2 < 0x1p60f && rnmax < 0x1p60f && (t0 - t1 > 2.f * emax * 1.0001f);
        hash[row] = clear ? j0 : -1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, tmem_cols);
}

// Stable counting sort of one (b,h) row of bucket ids per CTA. Warp w owns a
// contiguous slice of the row; per-warp histograms give each warp its start
// in every bucket, and the warp then scatters its slice in order, ranking
// equal ids inside each 32-element step with __match_any_sync.
//
// Rows longer than kSortChunk: CTA (row, chunk) sorts its chunk the same way,
// in three launches: mode 1 writes the chunk's bucket counts, mode 2 (one
// CTA per row, bucket_scan_kernel) turns them into the chunk's first output
// position per bucket and writes bucket_off, mode 2 scatters from those
// bases. Mode 0 is the whole row in one CTA.
//
// Ts > 0 (mode 0 only): the output is the tile-aligned layout directly (Ts
// rows per head): bucket b's rows start at bucket_off[b] = the sum over c < b
// of n_c rounded up to kTile, and the rows between a bucket's n_b rows and
// its next tile boundary, and all rows after the last bucket's tiles, are
// padding rows (position `pad`, bucket id b, nb - 1 after the last bucket).
__global__ void bucket_sort_kernel(const int32_t* __restrict__ hash, int T, int nb,
                                   int32_t* __restrict__ perm, int32_t* __restrict__ hash_sorted,
                                   int32_t* __restrict__ bucket_off, int mode, int chunk, int n_chunks,
                                   int32_t* __restrict__ chunk_ws, int Ts, int pad) {
  extern __shared__ int32_t hist[];  // [nwarps][nb], then [nb] totals, then [nb] counts (tile-aligned)
  __shared__ int s_end;              // tile-aligned: end of the last bucket's tiles
  const int nw = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool tiled = mode == 0 && Ts > 0;
  const int rs = tiled ? Ts : T;  // output rows per head
  const long long bh = mode == 0 ? blockIdx.x : blockIdx.x / n_chunks;
  const int ci = mode == 0 ? 0 : static_cast<int>(blockIdx.x % n_chunks);
  const int32_t* hrow = hash + bh * T;
  int32_t* prow = perm + bh * rs;
  int32_t* srow = hash_sorted + bh * rs;
  int32_t* orow = bucket_off + bh * (nb + 1);
  int32_t* cws = chunk_ws + (bh * n_chunks + ci) * nb;
  int32_t* tot = hist + nw * nb;
  int32_t* cnt = tot + nb;
  for (int i = threadIdx.x; i < (nw + 1) * nb; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int c_begin = mode == 0 ? 0 : min(T, ci * chunk);
  const int c_end = mode == 0 ? T : min(T, c_begin + chunk);
  const int len = c_end - c_begin;
  const int per = ((len + nw - 1) / nw + 31) / 32 * 32;
  const int b0 = c_begin + min(len, w * per), b1 = c_begin + min(len, w * per + per);
  int32_t* my = hist + w * nb;
  // the slice in steps of 32 ids, eight steps' ids loaded at once (one
  // memory latency per eight steps); an id outside [0, nb) takes no slot
  // (the id check reports it)
  constexpr int kSteps = 8;
  for (int base0 = b0; base0 < b1; base0 += 32 * kSteps) {
    int hv[kSteps];
#pragma unroll
    for (int u = 0; u < kSteps; ++u) {
      const int i = base0 + u * 32 + lane;
      const int h = i < b1 ? hrow[i] : -1;
      hv[u] = h >= nb ? -1 : h;
    }
#pragma unroll
    for (int u = 0; u < kSteps; ++u) {
      const int h = hv[u];
      const unsigned peers = __match_any_sync(0xffffffffu, h);
      if (h >= 0 && (peers & ((1u << lane) - 1u)) == 0) my[h] += __popc(peers);
      __syncwarp();
    }
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
  if (mode == 1) {
    for (int c = threadIdx.x; c < nb; c += blockDim.x) cws[c] = tot[c];
    return;
  }
  if (mode == 2) {
    for (int c = threadIdx.x; c < nb; c += blockDim.x) tot[c] = cws[c];
  } else if (w == 0) {
    // exclusive scan of the totals over buckets (warp 0), written to
    // bucket_off; tile-aligned, of the totals rounded up to kTile
    int run = 0;
    for (int base = 0; base < nb; base += 32) {
      const int c = base + lane;
      const int n_c = c < nb ? tot[c] : 0;
      const int v = tiled ? (n_c + kTile - 1) / kTile * kTile : n_c;
      int x = v;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (c < nb) {
        tot[c] = run + x - v;
        orow[c] = run + x - v;
        if (tiled) cnt[c] = n_c;
      }
      run += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) {
      orow[nb] = run;
      s_end = run;
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < nb; c += blockDim.x) {
    const int base = tot[c];
    for (int ww = 0; ww < nw; ++ww) hist[ww * nb + c] += base;
  }
  __syncthreads();
  for (int base0 = b0; base0 < b1; base0 += 32 * kSteps) {
    int hv[kSteps];
#pragma unroll
    for (int u = 0; u < kSteps; ++u) {
      const int i = base0 + u * 32 + lane;
      const int h = i < b1 ? hrow[i] : -1;
      hv[u] = h >= nb ? -1 : h;
    }
#pragma unroll
    for (int u = 0; u < kSteps; ++u) {
      const int i = base0 + u * 32 + lane;
      const int h = hv[u];
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
  if (tiled) {
    // padding rows: the rest of each bucket's last tile, then the tail
    for (int c = w; c < nb; c += nw) {
      const int a = tot[c] + cnt[c], e = tot[c] + (cnt[c] + kTile - 1) / kTile * kTile;
      for (int p = a + lane; p < e; p += 32) {
        prow[p] = pad;
        srow[p] = c;
      }
    }
    for (int p = s_end + threadIdx.x; p < Ts; p += blockDim.x) {
      prow[p] = pad;
      srow[p] = nb - 1;
    }
  }
}

// Per row (one CTA): bucket_off = exclusive scan over buckets of the summed
// chunk counts; each chunk's count is replaced by its first output position
// in that bucket (bucket start + counts of the earlier chunks).
__global__ void bucket_scan_kernel(int nb, int n_chunks, int32_t* __restrict__ chunk_ws,
                                   int32_t* __restrict__ bucket_off) {
  extern __shared__ int32_t tot2[];  // [nb]
  const long long bh = blockIdx.x;
  int32_t* cws = chunk_ws + bh * n_chunks * nb;
  int32_t* orow = bucket_off + bh * (nb + 1);
  for (int c = threadIdx.x; c < nb; c += blockDim.x) {
    int run = 0;
    for (int k = 0; k < n_chunks; ++k) {
      const int t = cws[k * nb + c];
      cws[k * nb + c] = run;
      run += t;
    }
    tot2[c] = run;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int run = 0;
    for (int base = 0; base < nb; base += 32) {
      const int c = base + lane;
      const int v = c < nb ? tot2[c] : 0;
      int x = v;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (c < nb) {
        tot2[c] = run + x - v;
        orow[c] = run + x - v;
      }
      run += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) orow[nb] = run;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < nb; c += blockDim.x) {
    const int start = tot2[c];
    for (int k = 0; k < n_chunks; ++k) cws[k * nb + c] += start;
  }
}

// 16-byte vector row moves between a sorted tensor of Ts rows per head and an
// original-order one of To rows per head. gather: sorted[s] = x[perm[s]], a
// zero row where perm[s] is outside [0, To) (a padding row); unsort:
// out[perm[s]] = sorted[s], skipping such rows.
__global__ void row_move_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ perm,
                                long long rows, int Ts, int To, int chunks, uint4* __restrict__ out, int unsort) {
  const long long n = rows * chunks;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < n; g += stride) {
    const long long row = g / chunks;  // sorted row over all heads
    const int ch = static_cast<int>(g - row * chunks);
    const long long bh = row / Ts;
    const int p = perm[row];
    const bool in = p >= 0 && p < To;
    const long long orig = (bh * To + p) * chunks + ch;
    if (unsort) {
      if (in) out[orig] = x[g];
    } else {
      out[g] = in ? x[orig] : make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

}  // namespace

bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, int D, long long T, long long BH);

__device__ int g_lsh_status;

int* lsh_scratch_status() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_lsh_status) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

template <int D>
static cudaError_t launch_lsh_tc(const uint16_t* x, const uint16_t* R, long long rows, const LshSegs& sg, int m,
                                 int32_t* hash, int* status, cudaStream_t st) {
  CUtensorMap tm;
  if (!make_tmap_bf16_3d(&tm, x, D, rows, 1)) return cudaErrorInvalidValue;
  const int m_pad = (m + 15) / 16 * 16;
  const size_t smem = sizeof(LshTcSmem<D>) + 1024;
  // four epilogue warpgroups when four accumulators fit in TMEM
  const int acc_cols = m_pad < 32 ? 32 : m_pad;
  const bool four = acc_cols * 4 <= 512;
  auto kern = four ? lsh_hash_tc_kernel<D, 4> : lsh_hash_tc_kernel<D, 2>;
  const int threads = 64 + 128 * (four ? 4 : 2);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // about one CTA per SM in all, split over the rotations
  const long long n_tiles = seg_units(sg, kTile);
  long long g = num_sms() / sg.n_heads;
  if (g > n_tiles) g = n_tiles;
  if (g < 1) g = 1;
  kern<<<dim3(static_cast<unsigned>(g), sg.n_heads), threads, smem, st>>>(tm, R, sg, m, m_pad, hash, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // certified second pass over the rows the first pass left at -1
  const size_t smem2 = static_cast<size_t>(D) * (((m + 3) & ~3) + kFixWarps) * sizeof(float);
  e = cudaFuncSetAttribute(lsh_fix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem2));
  if (e != cudaSuccess) return e;
  long long g2 = seg_units(sg, kFixSeg);
  const long long cap2 = 2LL * num_sms() / sg.n_heads;  // two CTAs per SM
  if (g2 > cap2) g2 = cap2;
  if (g2 < 1) g2 = 1;
  lsh_fix_kernel<<<dim3(static_cast<unsigned>(g2), sg.n_heads), kFixWarps * 32, smem2, st>>>(x, R, sg, D, m, hash);
  return cudaGetLastError();
}

static cudaError_t launch_lsh_segs(const uint16_t* x, const uint16_t* R, long long rows, const LshSegs& sg, int D,
                                   int m, int32_t* hash, int* status, cudaStream_t st) {
  // The tensor-core path needs D = 64 or 128, m a multiple of 8 (16-byte rows
  // of R), m <= 256 (one accumulator fits twice in TMEM) and a 16-byte aligned
  // x; other shapes take the CUDA-core kernel.
  const bool tc_ok = (D == 64 || D == 128) && m % 8 == 0 && m >= 8 && m <= 256 && status != nullptr &&
                     (reinterpret_cast<uintptr_t>(x) & 15u) == 0 && rows < (1ll << 31);
  if (tc_ok) return D == 64 ? launch_lsh_tc<64>(x, R, rows, sg, m, hash, status, st)
                            : launch_lsh_tc<128>(x, R, rows, sg, m, hash, status, st);
  const size_t smem = (static_cast<size_t>(D) * ((m + 3) & ~3) + static_cast<size_t>(kHashRows) * (D / 2 + 1)) *
                      sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(lsh_hash_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  long long g = seg_units(sg, kHashRows);
  const long long cap = static_cast<long long>(num_sms()) * 8 / sg.n_heads;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  lsh_hash_kernel<<<dim3(static_cast<unsigned>(g), sg.n_heads), kHashRows, smem, st>>>(x, R, sg, D, m, hash);
  return cudaGetLastError();
}

cudaError_t launch_lsh_hash(const uint16_t* x, const uint16_t* R, long long rows, int D, int m,
                            int32_t* hash, int* status, cudaStream_t st) {
  const LshSegs sg = {rows, 1, 1, 0};  // one rotation for every row
  return launch_lsh_segs(x, R, rows, sg, D, m, hash, status, st);
}

cudaError_t launch_lsh_hash_heads(const uint16_t* x, const uint16_t* R, int B, int H, int T, int D, int m,
                                  int32_t* hash, int* status, cudaStream_t st) {
  const LshSegs sg = {T, B, H, static_cast<long long>(D) * m};  // rotation h for the rows of head h
  return launch_lsh_segs(x, R, static_cast<long long>(B) * H * T, sg, D, m, hash, status, st);
}

cudaError_t launch_lsh_hash_cuda(const uint16_t* x, const uint16_t* R, long long rows, int D, int m,
                                 int32_t* hash, cudaStream_t st) {
  const LshSegs sg = {rows, 1, 1, 0};
  return launch_lsh_segs(x, R, rows, sg, D, m, hash, nullptr, st);
}

cudaError_t launch_bucket_sort(const int32_t* hash, int BH, int T, int nb,
                               int32_t* perm, int32_t* hash_sorted, int32_t* bucket_off, int32_t* chunk_ws,
                               cudaStream_t st, int Ts, int pad) {
  // per-warp histograms, the totals and (tile-aligned) the counts
  const int extra = Ts > 0 ? 2 : 1;
  const size_t budget = 160 * 1024;
  int nw = static_cast<int>(budget / (static_cast<size_t>(nb) * sizeof(int32_t))) - extra;
  if (nw > 32) nw = 32;
  if (nw < 1) nw = 1;
  const size_t smem = static_cast<size_t>(nw + extra) * nb * sizeof(int32_t);
  cudaError_t e = cudaFuncSetAttribute(bucket_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (Ts > 0) {
    // the tile-aligned layout straight from the sort: heads of one CTA only
    if (T > kSortChunk) return cudaErrorInvalidValue;
    bucket_sort_kernel<<<BH, nw * 32, smem, st>>>(hash, T, nb, perm, hash_sorted, bucket_off, 0, T, 1, nullptr, Ts,
                                                  pad);
    return cudaGetLastError();
  }
  if (T <= kSortChunk || chunk_ws == nullptr) {
    bucket_sort_kernel<<<BH, nw * 32, smem, st>>>(hash, T, nb, perm, hash_sorted, bucket_off, 0, T, 1, nullptr, 0, 0);
    return cudaGetLastError();
  }
  const int n_chunks = (T + kSortChunk - 1) / kSortChunk;
  const long long g = static_cast<long long>(BH) * n_chunks;
  bucket_sort_kernel<<<static_cast<int>(g), nw * 32, smem, st>>>(hash, T, nb, perm, hash_sorted, bucket_off, 1,
                                                                  kSortChunk, n_chunks, chunk_ws, 0, 0);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bucket_scan_kernel<<<BH, 256, static_cast<size_t>(nb) * sizeof(int32_t), st>>>(nb, n_chunks, chunk_ws, bucket_off);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bucket_sort_kernel<<<static_cast<int>(g), nw * 32, smem, st>>>(hash, T, nb, perm, hash_sorted, bucket_off, 2,
                                                                  kSortChunk, n_chunks, chunk_ws, 0, 0);
  return cudaGetLastError();
}

// Bucket ids given by the caller: any outside [0, nb) raises the status word.
__global__ void ids_check_kernel(const int32_t* __restrict__ ids, long long n, int nb, int* status) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  bool bad = false;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    bad |= ids[i] < 0 || ids[i] >= nb;
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) raise_status(status, SCFA_ERR_INVALID);
}

cudaError_t launch_ids_check(const int32_t* ids, long long n, int nb, int* status, cudaStream_t st) {
  long long g = (n + 255) / 256;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  ids_check_kernel<<<static_cast<int>(g), 256, 0, st>>>(ids, n, nb, status);
  return cudaGetLastError();
}

// Tile-aligned sorted layout. One warp per head: bucket b starts at row
// start[b] = sum over c < b of n_c rounded up to a multiple of kTile, so no
// tile holds two buckets; start[nb] is the end of the last bucket's tiles.
__global__ void tiled_offsets_kernel(const int32_t* __restrict__ off, int BH, int nb,
                                     int32_t* __restrict__ start) {
  const int lane = threadIdx.x & 31;
  const long long bh = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (bh >= BH) return;
  const int32_t* o = off + bh * (nb + 1);
  int32_t* s = start + bh * (nb + 1);
  int run = 0;
  for (int base = 0; base < nb; base += 32) {
    const int b = base + lane;
    const int v = b < nb ? (o[b + 1] - o[b] + kTile - 1) / kTile * kTile : 0;
    int x = v;
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += y;
    }
    if (b < nb) s[b] = run + x - v;
    run += __shfl_sync(0xffffffffu, x, 31);
  }
  if (lane == 0) s[nb] = run;
}

// Row p of the tile-aligned layout (Ts rows per head): the bucket b whose
// tiles hold p (the last start <= p), its rank r = p - start[b], and then
// either the r-th row of the bucket in the plain sorted order or, past the
// bucket's n_b rows and after the last bucket, a padding row: position `pad`
// and bucket id b (nb - 1 after the last bucket), so tile ranges keep one
// bucket each.
__global__ void tiled_spread_kernel(const int32_t* __restrict__ perm_u, const int32_t* __restrict__ off,
                                    const int32_t* __restrict__ start, int BH, int T, int Ts, int nb, int pad,
                                    int32_t* __restrict__ perm, int32_t* __restrict__ hash_sorted) {
  const long long n = static_cast<long long>(BH) * Ts;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < n; g += stride) {
    const long long bh = g / Ts;
    const int p = static_cast<int>(g - bh * Ts);
    const int32_t* s = start + bh * (nb + 1);
    const int32_t* o = off + bh * (nb + 1);
    int lo = 0, hi = nb - 1;  // last b in [0, nb) with s[b] <= p (s[0] = 0)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s[mid] <= p) lo = mid;
      else hi = mid - 1;
    }
    const int r = p - s[lo];
    const int n_b = o[lo + 1] - o[lo];
    perm[g] = r < n_b ? perm_u[bh * T + o[lo] + r] : pad;
    hash_sorted[g] = lo;
  }
}

cudaError_t launch_tiled_layout(const int32_t* perm_u, const int32_t* off_u, int BH, int T, int Ts, int nb, int pad,
                                int32_t* perm, int32_t* hash_sorted, int32_t* start, cudaStream_t st) {
  const int warps_per_block = 8;
  tiled_offsets_kernel<<<(BH + warps_per_block - 1) / warps_per_block, warps_per_block * 32, 0, st>>>(off_u, BH, nb,
                                                                                                      start);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long n = static_cast<long long>(BH) * Ts;
  long long g = (n + 255) / 256;
  const long long cap = static_cast<long long>(num_sms()) * 16;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  tiled_spread_kernel<<<static_cast<int>(g), 256, 0, st>>>(perm_u, off_u, start, BH, T, Ts, nb, pad, perm,
                                                           hash_sorted);
  return cudaGetLastError();
}

cudaError_t launch_gather(const uint16_t* x, const int32_t* perm, int BH, int Ts, int To, int D,
                          uint16_t* out, bool unsort, cudaStream_t st) {
  const int chunks = D / 8;
  const long long rows = static_cast<long long>(BH) * Ts;
  const long long n = rows * chunks;
  const int block = 256;
  long long g = (n + block - 1) / block;
  const long long cap = static_cast<long long>(num_sms()) * 16;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  row_move_kernel<<<static_cast<int>(g), block, 0, st>>>(reinterpret_cast<const uint4*>(x), perm, rows, Ts, To,
                                                         chunks, reinterpret_cast<uint4*>(out), unsort ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace scfa
