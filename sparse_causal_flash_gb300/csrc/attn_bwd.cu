// Attention backward over live tiles (dense / QK-sparse / hash-sparse), plus
// the row pre-pass (rowsum(dO * O), dQ accumulator reset) and the dQ
// finalisation.
//
// Page: "Faster Causal Attention Over Large Sequences Through Sparse Flash
// Attention" (deep-paper.org): the language-model training of section
// "实验与结果" runs SCFA inside training, so the kernels have a backward pass;
// the page prints no formula for it. With P = softmax(scale * Q K^T) under
// the mask, L = sum(O * dO): dV = P^T dO, dP = dO V^T,
// dS = P * (dP - rowsum(dO * O)), dQ = scale * dS K, dK = scale * dS^T Q.
//
// GB300 design: persistent CTAs walk the backward work order (key tiles by
// live count, longest first); each work item keeps K_j, V_j resident and
// streams the live query tiles of its CSC column:
//   warp 0      TMA producer: K_j, V_j once; Q_i, dO_i into a 2-stage ring.
//   warp 1      TMEM owner; lane 0 issues tcgen05.mma:
//               S^T = K Q^T and dP^T = V dO^T (TMEM, keys on lanes), then
//               dV += P^T dO, dK += dS^T Q (TMEM accumulators for the whole
//               item) and dQ_i = dS K (TMEM, queries on lanes).
//   warps 2-5   thread = key row: P^T = exp2(S^T - LSE) under the mask,
//               dS^T = P^T (dP^T - Drow) * scale, both written as bf16 to
//               shared memory; one buffer serves as K-major A operand of
//               dV / dK and as MN-major A operand (dS) of dQ.
//   warps 6-9   thread = query row: dQ_i from TMEM, added into an fp32
//               accumulator in the workspace with 16-byte vector atomics.
// The epilogue of each item writes dK, dV (bf16) straight from TMEM.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace scfa {
namespace {

constexpr int kSubBytes = kTile * 128;
constexpr int kBwdThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct __align__(1024) BwdSmem {
  uint8_t k[D / 64][kSubBytes];
  uint8_t v[D / 64][kSubBytes];
  uint8_t q[2][D / 64][kSubBytes];
  uint8_t dO[2][D / 64][kSubBytes];
  uint8_t pt[2][kSubBytes];   // P^T  [128 keys][128 queries] as two 64-query halves
  uint8_t dst[2][kSubBytes];  // dS^T [128 keys][128 queries]
  int32_t qidx[2][kTile];
  int32_t qhash[2][kTile];
  float lse2[2][kTile];
  float drow[2][kTile];
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full, dp_full, st_empty, ds_full, ds_empty, dq_full, dq_empty, dkv_full, dkv_empty, drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct BwdParams {
  int mode;
  int Tq, Tk, nKt;
  float scale, scale_log2;
  const int32_t* q_idx;
  const int32_t* k_idx;
  const int32_t* q_hash;
  const int32_t* k_hash;
  const float* lse;
  const float* drow;
  const int32_t* csc_ptr;
  const int32_t* csc_rows;
  const uint8_t* cflags;
  const int32_t* work;
  int n_work;
  float* dq_acc;
  uint16_t* dk;
  uint16_t* dv;
  int* status;
};

__device__ __forceinline__ void store_row_bf16(uint16_t* dst_row, const uint32_t* vals, int n) {
  uint4* dst = reinterpret_cast<uint4*>(dst_row);
  for (int c = 0; c < n / 8; ++c) {
    uint4 u;
    u.x = pack_bf16x2(__uint_as_float(vals[c * 8 + 0]), __uint_as_float(vals[c * 8 + 1]));
    u.y = pack_bf16x2(__uint_as_float(vals[c * 8 + 2]), __uint_as_float(vals[c * 8 + 3]));
    u.z = pack_bf16x2(__uint_as_float(vals[c * 8 + 4]), __uint_as_float(vals[c * 8 + 5]));
    u.w = pack_bf16x2(__uint_as_float(vals[c * 8 + 6]), __uint_as_float(vals[c * 8 + 7]));
    dst[c] = u;
  }
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(smem_raw + pad);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr uint32_t kColS = 0, kColDP = kTile, kColDV = 2 * kTile, kColDK = 2 * kTile + D, kColDQ = 2 * kTile + 2 * D;

  if (threadIdx.x == 0) {
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.dp_full, 1);
    mbar_init(&sm.st_empty, 128);
    mbar_init(&sm.ds_full, 128);
    mbar_init(&sm.ds_empty, 1);
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_empty, 128);
    mbar_init(&sm.dkv_full, 1);
    mbar_init(&sm.dkv_empty, 128);
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int q_it = 0, item = 0, last_kv = -1;
      for (int w = blockIdx.x; w < p.n_work; w += gridDim.x) {
        const int g = p.work[w];
        const int start = p.csc_ptr[g], n = p.csc_ptr[g + 1] - start;
        if (n == 0) continue;
        const int bh = g / p.nKt, j = g % p.nKt;
        if (!mbar_wait(&sm.kv_empty, (item & 1) ^ 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&sm.kv_full, 2 * D * kTile * 2);
        for (int sub = 0; sub < D / 64; ++sub) {
          tma_load_3d(sm.k[sub], &tm_k, &sm.kv_full, sub * 64, j * kTile, bh);
          tma_load_3d(sm.v[sub], &tm_v, &sm.kv_full, sub * 64, j * kTile, bh);
        }
        last_kv = item;
        bool ok = true;
        for (int t = 0; t < n; ++t) {
          const int i = p.csc_rows[start + t];
          const int s = q_it & 1;
          if (!mbar_wait(&sm.q_empty[s], ((q_it >> 1) & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&sm.q_full[s], 2 * D * kTile * 2);
          for (int sub = 0; sub < D / 64; ++sub) {
            tma_load_3d(sm.q[s][sub], &tm_q, &sm.q_full[s], sub * 64, i * kTile, bh);
            tma_load_3d(sm.dO[s][sub], &tm_do, &sm.q_full[s], sub * 64, i * kTile, bh);
          }
          ++q_it;
        }
        if (!ok) break;
        ++item;
      }
      for (int d = 1; d <= 2 && d <= q_it; ++d) {
        const int it = q_it - d;
        mbar_wait(&sm.q_full[it & 1], (it >> 1) & 1, abort_flag, p.status);
      }
      if (last_kv >= 0) mbar_wait(&sm.kv_full, last_kv & 1, abort_flag, p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kTile, kTile, 0, 0);
      constexpr uint32_t idesc_kv = idesc_bf16_f32(kTile, D, 0, 1);
      constexpr uint32_t idesc_q = idesc_bf16_f32(kTile, D, 1, 1);
      const uint32_t k_base = smem_u32(sm.k[0]);
      const uint32_t v_base = smem_u32(sm.v[0]);
      const uint32_t pt_base = smem_u32(sm.pt[0]);
      const uint32_t dst_base = smem_u32(sm.dst[0]);
      int q_it = 0, it = 0, item = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < p.n_work && ok; w += gridDim.x) {
        const int g = p.work[w];
        const int n = p.csc_ptr[g + 1] - p.csc_ptr[g];
        if (n == 0) continue;
        if (!mbar_wait(&sm.kv_full, item & 1, abort_flag, p.status)) break;
        for (int t = 0; t < n; ++t) {
          const int s = q_it & 1;
          if (!mbar_wait(&sm.q_full[s], (q_it >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
          if (!mbar_wait(&sm.st_empty, (it & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t q_base = smem_u32(sm.q[s][0]);
          const uint32_t do_base = smem_u32(sm.dO[s][0]);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kSubBytes + (kk & 3) * 32;
            mma_bf16_ss(tmem + kColS, smem_desc_sw128(k_base + off, 16, 1024),
                        smem_desc_sw128(q_base + off, 16, 1024), idesc_s, kk > 0);
          }
          tc_commit(&sm.s_full);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kSubBytes + (kk & 3) * 32;
            mma_bf16_ss(tmem + kColDP, smem_desc_sw128(v_base + off, 16, 1024),
                        smem_desc_sw128(do_base + off, 16, 1024), idesc_s, kk > 0);
          }
          tc_commit(&sm.dp_full);
          if (!mbar_wait(&sm.ds_full, it & 1, abort_flag, p.status)) { ok = false; break; }
          if (t == 0 && !mbar_wait(&sm.dkv_empty, (item & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
          if (!mbar_wait(&sm.dq_empty, (it & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t a_off = (kk >> 2) * kSubBytes + (kk & 3) * 32;
            const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
            mma_bf16_ss(tmem + kColDV, smem_desc_sw128(pt_base + a_off, 16, 1024),
                        smem_desc_sw128(do_base + kk * 2048, kSubBytes, 1024), idesc_kv, acc);
            mma_bf16_ss(tmem + kColDK, smem_desc_sw128(dst_base + a_off, 16, 1024),
                        smem_desc_sw128(q_base + kk * 2048, kSubBytes, 1024), idesc_kv, acc);
          }
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            mma_bf16_ss(tmem + kColDQ, smem_desc_sw128(dst_base + kk * 2048, kSubBytes, 1024),
                        smem_desc_sw128(k_base + kk * 2048, kSubBytes, 1024), idesc_q, kk > 0 ? 1u : 0u);
          }
          tc_commit(&sm.dq_full);
          tc_commit(&sm.q_empty[s]);
          tc_commit(&sm.ds_empty);
          ++q_it;
          ++it;
        }
        if (!ok) break;
        tc_commit(&sm.dkv_full);
        tc_commit(&sm.kv_empty);
        ++item;
      }
      tc_commit(&sm.drain);
      mbar_wait(&sm.drain, 0, abort_flag, p.status);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ P^T / dS^T warpgroup
    const int quarter = warp & 3;
    const int kr = quarter * 32 + lane;  // key row = TMEM lane
    const int tid = threadIdx.x - 64;    // 0..127
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    int it = 0, item = 0;
    for (int w = blockIdx.x; w < p.n_work; w += gridDim.x) {
      const int g = p.work[w];
      const int start = p.csc_ptr[g], n = p.csc_ptr[g + 1] - start;
      const int bh = g / p.nKt, j = g % p.nKt;
      const int key = j * kTile + kr;
      const bool kvalid = key < p.Tk;
      const long long gk = static_cast<long long>(bh) * p.Tk + key;
      if (n == 0) {
        if (kvalid) {
          uint4* a = reinterpret_cast<uint4*>(p.dk + gk * D);
          uint4* b = reinterpret_cast<uint4*>(p.dv + gk * D);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) {
            a[c] = make_uint4(0, 0, 0, 0);
            b[c] = make_uint4(0, 0, 0, 0);
          }
        }
        continue;
      }
      int ki, kh = 0;
      if (p.mode == SCFA_MODE_DENSE) ki = kvalid ? key : INT_MAX;
      else ki = kvalid ? p.k_idx[gk] : INT_MAX;
      if (p.mode == SCFA_MODE_HASH && kvalid) kh = p.k_hash[gk];
      bool ok = true;
      for (int t = 0; t < n; ++t) {
        const int i = p.csc_rows[start + t];
        const bool full = (p.cflags[start + t] & kFlagFull) != 0;
        const int b = it & 1;
        {
          const int qrow = i * kTile + tid;
          const bool qv = qrow < p.Tq;
          const long long gq = static_cast<long long>(bh) * p.Tq + qrow;
          int qid;
          if (p.mode == SCFA_MODE_DENSE) qid = qv ? qrow : INT_MIN;
          else qid = qv ? p.q_idx[gq] : INT_MIN;
          sm.qidx[b][tid] = qid;
          sm.qhash[b][tid] = (p.mode == SCFA_MODE_HASH && qv) ? p.q_hash[gq] : 0;
          sm.lse2[b][tid] = qv ? p.lse[gq] * kLog2e : 0.f;
          sm.drow[b][tid] = qv ? p.drow[gq] : 0.f;
        }
        named_bar_sync(1, 128);
        ok = mbar_wait(&sm.s_full, it & 1, abort_flag, p.status) &&
             mbar_wait(&sm.dp_full, it & 1, abort_flag, p.status) &&
             mbar_wait(&sm.ds_empty, (it & 1) ^ 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < kTile / 32; ++cc) {
          uint32_t sr[32], dr[32];
          tmem_ld32(lane_base + kColS + cc * 32, sr);
          tmem_ld32(lane_base + kColDP + cc * 32, dr);
          tmem_wait_ld();
          float pv[32], dsv[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int c = cc * 32 + e;
            bool adm = true;
            if (!full) {
              adm = sm.qidx[b][c] >= ki;
              if (p.mode == SCFA_MODE_HASH) adm = adm && (sm.qhash[b][c] == kh);
            }
            const float pe = ex2_approx(__uint_as_float(sr[e]) * p.scale_log2 - sm.lse2[b][c]);
            pv[e] = adm ? pe : 0.f;
            dsv[e] = pv[e] * (__uint_as_float(dr[e]) - sm.drow[b][c]) * p.scale;
          }
          const int h = cc >> 1;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int ch = (cc & 1) * 4 + u;
            uint4 a, d;
            a.x = pack_bf16x2(pv[u * 8 + 0], pv[u * 8 + 1]);
            a.y = pack_bf16x2(pv[u * 8 + 2], pv[u * 8 + 3]);
            a.z = pack_bf16x2(pv[u * 8 + 4], pv[u * 8 + 5]);
            a.w = pack_bf16x2(pv[u * 8 + 6], pv[u * 8 + 7]);
            d.x = pack_bf16x2(dsv[u * 8 + 0], dsv[u * 8 + 1]);
            d.y = pack_bf16x2(dsv[u * 8 + 2], dsv[u * 8 + 3]);
            d.z = pack_bf16x2(dsv[u * 8 + 4], dsv[u * 8 + 5]);
            d.w = pack_bf16x2(dsv[u * 8 + 6], dsv[u * 8 + 7]);
            *reinterpret_cast<uint4*>(sm.pt[h] + sw128_offset(kr, ch)) = a;
            *reinterpret_cast<uint4*>(sm.dst[h] + sw128_offset(kr, ch)) = d;
          }
        }
        tc_fence_before();
        mbar_arrive(&sm.st_empty);
        fence_proxy_async_smem();
        mbar_arrive(&sm.ds_full);
        ++it;
      }
      if (!ok) break;
      ok = mbar_wait(&sm.dkv_full, item & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      uint32_t dvr[D / 32][32], dkr[D / 32][32];
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        tmem_ld32(lane_base + kColDV + cc * 32, dvr[cc]);
        tmem_ld32(lane_base + kColDK + cc * 32, dkr[cc]);
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&sm.dkv_empty);
      if (kvalid) {
        store_row_bf16(p.dv + gk * D, &dvr[0][0], D);
        store_row_bf16(p.dk + gk * D, &dkr[0][0], D);
      }
      ++item;
    }
  } else {
    // ------------------------------------------------------------ dQ warpgroup
    const int quarter = warp & 3;
    const int qr = quarter * 32 + lane;  // query row = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    int it = 0;
    for (int w = blockIdx.x; w < p.n_work; w += gridDim.x) {
      const int g = p.work[w];
      const int start = p.csc_ptr[g], n = p.csc_ptr[g + 1] - start;
      if (n == 0) continue;
      const int bh = g / p.nKt;
      bool ok = true;
      for (int t = 0; t < n; ++t) {
        const int i = p.csc_rows[start + t];
        ok = mbar_wait(&sm.dq_full, it & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t qv[D / 32][32];
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(lane_base + kColDQ + cc * 32, qv[cc]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&sm.dq_empty);
        const int qrow = i * kTile + qr;
        if (qrow < p.Tq) {
          float4* dst = reinterpret_cast<float4*>(p.dq_acc + (static_cast<long long>(bh) * p.Tq + qrow) * D);
#pragma unroll
          for (int c = 0; c < D / 4; ++c) {
            const int e = c * 4;
            atomicAdd(dst + c, make_float4(__uint_as_float(qv[e >> 5][e & 31]), __uint_as_float(qv[e >> 5][(e + 1) & 31]),
                                           __uint_as_float(qv[e >> 5][(e + 2) & 31]), __uint_as_float(qv[e >> 5][(e + 3) & 31])));
          }
        }
        ++it;
      }
      if (!ok) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Drow[row] = sum_d dO * O (fp32) and dq_acc[row] = 0. D/8 lanes per row (one
// 16-byte chunk each), 32 / (D/8) rows per warp step; the loop is warp-uniform
// so the shuffle reduction always has the whole warp.
template <int D>
__global__ void bwd_pre_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dO, long long rows,
                               float* __restrict__ drow, float* __restrict__ dq_acc) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const int lane = threadIdx.x & 31;
  const long long warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long wg = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       wg * kRowsPerWarp < rows; wg += warps) {
    const long long row = wg * kRowsPerWarp + lane / kLanesPerRow;
    const int ch = lane % kLanesPerRow;
    const bool active = row < rows;
    float s = 0.f;
    if (active) {
      const uint4 a = reinterpret_cast<const uint4*>(o + row * D)[ch];
      const uint4 b = reinterpret_cast<const uint4*>(dO + row * D)[ch];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        s = fmaf(__uint_as_float(aw[u] << 16), __uint_as_float(bw[u] << 16), s);
        s = fmaf(__uint_as_float(aw[u] & 0xFFFF0000u), __uint_as_float(bw[u] & 0xFFFF0000u), s);
      }
    }
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (active) {
      if (ch == 0) drow[row] = s;
      float4* z = reinterpret_cast<float4*>(dq_acc + row * D) + ch * 2;
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

__global__ void dq_finalize_kernel(const float* __restrict__ dq_acc, long long n8, uint16_t* __restrict__ dq) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < n8; t += stride) {
    const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * t];
    const float4 b = reinterpret_cast<const float4*>(dq_acc)[2 * t + 1];
    uint4 u;
    u.x = pack_bf16x2(a.x, a.y);
    u.y = pack_bf16x2(a.z, a.w);
    u.z = pack_bf16x2(b.x, b.y);
    u.w = pack_bf16x2(b.z, b.w);
    reinterpret_cast<uint4*>(dq)[t] = u;
  }
}

}  // namespace

bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, int D, long long T, long long BH);

cudaError_t launch_attn_bwd(const AttnArgs& a, cudaStream_t st) {
  if (a.D != 64) return cudaErrorInvalidValue;
  constexpr int D = 64;
  const AttnWs& L = *a.L;
  const long long BH = static_cast<long long>(a.B) * a.H;
  const int sms = num_sms();
  float* dq_acc = reinterpret_cast<float*>(a.ws + L.dq_acc);
  float* drow = reinterpret_cast<float*>(a.ws + L.drow);
  const long long qrows = BH * a.Tq;
  {
    const long long work = (qrows * (D / 8) + 31) / 32 * 32;
    long long g = (work + 255) / 256;
    if (g > sms * 16LL) g = sms * 16LL;
    if (g < 1) g = 1;
    bwd_pre_kernel<D><<<static_cast<int>(g), 256, 0, st>>>(a.o, a.do_, qrows, drow, dq_acc);
  }
  CUtensorMap tq, tk, tv, tdo;
  if (!make_tmap_bf16_3d(&tq, a.q, D, a.Tq, BH) || !make_tmap_bf16_3d(&tk, a.k, D, a.Tk, BH) ||
      !make_tmap_bf16_3d(&tv, a.v, D, a.Tk, BH) || !make_tmap_bf16_3d(&tdo, a.do_, D, a.Tq, BH))
    return cudaErrorInvalidValue;
  BwdParams p;
  p.mode = a.mode;
  p.Tq = a.Tq;
  p.Tk = a.Tk;
  p.nKt = L.nKt;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.q_idx = a.q_idx;
  p.k_idx = a.k_idx;
  p.q_hash = a.q_hash;
  p.k_hash = a.k_hash;
  p.lse = a.lse_in;
  p.drow = drow;
  p.csc_ptr = reinterpret_cast<const int32_t*>(a.ws + L.csc_ptr);
  p.csc_rows = reinterpret_cast<const int32_t*>(a.ws + L.csc_rows);
  p.cflags = reinterpret_cast<const uint8_t*>(a.ws + L.cflags);
  p.work = reinterpret_cast<const int32_t*>(a.ws + L.work_bwd);
  p.n_work = static_cast<int>(L.n_ktiles);
  p.dq_acc = dq_acc;
  p.dk = a.dk;
  p.dv = a.dv;
  p.status = reinterpret_cast<int*>(a.ws + L.header);
  const size_t smem = sizeof(BwdSmem<D>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int grid = sms;
  if (grid > p.n_work) grid = p.n_work;
  if (grid < 1) grid = 1;
  record_kernel_event(1, true, st);
  attn_bwd_kernel<D><<<grid, kBwdThreads, smem, st>>>(tq, tk, tv, tdo, p);
  record_kernel_event(1, false, st);
  {
    const long long n8 = qrows * D / 8;
    long long g = (n8 + 255) / 256;
    if (g > sms * 16LL) g = sms * 16LL;
    if (g < 1) g = 1;
    dq_finalize_kernel<<<static_cast<int>(g), 256, 0, st>>>(dq_acc, n8, a.dq);
  }
  return cudaGetLastError();
}

}  // namespace scfa
