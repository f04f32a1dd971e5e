// Attention forward over live tiles (dense / QK-sparse / hash-sparse policies).
//
// Page: "Faster Causal Attention Over Large Sequences Through Sparse Flash
// Attention" (deep-paper.org): tiled exact attention that never materialises
// the T x T matrix ("FlashAttention 的兴起"), extended with original indices
// so whole tiles are skipped and the rest masked exactly ("SCFA 解决方案",
// parts 1 and 2). The online-softmax recurrence (running max, running sum,
// rescaled accumulator, stored log-sum-exp) is the standard way to keep that
// maths exact across tiles; the page does not print it.
//
// GB300 design: one persistent CTA per SM runs TWO independent pipelines, each
// walking its own share of the forward work order (query tiles by live count,
// longest first), so that one pipeline's MMAs keep the tensor core busy while
// the other pipeline's softmax runs. Per pipeline (6 warps):
//   producer warp  TMA: the Q tile once per work item, then K_j / V_j of each
//                  live key tile into a 2-stage ring (128-byte swizzle).
//   MMA warp       lane 0 issues tcgen05.mma: S = Q K_j^T into TMEM, then
//                  O += P V_j with P read from TMEM (it overwrites S in place
//                  as bf16 pairs), then S of the next tile into the same
//                  columns: the tensor core runs one thread's MMAs in order,
//                  so the next S cannot overtake the PV that reads P.
//   softmax WG     thread = query row = TMEM lane: reads S, applies the
//                  element mask only on tiles not flagged FULL, online softmax
//                  in the log2 domain with a lazy rescale (O is rescaled only
//                  when the row max grows by more than 2^8; S_j complete
//                  implies PV_{j-1} complete, so O is stable then), writes P,
//                  and at the end normalises O and writes O (bf16) and LSE.
// TMEM (512 columns): pipeline p uses S at [256 p, 256 p + 128) and O at
// [256 p + 128, 256 p + 128 + D). Every wait is bounded (1 s); on expiry the
// CTA raises the workspace status word, leaves its loops and frees TMEM.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace scfa {
namespace {

constexpr int kStages = 2;
constexpr int kPipes = 2;
constexpr int kSubBytes = kTile * 128;  // one [128 rows][64 bf16] swizzled sub-tile
constexpr int kWarpsPerPipe = 6;
constexpr int kFwdThreads = kPipes * kWarpsPerPipe * 32;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct __align__(1024) FwdPipe {
  uint8_t q[D / 64][kSubBytes];
  uint8_t k[kStages][D / 64][kSubBytes];
  uint8_t v[kStages][D / 64][kSubBytes];
  int32_t kidx[2][kTile];
  int32_t khash[2][kTile];
  uint64_t q_full, q_empty;
  uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
  uint64_t s_full, p_full, o_full, o_empty, drain;
};

template <int D>
struct __align__(1024) FwdSmem {
  FwdPipe<D> pipe[kPipes];
  uint32_t tmem_base;
  int abort_flag;
};

struct FwdParams {
  int mode;
  int Tq, Tk, nQt;
  float scale_log2;
  const int32_t* q_idx;
  const int32_t* k_idx;
  const int32_t* q_hash;
  const int32_t* k_hash;
  const int32_t* row_ptr;
  const int32_t* cols;
  const uint8_t* fflags;
  const int32_t* work;
  int n_work;
  uint16_t* o;
  float* lse;
  int* status;
};

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  FwdSmem<D>& sm = *reinterpret_cast<FwdSmem<D>*>(smem_raw + pad);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pi = warp / kWarpsPerPipe;      // pipeline of this warp
  const int role = warp % kWarpsPerPipe;    // 0 producer, 1 MMA, 2-5 softmax
  FwdPipe<D>& pp = sm.pipe[pi];

  if (threadIdx.x == 0) {
    for (int q = 0; q < kPipes; ++q) {
      FwdPipe<D>& P = sm.pipe[q];
      mbar_init(&P.q_full, 1);
      mbar_init(&P.q_empty, 1);
      for (int s = 0; s < kStages; ++s) {
        mbar_init(&P.k_full[s], 1);
        mbar_init(&P.v_full[s], 1);
        mbar_init(&P.kv_empty[s], 1);
      }
      mbar_init(&P.s_full, 1);
      mbar_init(&P.p_full, 128);
      mbar_init(&P.o_full, 1);
      mbar_init(&P.o_empty, 128);
      mbar_init(&P.drain, 1);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t colS = 256u * pi, colO = 256u * pi + 128u;
  volatile int* abort_flag = &sm.abort_flag;
  // this pipeline's share of the work order
  const int first = blockIdx.x * kPipes + pi;
  const int stride = gridDim.x * kPipes;

  if (role == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int kv_it = 0, item = 0, last_q = -1;
      for (int w = first; w < p.n_work; w += stride) {
        const int g = p.work[w];
        const int start = p.row_ptr[g], n = p.row_ptr[g + 1] - start;
        if (n == 0) continue;
        const int bh = g / p.nQt, i = g % p.nQt;
        if (!mbar_wait(&pp.q_empty, (item & 1) ^ 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&pp.q_full, D * kTile * 2);
        for (int sub = 0; sub < D / 64; ++sub) tma_load_3d(pp.q[sub], &tm_q, &pp.q_full, sub * 64, i * kTile, bh);
        last_q = item;
        bool ok = true;
        for (int t = 0; t < n; ++t) {
          const int j = p.cols[start + t];
          const int s = kv_it % kStages;
          const uint32_t ph = (kv_it / kStages) & 1;
          if (!mbar_wait(&pp.kv_empty[s], ph ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&pp.k_full[s], D * kTile * 2);
          for (int sub = 0; sub < D / 64; ++sub) tma_load_3d(pp.k[s][sub], &tm_k, &pp.k_full[s], sub * 64, j * kTile, bh);
          mbar_arrive_expect_tx(&pp.v_full[s], D * kTile * 2);
          for (int sub = 0; sub < D / 64; ++sub) tma_load_3d(pp.v[s][sub], &tm_v, &pp.v_full[s], sub * 64, j * kTile, bh);
          ++kv_it;
        }
        if (!ok) break;
        ++item;
      }
      // drain: every copy issued by this thread has landed before the CTA exits
      for (int d = 1; d <= kStages && d <= kv_it; ++d) {
        const int it = kv_it - d;
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        mbar_wait(&pp.k_full[s], ph, abort_flag, p.status);
        mbar_wait(&pp.v_full[s], ph, abort_flag, p.status);
      }
      if (last_q >= 0) mbar_wait(&pp.q_full, last_q & 1, abort_flag, p.status);
    }
  } else if (role == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kTile, kTile, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kTile, D, 0, 1);
      const uint32_t q_base = smem_u32(pp.q[0]);
      int kv_it = 0, p_it = 0, item = 0;
      bool ok = true;
      auto issue_s = [&](int kvi) -> bool {
        const int s = kvi % kStages;
        if (!mbar_wait(&pp.k_full[s], (kvi / kStages) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint32_t k_base = smem_u32(pp.k[s][0]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSubBytes + (kk & 3) * 32;
          mma_bf16_ss(tmem + colS, smem_desc_sw128(q_base + off, 16, 1024),
                      smem_desc_sw128(k_base + off, 16, 1024), idesc_s, kk > 0);
        }
        tc_commit(&pp.s_full);
        return true;
      };
      for (int w = first; w < p.n_work && ok; w += stride) {
        const int g = p.work[w];
        const int n = p.row_ptr[g + 1] - p.row_ptr[g];
        if (n == 0) continue;
        if (!mbar_wait(&pp.q_full, item & 1, abort_flag, p.status)) break;
        if (!issue_s(kv_it)) break;
        for (int t = 0; t < n; ++t) {
          const int s = kv_it % kStages;
          if (!mbar_wait(&pp.p_full, p_it & 1, abort_flag, p.status)) { ok = false; break; }
          if (t == 0 && !mbar_wait(&pp.o_empty, (item & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
          if (!mbar_wait(&pp.v_full[s], (kv_it / kStages) & 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t v_base = smem_u32(pp.v[s][0]);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_bf16_ts(tmem + colO, tmem + colS + kk * 8, smem_desc_sw128(v_base + kk * 2048, kSubBytes, 1024),
                        idesc_o, (t > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&pp.kv_empty[s]);
          ++kv_it;
          ++p_it;
          if (t + 1 < n && !issue_s(kv_it)) { ok = false; break; }
        }
        if (!ok) break;
        tc_commit(&pp.o_full);
        tc_commit(&pp.q_empty);
        ++item;
      }
      // drain: all MMAs issued by this thread are complete before TMEM is freed
      tc_commit(&pp.drain);
      mbar_wait(&pp.drain, 0, abort_flag, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroup
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;          // row of the tile = TMEM lane
    const int tid = (role - 2) * 32 + lane;     // 0..127 for cooperative staging
    const int bar_id = 1 + pi;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    int s_it = 0, item = 0;
    for (int w = first; w < p.n_work; w += stride) {
      const int g = p.work[w];
      const int start = p.row_ptr[g], n = p.row_ptr[g + 1] - start;
      const int bh = g / p.nQt, i = g % p.nQt;
      const int row = i * kTile + r;
      const bool valid = row < p.Tq;
      const long long grow = static_cast<long long>(bh) * p.Tq + row;
      int qi, qh = 0;
      if (p.mode == SCFA_MODE_DENSE) qi = valid ? row : INT_MIN;
      else qi = valid ? p.q_idx[grow] : INT_MIN;
      if (p.mode == SCFA_MODE_HASH && valid) qh = p.q_hash[grow];
      if (n == 0) {
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + grow * D);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
          p.lse[grow] = -INFINITY;
        }
        continue;
      }
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      for (int t = 0; t < n; ++t) {
        const int j = p.cols[start + t];
        const bool full = (p.fflags[start + t] & kFlagFull) != 0;
        const int b = s_it & 1;
        if (!full) {
          const int col = j * kTile + tid;
          const bool kv = col < p.Tk;
          const long long gk = static_cast<long long>(bh) * p.Tk + col;
          int kid;
          if (p.mode == SCFA_MODE_DENSE) kid = kv ? col : INT_MAX;
          else kid = kv ? p.k_idx[gk] : INT_MAX;
          pp.kidx[b][tid] = kid;
          if (p.mode == SCFA_MODE_HASH) pp.khash[b][tid] = kv ? p.k_hash[gk] : INT_MIN;
          named_bar_sync(bar_id, 128);
        }
        ok = mbar_wait(&pp.s_full, s_it & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        float sv[kTile];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t sr[32];
          tmem_ld32(lane_base + colS + cc * 32, sr);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[cc * 32 + c] = __uint_as_float(sr[c]) * p.scale_log2;
          if (!full) {
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const int4 k4 = *reinterpret_cast<const int4*>(&pp.kidx[b][cc * 32 + c4 * 4]);
              bool adm[4] = {qi >= k4.x, qi >= k4.y, qi >= k4.z, qi >= k4.w};
              if (p.mode == SCFA_MODE_HASH) {
                const int4 h4 = *reinterpret_cast<const int4*>(&pp.khash[b][cc * 32 + c4 * 4]);
                adm[0] = adm[0] && qh == h4.x;
                adm[1] = adm[1] && qh == h4.y;
                adm[2] = adm[2] && qh == h4.z;
                adm[3] = adm[3] && qh == h4.w;
              }
#pragma unroll
              for (int u = 0; u < 4; ++u)
                if (!adm[u]) sv[cc * 32 + c4 * 4 + u] = -INFINITY;
            }
          }
        }
        float mt = sv[0];
#pragma unroll
        for (int c = 1; c < kTile; ++c) mt = fmaxf(mt, sv[c]);
        const float m_new = fmaxf(m_used, mt);
        const bool resc = m_new > m_used + kRescaleThreshold;
        float alpha = 1.f;
        if (resc) {
          alpha = ex2_approx(m_used - m_new);
          m_used = m_new;
        }
        const float msub = (m_used == -INFINITY) ? 0.f : m_used;
        float rs = 0.f;
        // P (bf16 pairs) over the first 64 columns of S, one 64-key half at a time
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const float e0 = ex2_approx(sv[h * 64 + c] - msub);
            const float e1 = ex2_approx(sv[h * 64 + c + 1] - msub);
            rs += e0 + e1;
            pk[c >> 1] = pack_bf16x2(e0, e1);
          }
          tmem_st32(lane_base + colS + h * 32, pk);
        }
        l = l * alpha + rs;
        // rescale O (rare). S_t complete => PV_{t-1} complete (in-order tensor pipe): O is stable
        if (t > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t orr[32];
            tmem_ld32(lane_base + colO + cc * 32, orr);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
            tmem_st32(lane_base + colO + cc * 32, orr);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&pp.p_full);
        ++s_it;
      }
      if (!ok) break;
      // epilogue: O / l, LSE
      ok = mbar_wait(&pp.o_full, item & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      uint32_t orr[D / 32][32];
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(lane_base + colO + cc * 32, orr[cc]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&pp.o_empty);
      if (valid) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint4* dst = reinterpret_cast<uint4*>(p.o + grow * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const int e = c * 8;
          uint4 u;
          u.x = pack_bf16x2(__uint_as_float(orr[e >> 5][(e + 0) & 31]) * inv, __uint_as_float(orr[e >> 5][(e + 1) & 31]) * inv);
          u.y = pack_bf16x2(__uint_as_float(orr[e >> 5][(e + 2) & 31]) * inv, __uint_as_float(orr[e >> 5][(e + 3) & 31]) * inv);
          u.z = pack_bf16x2(__uint_as_float(orr[e >> 5][(e + 4) & 31]) * inv, __uint_as_float(orr[e >> 5][(e + 5) & 31]) * inv);
          u.w = pack_bf16x2(__uint_as_float(orr[e >> 5][(e + 6) & 31]) * inv, __uint_as_float(orr[e >> 5][(e + 7) & 31]) * inv);
          dst[c] = u;
        }
        p.lse[grow] = l > 0.f ? (m_used + log2f(l)) * kLn2 : -INFINITY;
      }
      ++item;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, int D, long long T, long long BH);

cudaError_t launch_attn_fwd(const AttnArgs& a, cudaStream_t st) {
  if (a.D != 64) return cudaErrorInvalidValue;
  constexpr int D = 64;
  const AttnWs& L = *a.L;
  const long long BH = static_cast<long long>(a.B) * a.H;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_bf16_3d(&tq, a.q, D, a.Tq, BH) || !make_tmap_bf16_3d(&tk, a.k, D, a.Tk, BH) ||
      !make_tmap_bf16_3d(&tv, a.v, D, a.Tk, BH))
    return cudaErrorInvalidValue;
  FwdParams p;
  p.mode = a.mode;
  p.Tq = a.Tq;
  p.Tk = a.Tk;
  p.nQt = L.nQt;
  p.scale_log2 = a.scale * kLog2e;
  p.q_idx = a.q_idx;
  p.k_idx = a.k_idx;
  p.q_hash = a.q_hash;
  p.k_hash = a.k_hash;
  p.row_ptr = reinterpret_cast<const int32_t*>(a.ws + L.row_ptr);
  p.cols = reinterpret_cast<const int32_t*>(a.ws + L.cols);
  p.fflags = reinterpret_cast<const uint8_t*>(a.ws + L.fflags);
  p.work = reinterpret_cast<const int32_t*>(a.ws + L.work_fwd);
  p.n_work = static_cast<int>(L.n_qtiles);
  p.o = a.o_out;
  p.lse = a.lse_out;
  p.status = reinterpret_cast<int*>(a.ws + L.header);
  const size_t smem = sizeof(FwdSmem<D>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int grid = num_sms();
  if (grid > (p.n_work + kPipes - 1) / kPipes) grid = (p.n_work + kPipes - 1) / kPipes;
  if (grid < 1) grid = 1;
  record_kernel_event(0, true, st);
  attn_fwd_kernel<D><<<grid, kFwdThreads, smem, st>>>(tq, tk, tv, p);
  record_kernel_event(0, false, st);
  return cudaGetLastError();
}

}  // namespace scfa
