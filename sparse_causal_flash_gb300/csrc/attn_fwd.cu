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
// GB300 design: one persistent CTA per SM walks the pair work order: a work
// item is a pair of adjacent query tiles (2m, 2m + 1) of one head, and the CTA
// streams the UNION of their live key-tile lists once, so each K / V tile load
// serves both query tiles. Roles (352 threads):
//   warp 0      producer: TMA of Q_2m and Q_2m+1 per item, then K_j / V_j of
//               each union tile into a ring (128-byte swizzle).
//   warps 1, 10 MMA issuers for query tile g = 0, 1 (lane 0; warp 1 also owns
//               TMEM): S_g = Q_g K_j^T into TMEM, then PV_g with P_g read from
//               TMEM. Two issuers keep one tile's S -> softmax -> PV chain from
//               waiting on the other's softmax. A tile live for only one query
//               tile skips the other's S and PV, but both issuers release every
//               ring stage (two arrivals).
//   warps 2-5, 6-9  softmax warpgroup g (query tile 2m + g); thread = query
//               row = TMEM lane: element mask only on tiles not flagged FULL,
//               online softmax in the log2 domain with a lazy rescale (O_g is
//               rescaled only when the row max grows by more than 2^8), P_g
//               written to TMEM as bf16 pairs, and the epilogue (O / l in bf16,
//               LSE in fp32, natural log). Max, argument and row sum use the
//               three-input max and packed f32x2 FMA / add.
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 [256+D,256+2D);
// at D = 64, P_0 [384,448) and P_1 [448,512), so S_g(j+1) is computed while the
// softmax of S_g(j) runs (the softmax frees S_g once it is in registers, and
// waits for PV_g(j-1) before overwriting P_g); at D = 128, P_g overwrites S_g
// and one issuer's in-order MMAs keep S_g(j+1) behind PV_g(j).
// Every wait is bounded (1 s); on expiry the CTA raises the workspace status
// word, leaves its loops and frees TMEM.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace scfa {
namespace {

// K / V ring depth: 4 stages of 32 KB at D = 64, 2 stages of 64 KB at D = 128
template <int D>
constexpr int fwd_stages() { return D == 64 ? 4 : 2; }
constexpr int kSubBytes = kTile * 128;  // one [128 rows][64 bf16] swizzled sub-tile
constexpr int kFwdThreads = 352;  // producer, MMA for tile 0, 2 x 4 softmax warps, MMA for tile 1
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// At D = 64, S_0, S_1, O_0, O_1 take 384 of the 512 TMEM columns and P_g gets
// its own 64 columns; then S_g(j+1) can be computed while the softmax of
// S_g(j) runs. At D = 128 the columns are all taken and P_g overwrites S_g.
template <int D>
constexpr bool fwd_separate_p() { return D == 64; }

template <int D>
struct __align__(1024) FwdSmem {
  static constexpr int kStages = fwd_stages<D>();
  uint8_t q[2][D / 64][kSubBytes];
  uint8_t k[kStages][D / 64][kSubBytes];
  uint8_t v[kStages][D / 64][kSubBytes];
  int32_t kidx[2][2][kTile];   // [softmax group][buffer][key]
  int32_t khash[2][2][kTile];
  uint64_t q_full, q_empty;
  uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], p_full[2], o_full[2], o_empty[2], drain[2];
  uint64_t s_free[2], pv_done[2];  // used when P has its own TMEM columns
  uint64_t kbar[2];                // the 128 softmax threads of query tile g around masked-tile keys
  uint32_t tmem_base;
  int abort_flag;
};

// fp32 copy of one O row (thread = row) for the backward's rowsum(dO * O);
// `scale` 0 writes zeros (a row with no admissible key, or one whose output
// row is outside [0, T) and therefore reads as zero)
template <int D>
__device__ __forceinline__ void store_o32_row(float* dst, const uint32_t (&orr)[D / 32][32], float scale) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int c = 0; c < D / 4; ++c) {
    const int e = c * 4;
    d[c] = make_float4(__uint_as_float(orr[e >> 5][(e + 0) & 31]) * scale, __uint_as_float(orr[e >> 5][(e + 1) & 31]) * scale,
                       __uint_as_float(orr[e >> 5][(e + 2) & 31]) * scale, __uint_as_float(orr[e >> 5][(e + 3) & 31]) * scale);
  }
}
template <int D>
__device__ __forceinline__ void zero_o32_row(float* dst) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int c = 0; c < D / 4; ++c) d[c] = make_float4(0.f, 0.f, 0.f, 0.f);
}

struct FwdParams {
  int mode;
  int Tq, Tk, nQt, nPairs;
  float scale_log2;
  const int32_t* q_idx;
  const int32_t* k_idx;
  const int32_t* q_hash;
  const int32_t* k_hash;
  const int32_t* row_ptr;
  const int32_t* work_pairs;
  const int32_t* pcount;
  int n_pairs;
  const int32_t* work;   // query tiles by live count descending (single-tile kernel)
  int n_work;
  int* sched;            // [0] next item, [1] CTAs done (single-tile kernel)
  uint16_t* o;
  const int32_t* o_rows;  // null, or the original row of each sorted query row
  int To;                 // rows per head of o when o_rows is set
  float* lse;
  float* o32;             // null, or an fp32 copy of O [B,H,Tq,D] in row order of q
  int stall;              // SCFA_FLAG_DEBUG_STALL: withhold the first K / V load
  int gather_q;           // q is an original-order tensor read by row gathers through q_idx (To rows per head)
  int gather_kv;          // k and v likewise through k_idx
  int* status;
};

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  FwdSmem<D>& sm = *reinterpret_cast<FwdSmem<D>*>(smem_raw + pad);
  constexpr int kStages = FwdSmem<D>::kStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // live-tile lists where the call that built them put them
  const int32_t* const cols = ws_list<int32_t>(p.status, kListCols);
  const uint8_t* const fflags = ws_list<uint8_t>(p.status, kListFflags);
  const int32_t* const ulist = ws_list<int32_t>(p.status, kListPairs);

  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 2);  // one commit from each MMA warp
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.kv_empty[s], 2);  // one commit from each MMA warp
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&sm.s_full[g], 1);
      mbar_init(&sm.p_full[g], 128);
      mbar_init(&sm.o_full[g], 1);
      mbar_init(&sm.o_empty[g], 128);
      mbar_init(&sm.s_free[g], 128);
      mbar_init(&sm.pv_done[g], 1);
      mbar_init(&sm.kbar[g], 128);
    }
    mbar_init(&sm.drain[0], 1);
    mbar_init(&sm.drain[1], 1);
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
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 0 && !p.gather_q && !p.gather_kv) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int kv_it = 0, item = 0, last_q = -1;
      for (int rnd = 0, w = work_item(0); w < p.n_pairs; w = work_item(++rnd)) {
        const int pid = p.work_pairs[w];
        const int cnt = p.pcount[pid];
        if (cnt == 0) continue;
        const int bh = pid / p.nPairs, m = pid % p.nPairs;
        const bool has1 = 2 * m + 1 < p.nQt;
        const long long g0 = static_cast<long long>(bh) * p.nQt + 2 * m;
        if (!mbar_wait(&sm.q_empty, (item & 1) ^ 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&sm.q_full, (has1 ? 2 : 1) * D * kTile * 2);
        for (int sub = 0; sub < D / 64; ++sub) {
          tma_load_3d(sm.q[0][sub], &tm_q, &sm.q_full, sub * 64, 2 * m * kTile, bh);
          if (has1) tma_load_3d(sm.q[1][sub], &tm_q, &sm.q_full, sub * 64, (2 * m + 1) * kTile, bh);
        }
        last_q = item;
        const int32_t* ul = ulist + p.row_ptr[g0];
        bool ok = !(p.stall && kv_it == 0);  // debug stall: no K / V load ever arrives
        for (int t = 0; t < cnt && ok; ++t) {
          const int j = ul[t] >> 4;
          const int s = kv_it % kStages;
          const uint32_t ph = (kv_it / kStages) & 1;
          if (!mbar_wait(&sm.kv_empty[s], ph ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&sm.k_full[s], D * kTile * 2);
          for (int sub = 0; sub < D / 64; ++sub) tma_load_3d(sm.k[s][sub], &tm_k, &sm.k_full[s], sub * 64, j * kTile, bh);
          mbar_arrive_expect_tx(&sm.v_full[s], D * kTile * 2);
          for (int sub = 0; sub < D / 64; ++sub) tma_load_3d(sm.v[s][sub], &tm_v, &sm.v_full[s], sub * 64, j * kTile, bh);
          ++kv_it;
        }
        if (!ok) break;
        ++item;
      }
      // drain: every copy issued by this thread has landed before the CTA
      // exits, also after an abort (K and V of one stage are issued together)
      for (int d = 1; d <= kStages && d <= kv_it; ++d) {
        const int it = kv_it - d;
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        mbar_wait_drain(&sm.k_full[s], ph, p.status);
        mbar_wait_drain(&sm.v_full[s], ph, p.status);
      }
      if (last_q >= 0) mbar_wait_drain(&sm.q_full, last_q & 1, p.status);
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer (row gathers)
    // The same walk with the whole warp: lane 0 waits on the stages and
    // issues the tiled loads, every lane issues four rows of each gathered
    // tile (p.gather_q: Q; p.gather_kv: K, V), their source rows loaded
    // before the stage wait.
    int kv_it = 0, item = 0, last_q = -1;
    for (int rnd = 0, w = work_item(0); w < p.n_pairs; w = work_item(++rnd)) {
      const int pid = p.work_pairs[w];
      const int cnt = p.pcount[pid];
      if (cnt == 0) continue;
      const int bh = pid / p.nPairs, m = pid % p.nPairs;
      const bool has1 = 2 * m + 1 < p.nQt;
      const long long g0 = static_cast<long long>(bh) * p.nQt + 2 * m;
      int r0[4], r1[4];
      if (p.gather_q) {
        gather_rows(p.q_idx, bh, p.Tq, p.To, 2 * m * kTile, lane, r0);
        if (has1) gather_rows(p.q_idx, bh, p.Tq, p.To, (2 * m + 1) * kTile, lane, r1);
      }
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(&sm.q_empty, (item & 1) ^ 1, abort_flag, p.status);
        if (ok) {
          mbar_arrive_expect_tx(&sm.q_full, (has1 ? 2 : 1) * D * kTile * 2);
          if (!p.gather_q) {
            for (int sub = 0; sub < D / 64; ++sub) {
              tma_load_3d(sm.q[0][sub], &tm_q, &sm.q_full, sub * 64, 2 * m * kTile, bh);
              if (has1) tma_load_3d(sm.q[1][sub], &tm_q, &sm.q_full, sub * 64, (2 * m + 1) * kTile, bh);
            }
          }
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      if (p.gather_q) {
        gather_issue(sm.q[0][0], kSubBytes, D / 64, &tm_q, &sm.q_full, r0, lane);
        if (has1) gather_issue(sm.q[1][0], kSubBytes, D / 64, &tm_q, &sm.q_full, r1, lane);
      }
      last_q = item;
      const int32_t* ul = ulist + p.row_ptr[g0];
      ok = !(p.stall && kv_it == 0);  // debug stall: no K / V load ever arrives
      for (int t = 0; t < cnt && ok; ++t) {
        const int j = ul[t] >> 4;
        const int s = kv_it % kStages;
        const uint32_t ph = (kv_it / kStages) & 1;
        int rr[4];
        if (p.gather_kv) gather_rows(p.k_idx, bh, p.Tk, p.To, j * kTile, lane, rr);  // K and V rows
        if (lane == 0) {
          ok = mbar_wait(&sm.kv_empty[s], ph ^ 1, abort_flag, p.status);
          if (ok) {
            mbar_arrive_expect_tx(&sm.k_full[s], D * kTile * 2);
            if (!p.gather_kv)
              for (int sub = 0; sub < D / 64; ++sub) tma_load_3d(sm.k[s][sub], &tm_k, &sm.k_full[s], sub * 64, j * kTile, bh);
            mbar_arrive_expect_tx(&sm.v_full[s], D * kTile * 2);
            if (!p.gather_kv)
              for (int sub = 0; sub < D / 64; ++sub) tma_load_3d(sm.v[s][sub], &tm_v, &sm.v_full[s], sub * 64, j * kTile, bh);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) { ok = false; break; }
        if (p.gather_kv) {
          gather_issue(sm.k[s][0], kSubBytes, D / 64, &tm_k, &sm.k_full[s], rr, lane);
          gather_issue(sm.v[s][0], kSubBytes, D / 64, &tm_v, &sm.v_full[s], rr, lane);
        }
        ++kv_it;
      }
      if (!ok) break;
      ++item;
    }
    if (lane == 0) {
      // drain: every copy issued by this warp has landed before the CTA
      // exits, also after an abort (K and V of one stage are issued together)
      for (int d = 1; d <= kStages && d <= kv_it; ++d) {
        const int it = kv_it - d;
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        mbar_wait_drain(&sm.k_full[s], ph, p.status);
        mbar_wait_drain(&sm.v_full[s], ph, p.status);
      }
      if (last_q >= 0) mbar_wait_drain(&sm.q_full, last_q & 1, p.status);
    }
  } else if (warp == 1 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues the MMAs of query tile 0 and warp 10 those of query tile
    // 1, so neither tile's S -> softmax -> PV chain waits on the other's
    // softmax; the tensor core interleaves the two instruction streams. Both
    // walk the same union list and release each K / V stage (2 arrivals).
    constexpr bool kSepP = fwd_separate_p<D>();
    const int g = warp == 1 ? 0 : 1;
    const int live_bit = g == 0 ? 1 : 4;
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kTile, kTile, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kTile, D, 0, 1);
      int kv_it = 0, item = 0, p_it = 0, o_it = 0, n_s = 0;
      bool ok = true;
      // descriptors built once; steps and stages are constant adds
      constexpr uint32_t kStage16 = (D / 64) * kSubBytes >> 4;
      const uint64_t qdesc = smem_desc_sw128(smem_u32(sm.q[g][0]), 16, 1024);
      const uint64_t kdesc = smem_desc_sw128(smem_u32(sm.k[0][0]), 16, 1024);
      const uint64_t vdesc = smem_desc_sw128(smem_u32(sm.v[0][0]), kSubBytes, 1024);
      const uint32_t dS = tmem + 128u * g, dO_ = tmem + 256u + D * g;
      const uint32_t aP = kSepP ? tmem + 384u + 64u * g : dS;
      auto issue_s = [&](int kvi) -> bool {
        const int s = kvi % kStages;
        // with its own P columns, S_g is overwritten once the softmax has read
        // the previous S_g; otherwise issue order behind PV_g protects it
        if (kSepP && n_s > 0 && !mbar_wait(&sm.s_free[g], (n_s - 1) & 1, abort_flag, p.status)) return false;
        if (!mbar_wait(&sm.k_full[s], (kvi / kStages) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint64_t b = kdesc + static_cast<uint64_t>(s * kStage16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(dS, qdesc + kstep_off16(kk, kSubBytes), b + kstep_off16(kk, kSubBytes), idesc_s, kk > 0);
        tc_commit(&sm.s_full[g]);
        ++n_s;
        return true;
      };
      for (int rnd = 0, w = work_item(0); w < p.n_pairs && ok; w = work_item(++rnd)) {
        const int pid = p.work_pairs[w];
        const int cnt = p.pcount[pid];
        if (cnt == 0) continue;
        const int bh = pid / p.nPairs, m = pid % p.nPairs;
        const long long g0 = static_cast<long long>(bh) * p.nQt + 2 * m;
        // union entries: current, next, and the one after, loaded two tiles
        // ahead so the list read stays off the issue chain
        const int32_t* ul = ulist + p.row_ptr[g0];
        int bits_cur = ul[0] & 15;
        int bits_nxt = cnt > 1 ? ul[1] & 15 : 0;
        if (!mbar_wait(&sm.q_full, item & 1, abort_flag, p.status)) break;
        if ((bits_cur & live_bit) && !issue_s(kv_it)) break;
        bool pv_first = true;
        for (int t = 0; t < cnt; ++t) {
          const bool more = t + 1 < cnt;
          const int bits_pre = t + 2 < cnt ? ul[t + 2] & 15 : 0;
          const bool s_next = more && (bits_nxt & live_bit);
          bool s_next_issued = false;
          const int s = kv_it % kStages;
          if (bits_cur & live_bit) {
            // S_g(j+1) ahead of PV_g(j) when the next union tile is live here
            // (its stage was filled before this one's release is needed)
            if (kSepP && s_next) {
              if (!issue_s(kv_it + 1)) { ok = false; break; }
              s_next_issued = true;
            }
            if (!mbar_wait(&sm.p_full[g], p_it & 1, abort_flag, p.status)) { ok = false; break; }
            if (pv_first && !mbar_wait(&sm.o_empty[g], (o_it & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
            if (!mbar_wait(&sm.v_full[s], (kv_it / kStages) & 1, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint64_t vb = vdesc + static_cast<uint64_t>(s * kStage16);
            const uint32_t acc0 = pv_first ? 0u : 1u;
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_bf16_ts(dO_, aP + kk * 8, vb + static_cast<uint64_t>(kk * 128), idesc_o, kk > 0 ? 1u : acc0);
            if (kSepP) tc_commit(&sm.pv_done[g]);
            pv_first = false;
            ++p_it;
          } else if (!mbar_wait(&sm.k_full[s], (kv_it / kStages) & 1, abort_flag, p.status)) {
            // a tile this query tile skips is still released only once it has
            // landed: without the wait this warp could run ahead through skipped
            // tiles and give both arrivals of a stage's release on its own
            ok = false;
            break;
          }
          tc_commit(&sm.kv_empty[s]);
          if (s_next && !s_next_issued && !issue_s(kv_it + 1)) { ok = false; break; }
          ++kv_it;
          bits_cur = bits_nxt;
          bits_nxt = bits_pre;
        }
        if (!ok) break;
        if (!pv_first) {
          tc_commit(&sm.o_full[g]);
          ++o_it;
        }
        tc_commit(&sm.q_empty);
        ++item;
      }
      // drain: all MMAs issued by this thread are complete before TMEM is freed
      tc_commit(&sm.drain[g]);
      mbar_wait_drain(&sm.drain[g], 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int grp = (warp - 2) >> 2;            // query tile 2m + grp
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;          // row of the tile = TMEM lane
    const int tid = (warp - 2 - 4 * grp) * 32 + lane;  // 0..127 for cooperative staging
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    constexpr bool kSepP = fwd_separate_p<D>();
    int x_it = 0;
    // bounded sync of this query tile's 128 softmax threads (a broken
    // pipeline ends in a status code instead of a hang at a named barrier)
    auto group_sync = [&]() -> bool {
      mbar_arrive(&sm.kbar[grp]);
      const bool r_ok = mbar_wait(&sm.kbar[grp], x_it & 1, abort_flag, p.status);
      ++x_it;
      return __all_sync(0xffffffffu, r_ok);
    };
    const uint32_t colS = 128u * grp, colO = 256u + D * grp;
    const uint32_t colP = kSepP ? 384u + 64u * grp : colS;
    int n_p = 0;  // P_g tiles written so far
    int s_it = 0, o_it = 0;
    for (int rnd = 0, w = work_item(0); w < p.n_pairs; w = work_item(++rnd)) {
      const int pid = p.work_pairs[w];
      const int bh = pid / p.nPairs, m = pid % p.nPairs;
      const int i = 2 * m + grp;
      const long long g0 = static_cast<long long>(bh) * p.nQt + 2 * m;
      const int row = i * kTile + r;
      const bool valid = i < p.nQt && row < p.Tq;
      const long long grow = static_cast<long long>(bh) * p.Tq + row;
      int qi = INT_MIN, qh = 0;
      if (valid) {
        qi = (p.mode == SCFA_MODE_DENSE) ? row : p.q_idx[grow];
        if (p.mode == SCFA_MODE_HASH) qh = p.q_hash[grow];
      }
      // this query tile's own live list; column, flag and key metadata of the
      // coming tiles are loaded ahead (column two tiles ahead, key index and
      // bucket one tile ahead) so no global load sits on the tile chain
      const int e_beg = i < p.nQt ? p.row_ptr[g0 + grp] : 0;
      const int e_end = i < p.nQt ? p.row_ptr[g0 + grp + 1] : 0;
      const long long kbase = static_cast<long long>(bh) * p.Tk;
      auto key_meta = [&](int j, int f, int& kid, int& kh) {
        kid = INT_MAX;
        kh = INT_MIN;
        if (f & kFlagFull) return;
        const int col = j * kTile + tid;
        const bool kv = col < p.Tk;
        if (p.mode == SCFA_MODE_DENSE) kid = kv ? col : INT_MAX;
        else kid = kv ? p.k_idx[kbase + col] : INT_MAX;
        if (p.mode == SCFA_MODE_HASH) kh = kv ? p.k_hash[kbase + col] : INT_MIN;
      };
      int j_c = 0, f_c = 0, kid_c = INT_MAX, kh_c = INT_MIN, j_n = 0, f_n = 0;
      if (e_beg < e_end) {
        j_c = cols[e_beg];
        f_c = fflags[e_beg];
        key_meta(j_c, f_c, kid_c, kh_c);
      }
      if (e_beg + 1 < e_end) {
        j_n = cols[e_beg + 1];
        f_n = fflags[e_beg + 1];
      }
      float m_used = -INFINITY, l = 0.f;
      float m_top = -INFINITY;  // largest score of the row so far (log2 units)
      bool ok = true, any = false;
      for (int e = e_beg; e < e_end; ++e) {
        const bool full = (f_c & kFlagFull) != 0;
        const int kid = kid_c, khv = kh_c;
        int kid_n = INT_MAX, kh_n = INT_MIN, j_nn = 0, f_nn = 0;
        if (e + 1 < e_end) key_meta(j_n, f_n, kid_n, kh_n);
        if (e + 2 < e_end) {
          j_nn = cols[e + 2];
          f_nn = fflags[e + 2];
        }
        const bool first_tile = !any;
        any = true;
        const int b = s_it & 1;
        if (!full) {
          sm.kidx[grp][b][tid] = kid;
          if (p.mode == SCFA_MODE_HASH) sm.khash[grp][b][tid] = khv;
          if (!group_sync()) { ok = false; break; }
        }
        ok = mbar_wait(&sm.s_full[grp], s_it & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        // raw scores of this row: four 32-column loads, one wait
        uint32_t sr[kTile];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          tmem_ld32(lane_base + colS + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[cc * 32]));
        tmem_wait_ld();
        tmem_ld_fence(sr);
        if (kSepP) {
          // S_g is in registers: the MMA warp may compute the next S_g
          tc_fence_before();
          mbar_arrive(&sm.s_free[grp]);
        }
        if (!full) {
#pragma unroll
          for (int c4 = 0; c4 < kTile / 4; ++c4) {
            const int4 k4 = *reinterpret_cast<const int4*>(&sm.kidx[grp][b][c4 * 4]);
            bool adm[4] = {qi >= k4.x, qi >= k4.y, qi >= k4.z, qi >= k4.w};
            if (p.mode == SCFA_MODE_HASH) {
              const int4 h4 = *reinterpret_cast<const int4*>(&sm.khash[grp][b][c4 * 4]);
              adm[0] = adm[0] && qh == h4.x;
              adm[1] = adm[1] && qh == h4.y;
              adm[2] = adm[2] && qh == h4.z;
              adm[3] = adm[3] && qh == h4.w;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (!adm[u]) sr[c4 * 4 + u] = 0xff800000u;  // -inf
          }
        }
        // row max: four independent chains of three-input maxima
        float mx0 = __uint_as_float(sr[0]), mx1 = __uint_as_float(sr[1]);
        float mx2 = __uint_as_float(sr[2]), mx3 = __uint_as_float(sr[3]);
#pragma unroll
        for (int c = 4; c < kTile; c += 8) {
          mx0 = max3f(mx0, __uint_as_float(sr[c + 0]), __uint_as_float(sr[c + 1]));
          mx1 = max3f(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
          mx2 = max3f(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
          mx3 = max3f(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
        }
        const float mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * p.scale_log2;
        const float m_new = fmaxf(m_used, mt);
        m_top = fmaxf(m_top, mt);
        const bool resc = m_new > m_used + kRescaleThreshold;
        float alpha = 1.f;
        if (resc) {
          alpha = ex2_approx(m_used - m_new);
          m_used = m_new;
        }
        const float msub = (m_used == -INFINITY) ? 0.f : m_used;
        // P = 2^(s * scale * log2(e) - m) as bf16 pairs over the first 64 columns
        // of S_g; the argument and the row sum run on packed f32 pairs
        const uint64_t sl2 = f2(p.scale_log2, p.scale_log2), nm2 = f2(-msub, -msub);
        if (kSepP && n_p > 0) {
          // the previous PV_g has read P_g (and finished adding into O_g)
          ok = mbar_wait(&sm.pv_done[grp], (n_p - 1) & 1, abort_flag, p.status);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
        }
        ++n_p;
        uint64_t rsum2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const uint64_t arg = fma2(f2(__uint_as_float(sr[h * 32 + c]), __uint_as_float(sr[h * 32 + c + 1])), sl2, nm2);
            float a0, a1;
            f2_split(arg, a0, a1);
            const float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
            rsum2[(c >> 1) & 3] = add2(rsum2[(c >> 1) & 3], f2(e0, e1));
            pk[c >> 1] = pack_bf16x2(e0, e1);
          }
          tmem_st16(lane_base + colP + h * 16, pk);
        }
        const uint64_t rs2 = add2(add2(rsum2[0], rsum2[1]), add2(rsum2[2], rsum2[3]));
        float rs_lo, rs_hi;
        f2_split(rs2, rs_lo, rs_hi);
        const float rs = rs_lo + rs_hi;
        l = l * alpha + rs;
        // rescale O (rare). PV_g(t-1) is complete here: with separate P columns
        // the wait above says so; otherwise S_g(t) complete implies it
        if (!first_tile && __any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t orr[32];
            tmem_ld32(lane_base + colO + cc * 32, orr);
            tmem_wait_ld();
            tmem_ld_fence(orr);
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
            tmem_st32(lane_base + colO + cc * 32, orr);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&sm.p_full[grp]);
        ++s_it;
        j_c = j_n;
        f_c = f_n;
        kid_c = kid_n;
        kh_c = kh_n;
        j_n = j_nn;
        f_n = f_nn;
      }
      if (!ok) break;
      if (!any) {
        if (valid) {
          const long long orow = mapped_row(p.o_rows, grow, bh, p.To);
          if (orow >= 0) {
            uint4* dst = reinterpret_cast<uint4*>(p.o + orow * D);
#pragma unroll
            for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
          }
          p.lse[grow] = -INFINITY;
          if (p.o32 && orow >= 0) zero_o32_row<D>(p.o32 + grow * D);
        }
        continue;
      }
      // epilogue: O / l, LSE
      ok = mbar_wait(&sm.o_full[grp], o_it & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      uint32_t orr[D / 32][32];
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(lane_base + colO + cc * 32, orr[cc]);
      tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) tmem_ld_fence(orr[cc]);
      tc_fence_before();
      mbar_arrive(&sm.o_empty[grp]);
      ++o_it;
      if (valid) {
        // O is normalised by the row sum as PV saw it for the largest score:
        // with the lazy rescale its weight 2^(m_top - m_used) need not be 1,
        // and PV used its bf16 rounding. Swapping that one term of l for the
        // rounded value makes a row with a single key return V exactly and
        // removes the largest coherent error of O on rows with few keys. LSE
        // keeps the unrounded sum (the backward recomputes P from it).
        float l_o = l;
        if (l > 0.f) {
          const float pm = ex2_approx(m_top - m_used);
          l_o = l - pm + __bfloat162float(__float2bfloat16_rn(pm));
        }
        const float inv = l_o > 0.f ? 1.f / l_o : 0.f;
        const long long orow = mapped_row(p.o_rows, grow, bh, p.To);
        uint4* dst = reinterpret_cast<uint4*>(p.o + (orow >= 0 ? orow : grow) * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const int e = c * 8;
          uint4 u;
          u.x = pack_bf16x2(__uint_as_float(orr[e >> 5][(e + 0) & 31]) * inv, __uint_as_float(orr[e >> 5][(e + 1) & 31]) * inv);
          u.y = pack_bf16x2(__uint_as_float(orr[e >> 5][(e + 2) & 31]) * inv, __uint_as_float(orr[e >> 5][(e + 3) & 31]) * inv);
          u.z = pack_bf16x2(__uint_as_float(orr[e >> 5][(e + 4) & 31]) * inv, __uint_as_float(orr[e >> 5][(e + 5) & 31]) * inv);
          u.w = pack_bf16x2(__uint_as_float(orr[e >> 5][(e + 6) & 31]) * inv, __uint_as_float(orr[e >> 5][(e + 7) & 31]) * inv);
          if (orow >= 0) dst[c] = u;
        }
        p.lse[grow] = l > 0.f ? (m_used + log2f(l)) * kLn2 : -INFINITY;
        // (a padding row of an original-order step has no O32 row: the
        // backward pre-pass skips it)
        if (p.o32 && orow >= 0) store_o32_row<D>(p.o32 + grow * D, orr, inv);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}


// ---------------------------------------------------------------------------
// Single-query-tile forward for D = 64: two CTAs per SM, each walking its own
// query tiles, so the two tiles an SM works on never wait on one another.
// Roles (192 threads): warp 0 producer (TMA: Q double-buffered, K and V in
// separate 2-stage rings so a K stage is released as soon as S has read it),
// warp 1 MMA issuer and TMEM owner (256 columns: S [0,128), O [128,192),
// P [192,256)), warps 2-5 softmax (thread = query row = TMEM lane). S(j+1) is
// computed while the softmax works on S(j): the softmax frees S once it is in
// registers and waits for PV(j-1) before overwriting P.
// ---------------------------------------------------------------------------
constexpr int kF1Threads = 192;
constexpr int kF1Stages = 2;
constexpr int kF1Slots = 4;  // work items handed from the producer to the other roles
constexpr uint32_t kF1TmemCols = 256;

struct __align__(1024) Fwd1Smem {
  uint8_t q[2][kSubBytes];
  uint8_t k[kF1Stages][kSubBytes];
  uint8_t v[kF1Stages][kSubBytes];
  int32_t kidx[2][kTile];
  int32_t khash[2][kTile];
  int32_t items[kF1Slots];
  uint64_t item_full[kF1Slots], item_empty[kF1Slots];
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kF1Stages], k_empty[kF1Stages], v_full[kF1Stages], v_empty[kF1Stages];
  uint64_t s_full, s_free, o_full, o_empty, kbar, drain;
  uint64_t p_full[2], pv_done[2];  // per key half: keys 0-63 (P columns 0-31), keys 64-127
  uint32_t tmem_base;
  int abort_flag;
};

__global__ void __launch_bounds__(kF1Threads, 2)
attn_fwd1_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  constexpr int D = 64;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  Fwd1Smem& sm = *reinterpret_cast<Fwd1Smem*>(smem_raw + pad);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // live-tile lists where the call that built them put them
  const int32_t* const cols = ws_list<int32_t>(p.status, kListCols);
  const uint8_t* const fflags = ws_list<uint8_t>(p.status, kListFflags);

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.q_full[b], 1);
      mbar_init(&sm.q_empty[b], 1);
    }
    for (int s = 0; s < kF1Stages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    for (int s = 0; s < kF1Slots; ++s) {
      mbar_init(&sm.item_full[s], 1);
      mbar_init(&sm.item_empty[s], 129);  // the MMA thread and the 128 softmax threads
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.s_free, 128);
    for (int hf = 0; hf < 2; ++hf) {
      mbar_init(&sm.p_full[hf], 128);
      mbar_init(&sm.pv_done[hf], 1);
    }
    mbar_init(&sm.o_full, 1);
    mbar_init(&sm.o_empty, 128);
    mbar_init(&sm.kbar, 128);
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, kF1TmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;
  constexpr uint32_t kColS = 0, kColO = 128, kColP = 192;

  if (warp == 0 && !p.gather_q && !p.gather_kv) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // Work items are taken from a global counter in list order (largest
      // first) as this CTA gets through its previous ones, and handed to the
      // MMA and softmax roles through a small slot ring; -1 ends the walk.
      int item = 0, kv = 0, slot_it = 0;
      int k_issued = 0, v_issued = 0, q_issued = 0;  // loads issued, for the drain
      for (;;) {
        const int slot = slot_it % kF1Slots;
        if (!mbar_wait(&sm.item_empty[slot], ((slot_it / kF1Slots) & 1) ^ 1, abort_flag, p.status)) break;
        const int w = atomicAdd(&p.sched[0], 1);
        sm.items[slot] = w < p.n_work ? w : -1;
        mbar_arrive(&sm.item_full[slot]);
        ++slot_it;
        if (w >= p.n_work) break;
        const int g = p.work[w];
        const int e0 = p.row_ptr[g], n = p.row_ptr[g + 1] - e0;
        if (n == 0) continue;
        const int bh = g / p.nQt, i = g % p.nQt;
        const int qb = item & 1;
        if (!mbar_wait(&sm.q_empty[qb], ((item >> 1) & 1) ^ 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&sm.q_full[qb], D * kTile * 2);
        tma_load_3d(sm.q[qb], &tm_q, &sm.q_full[qb], 0, i * kTile, bh);
        q_issued = item + 1;
        bool ok = !(p.stall && kv == 0);  // debug stall: no K / V load ever arrives
        for (int t = 0; t < n && ok; ++t) {
          const int j = cols[e0 + t];
          const int s = kv % kF1Stages;
          const uint32_t ph = ((kv / kF1Stages) & 1) ^ 1;
          if (!mbar_wait(&sm.k_empty[s], ph, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&sm.k_full[s], D * kTile * 2);
          tma_load_3d(sm.k[s], &tm_k, &sm.k_full[s], 0, j * kTile, bh);
          k_issued = kv + 1;
          if (!mbar_wait(&sm.v_empty[s], ph, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&sm.v_full[s], D * kTile * 2);
          tma_load_3d(sm.v[s], &tm_v, &sm.v_full[s], 0, j * kTile, bh);
          v_issued = kv + 1;
          ++kv;
        }
        if (!ok) break;
        ++item;
      }
      // drain: every copy issued by this thread has landed before the CTA
      // exits, also after an abort (the counts are of loads actually issued)
      for (int d = 1; d <= kF1Stages && d <= k_issued; ++d) {
        const int it = k_issued - d;
        mbar_wait_drain(&sm.k_full[it % kF1Stages], (it / kF1Stages) & 1, p.status);
      }
      for (int d = 1; d <= kF1Stages && d <= v_issued; ++d) {
        const int it = v_issued - d;
        mbar_wait_drain(&sm.v_full[it % kF1Stages], (it / kF1Stages) & 1, p.status);
      }
      for (int d = 1; d <= 2 && d <= q_issued; ++d) {
        const int it = q_issued - d;
        mbar_wait_drain(&sm.q_full[it & 1], (it >> 1) & 1, p.status);
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer (row gathers)
    // The same walk with the whole warp: lane 0 waits on the stages and
    // issues the tiled loads, every lane issues four rows of each gathered
    // tile (p.gather_q: Q; p.gather_kv: K, V), their source rows loaded a
    // tile ahead, before the stage wait. (Without gathers the single-lane
    // producer above is kept: the warp-wide loop cost the QK forward 4%.)
    int item = 0, kv = 0, slot_it = 0;
    int k_issued = 0, v_issued = 0, q_issued = 0;  // loads issued, for the drain
    for (;;) {
      const int slot = slot_it % kF1Slots;
      int w = INT_MAX;
      if (lane == 0 && mbar_wait(&sm.item_empty[slot], ((slot_it / kF1Slots) & 1) ^ 1, abort_flag, p.status)) {
        w = atomicAdd(&p.sched[0], 1);
        sm.items[slot] = w < p.n_work ? w : -1;
        mbar_arrive(&sm.item_full[slot]);
      }
      w = __shfl_sync(0xffffffffu, w, 0);
      ++slot_it;
      if (w >= p.n_work) break;
      const int g = p.work[w];
      const int e0 = p.row_ptr[g], n = p.row_ptr[g + 1] - e0;
      if (n == 0) continue;
      const int bh = g / p.nQt, i = g % p.nQt;
      const int qb = item & 1;
      int rr[4];
      if (p.gather_q) gather_rows(p.q_idx, bh, p.Tq, p.To, i * kTile, lane, rr);
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(&sm.q_empty[qb], ((item >> 1) & 1) ^ 1, abort_flag, p.status);
        if (ok) {
          mbar_arrive_expect_tx(&sm.q_full[qb], D * kTile * 2);
          if (!p.gather_q) tma_load_3d(sm.q[qb], &tm_q, &sm.q_full[qb], 0, i * kTile, bh);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      if (p.gather_q) gather_issue(sm.q[qb], 0, 1, &tm_q, &sm.q_full[qb], rr, lane);
      q_issued = item + 1;
      ok = !(p.stall && kv == 0);  // debug stall: no K / V load ever arrives
      // the item's key tiles are read 32 at a time (one per lane); with row
      // gathers the source rows of a tile are loaded a tile ahead
      int cj = lane < n ? cols[e0 + lane] : 0;
      int rk[4] = {0, 0, 0, 0};
      if (p.gather_kv) gather_rows(p.k_idx, bh, p.Tk, p.To, __shfl_sync(0xffffffffu, cj, 0) * kTile, lane, rk);
      for (int t = 0; t < n && ok; ++t) {
        const int j = __shfl_sync(0xffffffffu, cj, t & 31);
        const int s = kv % kF1Stages;
        const uint32_t ph = ((kv / kF1Stages) & 1) ^ 1;
        if (t + 1 < n) {
          if (((t + 1) & 31) == 0) cj = t + 1 + lane < n ? cols[e0 + t + 1 + lane] : 0;
          if (p.gather_kv)  // K and V rows of the next tile
            gather_rows(p.k_idx, bh, p.Tk, p.To, __shfl_sync(0xffffffffu, cj, (t + 1) & 31) * kTile, lane, rr);
        }
        if (lane == 0) {
          ok = mbar_wait(&sm.k_empty[s], ph, abort_flag, p.status);
          if (ok) {
            mbar_arrive_expect_tx(&sm.k_full[s], D * kTile * 2);
            if (!p.gather_kv) tma_load_3d(sm.k[s], &tm_k, &sm.k_full[s], 0, j * kTile, bh);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) { ok = false; break; }
        if (p.gather_kv) gather_issue(sm.k[s], 0, 1, &tm_k, &sm.k_full[s], rk, lane);
        k_issued = kv + 1;
        if (lane == 0) {
          ok = mbar_wait(&sm.v_empty[s], ph, abort_flag, p.status);
          if (ok) {
            mbar_arrive_expect_tx(&sm.v_full[s], D * kTile * 2);
            if (!p.gather_kv) tma_load_3d(sm.v[s], &tm_v, &sm.v_full[s], 0, j * kTile, bh);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) { ok = false; break; }
        if (p.gather_kv) {
          gather_issue(sm.v[s], 0, 1, &tm_v, &sm.v_full[s], rk, lane);
#pragma unroll
          for (int u = 0; u < 4; ++u) rk[u] = rr[u];
        }
        v_issued = kv + 1;
        ++kv;
      }
      if (!ok) break;
      ++item;
    }
    if (lane == 0) {
      // drain: every copy issued by this warp has landed before the CTA
      // exits, also after an abort (the counts are of loads actually issued)
      for (int d = 1; d <= kF1Stages && d <= k_issued; ++d) {
        const int it = k_issued - d;
        mbar_wait_drain(&sm.k_full[it % kF1Stages], (it / kF1Stages) & 1, p.status);
      }
      for (int d = 1; d <= kF1Stages && d <= v_issued; ++d) {
        const int it = v_issued - d;
        mbar_wait_drain(&sm.v_full[it % kF1Stages], (it / kF1Stages) & 1, p.status);
      }
      for (int d = 1; d <= 2 && d <= q_issued; ++d) {
        const int it = q_issued - d;
        mbar_wait_drain(&sm.q_full[it & 1], (it >> 1) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kTile, kTile, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kTile, D, 0, 1);
      const uint64_t qdesc = smem_desc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint64_t kdesc = smem_desc_sw128(smem_u32(sm.k[0]), 16, 1024);
      const uint64_t vdesc = smem_desc_sw128(smem_u32(sm.v[0]), kSubBytes, 1024);
      constexpr uint32_t kBuf16 = kSubBytes >> 4;
      int item = 0, kv = 0, n_s = 0, p_it = 0, o_it = 0;
      bool ok = true;
      auto issue_s = [&](int kvi, int qb) -> bool {
        const int s = kvi % kF1Stages;
        if (n_s > 0 && !mbar_wait(&sm.s_free, (n_s - 1) & 1, abort_flag, p.status)) return false;
        if (!mbar_wait(&sm.k_full[s], (kvi / kF1Stages) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint64_t a = qdesc + static_cast<uint64_t>(qb * kBuf16);
        const uint64_t b = kdesc + static_cast<uint64_t>(s * kBuf16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(tmem + kColS, a + kstep_off16(kk, kSubBytes), b + kstep_off16(kk, kSubBytes), idesc_s, kk > 0);
        tc_commit(&sm.s_full);
        tc_commit(&sm.k_empty[s]);  // K stage free once S has read it
        ++n_s;
        return true;
      };
      for (int slot_it = 0; ok; ++slot_it) {
        const int slot = slot_it % kF1Slots;
        if (!mbar_wait(&sm.item_full[slot], (slot_it / kF1Slots) & 1, abort_flag, p.status)) break;
        const int w = sm.items[slot];
        mbar_arrive(&sm.item_empty[slot]);
        if (w < 0) break;
        const int g = p.work[w];
        const int n = p.row_ptr[g + 1] - p.row_ptr[g];
        if (n == 0) continue;
        const int qb = item & 1;
        if (!mbar_wait(&sm.q_full[qb], (item >> 1) & 1, abort_flag, p.status)) break;
        if (!issue_s(kv, qb)) break;
        for (int t = 0; t < n; ++t) {
          const int s = kv % kF1Stages;
          if (t + 1 < n && !issue_s(kv + 1, qb)) { ok = false; break; }
          if (t == 0 && !mbar_wait(&sm.o_empty, (o_it & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
          if (!mbar_wait(&sm.v_full[s], (kv / kF1Stages) & 1, abort_flag, p.status)) { ok = false; break; }
          const uint64_t vb = vdesc + static_cast<uint64_t>(s * kBuf16);
          // PV in two halves of 64 keys, each as soon as the softmax has
          // written that half of P
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            if (!mbar_wait(&sm.p_full[hf], p_it & 1, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int kq = 0; kq < 4; ++kq) {
              const int kk = hf * 4 + kq;
              mma_bf16_ts(tmem + kColO, tmem + kColP + kk * 8, vb + static_cast<uint64_t>(kk * 128), idesc_o,
                          (kk > 0 || t > 0) ? 1u : 0u);
            }
            tc_commit(&sm.pv_done[hf]);
          }
          if (!ok) break;
          tc_commit(&sm.v_empty[s]);
          ++kv;
          ++p_it;
        }
        if (!ok) break;
        tc_commit(&sm.o_full);
        tc_commit(&sm.q_empty[qb]);
        ++o_it;
        ++item;
      }
      tc_commit(&sm.drain);
      mbar_wait_drain(&sm.drain, 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroup
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;          // row of the tile = TMEM lane
    const int tid = (warp - 2) * 32 + lane;     // 0..127
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    int s_it = 0, o_it = 0, x_it = 0;
    // the 128 softmax threads; a bounded wait (a broken pipeline ends in a
    // status code, not a hang)
    auto group_sync = [&]() -> bool {
      mbar_arrive(&sm.kbar);
      const bool r_ok = mbar_wait(&sm.kbar, x_it & 1, abort_flag, p.status);
      ++x_it;
      return __all_sync(0xffffffffu, r_ok);
    };
    for (int slot_it = 0;; ++slot_it) {
      const int slot = slot_it % kF1Slots;
      bool got = mbar_wait(&sm.item_full[slot], (slot_it / kF1Slots) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, got)) break;
      const int w = sm.items[slot];
      mbar_arrive(&sm.item_empty[slot]);
      if (w < 0) break;
      const int g = p.work[w];
      const int e_beg = p.row_ptr[g], e_end = p.row_ptr[g + 1];
      const int bh = g / p.nQt, i = g % p.nQt;
      const int row = i * kTile + r;
      const bool valid = row < p.Tq;
      const long long grow = static_cast<long long>(bh) * p.Tq + row;
      int qi = INT_MIN, qh = 0;
      if (valid) {
        qi = (p.mode == SCFA_MODE_DENSE) ? row : p.q_idx[grow];
        if (p.mode == SCFA_MODE_HASH) qh = p.q_hash[grow];
      }
      const long long kbase = static_cast<long long>(bh) * p.Tk;
      // key index / bucket of a masked tile, one per thread
      auto key_meta = [&](int j, int f, int& kid, int& kh) {
        kid = INT_MAX;
        kh = INT_MIN;
        if (f & kFlagFull) return;
        const int col = j * kTile + tid;
        const bool kvv = col < p.Tk;
        if (p.mode == SCFA_MODE_DENSE) kid = kvv ? col : INT_MAX;
        else kid = kvv ? p.k_idx[kbase + col] : INT_MAX;
        if (p.mode == SCFA_MODE_HASH) kh = kvv ? p.k_hash[kbase + col] : INT_MIN;
      };
      // column / flag two tiles ahead, key metadata one tile ahead
      int f_c = 0, j_n = 0, f_n = 0, kid_c = INT_MAX, kh_c = INT_MIN;
      if (e_beg < e_end) {
        f_c = fflags[e_beg];
        key_meta(cols[e_beg], f_c, kid_c, kh_c);
      }
      if (e_beg + 1 < e_end) {
        j_n = cols[e_beg + 1];
        f_n = fflags[e_beg + 1];
      }
      float m_used = -INFINITY, l = 0.f;
      float m_top = -INFINITY;  // largest score of the row so far (log2 units)
      bool ok = true, any = false;
      for (int e = e_beg; e < e_end; ++e) {
        const bool full = (f_c & kFlagFull) != 0;
        int kid_n = INT_MAX, kh_n = INT_MIN, j_nn = 0, f_nn = 0;
        if (e + 1 < e_end) key_meta(j_n, f_n, kid_n, kh_n);
        if (e + 2 < e_end) {
          j_nn = cols[e + 2];
          f_nn = fflags[e + 2];
        }
        const bool first_tile = !any;
        any = true;
        const int b = s_it & 1;
        if (!full) {
          sm.kidx[b][tid] = kid_c;
          if (p.mode == SCFA_MODE_HASH) sm.khash[b][tid] = kh_c;
          if (!group_sync()) { ok = false; break; }
        }
        ok = mbar_wait(&sm.s_full, s_it & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[kTile];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          tmem_ld32(lane_base + kColS + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[cc * 32]));
        tmem_wait_ld();
        tmem_ld_fence(sr);
        // S is in registers: the MMA warp may compute the next S
        tc_fence_before();
        mbar_arrive(&sm.s_free);
        if (!full) {
#pragma unroll
          for (int c4 = 0; c4 < kTile / 4; ++c4) {
            const int4 k4 = *reinterpret_cast<const int4*>(&sm.kidx[b][c4 * 4]);
            bool adm[4] = {qi >= k4.x, qi >= k4.y, qi >= k4.z, qi >= k4.w};
            if (p.mode == SCFA_MODE_HASH) {
              const int4 h4 = *reinterpret_cast<const int4*>(&sm.khash[b][c4 * 4]);
              adm[0] = adm[0] && qh == h4.x;
              adm[1] = adm[1] && qh == h4.y;
              adm[2] = adm[2] && qh == h4.z;
              adm[3] = adm[3] && qh == h4.w;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (!adm[u]) sr[c4 * 4 + u] = 0xff800000u;  // -inf
          }
        }
        float mx0 = __uint_as_float(sr[0]), mx1 = __uint_as_float(sr[1]);
        float mx2 = __uint_as_float(sr[2]), mx3 = __uint_as_float(sr[3]);
#pragma unroll
        for (int c = 4; c < kTile; c += 8) {
          mx0 = max3f(mx0, __uint_as_float(sr[c + 0]), __uint_as_float(sr[c + 1]));
          mx1 = max3f(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
          mx2 = max3f(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
          mx3 = max3f(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
        }
        const float mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * p.scale_log2;
        const float m_new = fmaxf(m_used, mt);
        m_top = fmaxf(m_top, mt);
        const bool resc = m_new > m_used + kRescaleThreshold;
        float alpha = 1.f;
        if (resc) {
          alpha = ex2_approx(m_used - m_new);
          m_used = m_new;
        }
        const float msub = (m_used == -INFINITY) ? 0.f : m_used;
        const uint64_t sl2 = f2(p.scale_log2, p.scale_log2), nm2 = f2(-msub, -msub);
        // P in two halves of 64 keys: each half waits for the previous PV's
        // half that read it, and is handed to the MMA warp as soon as written
        uint64_t rsum2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (s_it > 0) {
            ok = mbar_wait(&sm.pv_done[hf], (s_it - 1) & 1, abort_flag, p.status);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
          }
#pragma unroll
          for (int hq = 0; hq < 2; ++hq) {
            const int h = hf * 2 + hq;
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const uint64_t arg = fma2(f2(__uint_as_float(sr[h * 32 + c]), __uint_as_float(sr[h * 32 + c + 1])), sl2, nm2);
              float a0, a1;
              f2_split(arg, a0, a1);
              const float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
              rsum2[(c >> 1) & 3] = add2(rsum2[(c >> 1) & 3], f2(e0, e1));
              pk[c >> 1] = pack_bf16x2(e0, e1);
            }
            tmem_st16(lane_base + kColP + h * 16, pk);
          }
          // rescale O (rare) before the first half goes to the MMA warp; both
          // halves of the previous PV are complete (the second was waited for
          // only if needed here)
          if (hf == 0 && !first_tile && __any_sync(0xffffffffu, resc)) {
            ok = mbar_wait(&sm.pv_done[1], (s_it - 1) & 1, abort_flag, p.status);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t orr[32];
              tmem_ld32(lane_base + kColO + cc * 32, orr);
              tmem_wait_ld();
              tmem_ld_fence(orr);
#pragma unroll
              for (int e2 = 0; e2 < 32; ++e2) orr[e2] = __float_as_uint(__uint_as_float(orr[e2]) * alpha);
              tmem_st32(lane_base + kColO + cc * 32, orr);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&sm.p_full[hf]);
        }
        if (!ok) break;
        const uint64_t rs2 = add2(add2(rsum2[0], rsum2[1]), add2(rsum2[2], rsum2[3]));
        float rs_lo, rs_hi;
        f2_split(rs2, rs_lo, rs_hi);
        l = l * alpha + (rs_lo + rs_hi);
        ++s_it;
        f_c = f_n;
        kid_c = kid_n;
        kh_c = kh_n;
        j_n = j_nn;
        f_n = f_nn;
      }
      if (!ok) break;
      if (!any) {
        if (valid) {
          const long long orow = mapped_row(p.o_rows, grow, bh, p.To);
          if (orow >= 0) {
            uint4* dst = reinterpret_cast<uint4*>(p.o + orow * D);
#pragma unroll
            for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
          }
          p.lse[grow] = -INFINITY;
          if (p.o32 && orow >= 0) zero_o32_row<D>(p.o32 + grow * D);
        }
        continue;
      }
      // epilogue: O / l, LSE
      ok = mbar_wait(&sm.o_full, o_it & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      uint32_t orr[D / 32][32];
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(lane_base + kColO + cc * 32, orr[cc]);
      tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) tmem_ld_fence(orr[cc]);
      tc_fence_before();
      mbar_arrive(&sm.o_empty);
      ++o_it;
      if (valid) {
        // O is normalised by the row sum as PV saw it for the largest score:
        // with the lazy rescale its weight 2^(m_top - m_used) need not be 1,
        // and PV used its bf16 rounding. Swapping that one term of l for the
        // rounded value makes a row with a single key return V exactly and
        // removes the largest coherent error of O on rows with few keys. LSE
        // keeps the unrounded sum (the backward recomputes P from it).
        float l_o = l;
        if (l > 0.f) {
          const float pm = ex2_approx(m_top - m_used);
          l_o = l - pm + __bfloat162float(__float2bfloat16_rn(pm));
        }
        const float inv = l_o > 0.f ? 1.f / l_o : 0.f;
        const long long orow = mapped_row(p.o_rows, grow, bh, p.To);
        uint4* dst = reinterpret_cast<uint4*>(p.o + (orow >= 0 ? orow : grow) * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const int e = c * 8;
          uint4 u;
          u.x = pack_bf16x2(__uint_as_float(orr[e >> 5][(e + 0) & 31]) * inv, __uint_as_float(orr[e >> 5][(e + 1) & 31]) * inv);
          u.y = pack_bf16x2(__uint_as_float(orr[e >> 5][(e + 2) & 31]) * inv, __uint_as_float(orr[e >> 5][(e + 3) & 31]) * inv);
          u.z = pack_bf16x2(__uint_as_float(orr[e >> 5][(e + 4) & 31]) * inv, __uint_as_float(orr[e >> 5][(e + 5) & 31]) * inv);
          u.w = pack_bf16x2(__uint_as_float(orr[e >> 5][(e + 6) & 31]) * inv, __uint_as_float(orr[e >> 5][(e + 7) & 31]) * inv);
          if (orow >= 0) dst[c] = u;
        }
        p.lse[grow] = l > 0.f ? (m_used + log2f(l)) * kLn2 : -INFINITY;
        // (a padding row of an original-order step has no O32 row: the
        // backward pre-pass skips it)
        if (p.o32 && orow >= 0) store_o32_row<D>(p.o32 + grow * D, orr, inv);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kF1TmemCols);
  // the last CTA to finish (every CTA has stopped taking items by then)
  // leaves the counters at zero for the next launch on this workspace
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&p.sched[1], 1) == static_cast<int>(gridDim.x) - 1) {
      atomicExch(&p.sched[0], 0);
      atomicExch(&p.sched[1], 0);
    }
  }
}

}  // namespace

bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, int D, long long T, long long BH);

// tiled maps over the sorted q, k, v, or row-gather maps over the
// original-order ones
static bool make_fwd_maps(const AttnArgs& a, int D, long long BH, CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv) {
  const bool q_ok = a.gather_q ? make_tmap_bf16_rows(tq, a.q, D, BH * a.To) : make_tmap_bf16_3d(tq, a.q, D, a.Tq, BH);
  const bool kv_ok = a.gather_kv
                         ? make_tmap_bf16_rows(tk, a.k, D, BH * a.To) && make_tmap_bf16_rows(tv, a.v, D, BH * a.To)
                         : make_tmap_bf16_3d(tk, a.k, D, a.Tk, BH) && make_tmap_bf16_3d(tv, a.v, D, a.Tk, BH);
  return q_ok && kv_ok;
}

template <int D>
static cudaError_t launch_fwd_d(const AttnArgs& a, cudaStream_t st) {
  const AttnWs& L = *a.L;
  const long long BH = static_cast<long long>(a.B) * a.H;
  CUtensorMap tq, tk, tv;
  if (!make_fwd_maps(a, D, BH, &tq, &tk, &tv)) return cudaErrorInvalidValue;
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
  p.nPairs = L.nPairs;
  p.work_pairs = reinterpret_cast<const int32_t*>(a.ws + L.work_pairs);
  p.pcount = reinterpret_cast<const int32_t*>(a.ws + L.pcount);
  p.n_pairs = static_cast<int>(L.n_pairs);
  p.o = a.o_out;
  p.o_rows = a.q_rows;
  p.To = a.To;
  p.lse = a.lse_out;
  p.o32 = a.o32;
  p.stall = a.stall;
  p.gather_q = a.gather_q;
  p.gather_kv = a.gather_kv;
  p.status = reinterpret_cast<int*>(a.ws + L.header);
  const size_t smem = sizeof(FwdSmem<D>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int grid = num_sms();
  if (grid > p.n_pairs) grid = p.n_pairs;
  if (grid < 1) grid = 1;
  record_kernel_event(0, true, st);
  attn_fwd_kernel<D><<<grid, kFwdThreads, smem, st>>>(tq, tk, tv, p);
  record_kernel_event(0, false, st);
  return cudaGetLastError();
}

// D = 64: single-query-tile kernel, two CTAs per SM
static cudaError_t launch_fwd1(const AttnArgs& a, cudaStream_t st) {
  constexpr int D = 64;
  const AttnWs& L = *a.L;
  const long long BH = static_cast<long long>(a.B) * a.H;
  CUtensorMap tq, tk, tv;
  if (!make_fwd_maps(a, D, BH, &tq, &tk, &tv)) return cudaErrorInvalidValue;
  FwdParams p = {};
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
  p.work = reinterpret_cast<const int32_t*>(a.ws + L.work_fwd);
  p.n_work = static_cast<int>(L.n_qtiles);
  p.sched = reinterpret_cast<WsHeader*>(a.ws + L.header)->sched;
  p.o = a.o_out;
  p.o_rows = a.q_rows;
  p.To = a.To;
  p.lse = a.lse_out;
  p.o32 = a.o32;
  p.stall = a.stall;
  p.gather_q = a.gather_q;
  p.gather_kv = a.gather_kv;
  p.status = reinterpret_cast<int*>(a.ws + L.header);
  const size_t smem = sizeof(Fwd1Smem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int grid = 2 * num_sms();
  if (grid > p.n_work) grid = p.n_work;
  if (grid < 1) grid = 1;
  record_kernel_event(0, true, st);
  attn_fwd1_kernel<<<grid, kF1Threads, smem, st>>>(tq, tk, tv, p);
  record_kernel_event(0, false, st);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd(const AttnArgs& a, cudaStream_t st) {
  if (a.D == 64) return launch_fwd1(a, st);
  if (a.D == 128) return launch_fwd_d<128>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace scfa
