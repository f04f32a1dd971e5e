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
// GB300 design: persistent CTAs take key tiles from the backward work order
// through a global counter; each work item keeps K_j, V_j resident and
// streams the live query tiles i of its CSC column. Per query tile:
//   A(i): S^T = K Q_i^T and dP^T = V dO_i^T      (tcgen05, TMEM, keys on lanes)
//   compute(i): P^T = exp2(S^T - LSE) under the mask -> TMEM (bf16, the A
//         operand of the dV MMA); dS^T = P^T (dP^T - Drow) scale -> shared
//         memory (bf16, double-buffered)
//   B(i): dV += P^T dO_i (A from TMEM), dK += dS^T Q_i, dQ_i = dS K
// Head dimension 64 (attn_bwd_kernel<64>): the MMA warp issues A(i+1) as
// soon as compute(i) has read S^T / dP^T out of TMEM, so the tensor core runs
// A(i+1) and B(i-1) while compute(i) works. Roles (448 threads):
//   warp 0       producer: lane 0 issues the TMA loads of K_j, V_j (once per
//                item) and Q_i, dO_i (3-stage ring); all 32 lanes stage the
//                query metadata (position, bucket, LSE in log2 units,
//                rowsum * scale) of tile i next to it.
//   warp 1       TMEM owner (512 columns); lane 0 issues every tcgen05.mma.
//   warps 2-9    two compute warpgroups; thread = key row = TMEM lane; the
//                first group owns query columns 0-63, the second 64-127.
//   warps 10-13  dQ warpgroup; thread = query row: dQ_i from TMEM into a
//                swizzled fp32 shared tile, then one TMA reduce-add per
//                64-column half into the fp32 accumulator in the workspace.
// TMEM columns: S^T [0,128) dP^T [128,256) dV [256,320) dK [320,384)
// dQ [384,448) P^T (bf16 pairs) [448,512).
// Head dimension 128 (attn_bwd128_kernel): the same roles, but dV and dK
// take 128 TMEM columns each, so P^T and dQ overwrite S^T and dP^T once they
// have been read, and A(i+1) follows B(i); described at the kernel.
// Every wait is bounded.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace scfa {
namespace {

constexpr int kSubBytes = kTile * 128;
// Q / dO / query-metadata ring depth of attn_bwd_kernel (head dimension 64;
// head dimension 128 runs attn_bwd128_kernel), with one or two K / V buffers
template <int D, int KVB>
constexpr int bwd_qstages() {
  static_assert(D == 64, "attn_bwd_kernel is built for head dimension 64");
  static_assert(KVB == 1 || KVB == 2, "one or two K / V buffers");
  return 3;
}
// dS^T buffers: two with one K / V buffer; with two K / V buffers shared
// memory holds one, and the compute warps write dS^T(t) once the MMAs of
// tile t - 1 have read it (mostly done by the time tile t's math ends).
// Measured: the long QK columns need the second dS^T buffer, hash mode's
// short ones the second K / V buffer and the third query stage.
template <int KVB>
constexpr int bwd_dsbufs() {
  return KVB == 1 ? 2 : 1;
}
constexpr int kBwdThreads = 448;

constexpr int kBwdSlots = 4;  // work items handed from the producer to the other roles
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int D, int KVB>
struct __align__(1024) BwdSmem {
  static constexpr int kQStages = bwd_qstages<D, KVB>();
  static constexpr int kDsBufs = bwd_dsbufs<KVB>();
  uint8_t k[KVB][D / 64][kSubBytes];  // K / V of work item n in buffer n % KVB
  uint8_t v[KVB][D / 64][kSubBytes];
  uint8_t q[kQStages][D / 64][kSubBytes];
  uint8_t dO[kQStages][D / 64][kSubBytes];
  uint8_t dst[kDsBufs][2][kSubBytes];   // dS^T [buffer][query half][128 keys x 64 queries]
  uint8_t dqs[kSubBytes];         // dQ fp32 staging: one [128 rows x 32 floats] swizzled half at a time
  alignas(16) int32_t qidx[kQStages][kTile];
  alignas(16) int32_t qhash[kQStages][kTile];
  alignas(16) float lse2[kQStages][kTile];    // -LSE * log2(e)
  alignas(16) float drs[kQStages][kTile];     // -rowsum(dO * O) * scale
  uint64_t kv_full[KVB], kv_empty[KVB];
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t s_full, st_empty, ds_full, pt_free, ds_free[kDsBufs], dq_full, dq_empty, dkv_full, dkv_empty, drain;
  uint64_t dq_sync;  // the 128 threads of the dQ warpgroup around the staging tile
  int32_t items[kBwdSlots];
  int4 imeta[kBwdSlots];  // two K/V buffers (hash mode): the item's {key tile, first CSC entry, count}
  uint64_t item_full[kBwdSlots], item_empty[kBwdSlots];
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
  // per-query metadata (bwd_pre_kernel), four arrays of qm_n entries padded to
  // whole tiles (Tqp rows per head): -LSE*log2(e), -rowsum(dO*O)*scale, position, bucket
  const float* qm;
  long long qm_n;
  int Tqp;
  const int32_t* csc_ptr;
  const int32_t* work;
  int n_work;
  uint16_t* dk;
  uint16_t* dv;
  const int32_t* k_rows;  // null, or the original row of each sorted key row
  int To;                 // rows per head of dk / dv when k_rows is set
  int stall;   // SCFA_FLAG_DEBUG_STALL: withhold the first K / V load
  int gather_q;   // q and do are original-order tensors read by row gathers through q_idx (To rows per head)
  int gather_kv;  // k and v likewise through k_idx
  int* sched;  // [0] next work item, [1] CTAs done
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

template <int D, int KVB>
__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  BwdSmem<D, KVB>& sm = *reinterpret_cast<BwdSmem<D, KVB>*>(smem_raw + pad);
  constexpr int kQStages = BwdSmem<D, KVB>::kQStages;
  constexpr int kDsBufs = BwdSmem<D, KVB>::kDsBufs;
  constexpr int kHalves = D / 64;  // a work item = (key tile, 64-column half of D)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // live-tile lists where the call that built them put them
  const int32_t* const csc_rows = ws_list<int32_t>(p.status, kListCscRows);
  const uint8_t* const cflags = ws_list<uint8_t>(p.status, kListCflags);
  constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 320, kColDQ = 384, kColPT = 448;

  if (threadIdx.x == 0) {
    for (int b = 0; b < KVB; ++b) {
      mbar_init(&sm.kv_full[b], 1);
      mbar_init(&sm.kv_empty[b], 1);
    }
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 1);
    }
    for (int s = 0; s < kDsBufs; ++s) mbar_init(&sm.ds_free[s], 1);
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.st_empty, 256);
    mbar_init(&sm.ds_full, 256);
    mbar_init(&sm.pt_free, 1);
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_empty, 128);
    mbar_init(&sm.dkv_full, 1);
    mbar_init(&sm.dkv_empty, 256);
    mbar_init(&sm.drain, 1);
    mbar_init(&sm.dq_sync, 128);
    for (int s = 0; s < kBwdSlots; ++s) {
      mbar_init(&sm.item_full[s], 1);
      mbar_init(&sm.item_empty[s], 1 + 256 + 128);  // MMA thread, compute and dQ warpgroups
    }
    sm.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dq);
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer warp
    // Work items come from a global counter in list order (largest first) as
    // this CTA gets through its previous ones; lane 0 hands each to the other
    // roles through a slot ring, -1 ending the walk.
    int q_it = 0, item = 0, last_kv = -1;
    for (int slot_it = 0;; ++slot_it) {
      int w = INT_MAX;
      if (lane == 0) {
        const int slot = slot_it % kBwdSlots;
        if (mbar_wait(&sm.item_empty[slot], ((slot_it / kBwdSlots) & 1) ^ 1, abort_flag, p.status)) {
          w = atomicAdd(&p.sched[0], 1);
          sm.items[slot] = w < p.n_work ? w : -1;
          if constexpr (KVB == 2) {
            // short hash-mode items: the other roles take the item's key
            // tile and CSC range from the slot instead of loading them
            if (w < p.n_work) {
              const int gg = p.work[w / kHalves];
              const int s0 = p.csc_ptr[gg];
              sm.imeta[slot] = make_int4(gg, s0, p.csc_ptr[gg + 1] - s0, 0);
            }
          }
          mbar_arrive(&sm.item_full[slot]);
        }
      }
      w = __shfl_sync(0xffffffffu, w, 0);
      if (w >= p.n_work) break;
      const int g = p.work[w / kHalves];  // both halves load all of K, V, Q, dO
      const int start = p.csc_ptr[g], n = p.csc_ptr[g + 1] - start;
      if (n == 0) continue;
      const int bh = g / p.nKt, j = g % p.nKt;
      bool ok = true;
      const bool stall = p.stall && item == 0;  // debug stall: K / V never arrive
      // the item's query tiles are read 32 at a time (one per lane); with
      // row gathers (p.gather_q, p.gather_kv) every lane issues four rows of each tile, the
      // source rows of a tile loaded a tile ahead, before the stage wait
      int cq = lane < n ? csc_rows[start + lane] : 0;
      int rr[4], rq[4] = {0, 0, 0, 0}, rn[4] = {0, 0, 0, 0};
      if (p.gather_kv) gather_rows(p.k_idx, bh, p.Tk, p.To, j * kTile, lane, rr);
      if (p.gather_q) gather_rows(p.q_idx, bh, p.Tq, p.To, __shfl_sync(0xffffffffu, cq, 0) * kTile, lane, rq);
      const int kb = item % KVB;
      if (lane == 0 && !stall) {
        ok = mbar_wait(&sm.kv_empty[kb], ((item / KVB) & 1) ^ 1, abort_flag, p.status);
        if (ok) {
          mbar_arrive_expect_tx(&sm.kv_full[kb], 2 * D * kTile * 2);
          if (!p.gather_kv) {
            for (int sub = 0; sub < D / 64; ++sub) {
              tma_load_3d(sm.k[kb][sub], &tm_k, &sm.kv_full[kb], sub * 64, j * kTile, bh);
              tma_load_3d(sm.v[kb][sub], &tm_v, &sm.kv_full[kb], sub * 64, j * kTile, bh);
            }
          }
          last_kv = item;
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      if (p.gather_kv && !stall) {
        gather_issue(sm.k[kb][0], kSubBytes, D / 64, &tm_k, &sm.kv_full[kb], rr, lane);
        gather_issue(sm.v[kb][0], kSubBytes, D / 64, &tm_v, &sm.kv_full[kb], rr, lane);
      }
      const int n_steps = stall ? min(n, kQStages) : n;
      for (int t = 0; t < n_steps; ++t) {
        const int i = __shfl_sync(0xffffffffu, cq, t & 31);
        const int s = q_it % kQStages;
        if (t + 1 < n_steps) {
          if (((t + 1) & 31) == 0) cq = t + 1 + lane < n ? csc_rows[start + t + 1 + lane] : 0;
          if (p.gather_q)  // Q and dO rows of the next tile
            gather_rows(p.q_idx, bh, p.Tq, p.To, __shfl_sync(0xffffffffu, cq, (t + 1) & 31) * kTile, lane, rn);
        }
        if (lane == 0) {
          ok = mbar_wait(&sm.q_empty[s], ((q_it / kQStages) & 1) ^ 1, abort_flag, p.status);
          if (ok) {
            // Q_i, dO_i and the query metadata of tile i (four 512-byte rows
            // of the padded arrays) land on one barrier
            mbar_arrive_expect_tx(&sm.q_full[s], 2 * D * kTile * 2 + 4 * kTile * 4);
            if (!p.gather_q) {
              for (int sub = 0; sub < D / 64; ++sub) {
                tma_load_3d(sm.q[s][sub], &tm_q, &sm.q_full[s], sub * 64, i * kTile, bh);
                tma_load_3d(sm.dO[s][sub], &tm_do, &sm.q_full[s], sub * 64, i * kTile, bh);
              }
            }
            const float* m = p.qm + static_cast<long long>(bh) * p.Tqp + i * kTile;
            bulk_load(sm.lse2[s], m, kTile * 4, &sm.q_full[s]);
            bulk_load(sm.drs[s], m + p.qm_n, kTile * 4, &sm.q_full[s]);
            bulk_load(sm.qidx[s], m + 2 * p.qm_n, kTile * 4, &sm.q_full[s]);
            bulk_load(sm.qhash[s], m + 3 * p.qm_n, kTile * 4, &sm.q_full[s]);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) { ok = false; break; }
        if (p.gather_q) {
          gather_issue(sm.q[s][0], kSubBytes, D / 64, &tm_q, &sm.q_full[s], rq, lane);
          gather_issue(sm.dO[s][0], kSubBytes, D / 64, &tm_do, &sm.q_full[s], rq, lane);
#pragma unroll
          for (int u = 0; u < 4; ++u) rq[u] = rn[u];
        }
        ++q_it;
      }
      if (!ok || stall) break;
      ++item;
    }
    if (lane == 0) {
      // every copy issued by this thread lands before the CTA exits, also
      // after an abort (q_it counts the stages actually loaded)
      for (int d = 1; d <= kQStages && d <= q_it; ++d) {
        const int it = q_it - d;
        mbar_wait_drain(&sm.q_full[it % kQStages], (it / kQStages) & 1, p.status);
      }
      // (items load their K / V in order, so the last KVB loads are the
      // ones that can still be in flight)
      for (int d = 0; d < KVB && last_kv - d >= 0; ++d) {
        const int it = last_kv - d;
        mbar_wait_drain(&sm.kv_full[it % KVB], (it / KVB) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kTile, kTile, 0, 0);
      constexpr uint32_t idesc_kv = idesc_bf16_f32(kTile, 64, 0, 1);  // dV, dK: one 64-column half of D
      constexpr uint32_t idesc_q = idesc_bf16_f32(kTile, 64, 1, 1);   // dQ: one 64-column half of D
      // descriptors built once; steps, stages and buffers are constant adds
      constexpr uint32_t kStage16 = (D / 64) * kSubBytes >> 4;
      const uint64_t kdesc_k0 = smem_desc_sw128(smem_u32(sm.k[0][0]), 16, 1024);           // K, K-major
      const uint64_t vdesc_k0 = smem_desc_sw128(smem_u32(sm.v[0][0]), 16, 1024);           // V, K-major
      const uint64_t kdesc_mn0 = smem_desc_sw128(smem_u32(sm.k[0][0]), kSubBytes, 1024);   // K, MN-major
      constexpr uint32_t kKvBuf16 = (D / 64) * kSubBytes >> 4;  // one K (or V) buffer
      uint64_t kdesc_k = kdesc_k0, vdesc_k = vdesc_k0, kdesc_mn = kdesc_mn0;  // this item's buffer
      const uint64_t qdesc_k = smem_desc_sw128(smem_u32(sm.q[0][0]), 16, 1024);
      const uint64_t qdesc_mn = smem_desc_sw128(smem_u32(sm.q[0][0]), kSubBytes, 1024);
      const uint64_t odesc_k = smem_desc_sw128(smem_u32(sm.dO[0][0]), 16, 1024);
      const uint64_t odesc_mn = smem_desc_sw128(smem_u32(sm.dO[0][0]), kSubBytes, 1024);
      const uint64_t sdesc_k = smem_desc_sw128(smem_u32(sm.dst[0][0]), 16, 1024);      // dS^T, K-major
      const uint64_t sdesc_mn = smem_desc_sw128(smem_u32(sm.dst[0][0]), kSubBytes, 1024);  // dS, MN-major
      constexpr uint32_t kDsBuf16 = 2 * kSubBytes >> 4;
      int q_it = 0, it = 0, item = 0;
      bool ok = true;
      // A(i): S^T and dP^T of query tile stage s into TMEM
      auto issue_a = [&](int qi, int ii) -> bool {
        const int s = qi % kQStages;
        if (!mbar_wait(&sm.q_full[s], (qi / kQStages) & 1, abort_flag, p.status)) return false;
        if (!mbar_wait(&sm.st_empty, (ii & 1) ^ 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint64_t qb = qdesc_k + static_cast<uint64_t>(s * kStage16);
        const uint64_t ob = odesc_k + static_cast<uint64_t>(s * kStage16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(tmem + kColS, kdesc_k + kstep_off16(kk, kSubBytes), qb + kstep_off16(kk, kSubBytes), idesc_s, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(tmem + kColDP, vdesc_k + kstep_off16(kk, kSubBytes), ob + kstep_off16(kk, kSubBytes), idesc_s, kk > 0);
        tc_commit(&sm.s_full);
        return true;
      };
      for (int slot_it = 0; ok; ++slot_it) {
        const int slot = slot_it % kBwdSlots;
        if (!mbar_wait(&sm.item_full[slot], (slot_it / kBwdSlots) & 1, abort_flag, p.status)) break;
        const int w = sm.items[slot];
        int4 im = make_int4(0, 0, 0, 0);
        if constexpr (KVB == 2) im = sm.imeta[slot];
        mbar_arrive(&sm.item_empty[slot]);
        if (w < 0) break;
        const int hh = w % kHalves;
        int n;
        if constexpr (KVB == 2) {
          n = im.z;
        } else {
          const int g = p.work[w / kHalves];
          n = p.csc_ptr[g + 1] - p.csc_ptr[g];
        }
        if (n == 0) continue;
        const int kb = item % KVB;
        if (!mbar_wait(&sm.kv_full[kb], (item / KVB) & 1, abort_flag, p.status)) break;
        kdesc_k = kdesc_k0 + static_cast<uint64_t>(kb * kKvBuf16);
        vdesc_k = vdesc_k0 + static_cast<uint64_t>(kb * kKvBuf16);
        kdesc_mn = kdesc_mn0 + static_cast<uint64_t>(kb * kKvBuf16);
        if (!issue_a(q_it, it)) break;
        for (int t = 0; t < n; ++t) {
          const int s = q_it % kQStages;
          const int db = kDsBufs == 1 ? 0 : (it & 1);
          // A(t+1) before B(t) when it can go early: the compute warps free
          // the S^T / dP^T columns (st_empty) early in their step, long
          // before dS^T(t) is ready (ds_full), so wait for that first (the
          // thread sleeps in the barrier), and issue A(t+1) if its Q / dO have
          // landed; if they have not, B(t) goes first and A(t+1) after it.
          bool a_next = (t + 1 >= n);
          if (!a_next) {
            if (!mbar_wait(&sm.st_empty, ((it + 1) & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
            if (mbar_test(&sm.q_full[(q_it + 1) % kQStages], ((q_it + 1) / kQStages) & 1)) {
              if (!issue_a(q_it + 1, it + 1)) { ok = false; break; }
              a_next = true;
            }
          }
          // B(t): dS^T(t) written, dK / dV accumulators free at an item's
          // first tile, the previous dQ read out of TMEM
          if (!mbar_wait(&sm.ds_full, it & 1, abort_flag, p.status) ||
              (t == 0 && !mbar_wait(&sm.dkv_empty, (item & 1) ^ 1, abort_flag, p.status)) ||
              !mbar_wait(&sm.dq_empty, (it & 1) ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t half16 = static_cast<uint64_t>(hh * (kSubBytes >> 4));
          const uint64_t qmn = qdesc_mn + static_cast<uint64_t>(s * kStage16) + half16;
          const uint64_t omn = odesc_mn + static_cast<uint64_t>(s * kStage16) + half16;
          const uint64_t kmn = kdesc_mn + half16;
          const uint64_t dsk = sdesc_k + static_cast<uint64_t>(db * kDsBuf16);
          const uint64_t dsm = sdesc_mn + static_cast<uint64_t>(db * kDsBuf16);
          const uint32_t acc0 = t > 0 ? 1u : 0u;
          // dV += P^T dO (A = P^T in TMEM, two bf16 per column along the queries)
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_bf16_ts(tmem + kColDV, tmem + kColPT + kk * 8, omn + static_cast<uint64_t>(kk * 128), idesc_kv,
                        kk > 0 ? 1u : acc0);
          tc_commit(&sm.pt_free);
          // dK += dS^T Q
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_bf16_ss(tmem + kColDK, dsk + kstep_off16(kk, kSubBytes), qmn + static_cast<uint64_t>(kk * 128),
                        idesc_kv, kk > 0 ? 1u : acc0);
          // dQ_i = dS K (A = dS^T viewed MN-major: queries contiguous, keys along rows)
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_bf16_ss(tmem + kColDQ, dsm + static_cast<uint64_t>(kk * 128), kmn + static_cast<uint64_t>(kk * 128),
                        idesc_q, kk > 0 ? 1u : 0u);
          tc_commit(&sm.dq_full);
          tc_commit(&sm.q_empty[s]);
          tc_commit(&sm.ds_free[db]);
          if (!a_next && !issue_a(q_it + 1, it + 1)) { ok = false; break; }
          ++q_it;
          ++it;
        }
        if (!ok) break;
        tc_commit(&sm.dkv_full);
        tc_commit(&sm.kv_empty[item % KVB]);
        ++item;
      }
      tc_commit(&sm.drain);
      mbar_wait_drain(&sm.drain, 0, p.status);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ P^T / dS^T warpgroups
    const int grp = (warp - 2) >> 2;       // 0: query columns 0-63, 1: 64-127
    const int quarter = warp & 3;
    const int kr = quarter * 32 + lane;    // key row = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    int it = 0, q_it = 0, item = 0;
    for (int slot_it = 0;; ++slot_it) {
      const int slot = slot_it % kBwdSlots;
      const bool got = mbar_wait(&sm.item_full[slot], (slot_it / kBwdSlots) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, got)) break;
      const int w = sm.items[slot];
      int4 im = make_int4(0, 0, 0, 0);
      if constexpr (KVB == 2) im = sm.imeta[slot];
      mbar_arrive(&sm.item_empty[slot]);
      if (w < 0) break;
      int g, start, n;
      if constexpr (KVB == 2) {
        g = im.x;
        start = im.y;
        n = im.z;
      } else {
        g = p.work[w / kHalves];
        start = p.csc_ptr[g];
        n = p.csc_ptr[g + 1] - start;
      }
      const int hh = w % kHalves;  // which 64-column half of D
      const int bh = g / p.nKt, j = g % p.nKt;
      const int key = j * kTile + kr;
      const bool kvalid = key < p.Tk;
      const long long gk = static_cast<long long>(bh) * p.Tk + key;
      // dK / dV row within the head (-1: not written)
      const long long gko = kvalid ? mapped_row(p.k_rows, gk, bh, p.To) : -1;
      if (n == 0) {
        if (gko >= 0) {
          uint4* a = reinterpret_cast<uint4*>((grp == 0 ? p.dv : p.dk) + gko * D + 64 * hh);
#pragma unroll
          for (int c = 0; c < 8; ++c) a[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      int ki, kh = 0;
      if (p.mode == SCFA_MODE_DENSE) ki = kvalid ? key : INT_MAX;
      else ki = kvalid ? p.k_idx[gk] : INT_MAX;
      if (p.mode == SCFA_MODE_HASH && kvalid) kh = p.k_hash[gk];
      bool ok = true;
      for (int t = 0; t < n; ++t) {
        const bool full = (cflags[start + t] & kFlagFull) != 0;
        const int s = q_it % kQStages;
        const int db = kDsBufs == 1 ? 0 : (it & 1);
        ok = mbar_wait(&sm.q_full[s], (q_it / kQStages) & 1, abort_flag, p.status) &&
             mbar_wait(&sm.s_full, it & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const float* lse2 = sm.lse2[s] + grp * 64;
        const float* drs = sm.drs[s] + grp * 64;
        const int* qid = sm.qidx[s] + grp * 64;
        const int* qhs = sm.qhash[s] + grp * 64;
        // one 32-query chunk: P^T and dS^T as packed bf16 pairs. The
        // arithmetic runs on packed f32 pairs (same operations and rounding
        // as the scalar form); tiles not flagged FULL then zero the pairs
        // that are not admissible.
        const uint64_t sl2 = f2(p.scale_log2, p.scale_log2), sc2 = f2(p.scale, p.scale);
        auto chunk = [&](int c, const uint32_t (&sr)[32], const uint32_t (&dr)[32], uint32_t (&pk)[16],
                         uint32_t (&dk16)[16]) {
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const int e = e4 * 4;
            const float4 l4 = *reinterpret_cast<const float4*>(lse2 + c * 32 + e);
            const float4 d4 = *reinterpret_cast<const float4*>(drs + c * 32 + e);
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
              const uint64_t nl = u == 0 ? f2(l4.x, l4.y) : f2(l4.z, l4.w);
              const uint64_t nd = u == 0 ? f2(d4.x, d4.y) : f2(d4.z, d4.w);
              float a0, a1;
              f2_split(fma2(f2(__uint_as_float(sr[e + u]), __uint_as_float(sr[e + u + 1])), sl2, nl), a0, a1);
              const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
              const uint64_t t = fma2(f2(__uint_as_float(dr[e + u]), __uint_as_float(dr[e + u + 1])), sc2, nd);
              float d0, d1;
              f2_split(mul2(f2(p0, p1), t), d0, d1);
              pk[e4 * 2 + u / 2] = pack_bf16x2(p0, p1);
              dk16[e4 * 2 + u / 2] = pack_bf16x2(d0, d1);
            }
          }
          if (!full) {
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
              const int e = e4 * 4;
              const int4 q4 = *reinterpret_cast<const int4*>(qid + c * 32 + e);
              bool adm[4] = {q4.x >= ki, q4.y >= ki, q4.z >= ki, q4.w >= ki};
              if (p.mode == SCFA_MODE_HASH) {
                const int4 h4 = *reinterpret_cast<const int4*>(qhs + c * 32 + e);
                adm[0] = adm[0] && h4.x == kh;
                adm[1] = adm[1] && h4.y == kh;
                adm[2] = adm[2] && h4.z == kh;
                adm[3] = adm[3] && h4.w == kh;
              }
#pragma unroll
              for (int u = 0; u < 4; u += 2) {
                const uint32_t keep = (adm[u] ? 0x0000ffffu : 0u) | (adm[u + 1] ? 0xffff0000u : 0u);
                pk[e4 * 2 + u / 2] &= keep;
                dk16[e4 * 2 + u / 2] &= keep;
              }
            }
          }
        };
        uint32_t pk[2][16], dsk[2][16];
        {
          uint32_t sr[32], dr[32];
          tmem_ld32(lane_base + kColS + grp * 64, sr);
          tmem_ld32(lane_base + kColDP + grp * 64, dr);
          tmem_wait_ld();
          tmem_ld_fence(sr);
          tmem_ld_fence(dr);
          chunk(0, sr, dr, pk[0], dsk[0]);
        }
        {
          uint32_t sr[32], dr[32];
          tmem_ld32(lane_base + kColS + grp * 64 + 32, sr);
          tmem_ld32(lane_base + kColDP + grp * 64 + 32, dr);
          tmem_wait_ld();
          tmem_ld_fence(sr);
          tmem_ld_fence(dr);
          tc_fence_before();
          mbar_arrive(&sm.st_empty);  // S^T / dP^T may now be overwritten by the next A
          chunk(1, sr, dr, pk[1], dsk[1]);
        }
        // the previous dV MMA must have read P^T, the MMAs kDsBufs tiles back dS^T[db]
        ok = mbar_wait(&sm.pt_free, (it & 1) ^ 1, abort_flag, p.status) &&
             mbar_wait(&sm.ds_free[db], (kDsBufs == 1 ? (it & 1) : ((it >> 1) & 1)) ^ 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        uint8_t* dsh = sm.dst[db][grp];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          // P^T (bf16 pairs) -> TMEM columns of this group's queries
          tmem_st16(lane_base + kColPT + grp * 32 + c * 16, pk[c]);
          // dS^T -> shared memory, 128-byte swizzle, K-major over queries
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(dsh + sw128_offset(kr, c * 4 + u)) =
                make_uint4(dsk[c][u * 4], dsk[c][u * 4 + 1], dsk[c][u * 4 + 2], dsk[c][u * 4 + 3]);
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&sm.ds_full);
        ++it;
        ++q_it;
      }
      if (!ok) break;
      // item epilogue: group 0 writes dV, group 1 writes dK
      ok = mbar_wait(&sm.dkv_full, item & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      uint32_t acc[2][32];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) tmem_ld32(lane_base + (grp == 0 ? kColDV : kColDK) + cc * 32, acc[cc]);
      tmem_wait_ld();
      tmem_ld_fence(acc[0]);
      tmem_ld_fence(acc[1]);
      tc_fence_before();
      mbar_arrive(&sm.dkv_empty);
      if (gko >= 0)
        store_row_bf16((grp == 0 ? p.dv : p.dk) + gko * D + 64 * hh, &acc[0][0], 64);
      ++item;
    }
  } else {
    // ------------------------------------------------------------ dQ warpgroup
    const int quarter = warp & 3;
    const int qr = quarter * 32 + lane;  // query row = TMEM lane
    const int tid = threadIdx.x - 320;   // 0..127
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    int it = 0, x_it = 0;
    // bounded sync of the dQ warpgroup (a broken pipeline ends in a status
    // code instead of a hang at a named barrier)
    auto dq_group_sync = [&]() -> bool {
      mbar_arrive(&sm.dq_sync);
      const bool r_ok = mbar_wait(&sm.dq_sync, x_it & 1, abort_flag, p.status);
      ++x_it;
      return __all_sync(0xffffffffu, r_ok);
    };
    for (int slot_it = 0;; ++slot_it) {
      const int slot = slot_it % kBwdSlots;
      const bool got = mbar_wait(&sm.item_full[slot], (slot_it / kBwdSlots) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, got)) break;
      const int w = sm.items[slot];
      int4 im = make_int4(0, 0, 0, 0);
      if constexpr (KVB == 2) im = sm.imeta[slot];
      mbar_arrive(&sm.item_empty[slot]);
      if (w < 0) break;
      int g, start, n;
      if constexpr (KVB == 2) {
        g = im.x;
        start = im.y;
        n = im.z;
      } else {
        g = p.work[w / kHalves];
        start = p.csc_ptr[g];
        n = p.csc_ptr[g + 1] - start;
      }
      const int hh = w % kHalves;  // which 64-column half of D
      if (n == 0) continue;
      const int bh = g / p.nKt;
      bool ok = true;
      for (int t = 0; t < n; ++t) {
        const int i = csc_rows[start + t];
        ok = mbar_wait(&sm.dq_full, it & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t qv[2][32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) tmem_ld32(lane_base + kColDQ + cc * 32, qv[cc]);
        tmem_wait_ld();
        tmem_ld_fence(qv[0]);
        tmem_ld_fence(qv[1]);
        tc_fence_before();
        mbar_arrive(&sm.dq_empty);
        // the two 32-column halves go through one 16 KB staging tile; the
        // previous reduce must have read it before it is rewritten
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (tid == 0) bulk_wait_group_read0();
          if (!dq_group_sync()) { ok = false; break; }
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(sm.dqs + sw128_offset(qr, c)) =
                make_uint4(qv[h][c * 4], qv[h][c * 4 + 1], qv[h][c * 4 + 2], qv[h][c * 4 + 3]);
          fence_proxy_async_smem();
          if (!dq_group_sync()) { ok = false; break; }
          if (tid == 0) {
            tma_reduce_add_3d(&tm_dq, sm.dqs, 64 * hh + h * 32, i * kTile, bh);
            bulk_commit_group();
          }
        }
        if (!ok) break;
        ++it;
      }
      if (!ok) break;
    }
    if (tid == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
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


// ---------------------------------------------------------------------------
// Head dimension 128, one work item per key tile (the whole of D). TMEM:
// S^T [0,128) with P^T overwriting its first 64 columns once both compute
// warpgroups have read S^T; dP^T [128,256) with dQ overwriting it once read;
// dV [256,384) and dK [384,512) accumulate over the key tile's query tiles.
// Per query tile the MMA warp issues S^T (once dV of the previous tile has
// read P^T) and dP^T (once the dQ warpgroup has read the previous dQ), then
// dV, dK, dQ. Q has two stages, so the next tile's Q is in place a whole step
// ahead; dO has one, refilled as soon as dV has read it (dV runs first). The
// producer loads each tile's row metadata before it waits for a stage. dQ
// leaves TMEM in two rounds of 64 columns through two 16 KB staging tiles and
// TMA reduce-adds; the staging tiles share their shared memory with dS^T (the
// next dS^T is written once the reduces have read the staged dQ).
// ---------------------------------------------------------------------------
struct __align__(1024) Bwd128Smem {
  uint8_t k[2][kSubBytes];
  uint8_t v[2][kSubBytes];
  uint8_t q[2][2][kSubBytes];  // [stage][64-column half of D]
  uint8_t dO[2][kSubBytes];
  uint8_t dsq[2][kSubBytes];   // dS^T [query half][128 keys x 64 queries] (bf16), then
                               // the dQ staging tiles [128 rows x 32 floats] (fp32)
  alignas(16) int32_t qidx[2][kTile];      // query metadata by step parity
  alignas(16) int32_t qhash[2][kTile];
  alignas(16) float lse2[2][kTile];        // -LSE * log2(e)
  alignas(16) float drs[2][kTile];         // -rowsum(dO * O) * scale
  uint64_t kv_full, kv_empty, q_full[2], q_empty[2], do_full, do_empty, s_full, loaded, ds_full;
  uint64_t dq_full, dq_empty, dqs_free, dkv_full, dkv_empty, drain, dq_sync;
  int32_t items[kBwdSlots];
  uint64_t item_full[kBwdSlots], item_empty[kBwdSlots];
  uint32_t tmem_base;
  int abort_flag;
};

__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  Bwd128Smem& sm = *reinterpret_cast<Bwd128Smem*>(smem_raw + pad);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // live-tile lists where the call that built them put them
  const int32_t* const csc_rows = ws_list<int32_t>(p.status, kListCscRows);
  const uint8_t* const cflags = ws_list<uint8_t>(p.status, kListCflags);
  constexpr uint32_t kColS = 0, kColPT = 0, kColDP = 128, kColDQ = 128, kColDV = 256, kColDK = 384;

  if (threadIdx.x == 0) {
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 1);
    }
    mbar_init(&sm.do_full, 1);
    mbar_init(&sm.do_empty, 1);
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.loaded, 256);
    mbar_init(&sm.ds_full, 256);
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_empty, 128);
    mbar_init(&sm.dqs_free, 1);
    mbar_init(&sm.dkv_full, 1);
    mbar_init(&sm.dkv_empty, 256);
    mbar_init(&sm.drain, 1);
    mbar_init(&sm.dq_sync, 128);
    for (int s = 0; s < kBwdSlots; ++s) {
      mbar_init(&sm.item_full[s], 1);
      mbar_init(&sm.item_empty[s], 1 + 256 + 128);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dq);
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer warp
    int qt = 0, item = 0, last_kv = -1;
    int q_issued = 0, do_issued = 0;  // loads issued, for the drain
    for (int slot_it = 0;; ++slot_it) {
      int w = INT_MAX;
      if (lane == 0) {
        const int slot = slot_it % kBwdSlots;
        if (mbar_wait(&sm.item_empty[slot], ((slot_it / kBwdSlots) & 1) ^ 1, abort_flag, p.status)) {
          w = atomicAdd(&p.sched[0], 1);
          sm.items[slot] = w < p.n_work ? w : -1;
          mbar_arrive(&sm.item_full[slot]);
        }
      }
      w = __shfl_sync(0xffffffffu, w, 0);
      if (w >= p.n_work) break;
      const int g = p.work[w];
      const int start = p.csc_ptr[g], n = p.csc_ptr[g + 1] - start;
      if (n == 0) continue;
      const int bh = g / p.nKt, j = g % p.nKt;
      bool ok = true;
      const bool stall = p.stall && item == 0;  // debug stall: K / V never arrive
      // the item's query tiles are read 32 at a time (one per lane); with
      // row gathers (p.gather_q, p.gather_kv) every lane issues four rows of each tile, the
      // source rows of a tile loaded a tile ahead, before the stage wait
      int cq = lane < n ? csc_rows[start + lane] : 0;
      int rr[4], rq[4] = {0, 0, 0, 0}, rn[4] = {0, 0, 0, 0};
      if (p.gather_kv) gather_rows(p.k_idx, bh, p.Tk, p.To, j * kTile, lane, rr);
      if (p.gather_q) gather_rows(p.q_idx, bh, p.Tq, p.To, __shfl_sync(0xffffffffu, cq, 0) * kTile, lane, rq);
      if (lane == 0 && !stall) {
        ok = mbar_wait(&sm.kv_empty, (item & 1) ^ 1, abort_flag, p.status);
        if (ok) {
          mbar_arrive_expect_tx(&sm.kv_full, 2 * D * kTile * 2);
          if (!p.gather_kv) {
            for (int sub = 0; sub < 2; ++sub) {
              tma_load_3d(sm.k[sub], &tm_k, &sm.kv_full, sub * 64, j * kTile, bh);
              tma_load_3d(sm.v[sub], &tm_v, &sm.kv_full, sub * 64, j * kTile, bh);
            }
          }
          last_kv = item;
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      if (p.gather_kv && !stall) {
        gather_issue(sm.k[0], kSubBytes, 2, &tm_k, &sm.kv_full, rr, lane);
        gather_issue(sm.v[0], kSubBytes, 2, &tm_v, &sm.kv_full, rr, lane);
      }
      const int n_steps = stall ? 1 : n;
      for (int t = 0; t < n_steps; ++t) {
        const int i = __shfl_sync(0xffffffffu, cq, t & 31);
        const int mb = qt & 1, s = qt & 1;
        if (t + 1 < n_steps) {
          if (((t + 1) & 31) == 0) cq = t + 1 + lane < n ? csc_rows[start + t + 1 + lane] : 0;
          if (p.gather_q)  // Q and dO rows of the next tile
            gather_rows(p.q_idx, bh, p.Tq, p.To, __shfl_sync(0xffffffffu, cq, (t + 1) & 31) * kTile, lane, rn);
        }
        if (lane == 0) {
          // Q into its stage once dK two tiles back has read it
          ok = mbar_wait(&sm.q_empty[s], ((qt >> 1) & 1) ^ 1, abort_flag, p.status);
          if (ok) {
            mbar_arrive_expect_tx(&sm.q_full[s], D * kTile * 2);
            if (!p.gather_q)
              for (int sub = 0; sub < 2; ++sub)
                tma_load_3d(sm.q[s][sub], &tm_q, &sm.q_full[s], sub * 64, i * kTile, bh);
            q_issued = qt + 1;
          }
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) { ok = false; break; }
        if (p.gather_q) gather_issue(sm.q[s][0], kSubBytes, 2, &tm_q, &sm.q_full[s], rq, lane);
        if (lane == 0) {
          // dO and the query metadata (four 512-byte rows of the padded
          // arrays, kept by step parity) once dV of the previous tile has
          // read dO
          ok = mbar_wait(&sm.do_empty, (qt & 1) ^ 1, abort_flag, p.status);
          if (ok) {
            mbar_arrive_expect_tx(&sm.do_full, D * kTile * 2 + 4 * kTile * 4);
            if (!p.gather_q)
              for (int sub = 0; sub < 2; ++sub) tma_load_3d(sm.dO[sub], &tm_do, &sm.do_full, sub * 64, i * kTile, bh);
            const float* m = p.qm + static_cast<long long>(bh) * p.Tqp + i * kTile;
            bulk_load(sm.lse2[mb], m, kTile * 4, &sm.do_full);
            bulk_load(sm.drs[mb], m + p.qm_n, kTile * 4, &sm.do_full);
            bulk_load(sm.qidx[mb], m + 2 * p.qm_n, kTile * 4, &sm.do_full);
            bulk_load(sm.qhash[mb], m + 3 * p.qm_n, kTile * 4, &sm.do_full);
            do_issued = qt + 1;
          }
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) { ok = false; break; }
        if (p.gather_q) {
          gather_issue(sm.dO[0], kSubBytes, 2, &tm_do, &sm.do_full, rq, lane);
#pragma unroll
          for (int u = 0; u < 4; ++u) rq[u] = rn[u];
        }
        ++qt;
      }
      if (!ok || stall) break;
      ++item;
    }
    if (lane == 0) {
      // no load may still be in flight when the CTA exits, also after an
      // abort (the counts are of loads actually issued)
      if (do_issued > 0) mbar_wait_drain(&sm.do_full, (do_issued - 1) & 1, p.status);
      for (int d = 1; d <= 2 && d <= q_issued; ++d) {
        const int it = q_issued - d;
        mbar_wait_drain(&sm.q_full[it & 1], (it >> 1) & 1, p.status);
      }
      if (last_kv >= 0) mbar_wait_drain(&sm.kv_full, last_kv & 1, p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kTile, kTile, 0, 0);
      constexpr uint32_t idesc_kv = idesc_bf16_f32(kTile, D, 0, 1);  // dV, dK: N = D, B MN-major
      constexpr uint32_t idesc_q = idesc_bf16_f32(kTile, D, 1, 1);   // dQ: A = dS (MN-major), B = K (MN-major)
      const uint64_t kdesc_k = smem_desc_sw128(smem_u32(sm.k[0]), 16, 1024);
      const uint64_t vdesc_k = smem_desc_sw128(smem_u32(sm.v[0]), 16, 1024);
      const uint64_t kdesc_mn = smem_desc_sw128(smem_u32(sm.k[0]), kSubBytes, 1024);
      const uint64_t qdesc_k = smem_desc_sw128(smem_u32(sm.q[0][0]), 16, 1024);
      const uint64_t qdesc_mn = smem_desc_sw128(smem_u32(sm.q[0][0]), kSubBytes, 1024);
      constexpr uint32_t kQStage16 = (2 * kSubBytes) >> 4;
      const uint64_t odesc_k = smem_desc_sw128(smem_u32(sm.dO[0]), 16, 1024);
      const uint64_t odesc_mn = smem_desc_sw128(smem_u32(sm.dO[0]), kSubBytes, 1024);
      const uint64_t sdesc_k = smem_desc_sw128(smem_u32(sm.dsq[0]), 16, 1024);
      const uint64_t sdesc_mn = smem_desc_sw128(smem_u32(sm.dsq[0]), kSubBytes, 1024);
      int it = 0, item = 0;
      bool ok = true;
      for (int slot_it = 0; ok; ++slot_it) {
        const int slot = slot_it % kBwdSlots;
        if (!mbar_wait(&sm.item_full[slot], (slot_it / kBwdSlots) & 1, abort_flag, p.status)) break;
        const int w = sm.items[slot];
        mbar_arrive(&sm.item_empty[slot]);
        if (w < 0) break;
        const int g = p.work[w];
        const int n = p.csc_ptr[g + 1] - p.csc_ptr[g];
        if (n == 0) continue;
        if (!mbar_wait(&sm.kv_full, item & 1, abort_flag, p.status)) break;
        for (int t = 0; t < n; ++t) {
          // S^T = K Q^T once dV of the previous tile has read P^T (the same
          // columns), then dP^T = V dO^T once dQ of the previous tile is out
          // of TMEM
          const int s = it & 1;
          const uint64_t qs16 = static_cast<uint64_t>(s * kQStage16);
          if (!mbar_wait(&sm.q_full[s], (it >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
          if (it > 0 && !mbar_wait(&sm.do_empty, (it - 1) & 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_ss(tmem + kColS, kdesc_k + kstep_off16(kk, kSubBytes),
                        qdesc_k + qs16 + kstep_off16(kk, kSubBytes), idesc_s, kk > 0);
          if (!mbar_wait(&sm.do_full, it & 1, abort_flag, p.status)) { ok = false; break; }
          if (it > 0 && !mbar_wait(&sm.dq_empty, (it - 1) & 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_ss(tmem + kColDP, vdesc_k + kstep_off16(kk, kSubBytes), odesc_k + kstep_off16(kk, kSubBytes),
                        idesc_s, kk > 0);
          tc_commit(&sm.s_full);
          // P^T in TMEM and dS^T in shared memory from the compute warps
          if (!mbar_wait(&sm.ds_full, it & 1, abort_flag, p.status)) { ok = false; break; }
          if (t == 0 && !mbar_wait(&sm.dkv_empty, (item & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t acc0 = t > 0 ? 1u : 0u;
          // dV += P^T dO (A = P^T in TMEM)
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_bf16_ts(tmem + kColDV, tmem + kColPT + kk * 8, odesc_mn + static_cast<uint64_t>(kk * 128), idesc_kv,
                        kk > 0 ? 1u : acc0);
          tc_commit(&sm.do_empty);
          // dK += dS^T Q
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_bf16_ss(tmem + kColDK, sdesc_k + kstep_off16(kk, kSubBytes),
                        qdesc_mn + qs16 + static_cast<uint64_t>(kk * 128), idesc_kv, kk > 0 ? 1u : acc0);
          tc_commit(&sm.q_empty[s]);
          // dQ_i = dS K into the dP^T columns (read by now)
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_bf16_ss(tmem + kColDQ, sdesc_mn + static_cast<uint64_t>(kk * 128),
                        kdesc_mn + static_cast<uint64_t>(kk * 128), idesc_q, kk > 0 ? 1u : 0u);
          tc_commit(&sm.dq_full);
          ++it;
        }
        if (!ok) break;
        tc_commit(&sm.dkv_full);
        tc_commit(&sm.kv_empty);
        ++item;
      }
      tc_commit(&sm.drain);
      mbar_wait_drain(&sm.drain, 0, p.status);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ P^T / dS^T warpgroups
    const int grp = (warp - 2) >> 2;       // 0: query columns 0-63, 1: 64-127
    const int quarter = warp & 3;
    const int kr = quarter * 32 + lane;    // key row = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    int it = 0, item = 0;
    for (int slot_it = 0;; ++slot_it) {
      const int slot = slot_it % kBwdSlots;
      const bool got = mbar_wait(&sm.item_full[slot], (slot_it / kBwdSlots) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, got)) break;
      const int w = sm.items[slot];
      mbar_arrive(&sm.item_empty[slot]);
      if (w < 0) break;
      const int g = p.work[w];
      const int start = p.csc_ptr[g], n = p.csc_ptr[g + 1] - start;
      const int bh = g / p.nKt, j = g % p.nKt;
      const int key = j * kTile + kr;
      const bool kvalid = key < p.Tk;
      const long long gk = static_cast<long long>(bh) * p.Tk + key;
      const long long gko = kvalid ? mapped_row(p.k_rows, gk, bh, p.To) : -1;  // dK / dV row
      if (n == 0) {
        if (gko >= 0) {
          uint4* a = reinterpret_cast<uint4*>((grp == 0 ? p.dv : p.dk) + gko * D);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) a[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      int ki, kh = 0;
      if (p.mode == SCFA_MODE_DENSE) ki = kvalid ? key : INT_MAX;
      else ki = kvalid ? p.k_idx[gk] : INT_MAX;
      if (p.mode == SCFA_MODE_HASH && kvalid) kh = p.k_hash[gk];
      bool ok = true;
      for (int t = 0; t < n; ++t) {
        const bool full = (cflags[start + t] & kFlagFull) != 0;
        const int mb = it & 1;
        ok = mbar_wait(&sm.do_full, it & 1, abort_flag, p.status) &&
             mbar_wait(&sm.s_full, it & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const float* lse2 = sm.lse2[mb] + grp * 64;
        const float* drs = sm.drs[mb] + grp * 64;
        const int* qid = sm.qidx[mb] + grp * 64;
        const int* qhs = sm.qhash[mb] + grp * 64;
        const uint64_t sl2 = f2(p.scale_log2, p.scale_log2), sc2 = f2(p.scale, p.scale);
        auto chunk = [&](int c, const uint32_t (&sr)[32], const uint32_t (&dr)[32], uint32_t (&pk)[16],
                         uint32_t (&dk16)[16]) {
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const int e = e4 * 4;
            const float4 l4 = *reinterpret_cast<const float4*>(lse2 + c * 32 + e);
            const float4 d4 = *reinterpret_cast<const float4*>(drs + c * 32 + e);
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
              const uint64_t nl = u == 0 ? f2(l4.x, l4.y) : f2(l4.z, l4.w);
              const uint64_t nd = u == 0 ? f2(d4.x, d4.y) : f2(d4.z, d4.w);
              float a0, a1;
              f2_split(fma2(f2(__uint_as_float(sr[e + u]), __uint_as_float(sr[e + u + 1])), sl2, nl), a0, a1);
              const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
              const uint64_t tt = fma2(f2(__uint_as_float(dr[e + u]), __uint_as_float(dr[e + u + 1])), sc2, nd);
              float d0, d1;
              f2_split(mul2(f2(p0, p1), tt), d0, d1);
              pk[e4 * 2 + u / 2] = pack_bf16x2(p0, p1);
              dk16[e4 * 2 + u / 2] = pack_bf16x2(d0, d1);
            }
          }
          if (!full) {
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
              const int e = e4 * 4;
              const int4 q4 = *reinterpret_cast<const int4*>(qid + c * 32 + e);
              bool adm[4] = {q4.x >= ki, q4.y >= ki, q4.z >= ki, q4.w >= ki};
              if (p.mode == SCFA_MODE_HASH) {
                const int4 h4 = *reinterpret_cast<const int4*>(qhs + c * 32 + e);
                adm[0] = adm[0] && h4.x == kh;
                adm[1] = adm[1] && h4.y == kh;
                adm[2] = adm[2] && h4.z == kh;
                adm[3] = adm[3] && h4.w == kh;
              }
#pragma unroll
              for (int u = 0; u < 4; u += 2) {
                const uint32_t keep = (adm[u] ? 0x0000ffffu : 0u) | (adm[u + 1] ? 0xffff0000u : 0u);
                pk[e4 * 2 + u / 2] &= keep;
                dk16[e4 * 2 + u / 2] &= keep;
              }
            }
          }
        };
        uint32_t pk[2][16], dsk[2][16];
        {
          uint32_t sr[32], dr[32];
          tmem_ld32(lane_base + kColS + grp * 64, sr);
          tmem_ld32(lane_base + kColDP + grp * 64, dr);
          tmem_wait_ld();
          tmem_ld_fence(sr);
          tmem_ld_fence(dr);
          chunk(0, sr, dr, pk[0], dsk[0]);
        }
        {
          uint32_t sr[32], dr[32];
          tmem_ld32(lane_base + kColS + grp * 64 + 32, sr);
          tmem_ld32(lane_base + kColDP + grp * 64 + 32, dr);
          tmem_wait_ld();
          tmem_ld_fence(sr);
          tmem_ld_fence(dr);
          tc_fence_before();
          mbar_arrive(&sm.loaded);  // this thread's S^T / dP^T columns are in registers
          chunk(1, sr, dr, pk[1], dsk[1]);
        }
        // P^T overwrites S^T columns 0-63: both warpgroups must have read them
        ok = mbar_wait(&sm.loaded, it & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) tmem_st16(lane_base + kColPT + grp * 32 + c * 16, pk[c]);
        // dS^T replaces the previous tile's staged dQ once its reduces have read it
        ok = mbar_wait(&sm.dqs_free, (it & 1) ^ 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        uint8_t* dsh = sm.dsq[grp];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(dsh + sw128_offset(kr, c * 4 + u)) =
                make_uint4(dsk[c][u * 4], dsk[c][u * 4 + 1], dsk[c][u * 4 + 2], dsk[c][u * 4 + 3]);
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&sm.ds_full);
        ++it;
      }
      if (!ok) break;
      // item epilogue: group 0 writes dV, group 1 writes dK, 64 columns at a time
      ok = mbar_wait(&sm.dkv_full, item & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t col = grp == 0 ? kColDV : kColDK;
      uint16_t* orow = (grp == 0 ? p.dv : p.dk) + (gko >= 0 ? gko : 0) * D;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t acc[2][32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) tmem_ld32(lane_base + col + hf * 64 + cc * 32, acc[cc]);
        tmem_wait_ld();
        tmem_ld_fence(acc[0]);
        tmem_ld_fence(acc[1]);
        if (hf == 1) {
          tc_fence_before();
          mbar_arrive(&sm.dkv_empty);
        }
        if (gko >= 0) store_row_bf16(orow + 64 * hf, &acc[0][0], 64);
      }
      ++item;
    }
  } else {
    // ------------------------------------------------------------ dQ warpgroup
    const int quarter = warp & 3;
    const int qr = quarter * 32 + lane;  // query row = TMEM lane
    const int tid = threadIdx.x - 320;   // 0..127
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    int it = 0, x_it = 0;
    auto dq_group_sync = [&]() -> bool {
      mbar_arrive(&sm.dq_sync);
      const bool r_ok = mbar_wait(&sm.dq_sync, x_it & 1, abort_flag, p.status);
      ++x_it;
      return __all_sync(0xffffffffu, r_ok);
    };
    for (int slot_it = 0;; ++slot_it) {
      const int slot = slot_it % kBwdSlots;
      const bool got = mbar_wait(&sm.item_full[slot], (slot_it / kBwdSlots) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, got)) break;
      const int w = sm.items[slot];
      mbar_arrive(&sm.item_empty[slot]);
      if (w < 0) break;
      const int g = p.work[w];
      const int start = p.csc_ptr[g], n = p.csc_ptr[g + 1] - start;
      if (n == 0) continue;
      const int bh = g / p.nKt;
      bool ok = true;
      for (int t = 0; t < n; ++t) {
        const int i = csc_rows[start + t];
        ok = mbar_wait(&sm.dq_full, it & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        // two rounds of 64 columns; the second round's loads free the TMEM
#pragma unroll
        for (int rd = 0; rd < 2; ++rd) {
          uint32_t qv[2][32];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) tmem_ld32(lane_base + kColDQ + rd * 64 + cc * 32, qv[cc]);
          tmem_wait_ld();
          tmem_ld_fence(qv[0]);
          tmem_ld_fence(qv[1]);
          if (rd == 1) {
            tc_fence_before();
            mbar_arrive(&sm.dq_empty);
          }
          // the staging tiles are free once the first round's reduces have read them
          if (tid == 0) bulk_wait_group_read0();
          if (!dq_group_sync()) { ok = false; break; }
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(&sm.dsq[h][0] + sw128_offset(qr, c)) =
                  make_uint4(qv[h][c * 4], qv[h][c * 4 + 1], qv[h][c * 4 + 2], qv[h][c * 4 + 3]);
          fence_proxy_async_smem();
          if (!dq_group_sync()) { ok = false; break; }
          if (tid == 0) {
            tma_reduce_add_3d(&tm_dq, &sm.dsq[0][0], rd * 64, i * kTile, bh);
            tma_reduce_add_3d(&tm_dq, &sm.dsq[1][0], rd * 64 + 32, i * kTile, bh);
            bulk_commit_group();
          }
        }
        if (!ok) break;
        // the staging tiles go back to dS^T once the reduces have read them
        if (tid == 0) {
          bulk_wait_group_read0();
          mbar_arrive(&sm.dqs_free);
        }
        ++it;
      }
      if (!ok) break;
    }
    if (tid == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&p.sched[1], 1) == static_cast<int>(gridDim.x) - 1) {
      atomicExch(&p.sched[0], 0);
      atomicExch(&p.sched[1], 0);
    }
  }
}

// Per query row: Drow = sum_d dO * O (fp32) and dq_acc[row] = 0, and the
// metadata that the backward's producer copies next to each Q / dO tile,
// written into four arrays padded to whole tiles of 128 rows (Tqp rows per
// head): -LSE * log2(e), -Drow * scale, the position (the row itself in dense
// mode) and the bucket id. Padding rows get position INT_MIN (never
// admissible) and zeros. D/8 lanes per row (one 16-byte chunk each),
// 32 / (D/8) rows per warp step; the loop is warp-uniform so the shuffle
// reduction always has the whole warp.
// With o32 (the forward's fp32 copy of O, kept in the dQ accumulator's place)
// the sum is taken from it instead of the bf16 o: the bf16 store of O is the
// largest error term of dS otherwise. Each lane reads its chunk of o32 before
// zeroing it.
struct PreParams {
  const uint16_t* o;
  const uint16_t* dO;
  const float* o32;
  const int32_t* o_rows;
  const int32_t* do_rows;  // null, or the original row of each sorted row of dO (row gathers)
  int To;             // rows per head of o (and dO) when o_rows (do_rows) is set
  const float* lse;
  const int32_t* q_idx;
  const int32_t* q_hash;
  float* dq_acc;
  float* qm;          // four arrays of n_pad entries
  long long n_pad;    // B*H*Tqp
  int Tq, Tqp, mode;
  float scale;
};

template <int D>
__global__ void bwd_pre_kernel(const PreParams p) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const int lane = threadIdx.x & 31;
  const long long warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long wg = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       wg * kRowsPerWarp < p.n_pad; wg += warps) {
    const long long rp = wg * kRowsPerWarp + lane / kLanesPerRow;  // padded row
    const int ch = lane % kLanesPerRow;
    const long long bh = rp / p.Tqp;
    const int r = static_cast<int>(rp - bh * p.Tqp);
    const bool inside = rp < p.n_pad;
    const long long row = bh * p.Tq + r;
    // with original-order outputs a sorted row whose index falls outside
    // [0, To) (a padding row) has no output: no dO / O reads and no dQ reset
    // for it, and metadata that masks it (position INT_MIN)
    const bool active = inside && r < p.Tq && (p.o_rows == nullptr || mapped_row(p.o_rows, row, bh, p.To) >= 0);
    float s = 0.f;
    if (active) {
      const long long drow = mapped_row(p.do_rows, row, bh, p.To);
      const uint4 b = drow >= 0 ? reinterpret_cast<const uint4*>(p.dO + drow * D)[ch] : make_uint4(0, 0, 0, 0);
      const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
      if (p.o32 != nullptr) {
        const float4 a0 = reinterpret_cast<const float4*>(p.o32 + row * D)[ch * 2];
        const float4 a1 = reinterpret_cast<const float4*>(p.o32 + row * D)[ch * 2 + 1];
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          s = fmaf(av[2 * u], __uint_as_float(bw[u] << 16), s);
          s = fmaf(av[2 * u + 1], __uint_as_float(bw[u] & 0xFFFF0000u), s);
        }
      } else {
        // O may be stored in original row order (o_rows maps sorted -> original)
        const long long orow = mapped_row(p.o_rows, row, bh, p.To);
        const uint4 a = orow >= 0 ? reinterpret_cast<const uint4*>(p.o + orow * D)[ch] : make_uint4(0, 0, 0, 0);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          s = fmaf(__uint_as_float(aw[u] << 16), __uint_as_float(bw[u] << 16), s);
          s = fmaf(__uint_as_float(aw[u] & 0xFFFF0000u), __uint_as_float(bw[u] & 0xFFFF0000u), s);
        }
      }
    }
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (inside && ch == 0) {
      float* m = p.qm + rp;
      int32_t* mi = reinterpret_cast<int32_t*>(p.qm) + rp;
      if (active) {
        m[0] = -(p.lse[row] * kLog2e);
        m[p.n_pad] = -(s * p.scale);
        mi[2 * p.n_pad] = p.mode == SCFA_MODE_DENSE ? r : p.q_idx[row];
        mi[3 * p.n_pad] = p.mode == SCFA_MODE_HASH ? p.q_hash[row] : 0;
      } else {
        m[0] = 0.f;
        m[p.n_pad] = 0.f;
        mi[2 * p.n_pad] = INT_MIN;
        mi[3 * p.n_pad] = 0;
      }
    }
    if (active) {
      float4* z = reinterpret_cast<float4*>(p.dq_acc + row * D) + ch * 2;
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

__global__ void dq_finalize_kernel(const float* __restrict__ dq_acc, long long n8, uint16_t* __restrict__ dq,
                                   const int32_t* __restrict__ q_rows, int T, int To, int chunks) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < n8; t += stride) {
    // dQ may be stored in original row order (q_rows maps sorted -> original)
    long long out = t;
    if (q_rows != nullptr) {
      const long long row = t / chunks;
      const long long orow = mapped_row(q_rows, row, row / T, To);
      if (orow < 0) continue;
      out = orow * chunks + (t - row * chunks);
    }
    const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * t];
    const float4 b = reinterpret_cast<const float4*>(dq_acc)[2 * t + 1];
    uint4 u;
    u.x = pack_bf16x2(a.x, a.y);
    u.y = pack_bf16x2(a.z, a.w);
    u.z = pack_bf16x2(b.x, b.y);
    u.w = pack_bf16x2(b.z, b.w);
    reinterpret_cast<uint4*>(dq)[out] = u;
  }
}

}  // namespace

bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, int D, long long T, long long BH);
bool make_tmap_f32_3d(CUtensorMap* map, void* base, int D, long long T, long long BH);

template <int D>
static cudaError_t launch_bwd_d(const AttnArgs& a, cudaStream_t st) {
  const AttnWs& L = *a.L;
  const long long BH = static_cast<long long>(a.B) * a.H;
  const int sms = num_sms();
  float* dq_acc = reinterpret_cast<float*>(a.ws + L.dq_acc);
  float* qm = reinterpret_cast<float*>(a.ws + L.qmeta);
  const int Tqp = L.nQt * kTile;
  const long long qrows = BH * a.Tq;
  const long long n_pad = BH * Tqp;
  {
    PreParams pp;
    pp.o = a.o;
    pp.dO = a.do_;
    pp.o32 = a.o32;
    pp.o_rows = a.q_rows;
    pp.do_rows = a.gather_q ? a.q_idx : nullptr;
    pp.To = a.To;
    pp.lse = a.lse_in;
    pp.q_idx = a.q_idx;
    pp.q_hash = a.q_hash;
    pp.dq_acc = dq_acc;
    pp.qm = qm;
    pp.n_pad = n_pad;
    pp.Tq = a.Tq;
    pp.Tqp = Tqp;
    pp.mode = a.mode;
    pp.scale = a.scale;
    const long long work = (n_pad * (D / 8) + 31) / 32 * 32;
    long long g = (work + 255) / 256;
    if (g > sms * 16LL) g = sms * 16LL;
    if (g < 1) g = 1;
    bwd_pre_kernel<D><<<static_cast<int>(g), 256, 0, st>>>(pp);
  }
  CUtensorMap tq, tk, tv, tdo, tdq;
  // tiled maps over the sorted q, k, v, dO, or row-gather maps over the
  // original-order ones
  const bool maps_ok =
      (a.gather_q ? (make_tmap_bf16_rows(&tq, a.q, D, BH * a.To) && make_tmap_bf16_rows(&tdo, a.do_, D, BH * a.To))
                  : (make_tmap_bf16_3d(&tq, a.q, D, a.Tq, BH) && make_tmap_bf16_3d(&tdo, a.do_, D, a.Tq, BH))) &&
      (a.gather_kv ? (make_tmap_bf16_rows(&tk, a.k, D, BH * a.To) && make_tmap_bf16_rows(&tv, a.v, D, BH * a.To))
                   : (make_tmap_bf16_3d(&tk, a.k, D, a.Tk, BH) && make_tmap_bf16_3d(&tv, a.v, D, a.Tk, BH)));
  if (!maps_ok || !make_tmap_f32_3d(&tdq, dq_acc, D, a.Tq, BH)) return cudaErrorInvalidValue;
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
  p.qm = qm;
  p.qm_n = n_pad;
  p.Tqp = Tqp;
  p.csc_ptr = reinterpret_cast<const int32_t*>(a.ws + L.csc_ptr);
  p.work = reinterpret_cast<const int32_t*>(a.ws + L.work_bwd);
  p.n_work = static_cast<int>(L.n_ktiles);  // one work item per key tile
  p.dk = a.dk;
  p.dv = a.dv;
  p.k_rows = a.k_rows;
  p.To = a.To;
  p.stall = a.stall;
  p.gather_q = a.gather_q;
  p.gather_kv = a.gather_kv;
  p.status = reinterpret_cast<int*>(a.ws + L.header);
  p.sched = reinterpret_cast<WsHeader*>(a.ws + L.header)->sched + 2;
  int grid = sms;
  if (grid > p.n_work) grid = p.n_work;
  if (grid < 1) grid = 1;
  if constexpr (D == 128) {
    const size_t smem = sizeof(Bwd128Smem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(attn_bwd128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    record_kernel_event(1, true, st);
    attn_bwd128_kernel<<<grid, kBwdThreads, smem, st>>>(tq, tk, tv, tdo, tdq, p);
    record_kernel_event(1, false, st);
  } else {
    // hash mode: about three query tiles per key tile, so a second K / V
    // buffer (loaded while the previous item runs) is worth the second dS^T
    // buffer; the long columns of the other modes keep that one
    static_assert(sizeof(BwdSmem<D, 2>) + 1024 <= 227 * 1024 && sizeof(BwdSmem<D, 1>) + 1024 <= 227 * 1024,
                  "shared memory per CTA");
    const bool two_kv = a.mode == SCFA_MODE_HASH;
    const size_t smem = (two_kv ? sizeof(BwdSmem<D, 2>) : sizeof(BwdSmem<D, 1>)) + 1024;
    auto kern = two_kv ? attn_bwd_kernel<D, 2> : attn_bwd_kernel<D, 1>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    record_kernel_event(1, true, st);
    kern<<<grid, kBwdThreads, smem, st>>>(tq, tk, tv, tdo, tdq, p);
    record_kernel_event(1, false, st);
  }
  {
    const long long n8 = qrows * D / 8;
    long long g = (n8 + 255) / 256;
    if (g > sms * 16LL) g = sms * 16LL;
    if (g < 1) g = 1;
    dq_finalize_kernel<<<static_cast<int>(g), 256, 0, st>>>(dq_acc, n8, a.dq, a.q_rows, a.Tq, a.To, D / 8);
  }
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const AttnArgs& a, cudaStream_t st) {
  if (a.D == 64) return launch_bwd_d<64>(a, st);
  if (a.D == 128) return launch_bwd_d<128>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace scfa
