// Shared device helpers for the SCFA kernels: inline PTX for mbarriers, TMA,
// tcgen05 (TMEM allocation, MMA, loads/stores), fences, and the bounded wait
// that turns a stuck pipeline into a status code instead of a hang.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/scfa.h"

namespace scfa {

constexpr int kTile = SCFA_TILE;       // 128 rows per query tile and per key tile
constexpr uint32_t kFlagFull = 1u;     // tile flag bit: every pair admissible

// Workspace header (first 256 bytes of every attention / sort workspace).
struct WsHeader {
  int status;       // SCFA_OK or the first device-side error
  int n_live;       // total live tiles (written by the tile pass)
  // work counters of the dynamically scheduled kernels: [0] next forward
  // item, [1] forward CTAs done, [2] next backward item, [3] backward CTAs
  // done; zeroed with the header by the tile pass and again by the last CTA
  // of each launch
  int sched[4];
  // where the call that built the live-tile lists put them (byte offsets from
  // the workspace start: cols, csc_rows, fflags, cflags, pair lists) and how
  // many entries each holds; calls that reuse the lists read them from here
  long long list_off[5];
  long long list_cap;
  int pad[46];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");
enum { kListCols = 0, kListCscRows = 1, kListFflags = 2, kListCflags = 3, kListPairs = 4 };
template <typename T>
__device__ __forceinline__ const T* ws_list(const int* status, int which) {
  const WsHeader* h = reinterpret_cast<const WsHeader*>(status);
  return reinterpret_cast<const T*>(reinterpret_cast<const char*>(h) + h->list_off[which]);
}

// ---------------------------------------------------------------------------
// Generic helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void raise_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// maximum of three. Written as two fmaxf so that the compiler picks the
// instruction: a hand-written three-input max.f32 on scores fresh from a TMEM
// load returned stale values in the softmax loop (a row whose every key was
// masked got a tiny denormal instead of -inf as its tile maximum), which made
// the low bits of O and LSE depend on the launch.
__device__ __forceinline__ float max3f(float a, float b, float c) { return fmaxf(fmaxf(a, b), c); }

// packed pairs of f32: one instruction does two lanes' worth of FMA / add / mul
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
  return v;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Work item of round r for this CTA of a persistent grid walking a list sorted
// by size, largest first: rounds alternate direction (CTA b takes item b of
// round 0, item G - 1 - b of round 1, ...), so no CTA gets the largest item
// of every round. Every role of a CTA calls it with the same r sequence.
__device__ __forceinline__ int work_item(int r) {
  const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  return r * G + ((r & 1) ? (G - 1 - b) : b);
}

// Output row of the row `grow` of head `bh` of a sorted tensor: grow itself
// without a row map, else row rows[grow] of that head in an original-order
// tensor of To rows per head; -1 when the map points outside [0, To) (such
// rows are neither written nor read).
__device__ __forceinline__ long long mapped_row(const int32_t* rows, long long grow, long long bh, int To) {
  if (rows == nullptr) return grow;
  const int t = rows[grow];
  return (t >= 0 && t < To) ? bh * To + t : -1;
}

// named barrier among `count` threads (ids 1..15; 0 is __syncthreads)
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may sleep until the phase completes (up to
// about `hint_ns`) instead of returning at once, so a waiting warp takes no
// issue slots from the warps that share its scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns) : "memory");
  return ok != 0;
}

// non-blocking test of phase `parity`
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Wall-clock limit of one pipeline wait. Every stage of every kernel finishes
// in microseconds, so a wait this long means the pipeline is broken.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s
// longest sleep of one try inside a wait; the abort flag and the limit are
// checked between tries
constexpr uint32_t kWaitSleepNs = 20000u;  // 20 us

// Bounded wait on phase `parity` of `bar`. Returns false if the CTA abort
// flag is raised or the time limit passes (then it raises the status word
// and the abort flag so that every role of the CTA leaves its loop).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      raise_status(status, SCFA_ERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

// Wait used when a role leaves: for copies and MMAs this thread has already
// issued, which complete on their own. It ignores the abort flag (so a CTA
// that is aborting still lets its in-flight TMA loads land and its MMAs
// finish before it releases shared memory and TMEM) and is bounded by the
// same limit.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      raise_status(status, SCFA_ERR_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA (tensor copies, global -> shared), completion counted on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      :: "r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)),
         "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// four rows of a 2-D map whose box is one row high (tile::gather4): rows
// r0..r3, columns x .. x + box width, landing as consecutive box rows at
// smem_dst with the map's swizzle (the same bytes a tiled load of those rows
// would write there)
__device__ __forceinline__ void tma_gather4(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int r0,
                                            int r1, int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
      :: "r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2),
         "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

// Row gathers of one 128-row tile by a whole warp, from an original-order
// tensor (a 2-D map over its BH * To rows, 64-column boxes one row high):
// sorted slot row0 + r of head bh is row idx[bh * Ts + row0 + r] of that
// head. A slot at or past Ts, or whose index falls outside [0, To), is a
// padding row and reads the head's first row instead (every score against a
// padding row is masked, so its values only ever meet exact zeros).
// gather_rows: lane l's four source rows 4l .. 4l + 3 (loaded ahead of the
// stage wait); gather_issue: lane l's gathers into each 64-column sub-tile
// (sub-tiles sub_bytes apart), completing on `bar`, whose expected byte
// count the caller has set.
__device__ __forceinline__ void gather_rows(const int32_t* __restrict__ idx, long long bh, int Ts, int To, int row0,
                                            int lane, int (&rr)[4]) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int slot = row0 + 4 * lane + u;
    int src = slot < Ts ? __ldg(idx + bh * Ts + slot) : -1;
    if (src < 0 || src >= To) src = 0;
    rr[u] = static_cast<int>(bh * To + src);
  }
}
__device__ __forceinline__ void gather_issue(uint8_t* dst, uint32_t sub_bytes, int n_sub, const CUtensorMap* map,
                                             uint64_t* bar, const int (&rr)[4], int lane) {
  for (int sub = 0; sub < n_sub; ++sub)
    tma_gather4(dst + sub * sub_bytes + 512 * lane, map, bar, sub * 64, rr[0], rr[1], rr[2], rr[3]);
}

// untiled bulk copy global -> shared of `bytes` bytes (both addresses 16-byte
// aligned, bytes a multiple of 16), completion counted on `bar`
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// element-wise add of a shared-memory tile into a global tensor (TMA reduce),
// tracked by the issuing thread's bulk async-group
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* smem_src, int x, int y, int z) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3}], [%4];"
      :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(smem_src)) : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until every committed bulk group has finished READING its shared-memory source
__device__ __forceinline__ void bulk_wait_group_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// wait until every committed bulk group has completed
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// generic-proxy shared-memory writes -> visible to the async proxy (MMA/TMA)
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, loads / stores
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(smem_u32(slot_smem)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive on `bar` once every tcgen05 async operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(smem_u32(bar)) : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T: A (M x K, K-major) read from tensor memory,
// two bf16 per 32-bit column along K
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (16-byte units), fixed version bits 46-48 = 0b001,
// swizzle mode 2 (128-byte swizzle) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Byte offset of 16-element K step kk inside a K-major tile made of
// [128 rows][64 bf16] swizzled sub-tiles, in descriptor units (16 bytes):
// added to a descriptor it moves the start address (bits 0-13) only, since
// every shared-memory address is below 256 KB.
__host__ __device__ constexpr uint64_t kstep_off16(int kk, int sub_bytes) {
  return static_cast<uint64_t>(((kk >> 2) * sub_bytes + (kk & 3) * 32) >> 4);
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D.
// a_mn / b_mn: operand is MN-major (1) instead of K-major (0).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                                   // D format: f32
       | (1u << 7)                                   // A format: bf16
       | (1u << 10)                                  // B format: bf16
       | (static_cast<uint32_t>(a_mn) << 15)
       | (static_cast<uint32_t>(b_mn) << 16)
       | (static_cast<uint32_t>(N >> 3) << 17)
       | (static_cast<uint32_t>(M >> 4) << 24);
}

// 32 lanes x 32 bits, 32 consecutive columns -> 32 registers per thread
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 32 lanes x 32 bits, 16 consecutive columns -> 16 registers per thread
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      :: "r"(taddr),
         "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
         "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
         "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
         "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// 32 lanes x 32 bits, 16 consecutive columns <- 16 registers per thread
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      :: "r"(taddr),
         "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
         "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// tcgen05.ld fills its destination registers asynchronously, but to the
// compiler they are defined when the load issues: register-only arithmetic on
// them (a max, an FMA) may be scheduled above tcgen05.wait::ld and then reads
// values the load has not written yet. After each wait, pass every register
// loaded since the previous wait through this empty volatile asm: it comes
// after the wait (volatile asm keeps its order) and redefines the registers,
// so every use of them follows it.
template <int N>
__device__ __forceinline__ void tmem_ld_fence(uint32_t (&r)[N]) {
  static_assert(N % 8 == 0, "fence registers in groups of 8");
#pragma unroll
  for (int i = 0; i < N; i += 8)
    asm volatile("" : "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), "+r"(r[i + 5]),
                 "+r"(r[i + 6]), "+r"(r[i + 7]));
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Offset of element (row, col) of a [rows][64] bf16 tile stored with the
// 128-byte swizzle (16-byte chunk index XOR row % 8), as TMA writes it and as
// the MMA descriptors above read it.
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk16) {
  return static_cast<uint32_t>(row * 128 + ((chunk16 ^ (row & 7)) << 4));
}

}  // namespace scfa
