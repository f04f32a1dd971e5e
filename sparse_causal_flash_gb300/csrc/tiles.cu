// Tile metadata and the live-tile work list.
//
// Page: "Faster Causal Attention Over Large Sequences Through Sparse Flash
// Attention" (deep-paper.org), section "SCFA 解决方案": tile pruning by
// max(q_idx_i) < min(k_idx_j) (part 1), bucket and causal pruning (part 2).
// Tiles are 128 x 128. Per tile the pass records min / max of the original
// positions and of the bucket ids over its valid rows, tests every candidate
// (query tile, key tile) pair, and emits CSR (by query tile), CSC (by key
// tile), a FULL flag per entry (all 128 x 128 pairs admissible: no element
// mask needed), and the work orders that the persistent attention kernels
// walk: tile ids by live count descending, then id ascending, except that the
// key-tile list keeps its natural order when its total work is at least
// 4,096 times its largest item.
//
// All passes are integer and tiny next to the attention itself. In hash mode
// the bucket ids are non-decreasing along the sorted rows, so the key tiles
// whose bucket range can overlap a query tile's form one contiguous run found
// by binary search; QK and dense modes test every pair of tiles of a head.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace scfa {
namespace {

__device__ __forceinline__ int warp_min(int v) {
  for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_max(int v) {
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One side of the tile statistics pass: index and bucket arrays, tiles.
struct StatSide {
  const int32_t* idx;
  const int32_t* hash;
  long long n_tiles;
  int T, nT;
  int4* out;
};
// Where the call puts the live-tile lists and how many entries they hold.
struct HdrInit {
  long long off[5];
  long long cap;
};

// One warp per tile: {min idx, max idx, min hash, max hash} over valid rows,
// query tiles first, then key tiles. Thread 0 of block 0 also clears the
// status word, counters and schedule and records the list layout (the
// header is read only by later launches).
__global__ void tile_stats_kernel(int mode, StatSide qs, StatSide ks, WsHeader* hdr, HdrInit hi) {
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    hdr->status = 0;
    hdr->n_live = 0;
    for (int i = 0; i < 4; ++i) hdr->sched[i] = 0;
    for (int i = 0; i < 5; ++i) hdr->list_off[i] = hi.off[i];
    hdr->list_cap = hi.cap;
  }
  const int lane = threadIdx.x & 31;
  const long long warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < qs.n_tiles + ks.n_tiles;
       w += warps) {
    const bool q_side = w < qs.n_tiles;
    const StatSide& sd = q_side ? qs : ks;
    const long long t = q_side ? w : w - qs.n_tiles;
    const long long bh = t / sd.nT;
    const int r0 = static_cast<int>(t % sd.nT) * kTile;
    const int rows = min(kTile, sd.T - r0);
    int mn = INT_MAX, mx = INT_MIN, hmn = INT_MAX, hmx = INT_MIN;
    for (int r = lane; r < rows; r += 32) {
      const long long g = bh * sd.T + r0 + r;
      const int id = (mode == SCFA_MODE_DENSE) ? (r0 + r) : sd.idx[g];
      mn = min(mn, id);
      mx = max(mx, id);
      if (mode == SCFA_MODE_HASH) {
        const int h = sd.hash[g];
        hmn = min(hmn, h);
        hmx = max(hmx, h);
      }
    }
    mn = warp_min(mn);
    mx = warp_max(mx);
    hmn = warp_min(hmn);
    hmx = warp_max(hmx);
    if (lane == 0) sd.out[t] = make_int4(mn, mx, hmn, hmx);
  }
}

struct TileCtx {
  int mode;
  unsigned flags;
  int Tq, Tk, nQt, nKt;
  const int4* qstat;
  const int4* kstat;
};

__device__ __forceinline__ bool tile_live(const TileCtx& c, const int4& qs, const int4& ks) {
  if (c.flags & SCFA_FLAG_NO_PRUNE) return true;
  bool live = qs.y >= ks.x;
  if (c.mode == SCFA_MODE_HASH) live = live && (qs.z <= ks.w) && (ks.z <= qs.w);
  return live;
}
__device__ __forceinline__ bool tile_full(const TileCtx& c, int i, int j, const int4& qs, const int4& ks) {
  const bool complete = (min(kTile, c.Tq - i * kTile) == kTile) && (min(kTile, c.Tk - j * kTile) == kTile);
  bool full = complete && (qs.x >= ks.y);
  if (c.mode == SCFA_MODE_HASH) full = full && (qs.z == qs.w) && (ks.z == ks.w) && (qs.z == ks.z);
  return full;
}

// first index in [0, n) with key(i) >= v, for a non-decreasing key
template <typename F>
__device__ __forceinline__ int lower_bound_by(int n, int v, F key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (key(mid) < v) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Candidate range [lo, hi) of partner tiles of one tile.
__device__ __forceinline__ void partner_range(const TileCtx& c, bool by_q, const int4& self, long long bh,
                                              int* lo, int* hi) {
  const int n = by_q ? c.nKt : c.nQt;
  if (c.mode != SCFA_MODE_HASH || (c.flags & SCFA_FLAG_NO_PRUNE)) {
    *lo = 0;
    *hi = n;
    return;
  }
  const int4* other = (by_q ? c.kstat : c.qstat) + bh * n;
  // partners with max hash >= my min hash, and min hash <= my max hash
  *lo = lower_bound_by(n, self.z, [&](int t) { return other[t].w; });
  *hi = lower_bound_by(n, self.w + 1, [&](int t) { return other[t].z; });
  if (self.w == INT_MAX) *hi = n;
}

// One warp per query tile (first B*H*nQt ids) or key tile (next B*H*nKt):
// the lanes test 32 partner tiles at a time.
__global__ void tile_count_kernel(TileCtx c, long long n_q, long long n_k,
                                  int32_t* __restrict__ qcount, int32_t* __restrict__ kcount) {
  const int lane = threadIdx.x & 31;
  const long long warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long t = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < n_q + n_k; t += warps) {
    const bool by_q = t < n_q;
    const long long id = by_q ? t : t - n_q;
    const int nself = by_q ? c.nQt : c.nKt;
    const long long bh = id / nself;
    const int4 self = (by_q ? c.qstat : c.kstat)[id];
    int lo, hi;
    partner_range(c, by_q, self, bh, &lo, &hi);
    const int4* other = (by_q ? c.kstat : c.qstat) + bh * (by_q ? c.nKt : c.nQt);
    int cnt = 0;
    for (int p0 = lo; p0 < hi; p0 += 32) {
      const int p = p0 + lane;
      bool live = false;
      if (p < hi) {
        const int4 o = other[p];
        live = by_q ? tile_live(c, self, o) : tile_live(c, o, self);
      }
      cnt += __popc(__ballot_sync(0xffffffffu, live));
    }
    if (lane == 0) (by_q ? qcount : kcount)[id] = cnt;
  }
}

// Exclusive scans: block 0 -> row_ptr from qcount, block 1 -> csc_ptr from
// kcount. If the total exceeds the lists' capacity `cap`, every pointer is 0
// (all lists empty, so nothing reads or writes past them) and the status word
// says SCFA_ERR_WORKSPACE.
struct ScanArgs {
  const int32_t* qcount;
  long long n_q;
  int32_t* row_ptr;
  const int32_t* kcount;
  long long n_k;
  int32_t* csc_ptr;
  WsHeader* hdr;
  long long cap;
};
__device__ void tile_scan_block(const ScanArgs& a, int blk) {
  const int32_t* in = blk == 0 ? a.qcount : a.kcount;
  int32_t* out = blk == 0 ? a.row_ptr : a.csc_ptr;
  const long long n = blk == 0 ? a.n_q : a.n_k;
  WsHeader* hdr = a.hdr;
  const long long cap = a.cap;
  const int tid = threadIdx.x, nt = blockDim.x;
  const long long per = (n + nt - 1) / nt;
  const long long b = min(n, per * tid), e = min(n, b + per);
  long long sum = 0;
  for (long long i = b; i < e; ++i) sum += in[i];
  __shared__ long long wsum[32];
  // block exclusive scan of the per-thread sums
  long long x = sum;
  const int lane = tid & 31, w = tid >> 5;
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  if (w == 0) {
    long long s = (lane < (nt >> 5)) ? wsum[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    wsum[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const bool over = wsum[(nt >> 5) - 1] > cap;
  long long run = over ? 0 : x - sum + (w > 0 ? wsum[w - 1] : 0);
  for (long long i = b; i < e; ++i) {
    out[i] = static_cast<int32_t>(run);
    if (!over) run += in[i];
  }
  if (tid == nt - 1) {
    out[n] = static_cast<int32_t>(run);
    if (blk == 0) {
      hdr->n_live = static_cast<int>(run);
      if (over) raise_status(&hdr->status, SCFA_ERR_WORKSPACE);
    }
  }
}

// One warp per tile, as the count pass: live partners are written in
// ascending order at ballot prefix positions.
__global__ void tile_fill_kernel(TileCtx c, long long n_q, long long n_k,
                                 const int32_t* __restrict__ row_ptr, int32_t* __restrict__ cols,
                                 uint8_t* __restrict__ fflags,
                                 const int32_t* __restrict__ csc_ptr, int32_t* __restrict__ csc_rows,
                                 uint8_t* __restrict__ cflags) {
  const int lane = threadIdx.x & 31;
  const long long warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long t = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < n_q + n_k; t += warps) {
    const bool by_q = t < n_q;
    const long long id = by_q ? t : t - n_q;
    const int nself = by_q ? c.nQt : c.nKt;
    const long long bh = id / nself;
    const int me = static_cast<int>(id % nself);
    const int4 self = (by_q ? c.qstat : c.kstat)[id];
    int lo, hi;
    partner_range(c, by_q, self, bh, &lo, &hi);
    const int4* other = (by_q ? c.kstat : c.qstat) + bh * (by_q ? c.nKt : c.nQt);
    const long long first = by_q ? row_ptr[id] : csc_ptr[id];
    // entries this tile may write (0 for every tile when the lists overflowed)
    const long long budget = (by_q ? row_ptr[id + 1] : csc_ptr[id + 1]) - first;
    long long pos = first;
    for (int p0 = lo; p0 < hi; p0 += 32) {
      const int p = p0 + lane;
      bool live = false;
      uint8_t f = 0;
      if (p < hi) {
        const int4 o = other[p];
        const int4 qs = by_q ? self : o;
        const int4 ks = by_q ? o : self;
        live = tile_live(c, qs, ks);
        f = tile_full(c, by_q ? me : p, by_q ? p : me, qs, ks) ? kFlagFull : 0;
      }
      const unsigned m = __ballot_sync(0xffffffffu, live);
      if (live && pos + __popc(m & ((1u << lane) - 1u)) - first < budget) {
        const long long at = pos + __popc(m & ((1u << lane) - 1u));
        if (by_q) {
          cols[at] = p;
          fflags[at] = f;
        } else {
          csc_rows[at] = p;
          cflags[at] = f;
        }
      }
      pos += __popc(m);
    }
  }
}

// Union list of each query-tile pair (2m, 2m + 1), one warp per pair. Both
// CSR rows are strictly ascending; an entry's place in the union is its index
// in its own row, plus the entries of the other row below it (binary search),
// minus the columns common to both rows below it (a running ballot count in
// row order). A common column is written once, from row 2m.
__global__ void pair_list_kernel(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ cols,
                                 const uint8_t* __restrict__ fflags, int nQt, int nPairs, long long n_pairs,
                                 int32_t* __restrict__ pcount, int32_t* __restrict__ ulist) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  const long long warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long pid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; pid < n_pairs;
       pid += warps) {
    const long long bh = pid / nPairs;
    const int m = static_cast<int>(pid % nPairs);
    const long long g0 = bh * nQt + 2 * m;
    const int a0 = row_ptr[g0], na = row_ptr[g0 + 1] - a0;
    const bool has1 = 2 * m + 1 < nQt;
    const int b0 = has1 ? row_ptr[g0 + 1] : 0, nb = has1 ? row_ptr[g0 + 2] - b0 : 0;
    const int32_t* A = cols + a0;
    const int32_t* Bc = cols + b0;
    // the union is no longer than the two rows together, so it fits in their
    // slots, which start at row_ptr[g0]
    int32_t* out = ulist + a0;
    int common = 0;
    for (int c0 = 0; c0 < na; c0 += 32) {
      const int ia = c0 + lane;
      bool both = false;
      int x = 0, kb = 0;
      if (ia < na) {
        x = A[ia];
        kb = lower_bound_by(nb, x, [&](int t) { return Bc[t]; });
        both = kb < nb && Bc[kb] == x;
      }
      const unsigned mk = __ballot_sync(0xffffffffu, both);
      if (ia < na) {
        int bits = 1 | ((fflags[a0 + ia] & kFlagFull) ? 2 : 0);
        if (both) bits |= 4 | ((fflags[b0 + kb] & kFlagFull) ? 8 : 0);
        out[ia + kb - (common + __popc(mk & lt))] = (x << 4) | bits;
      }
      common += __popc(mk);
    }
    int common_b = 0;
    for (int c0 = 0; c0 < nb; c0 += 32) {
      const int ib = c0 + lane;
      bool both = false;
      int y = 0, ka = 0;
      if (ib < nb) {
        y = Bc[ib];
        ka = lower_bound_by(na, y, [&](int t) { return A[t]; });
        both = ka < na && A[ka] == y;
      }
      const unsigned mk = __ballot_sync(0xffffffffu, both);
      if (ib < nb && !both)
        out[ib + ka - (common_b + __popc(mk & lt))] = (y << 4) | 4 | ((fflags[b0 + ib] & kFlagFull) ? 8 : 0);
      common_b += __popc(mk);
    }
    if (lane == 0) pcount[pid] = na + nb - common;
  }
}

struct OrderList {
  const int32_t* count;
  long long n;
  int maxc;
  int32_t* out;
  int32_t* gcur;
  bool may_keep_natural;
};

constexpr int kOrderChunk = 4096;     // counts staged in shared memory per scatter round
// A key-tile list whose total work is at least this many times its largest
// item keeps the natural (head, tile) order: the tail left by the largest item
// is then small, and key tiles taken at the same time share their query tiles
// in L2. (The forward lists stay sorted: the query-tile-pair forward hands its
// items out in fixed rounds, where the sorted order balances better.)
constexpr long long kNaturalOrderRatio = 4096;
constexpr int kOrderWarpBins = 8192;  // per-warp bin offsets (few distinct counts)

// Stable counting sort of ids by count, descending: block 0 builds the
// forward order (query tiles), block 1 the backward order (key tiles), block
// 2 the order of query-tile pairs. The whole block histograms; warp 0 scans
// and scatters in id order (stable by construction), reading the counts from
// shared memory, where the whole block stages them one chunk at a time.
__device__ void work_order_block(const OrderList& L, int smem_bins) {
  extern __shared__ int32_t scur[];
  const int32_t* cnt = L.count;
  const long long n = L.n;
  const int maxc = L.maxc;
  int32_t* out = L.out;
  int32_t* cur = (maxc + 1 <= smem_bins) ? scur : L.gcur;
  int32_t* chunk = scur + smem_bins;
  if (L.may_keep_natural) {
    __shared__ unsigned long long s_total;
    __shared__ int s_max;
    if (threadIdx.x == 0) {
      s_total = 0;
      s_max = 0;
    }
    __syncthreads();
    unsigned long long tot = 0;
    int mx = 0;
    for (long long i = threadIdx.x; i < n; i += blockDim.x) {
      const int c = max(cnt[i], 0);
      tot += static_cast<unsigned long long>(c);
      mx = max(mx, c);
    }
    for (int o = 16; o > 0; o >>= 1) {
      tot += __shfl_xor_sync(0xffffffffu, tot, o);
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if ((threadIdx.x & 31) == 0) {
      atomicAdd(&s_total, tot);
      atomicMax(&s_max, mx);
    }
    __syncthreads();
    const bool natural = n > 0 && static_cast<unsigned long long>(s_max) * kNaturalOrderRatio <= s_total;
    if (natural) {
      for (long long i = threadIdx.x; i < n; i += blockDim.x) out[i] = static_cast<int32_t>(i);
      return;
    }
  }
  for (int cc = threadIdx.x; cc <= maxc; cc += blockDim.x) cur[cc] = 0;
  __syncthreads();
  for (long long i = threadIdx.x; i < n; i += blockDim.x) atomicAdd(&cur[min(max(cnt[i], 0), maxc)], 1);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    // start[c] = number of ids with a larger count
    int running = 0;
    for (int base = maxc; base >= 0; base -= 32) {
      const int cc = base - lane;
      const int v = cc >= 0 ? cur[cc] : 0;
      int x = v;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (cc >= 0) cur[cc] = running + x - v;
      running += __shfl_sync(0xffffffffu, x, 31);
    }
  }
  // few distinct counts: all 32 warps scatter, each a contiguous slice of the
  // chunk, from per-warp bin offsets (earlier slices first: stable)
  const int nwarps = static_cast<int>(blockDim.x >> 5), wid = static_cast<int>(threadIdx.x >> 5);
  int32_t* hw = chunk + kOrderChunk;  // [nwarps][maxc + 1]
  const bool parallel = (maxc + 1) * nwarps <= kOrderWarpBins;
  for (long long c0 = 0; c0 < n; c0 += kOrderChunk) {
    const int len = static_cast<int>(min(static_cast<long long>(kOrderChunk), n - c0));
    __syncthreads();  // the previous chunk is scattered (and the scan above is done)
    for (int t = threadIdx.x; t < len; t += blockDim.x) chunk[t] = min(max(cnt[c0 + t], 0), maxc);
    if (parallel) {
      for (int i = threadIdx.x; i < (maxc + 1) * nwarps; i += blockDim.x) hw[i] = 0;
      __syncthreads();
      const int per = (len + nwarps - 1) / nwarps;
      const int s0 = min(len, wid * per), s1 = min(len, s0 + per);
      int32_t* my = hw + wid * (maxc + 1);
      for (int base = s0; base < s1; base += 32) {
        const int t = base + lane;
        const int cc = t < s1 ? chunk[t] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, cc);
        if (cc >= 0 && (peers & ((1u << lane) - 1u)) == 0) my[cc] += __popc(peers);
        __syncwarp();
      }
      __syncthreads();
      for (int c = threadIdx.x; c <= maxc; c += blockDim.x) {
        int run = cur[c];
        for (int w = 0; w < nwarps; ++w) {
          const int t = hw[w * (maxc + 1) + c];
          hw[w * (maxc + 1) + c] = run;
          run += t;
        }
        cur[c] = run;
      }
      __syncthreads();
      for (int base = s0; base < s1; base += 32) {
        const int t = base + lane;
        const bool active = t < s1;
        const int cc = active ? chunk[t] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, cc);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        const int start = active ? my[cc] : 0;
        __syncwarp();
        if (active) {
          out[start + rank] = static_cast<int32_t>(c0 + t);
          if (rank == 0) my[cc] = start + __popc(peers);
        }
        __syncwarp();
      }
      continue;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      for (int base = 0; base < len; base += 32) {
        const int t = base + lane;
        const bool active = t < len;
        const int cc = active ? chunk[t] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, cc);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        const int start = active ? cur[cc] : 0;
        __syncwarp();
        if (active) {
          out[start + rank] = static_cast<int32_t>(c0 + t);
          if (rank == 0) cur[cc] = start + __popc(peers);
        }
        __syncwarp();
      }
    }
  }
}

// The two exclusive scans (blocks 0 and 1: row_ptr, csc_ptr) and the work
// orders of the query and key tiles (blocks 2 and 3) in one launch: the
// orders read only the counts, so they need not wait for the scans. A launch
// of two blocks runs the scans alone.
__global__ void tile_scan_order_kernel(ScanArgs sa, OrderList lq, OrderList lk, int smem_bins) {
  if (blockIdx.x < 2) {
    tile_scan_block(sa, blockIdx.x);
  } else {
    work_order_block(blockIdx.x == 2 ? lq : lk, smem_bins);
  }
}

// The order of the query-tile pairs (head dimension 128), once their union
// lists are counted.
__global__ void pair_order_kernel(OrderList lp, int smem_bins) { work_order_block(lp, smem_bins); }

// SCFA_FLAG_VALIDATE: checks the documented contracts of the index inputs and
// raises SCFA_ERR_INVALID in the status word on the first violation (nothing
// traps; the attention still runs and its results are then undefined).
//   QK: per head, the kept positions (q_idx >= 0, k_idx < INT32_MAX) strictly
//       ascending, padding sentinels (-1 / INT32_MAX) only after them.
//   hash: per head, q_hash and k_hash non-decreasing and >= 0; with
//       `original` (SCFA_FLAG_ORIGINAL_ORDER) no index in [0, T) twice
//       (two rows would write the same output row), checked with one bit per
//       row in `bits` (zeroed by the caller).
__global__ void validate_kernel(int mode, int original, const int32_t* __restrict__ q_idx,
                                const int32_t* __restrict__ k_idx, const int32_t* __restrict__ q_hash,
                                const int32_t* __restrict__ k_hash, long long BH, int Tq, int Tk, int To,
                                uint32_t* __restrict__ bits, int* status) {
  const long long nq = BH * Tq, n = nq + BH * Tk;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < n; t += stride) {
    const bool is_q = t < nq;
    const long long u = is_q ? t : t - nq;
    const int T = is_q ? Tq : Tk;
    const long long bh = u / T;
    const int r = static_cast<int>(u - bh * T);
    const int32_t* idx = (is_q ? q_idx : k_idx) + bh * T;
    bool bad = false;
    if (mode == SCFA_MODE_QK) {
      const int32_t sent = is_q ? -1 : INT_MAX;
      const int32_t v = idx[r];
      if (v != sent && v < 0) bad = true;
      if (r > 0) {
        const int32_t w = idx[r - 1];
        if (w == sent && v != sent) bad = true;         // a kept row after padding
        if (w != sent && v != sent && w >= v) bad = true;  // not strictly ascending
      }
    } else if (mode == SCFA_MODE_HASH) {
      const int32_t* h = (is_q ? q_hash : k_hash) + bh * T;
      if (h[r] < 0 || (r > 0 && h[r - 1] > h[r])) bad = true;
      if (original) {
        const int32_t v = idx[r];
        if (v >= 0 && v < To) {  // ids outside [0, To) are rows that are not written
          const long long words = (static_cast<long long>(T) + 31) / 32;
          uint32_t* b = bits + (is_q ? 0 : BH * ((static_cast<long long>(Tq) + 31) / 32)) + bh * words + v / 32;
          const uint32_t m = 1u << (v & 31);
          if (atomicOr(b, m) & m) bad = true;  // this index seen before in this head
        }
      }
    }
    if (bad) raise_status(status, SCFA_ERR_INVALID);
  }
}

inline int grid_for(long long work, int block, int max_blocks) {
  long long g = (work + block - 1) / block;
  if (g < 1) g = 1;
  if (g > max_blocks) g = max_blocks;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_validate(int mode, bool original, const int32_t* q_idx, const int32_t* k_idx,
                            const int32_t* q_hash, const int32_t* k_hash, int B, int H, int Tq, int Tk, int To,
                            char* ws, const AttnWs& L, cudaStream_t st) {
  if (mode == SCFA_MODE_DENSE) return cudaSuccess;
  const long long BH = static_cast<long long>(B) * H;
  uint32_t* bits = reinterpret_cast<uint32_t*>(ws + L.vbits);
  if (original) {
    cudaError_t e = cudaMemsetAsync(bits, 0, L.vbits_bytes, st);
    if (e != cudaSuccess) return e;
  }
  const long long n = BH * (static_cast<long long>(Tq) + Tk);
  validate_kernel<<<grid_for(n, 256, num_sms() * 8), 256, 0, st>>>(mode, original ? 1 : 0, q_idx, k_idx, q_hash,
                                                                    k_hash, BH, Tq, Tk, To, bits,
                                                                    reinterpret_cast<int*>(ws + L.header));
  return cudaGetLastError();
}

cudaError_t launch_tiles(int mode, const int32_t* q_idx, const int32_t* k_idx,
                         const int32_t* q_hash, const int32_t* k_hash,
                         int B, int H, int Tq, int Tk, unsigned flags,
                         char* ws, const AttnWs& L, cudaStream_t st, bool with_pairs, bool count_only) {
  const int sms = num_sms();
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws + L.header);
  int4* qstat = reinterpret_cast<int4*>(ws + L.qstat);
  int4* kstat = reinterpret_cast<int4*>(ws + L.kstat);
  int32_t* qcount = reinterpret_cast<int32_t*>(ws + L.qcount);
  int32_t* kcount = reinterpret_cast<int32_t*>(ws + L.kcount);
  int32_t* row_ptr = reinterpret_cast<int32_t*>(ws + L.row_ptr);
  int32_t* csc_ptr = reinterpret_cast<int32_t*>(ws + L.csc_ptr);

  // header + tile statistics of both sides; counts; scans with the two
  // work orders; lists (+ pair unions and their order at D = 128)
  const HdrInit hi{{static_cast<long long>(L.cols), static_cast<long long>(L.csc_rows),
                    static_cast<long long>(L.fflags), static_cast<long long>(L.cflags),
                    static_cast<long long>(L.ulist)},
                   L.cap};
  const StatSide sq{q_idx, q_hash, L.n_qtiles, Tq, L.nQt, qstat};
  const StatSide sk{k_idx, k_hash, L.n_ktiles, Tk, L.nKt, kstat};
  const long long nt = L.n_qtiles + L.n_ktiles;
  tile_stats_kernel<<<grid_for(nt * 32, 256, sms * 8), 256, 0, st>>>(mode, sq, sk, hdr, hi);
  TileCtx c{mode, flags, Tq, Tk, L.nQt, L.nKt, qstat, kstat};
  tile_count_kernel<<<grid_for(nt * 32, 256, sms * 8), 256, 0, st>>>(c, L.n_qtiles, L.n_ktiles, qcount, kcount);
  const ScanArgs sa{qcount, L.n_qtiles, row_ptr, kcount, L.n_ktiles, csc_ptr, hdr, count_only ? LLONG_MAX : L.cap};
  const int smem_bins = 12 * 1024;  // 48 KB of shared memory; larger histograms use the workspace
  const size_t smem = static_cast<size_t>(smem_bins + kOrderChunk + kOrderWarpBins) * sizeof(int32_t);
  static bool order_smem_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !order_smem_set[dev]) {
    e = cudaFuncSetAttribute(tile_scan_order_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(pair_order_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) order_smem_set[dev] = true;
  }
  int32_t* gcur = reinterpret_cast<int32_t*>(ws + L.cursor);
  OrderList lf{qcount, L.n_qtiles, L.nKt, reinterpret_cast<int32_t*>(ws + L.work_fwd), gcur, false};
  OrderList lb{kcount, L.n_ktiles, L.nQt, reinterpret_cast<int32_t*>(ws + L.work_bwd), gcur + L.nKt + 1, true};
  tile_scan_order_kernel<<<count_only ? 2 : 4, 1024, smem, st>>>(sa, lf, lb, smem_bins);
  if (count_only) return cudaGetLastError();
  tile_fill_kernel<<<grid_for(nt * 32, 256, sms * 8), 256, 0, st>>>(
      c, L.n_qtiles, L.n_ktiles, row_ptr, reinterpret_cast<int32_t*>(ws + L.cols),
      reinterpret_cast<uint8_t*>(ws + L.fflags), csc_ptr, reinterpret_cast<int32_t*>(ws + L.csc_rows),
      reinterpret_cast<uint8_t*>(ws + L.cflags));
  if (with_pairs) {
    pair_list_kernel<<<grid_for(L.n_pairs * 32, 256, sms * 8), 256, 0, st>>>(
        row_ptr, reinterpret_cast<const int32_t*>(ws + L.cols), reinterpret_cast<const uint8_t*>(ws + L.fflags),
        L.nQt, L.nPairs, L.n_pairs, reinterpret_cast<int32_t*>(ws + L.pcount), reinterpret_cast<int32_t*>(ws + L.ulist));
    OrderList lp{reinterpret_cast<const int32_t*>(ws + L.pcount), L.n_pairs, L.nKt,
                 reinterpret_cast<int32_t*>(ws + L.work_pairs), gcur + L.nKt + L.nQt + 2, false};
    pair_order_kernel<<<1, 1024, smem, st>>>(lp, smem_bins);
  }
  return cudaGetLastError();
}

}  // namespace scfa
