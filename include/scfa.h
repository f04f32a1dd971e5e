/*
 * scfa.h — C ABI of libscfa.so: sparse causal flash attention (SCFA) on
 * NVIDIA GB300 (sm_103a).
 *
 * The operation: exact causal softmax attention, forward and backward, over
 * irregular dynamic-sparse layouts ("Faster Causal Attention Over Large
 * Sequences Through Sparse Flash Attention", summary page on deep-paper.org
 * of arXiv 2306.01160, section "SCFA 解决方案"):
 *   - QK-sparse: queries and keys were dropped and the kept rows compacted;
 *     q_idx / k_idx hold their original positions; a 128 x 128 tile is skipped
 *     when max(q_idx) < min(k_idx), and inside live tiles an element is kept
 *     iff q_idx >= k_idx  (part 1 "QK-Sparse").
 *   - Hash-sparse: tokens are bucket-sorted by an LSH id (q_hash / k_hash);
 *     tiles whose bucket ranges do not overlap, or that are wholly acausal,
 *     are skipped, and inside live tiles an element is kept iff it is causal
 *     in original positions AND in the same bucket (part 2 "Hash-Sparse").
 *   - Dense causal (the comparator of section "FlashAttention 的兴起"): the
 *     same kernels with q_idx = k_idx = position.
 *
 * Conventions for every entry point below:
 *   - Tensor pointers are DEVICE pointers to contiguous row-major arrays.
 *     bf16 tensors are passed as uint16_t (IEEE bfloat16 bit patterns).
 *     Q/K/V/O/dO/dQ/dK/dV have layout [B][H][T][D]; LSE, idx and hash arrays
 *     [B][H][T]. bf16 tensor pointers must be 16-byte aligned.
 *   - D is the head dimension (64 or 128 where stated); scale multiplies QK^T
 *     (normally 1/sqrt(D)). LSE is the natural-log softmax denominator, fp32.
 *   - A query row with no admissible key gets O = 0, LSE = -inf and passes no
 *     gradient; a key no query may see gets dK = dV = 0. Outputs are fully
 *     overwritten. Inputs are read only. Inputs and outputs must not alias.
 *   - The caller owns all memory. The library never allocates, frees or
 *     synchronises, except scfa_get_device_status (which synchronises the
 *     stream) and SCFA_FLAG_DEBUG_SYNC. Scratch space is the caller's
 *     workspace `ws` of `ws_bytes` bytes (256-byte aligned), sized by the
 *     *_workspace_size functions. One workspace must not be used by two calls
 *     that may run at the same time.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every
 *     call is asynchronous on that stream.
 *   - Errors: arguments are validated on the host before any launch and a bad
 *     argument returns SCFA_ERR_INVALID / SCFA_ERR_UNSUPPORTED /
 *     SCFA_ERR_WORKSPACE with nothing launched. A failed launch returns
 *     SCFA_ERR_CUDA. Device-side failures (a pipeline wait that ran past its
 *     time limit) are written to a status word in the workspace and read with
 *     scfa_get_device_status; kernels never trap.
 */
#ifndef SCFA_H
#define SCFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int scfa_status;
enum {
  SCFA_OK = 0,
  SCFA_ERR_INVALID = 1,      /* null pointer, bad size, misaligned pointer */
  SCFA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. head dim) */
  SCFA_ERR_WORKSPACE = 3,    /* workspace too small or misaligned */
  SCFA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  SCFA_ERR_TIMEOUT = 5       /* device: a pipeline wait passed its limit */
};

/* attention modes */
enum { SCFA_MODE_DENSE = 0, SCFA_MODE_QK = 1, SCFA_MODE_HASH = 2 };

/* flags */
enum {
  SCFA_FLAG_NO_PRUNE = 1,    /* treat every tile as live (results unchanged) */
  SCFA_FLAG_VALIDATE = 2,    /* check the index contracts on the device first and
                                raise SCFA_ERR_INVALID in the status word on a
                                violation (the call still runs; its results are
                                then undefined): QK: per head the kept positions
                                strictly ascending, sentinels only after them;
                                hash: q_hash / k_hash non-decreasing and >= 0,
                                and with SCFA_FLAG_ORIGINAL_ORDER no index in
                                [0, T) twice. */
  SCFA_FLAG_DEBUG_SYNC = 4,  /* synchronise the stream after every launch */
  SCFA_FLAG_REUSE_TILES = 8,  /* the workspace already holds the live-tile list
                                 of these exact indices and shape (built by
                                 scfa_tiles or an earlier call on the same
                                 workspace): skip the metadata pass. One
                                 backward-sized workspace may then serve the
                                 forward and the backward call of a step. */
  SCFA_FLAG_ORIGINAL_ORDER = 16, /* hash mode only: the row tensors o (forward
                                 output and backward input), dq, dk and dv are
                                 in ORIGINAL row order: sorted query row s of
                                 head (b,h) is row q_idx[b,h,s] of o and dq,
                                 sorted key row s is row k_idx[b,h,s] of dk and
                                 dv (within each head, the q_idx / k_idx that
                                 fall in [0, T_orig) must be distinct; rows
                                 whose index falls outside are not written,
                                 and read as zero).
                                 q, k, v, do, lse stay in sorted order. This
                                 replaces the lsh_unsort passes. */
  SCFA_FLAG_KEEP_O32 = 32,       /* forward: also store O in fp32 in the
                                 workspace, which must then be sized for the
                                 backward (scfa_attn_workspace_size(mode, 1,
                                 ...)); backward: take rowsum(dO * O) from that
                                 copy instead of the bf16 o. Pass it to the
                                 forward and the backward of one step on the
                                 same workspace. The bf16 rounding of O is
                                 otherwise the largest error term of dS. */
  SCFA_FLAG_DEBUG_STALL = 64,    /* debug: the main attention kernel of the call
                                 withholds the first K / V load of every CTA,
                                 so its pipeline waits on a barrier that
                                 nothing completes; each wait gives up after
                                 its limit (1 s), the status word reads
                                 SCFA_ERR_TIMEOUT and the results are invalid.
                                 For testing the timeout path: the CTAs drain
                                 their issued copies and MMAs and exit, and the
                                 device stays usable. */
  SCFA_FLAG_GATHER_Q = 128,      /* hash mode, with SCFA_FLAG_ORIGINAL_ORDER:
                                 q (and do in the backward) are also in
                                 ORIGINAL row order, [B,H,T_orig,D]; the
                                 attention kernels load sorted query row s of
                                 head (b,h) from row q_idx[b,h,s] (tile-row
                                 gathers), so no sorted copy is made. A sorted
                                 row whose index falls outside [0, T_orig)
                                 (padding) reads some row of the same head:
                                 its scores are masked, so for finite inputs
                                 the results equal those computed from sorted
                                 copies with zero padding rows. Needs
                                 B*H*T_orig < 2^31. lse stays in sorted
                                 order. */
  SCFA_FLAG_GATHER_KV = 256      /* the same for k and v, through k_idx. */
};

/* Tiles are SCFA_TILE rows of queries by SCFA_TILE rows of keys. */
#define SCFA_TILE 128

/* Human-readable name of a status code (static string). */
const char* scfa_status_string(scfa_status s);

/* ----------------------------------------------------------------------------
 * Workspace sizing.
 * scfa_attn_workspace_size: bytes needed by scfa_{dense,qk,hash}_{fwd,bwd} and
 * scfa_tiles for the given mode (SCFA_MODE_*), direction (backward = 0 / 1)
 * and shape. Tq = Tk = T for dense and hash modes. Returns 0 on bad sizes.
 * ------------------------------------------------------------------------- */
size_t scfa_attn_workspace_size(int mode, int backward, int B, int H, int Tq, int Tk, int D);

/* The live-tile lists of a workspace hold as many entries as fit past its
 * fixed part; scfa_attn_workspace_size leaves room for every tile pair (the
 * worst case), which at long T dominates (8 heads of 2^20 tokens: 7.5 GB).
 * The layout of a workspace depends on its size alone, never on the call: a
 * workspace that holds the backward's fixed part (the fp32 dQ accumulator
 * and the per-row metadata) lays them out for every call, forward included,
 * and the lists follow them; so a forward and a SCFA_FLAG_REUSE_TILES
 * backward on one workspace always agree on where the lists are. (So a
 * forward-only workspace grown past that fixed part holds fewer entries than
 * one just below it; the sizes returned below never fall in that gap.)
 * scfa_attn_workspace_size_live sizes a workspace whose lists hold n_live
 * entries for a call of the given kind; scfa_attn_workspace_capacity returns
 * how many entries a workspace of ws_bytes holds (-1: not even the fixed part
 * the call needs fits). Both are host-only arithmetic. scfa_tiles_count writes
 * the live count of a problem (an int32 on the DEVICE, asynchronously on
 * `stream`) using a workspace of at least
 * scfa_attn_workspace_size_live(mode, 0, ..., 0) bytes. A call whose lists
 * need more entries than its workspace holds leaves every list empty, so no
 * tile is computed and nothing is read or written past the lists, and raises
 * SCFA_ERR_WORKSPACE in the status word. A call that reuses a list
 * (SCFA_FLAG_REUSE_TILES) finds it where the building call recorded it in
 * the workspace header. */
size_t scfa_attn_workspace_size_live(int mode, int backward, int B, int H, int Tq, int Tk, int D,
                                     long long n_live);
long long scfa_attn_workspace_capacity(int mode, int backward, int B, int H, int Tq, int Tk, int D,
                                       size_t ws_bytes);
scfa_status scfa_tiles_count(int mode, const int32_t* q_idx, const int32_t* k_idx,
                             const int32_t* q_hash, const int32_t* k_hash,
                             int B, int H, int Tq, int Tk, void* ws, size_t ws_bytes,
                             int32_t* n_live, void* stream);

/* ----------------------------------------------------------------------------
 * Dense causal attention (comparator; page section "FlashAttention 的兴起":
 * a token sees only earlier tokens). q, k, v, o, do_, dq, dk, dv: [B,H,T,D]
 * bf16; lse: [B,H,T] fp32. D = 64 or 128.
 * ------------------------------------------------------------------------- */
scfa_status scfa_dense_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           int B, int H, int T, int D, float scale,
                           uint16_t* o, float* lse,
                           void* ws, size_t ws_bytes, unsigned flags, void* stream);
scfa_status scfa_dense_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const uint16_t* o, const float* lse, const uint16_t* do_,
                           int B, int H, int T, int D, float scale,
                           uint16_t* dq, uint16_t* dk, uint16_t* dv,
                           void* ws, size_t ws_bytes, unsigned flags, void* stream);

/* ----------------------------------------------------------------------------
 * QK-sparse attention (page section "SCFA 解决方案", part 1 "QK-Sparse").
 * q, o, do_, dq: [B,H,Tq,D]; k, v, dk, dv: [B,H,Tk,D]; q_idx [B,H,Tq] and
 * k_idx [B,H,Tk] int32 original positions, ascending within each (b,h) over
 * the kept rows. Heads keep different counts, so rows past a head's count are
 * padding with sentinels: q_idx = -1 for padded queries, k_idx = INT32_MAX
 * for padded keys (never admissible). Outputs are in compacted order. D = 64 or 128.
 * ------------------------------------------------------------------------- */
scfa_status scfa_qk_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const int32_t* q_idx, const int32_t* k_idx,
                        int B, int H, int Tq, int Tk, int D, float scale,
                        uint16_t* o, float* lse,
                        void* ws, size_t ws_bytes, unsigned flags, void* stream);
scfa_status scfa_qk_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const uint16_t* o, const float* lse, const uint16_t* do_,
                        const int32_t* q_idx, const int32_t* k_idx,
                        int B, int H, int Tq, int Tk, int D, float scale,
                        uint16_t* dq, uint16_t* dk, uint16_t* dv,
                        void* ws, size_t ws_bytes, unsigned flags, void* stream);

/* The selection step in front of QK-sparse attention (same page section:
 * dropped queries and keys leave compacted Q/K/V with their original
 * positions). keep [B,H,T] uint8 (nonzero = kept; the policy that sets it is
 * the caller's). idx [B,H,Tc] int32: the positions of the kept tokens of
 * each head in ascending order, then `sentinel` (which must lie outside
 * [0, T): -1 for queries, INT32_MAX for keys); count [B,H] int32: the kept
 * count, also when it exceeds Tc (then only the first Tc positions are
 * written: size Tc to the largest count). The rows move with lsh_gather
 * (x_c = x gathered by idx, zero rows at the sentinels: T = T, T_sorted =
 * Tc) and gradients go back to full length with lsh_unsort. */
scfa_status scfa_qk_select(const uint8_t* keep, int B, int H, int T, int Tc, int32_t sentinel,
                           int32_t* idx, int32_t* count, void* stream);

/* ----------------------------------------------------------------------------
 * Hash-sparse attention on bucket-sorted rows (page section "SCFA 解决方案",
 * part 2 "Hash-Sparse"). All row tensors are in SORTED order, as produced by
 * lsh_bucket_sort / lsh_gather: q_s, o_s, do_s, dq_s use the query order,
 * k_s, v_s, dk_s, dv_s the key order. q_idx / k_idx [B,H,T] are the original
 * positions of the sorted rows (the perm of lsh_bucket_sort) and q_hash /
 * k_hash [B,H,T] their bucket ids, non-decreasing within each (b,h).
 * T is the row count per head of the sorted tensors; T_orig that of the
 * original-order tensors (T_orig <= T; equal to T unless the sorted layout
 * has padding rows, as lsh_bucket_sort_tiled's does).
 * Put results back in original order with lsh_unsort, or pass
 * SCFA_FLAG_ORIGINAL_ORDER to have the kernels write o / dq / dk / dv (and
 * read o) in original order directly, as [B,H,T_orig,D] tensors. Without
 * that flag T_orig must equal T. D = 64 or 128.
 * ------------------------------------------------------------------------- */
scfa_status scfa_hash_fwd(const uint16_t* q_s, const uint16_t* k_s, const uint16_t* v_s,
                          const int32_t* q_idx, const int32_t* k_idx,
                          const int32_t* q_hash, const int32_t* k_hash,
                          int B, int H, int T, int T_orig, int D, float scale,
                          uint16_t* o_s, float* lse_s,
                          void* ws, size_t ws_bytes, unsigned flags, void* stream);
scfa_status scfa_hash_bwd(const uint16_t* q_s, const uint16_t* k_s, const uint16_t* v_s,
                          const uint16_t* o_s, const float* lse_s, const uint16_t* do_s,
                          const int32_t* q_idx, const int32_t* k_idx,
                          const int32_t* q_hash, const int32_t* k_hash,
                          int B, int H, int T, int T_orig, int D, float scale,
                          uint16_t* dq_s, uint16_t* dk_s, uint16_t* dv_s,
                          void* ws, size_t ws_bytes, unsigned flags, void* stream);

/* ----------------------------------------------------------------------------
 * LSH bucketing (page section "动态稀疏性为何会破坏它", item 2: similar tokens
 * are grouped into buckets with LSH as in Reformer, and reordered by bucket).
 * Construction: h(x) = argmax_j v_j with v = [x R, -x R], R a [D, m] bf16
 * random rotation shared by queries and keys, n_buckets = 2 m. The argmax is
 * of the EXACT real values (ties -> smallest j); L2 normalisation of x does
 * not change it and is not applied. Inputs must be finite.
 * x: [B,H,T,D] bf16, D a multiple of 8 and <= 256; 2 <= n_buckets <= 32768,
 * even.
 *
 * lsh_hash: hash [B,H,T] int32 in original order.
 * lsh_bucket_sort: per (b,h) stable sort by (bucket, position). perm [B,H,T]:
 *   sorted slot -> original position; hash_sorted [B,H,T]; bucket_off
 *   [B,H,n_buckets+1]: number of tokens with a smaller bucket id; x_sorted
 *   (nullable) [B,H,T,D] = x gathered by perm. Workspace:
 *   lsh_workspace_size.
 * lsh_bucket_sort_tiled: the same order, laid out so that every bucket
 *   starts on a multiple of 128 rows (the attention tile height): no tile then
 *   holds two buckets, so far fewer (query tile, key tile) pairs stay live.
 *   Bucket b's n_b rows start at bucket_start[b,h,b] = the sum over c < b of
 *   n_c rounded up to a multiple of 128; bucket_start[b,h,n_buckets] is where
 *   the last bucket's tiles end. The rows between a bucket's n_b rows and its
 *   next multiple of 128, and all rows after the last bucket up to T_sorted,
 *   are padding: perm = pad, hash_sorted = the bucket's id (n_buckets - 1
 *   after the last bucket) and x_sorted a zero row. pad must lie outside
 *   [0, T): pass -1 for queries (a query row that sees no key) and INT32_MAX
 *   for keys (a key row no query sees), the QK-mode sentinels. perm,
 *   hash_sorted [B,H,T_sorted]; x_sorted [B,H,T_sorted,D];
 *   T_sorted >= scfa_tiled_rows(T, n_buckets), the largest such layout
 *   (T + 127 per non-empty bucket, rounded up to 128). Same workspace as
 *   lsh_bucket_sort.
 * lsh_sort_ids: the stable sort of bucket ids given by the caller (hash
 *   [B,H,T] in original order, each in [0, n_buckets); 1 <= n_buckets <=
 *   32768), without hashing: T_sorted == T gives the plain layout of
 *   lsh_bucket_sort (bucket_start = bucket_off, pad unused), T_sorted >=
 *   scfa_tiled_rows(T, n_buckets) the tile-aligned one of
 *   lsh_bucket_sort_tiled. Shared-QK hashing sorts the keys by their queries'
 *   ids this way. An id outside [0, n_buckets) raises SCFA_ERR_INVALID in the
 *   workspace's status word (scfa_get_device_status) and takes no slot; the
 *   outputs are then undefined. Same workspace as lsh_bucket_sort.
 * lsh_gather: x_sorted[b,h,s,:] = x[b,h,perm[b,h,s],:] for the T_sorted rows
 *   s of each head (x has T rows per head); a zero row where perm[b,h,s] is
 *   outside [0, T).
 * lsh_unsort: y[b,h,perm[b,h,s],:] = y_sorted[b,h,s,:]. Rows whose perm entry
 *   is out of [0, T) are skipped. T_sorted (rows per head of the sorted
 *   tensor and of perm) may be anything >= 1: T for the plain layout, more
 *   for the tile-aligned one, fewer for a QK compaction (scfa_qk_select).
 * ------------------------------------------------------------------------- */
size_t lsh_workspace_size(int B, int H, int T, int n_buckets);
scfa_status lsh_hash(const uint16_t* x, const uint16_t* R, int B, int H, int T, int D,
                     int n_buckets, int32_t* hash, void* stream);
/* lsh_hash_heads: lsh_hash with one rotation per head: R is [H][D][n_buckets/2]
 * bf16 and head h of every batch is hashed with R[h] (the same construction,
 * the same exact argmax). Sort the ids with lsh_sort_ids. */
scfa_status lsh_hash_heads(const uint16_t* x, const uint16_t* R, int B, int H, int T, int D,
                           int n_buckets, int32_t* hash, void* stream);
scfa_status lsh_bucket_sort(const uint16_t* x, const uint16_t* R, int B, int H, int T, int D,
                            int n_buckets, int32_t* hash_sorted, int32_t* perm,
                            int32_t* bucket_off, uint16_t* x_sorted,
                            void* ws, size_t ws_bytes, unsigned flags, void* stream);
int scfa_tiled_rows(int T, int n_buckets);
scfa_status lsh_bucket_sort_tiled(const uint16_t* x, const uint16_t* R, int B, int H, int T, int D,
                                  int n_buckets, int T_sorted, int32_t pad, int32_t* hash_sorted,
                                  int32_t* perm, int32_t* bucket_start, uint16_t* x_sorted,
                                  void* ws, size_t ws_bytes, unsigned flags, void* stream);
scfa_status lsh_sort_ids(const int32_t* hash, int B, int H, int T, int n_buckets, int T_sorted,
                         int32_t pad, int32_t* hash_sorted, int32_t* perm, int32_t* bucket_start,
                         void* ws, size_t ws_bytes, unsigned flags, void* stream);
scfa_status lsh_gather(const uint16_t* x, const int32_t* perm, int B, int H, int T, int T_sorted,
                       int D, uint16_t* x_sorted, void* stream);
scfa_status lsh_unsort(const uint16_t* y_sorted, const int32_t* perm, int B, int H, int T, int T_sorted,
                       int D, uint16_t* y, void* stream);

/* ----------------------------------------------------------------------------
 * Tile metadata and the live-tile work list (page section "SCFA 解决方案":
 * tile pruning of part 1, bucket and causal pruning of part 2). Normally run
 * inside the attention calls; exposed for inspection and tests. Writes into
 * the workspace (sized for `mode`, backward = 1). Index arguments as for the
 * attention call of that mode (NULL where the mode has none).
 * Definitions, over the valid rows of each 128-row tile:
 *   QK / dense: live(i,j) = max q_idx(i) >= min k_idx(j).
 *   hash: live(i,j) = bucket ranges overlap AND max q_idx(i) >= min k_idx(j).
 *   FULL(i,j) (no element mask needed): both tiles have 128 valid rows, min
 *   q_idx(i) >= max k_idx(j) and, in hash mode, all four bucket bounds equal.
 * scfa_tile_view_get fills device pointers into the workspace (it reads the
 * workspace header, synchronously, to find the lists):
 *   row_ptr [B*H*nQt+1], cols, fflags (CSR over q tiles, columns ascending);
 *   csc_ptr [B*H*nKt+1], csc_rows, cflags (CSC over k tiles, rows ascending);
 *   flag bit 0 = FULL; work_fwd [B*H*nQt] and work_bwd [B*H*nKt]: every tile
 *   id sorted by live count descending, then id ascending, except that
 *   work_bwd keeps the natural id order when its summed live counts reach
 *   4096 times its largest count.
 *   Forward schedule over pairs of query tiles (2m, 2m + 1) of one head, pair
 *   id = (b*H + h) * ceil(nQt / 2) + m: pair_count [pairs] = size of the union
 *   of the two live lists; pair_list holds that union, key tiles ascending,
 *   from index row_ptr[(b*H + h)*nQt + 2m], one int32 per tile:
 *   (key tile << 4) | bit 0 live for 2m | bit 1 FULL for 2m | bit 2 live for
 *   2m + 1 | bit 3 FULL for 2m + 1; work_pairs [pairs]: pair ids by
 *   pair_count descending, then id ascending.
 * ------------------------------------------------------------------------- */
scfa_status scfa_tiles(int mode, const int32_t* q_idx, const int32_t* k_idx,
                       const int32_t* q_hash, const int32_t* k_hash,
                       int B, int H, int Tq, int Tk, int D,
                       void* ws, size_t ws_bytes, unsigned flags, void* stream);

typedef struct {
  const int32_t* row_ptr;
  const int32_t* cols;
  const uint8_t* fflags;
  const int32_t* csc_ptr;
  const int32_t* csc_rows;
  const uint8_t* cflags;
  const int32_t* work_fwd;
  const int32_t* work_bwd;
  const int32_t* pair_count;
  const int32_t* pair_list;
  const int32_t* work_pairs;
  int n_q_tiles;   /* per head */
  int n_k_tiles;   /* per head */
} scfa_tile_view;

scfa_status scfa_tile_view_get(const void* ws, int mode, int B, int H, int Tq, int Tk, int D,
                               scfa_tile_view* out);

/* ----------------------------------------------------------------------------
 * Pair counts (page section "实验与结果": SCFA hash-sparse attention covers
 * 100% of the bucket collisions, Reformer's chunked attention does not). A
 * pair (query row r, key row c) is admissible when the mode's element mask
 * keeps it: q_idx[r] >= k_idx[c] (QK), r >= c (dense), and in hash mode also
 * q_hash[r] == k_hash[c]. Results are written to *count, a DEVICE uint64,
 * asynchronously on `stream`.
 *
 * scfa_count_pairs: admissible pairs inside the live tiles of the list that
 *   `ws` holds (built by scfa_tiles or by an attention call with the same
 *   mode, indices and shape; ws sized for that mode). With full coverage this
 *   is the number of admissible pairs of the whole problem, the basis of the
 *   useful-FLOP count (4 D forward, 10 D backward per pair).
 * scfa_count_chunked_pairs: hash mode on bucket-sorted rows (q_idx / k_idx the
 *   original positions, q_hash / k_hash the sorted bucket ids, [B,H,T]):
 *   admissible pairs whose key's sorted slot lies in the query's chunk of
 *   `chunk` slots or in the chunk before it, i.e. the pairs a Reformer-style
 *   chunked attention over the same sort would see.
 * ------------------------------------------------------------------------- */
scfa_status scfa_count_pairs(int mode, const int32_t* q_idx, const int32_t* k_idx,
                             const int32_t* q_hash, const int32_t* k_hash,
                             int B, int H, int Tq, int Tk, int D, const void* ws, size_t ws_bytes,
                             unsigned long long* count, void* stream);
scfa_status scfa_count_chunked_pairs(const int32_t* q_idx, const int32_t* k_idx,
                                     const int32_t* q_hash, const int32_t* k_hash,
                                     int B, int H, int T, int chunk,
                                     unsigned long long* count, void* stream);

/* ----------------------------------------------------------------------------
 * Profiling hook: when set, every later attention call records
 * `start_event` (cudaEvent_t) on its stream right before launching the main
 * attention kernel (forward: the fused forward kernel; backward: the fused
 * backward kernel) and `stop_event` right after it, so the caller can time
 * that kernel alone with cudaEventElapsedTime. `which` = 0 sets the events of
 * forward kernels, 1 of backward kernels; NULL events switch the hook off.
 * Process-wide setting; not synchronised between host threads.
 * ------------------------------------------------------------------------- */
scfa_status scfa_set_kernel_events(int which, void* start_event, void* stop_event);

/* ----------------------------------------------------------------------------
 * Device status word of a workspace: SCFA_OK, or the first device-side error
 * (SCFA_ERR_TIMEOUT) raised by the last attention call that used `ws`.
 * Synchronises `stream`. Returns SCFA_ERR_CUDA if the copy fails.
 * ------------------------------------------------------------------------- */
scfa_status scfa_get_device_status(const void* ws, void* stream);

/* ----------------------------------------------------------------------------
 * Allocation-free QK-sparse forward (the paper has no counterpart: this is a
 * packaging variant for callers that cannot allocate device memory).
 *
 * Same operation, arguments, layouts and results as scfa_qk_fwd, without the
 * workspace: the forward's scratch (the live-tile metadata) is a
 * SCFA_NOALLOC_SCRATCH_BYTES array compiled into the library, which every GPU
 * that loads the library keeps until the process exits. For callers that may
 * not call cudaMalloc where they run attention: servers whose allocator hands
 * out one fixed pool at start-up and refuses later requests, and plugins in a
 * host framework that forbids allocation inside its callbacks. The call
 * allocates nothing (no cudaMalloc / cudaFree, no allocating library call).
 *
 * - Shapes whose forward scratch exceeds SCFA_NOALLOC_SCRATCH_BYTES (see
 *   scfa_attn_workspace_size(SCFA_MODE_QK, 0, ...)) are rejected on the host
 *   with SCFA_ERR_WORKSPACE before anything is launched.
 * - The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture begins.
 * - Every call shares the one array: calls that overlap on the GPU (e.g. on
 *   two unordered streams) race. Each call clears and rewrites all the
 *   scratch it reads.
 * - The device status word lives in the array: scfa_qk_fwd_noalloc_status
 *   synchronises `stream` and returns it (SCFA_OK, or the SCFA_ERR_* a
 *   device-side check or a pipeline timeout of the last call raised), as
 *   scfa_get_device_status does for a workspace.
 * ------------------------------------------------------------------------- */
#define SCFA_NOALLOC_SCRATCH_BYTES (16u << 20)

scfa_status scfa_qk_fwd_noalloc(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                const int32_t* q_idx, const int32_t* k_idx,
                                int B, int H, int Tq, int Tk, int D, float scale,
                                uint16_t* o, float* lse, void* stream);
scfa_status scfa_qk_fwd_noalloc_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SCFA_H */
