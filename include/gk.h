/*
 * gk.h -- C ABI of the shared-prefix paged decode-attention library (libgk.so).
 *
 * Storage follows "GraniKV: Asymmetric Granularity KV-Cache Paging for
 * Multi-Agent Systems with Long Shared Prefix": a shared prefix lives in a
 * contiguous HOT pool (Section 3.2) and each request's own tokens live in a
 * token-granular COLD pool (Section 3.3) reached through a block table whose
 * bookkeeping is the refcounted copy-on-write block manager of "Paged KV cache"
 * (How it works; Code).
 *
 * Conventions for every call:
 *  - The return value is a gk_status; GK_OK is 0.  On failure the pool's
 *    gk_last_error() text says what was wrong.  No C++ exception crosses the ABI.
 *  - "device" pointers are CUDA global-memory addresses owned by the caller;
 *    the library never frees them.  "host" pointers are ordinary memory.
 *  - Device work is enqueued on the caller's stream (a cudaStream_t passed as
 *    void*; NULL is the legacy default stream) and returns before it finishes.
 *  - Host metadata (block tables, refcounts, HOT free list, plans) is owned by
 *    the library.  A pool and its plans are not thread-safe.
 *  - bf16 is passed as raw 16-bit storage (void*); fp32 as float*.
 *
 * Layouts (all row-major, d = head_dim, Hkv = num_kv_heads, L = num_layers):
 *  - HOT K and V: [hot_tokens * L * Hkv * d] bf16 each.  A prefix at token base
 *    b with Lp tokens owns elements [b*L*Hkv*d, (b+Lp)*L*Hkv*d), laid out
 *    [L][Hkv][Lp][d], so the (layer, head) slice is one contiguous [Lp][d]
 *    block ("base + l*Lp*Hkv + h*Lp" of Section 3.2 with the allocator
 *    counting tokens).
 *  - COLD K and V: [L][cold_slots][Hkv][d] bf16 each; the slot of token t of a
 *    sequence is table[t / P] * P + t % P with P = cold_page_size
 *    ("Paged KV cache", How it works).
 *  - Queries [B][Hq][d] bf16, outputs [B][Hq][d] fp32, LSE [B][Hq] fp32
 *    (natural log).  Query head qh reads KV head qh / (Hq / Hkv).
 */
#ifndef GK_H_
#define GK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gk_status {
  GK_OK = 0,
  GK_ERR_INVALID = 1,        /* bad argument, unknown id, inconsistent sizes */
  GK_ERR_OOM = 2,            /* COLD pool out of blocks: preempt a sequence ("Paged KV cache", step 4) */
  GK_ERR_HOT_FULL = 3,       /* no HOT range fits: place the prefix in COLD (GraniKV Appendix B.10) */
  GK_ERR_CUDA = 4,           /* a CUDA runtime or driver call failed */
  GK_ERR_DEVICE_BOUNDS = 5,  /* a kernel met an out-of-range block or slot id and skipped it */
  GK_ERR_TIMEOUT = 6,        /* a kernel's bounded wait ran out; its results are not valid */
  GK_ERR_UNSUPPORTED = 7     /* geometry the kernels were not built for */
} gk_status;

typedef enum gk_backend {
  GK_BACKEND_DENSE = 0,      /* flat paged attention: every request reads its whole context */
  GK_BACKEND_CASCADE = 1     /* shared-prefix contraction + suffix gather + LSE merge */
} gk_backend;

typedef struct gk_pool gk_pool;
typedef struct gk_plan gk_plan;

typedef struct gk_pool_config {
  int32_t num_layers;
  int32_t num_q_heads;
  int32_t num_kv_heads;      /* 1..8, divides num_q_heads */
  int32_t head_dim;          /* 64 or 128; Hq/Hkv in {1,2,4} at 64, {1,2,4,5,8} at 128 */
  int64_t hot_tokens;        /* HOT capacity in tokens */
  int64_t cold_slots;        /* COLD capacity in token slots; a multiple of cold_page_size, at most 2^31 - 1 */
  int32_t cold_page_size;    /* P: tokens per COLD block (GraniKV uses 1; "Paged KV cache" uses 16) */
  int32_t reserved0;
  uint64_t seed;             /* 0: blocks are handed out 0,1,2,...; otherwise in a splitmix64-driven
                                Fisher-Yates order (shuffled physical slots) */
  void *hot_k, *hot_v;       /* device, layouts above; all four NULL = host-only pool (bookkeeping,
                                planning and dispatch work without a GPU) */
  void *cold_k, *cold_v;
} gk_pool_config;

/* ---- pool ------------------------------------------------------------------ */

/* Create a pool over caller-allocated storage.  Does not touch the device
 * contents.  *out is owned by the caller and freed with gk_pool_destroy. */
gk_status gk_pool_create(const gk_pool_config* cfg, gk_pool** out);
void gk_pool_destroy(gk_pool* pool);
/* Text of the pool's last error ("" if none); valid until the next call on the pool. */
const char* gk_last_error(const gk_pool* pool);
const char* gk_status_string(gk_status s);

/* ---- HOT pool (GraniKV Section 3.2; first-fit packing, Appendix B.8b) -------- */

/* Reserve prefix_len contiguous tokens: first fit over the address-ordered,
 * coalesced free list, else the bump pointer.  GK_ERR_HOT_FULL when nothing fits
 * (the caller keeps the prefix in COLD; no demotion, Appendix B.10). */
gk_status gk_prefix_alloc(gk_pool* pool, int64_t prefix_len, int64_t* hot_base);
/* Return a prefix's range; it merges with adjacent free ranges, and a range
 * ending at the bump pointer lowers it.  GK_ERR_INVALID for a range held by the
 * prefix cache below (those leave through gk_prefix_unref and eviction). */
gk_status gk_prefix_release(gk_pool* pool, int64_t hot_base);
gk_status gk_hot_stats(const gk_pool* pool, int64_t* bump_top, int64_t* free_ranges,
                       int64_t* free_tokens);

/* HOT prefix cache (GraniKV Section 3.2: a prefix's slab is reference counted;
 * at zero references it becomes evictable, and LRU eviction returns its range
 * to the free list, merged with its neighbours, under memory pressure).
 * key names the prefix's contents (the caller's hash of its tokens).
 * gk_prefix_acquire: a cached key gains a reference and *hit = 1 (its K/V are
 * already in the slab).  Otherwise a range is allocated as gk_prefix_alloc
 * does; while nothing fits, the slab idle longest (no reference since its last
 * use) is evicted and the allocation retried; the new slab has one reference
 * and *hit = 0 (the caller writes its K/V, gk_write_prefix_kv).  GK_ERR_HOT_FULL
 * when nothing fits even after every idle slab is evicted (those stay
 * evicted); GK_ERR_INVALID when key is cached with another prefix_len.  gk_prefix_unref drops one reference (GK_ERR_INVALID if
 * the key holds none).  Acquire and unref both count as a use for the LRU
 * order.  Host only. */
gk_status gk_prefix_acquire(gk_pool* pool, uint64_t key, int64_t prefix_len, int64_t* hot_base, int32_t* hit);
gk_status gk_prefix_unref(gk_pool* pool, uint64_t key);
/* Slabs in the cache, those of them idle, and the tokens the idle ones hold. */
gk_status gk_hot_cache_stats(const gk_pool* pool, int64_t* cached, int64_t* idle, int64_t* idle_tokens);

/* ---- COLD pool block manager ("Paged KV cache", How it works steps 1-4; Code) - */

gk_status gk_seq_create(gk_pool* pool, int32_t* seq);
/* Child shares every block of parent (refcount + 1); nothing is copied. */
gk_status gk_seq_fork(gk_pool* pool, int32_t parent, int32_t* child);
/* Drop one reference to every block of seq; blocks reaching zero return to the
 * free list (most recently freed is handed out first).  The id becomes invalid. */
gk_status gk_seq_release(gk_pool* pool, int32_t seq);
/* Borrow seq's block table (valid until the next call that changes the pool). */
gk_status gk_seq_table(const gk_pool* pool, int32_t seq, const int32_t** table, int32_t* nblocks,
                       int64_t* len);
/* Reserve one slot for each entry of seqs[0..n) in order (a sequence may repeat).
 * slot_mapping_out[i] receives the slot of that token.  When the token lands in
 * a shared partial block, the sequence first takes a fresh block; the pair
 * (shared, fresh) is appended to cow_pairs_out (capacity 2*n int32) and counted
 * in *n_cow.  GK_ERR_OOM: the first failing entry is reported in *n_done and the
 * entries before it stay applied (so the caller can preempt and retry the rest);
 * *n_done = n on success.  n_done may be NULL. */
gk_status gk_seq_append_slots(gk_pool* pool, int32_t n, const int32_t* seqs, int64_t* slot_mapping_out,
                              int32_t* n_cow, int32_t* cow_pairs_out, int32_t* n_done);
/* Block tables of n sequences as one row-major [n][max_blocks] int32 array
 * (rows padded with block 0 past each table's end; the padding is never read
 * because a request reads only its own length) and their lengths in tokens.
 * GK_ERR_INVALID if a table is longer than max_blocks. */
gk_status gk_seq_tables(const gk_pool* pool, int32_t n, const int32_t* seqs, int32_t max_blocks,
                        int32_t* table_out, int32_t* len_out);
gk_status gk_cold_stats(const gk_pool* pool, int64_t* free_blocks, int64_t* total_blocks);
/* A block's references: one per sequence holding it, plus one while it is cached. */
gk_status gk_block_refcount(const gk_pool* pool, int32_t block, int32_t* refcount);

/* COLD prefix caching ("Paged KV cache", How it works, step 5): each full block
 * is keyed by a hash of its parent block's key and its page_size token ids,
 *   key(block i) = H(key(block i - 1), tokens[i P .. i P + P)),  key(block -1) = 0,
 *   H(parent, t[0..P)) = h_P where h_0 = mix(parent + G) and h_{j+1} = mix(h_j XOR t_j * G)
 * (64-bit arithmetic, t_j taken as an unsigned 32-bit value, G = 0x9E3779B97F4A7C15,
 * mix = the output function of splitmix64).  The cache holds one reference on
 * each cached block, so a cached block outlives the sequences that used it;
 * when the free list is empty, taking a block first releases the least
 * recently used cached block that no sequence holds (creation of a cached
 * sequence and caching count as uses).
 * gk_seq_create_cached: a new sequence that starts with the longest chain of
 * cached blocks matching tokens[0..n) block by block (each gains a reference);
 * *n_cached = its length in tokens (a multiple of the page size; their K/V are
 * already in the pool).  The caller appends and writes the remaining tokens.
 * gk_seq_cache_blocks: caches seq's full blocks covering tokens[0..n) (at most
 * its length), skipping keys already cached and blocks cached under another
 * key; *n_new (may be NULL) = blocks added.  Host only. */
gk_status gk_seq_create_cached(gk_pool* pool, int32_t n_tokens, const int32_t* tokens, int32_t* seq, int64_t* n_cached);
gk_status gk_seq_cache_blocks(gk_pool* pool, int32_t seq, int32_t n_tokens, const int32_t* tokens, int32_t* n_new);
/* Blocks in the cache, and those of them no sequence holds (evictable). */
gk_status gk_cold_cache_stats(const gk_pool* pool, int64_t* cached_blocks, int64_t* evictable_blocks);

/* ---- KV writes (device) ---------------------------------------------------- */

/* reshape_and_cache ("Paged KV cache", step 1) for one layer: first copy every
 * copy-on-write pair's whole source block to its destination block, then write
 * token i's K and V [Hkv][d] to COLD slot d_slot_mapping[i].
 * d_slot_mapping: device int64 [n]; d_k, d_v: device bf16 [n][Hkv][d];
 * d_cow_pairs: device int32 [n_cow][2] (src, dst) or NULL when n_cow = 0.
 * Out-of-range slots or blocks are skipped and reported as GK_ERR_DEVICE_BOUNDS
 * by gk_device_error(). */
gk_status gk_append_kv(gk_pool* pool, void* stream, int32_t layer, int32_t n, const int64_t* d_slot_mapping,
                       const void* d_k, const void* d_v, int32_t n_cow, const int32_t* d_cow_pairs);
/* Write prefix tokens [t0, t0+n) of one layer into the HOT slab at hot_base
 * (a range from gk_prefix_alloc of prefix_len tokens).  d_k, d_v: device bf16
 * [n][Hkv][d] (token-major, the same input layout as gk_append_kv). */
gk_status gk_write_prefix_kv(gk_pool* pool, void* stream, int32_t layer, int64_t hot_base,
                             int64_t prefix_len, int64_t t0, int64_t n, const void* d_k, const void* d_v);

/* ---- one decode step ------------------------------------------------------- */

typedef struct gk_batch {
  int32_t num_requests;           /* B */
  int32_t max_blocks;             /* row stride of d_block_table */
  const int64_t* prefix_hot_base; /* host [B]: HOT base of the request's shared prefix, -1 = none */
  const int32_t* prefix_len;      /* host [B]: its length in tokens (0 when the base is -1) */
  const int32_t* suffix_len;      /* host [B]: tokens the request reads from COLD */
  const int32_t* d_block_table;   /* device [B][max_blocks]: COLD block ids of each request */
  const void* d_q;                /* device bf16 [B][Hq][d] (this layer's queries) */
  float* d_out;                   /* device fp32 [B][Hq][d] */
  float* d_lse;                   /* device fp32 [B][Hq], natural log; may be NULL */
  /* Optional fused append ("Paged KV cache", How it works step 2: reshape_and_cache),
   * both NULL or both set: this layer's new token of every request, device bf16
   * [B][Hkv][d].  Each request's last COLD token (suffix position suffix_len - 1,
   * reserved by gk_seq_append_slots and present in the block table) is then read
   * from here instead of the pool, and the decode writes it into the pool slot the
   * table gives -- what gk_append_kv would have written -- so no separate scatter
   * launch is needed.  Copy-on-write pairs of the step must be copied first
   * (gk_append_kv with n = 0).  Requests with suffix_len 0 are unaffected. */
  const void* d_new_k;
  const void* d_new_v;
} gk_batch;

typedef struct gk_plan_summary {
  int32_t num_requests;
  int32_t num_groups;             /* distinct HOT prefixes in the step */
  int32_t max_m_eff;              /* largest M_eff = B_g * Hq/Hkv over the groups (GraniKV Eq. 2) */
  int32_t prefix_ctas;            /* cascade prefix-kernel CTAs per layer */
  int32_t suffix_ctas;            /* suffix-gather CTAs per layer */
  int32_t dense_ctas;             /* flat-gather CTAs per layer */
  int32_t num_partials;           /* partial (O, LSE) states the merge combines per layer */
  int32_t dense_merge;            /* 1 if gk_decode_dense launches a merge (a request spans CTAs) */
  int64_t prefix_bytes;           /* algorithmic bytes per layer: HOT K+V read once per group */
  int64_t prefix_flops;           /* 4 * B_g * Hq * Lp * d summed over groups */
  int64_t suffix_bytes;           /* COLD K+V of all suffixes */
  int64_t dense_bytes;            /* K+V of every request's whole context */
  int32_t cascade_split;          /* 1: gk_decode_cascade runs the prefix items (prefix_ctas SMs) and
                                     the suffix gather (suffix_ctas SMs) side by side in one launch;
                                     0: one after the other, each over every SM */
  int32_t prefix_tiles_per_item;  /* 128-key tiles of the longest prefix work item */
  int32_t prefix_kernel;          /* prefix work items: GK_PREFIX_TENSOR or GK_PREFIX_WARP */
  int32_t prefix_rows_per_item;   /* stacked query rows per prefix work item: 256 or 128 */
  int32_t prefix_row_groups;      /* warp items: 16-row groups of the fullest item, rounded up to
                                     1, 2, 4 or 8; 0 for tensor-core items */
  int32_t prefix_ctas_gather;     /* split plans: 1 when the prefix CTAs also gather a share of the
                                     suffix after their items, 0 when only the other CTAs gather */
  int32_t sm_slots;               /* split plans: 1 when the slots are planned per SM from the pool's
                                     SM speeds (gk_pool_set_sm_speeds), 0 when CTA b takes slot b */
} gk_plan_summary;

/* Plan one decode step: group requests by HOT prefix (stable, first appearance),
 * split the prefix contraction and the gathers into balanced CTA work lists,
 * and lay out the partial states.  The grouping is GraniKV Section 3.6's: the
 * requests that share one HOT prefix stack their B_g * Hq/Hkv query rows per KV
 * head into one matrix (M_eff of Eq. 2, which also drives gk_dispatch).  Depends
 * only on the host arrays of the batch, which every layer of a step shares, so
 * one plan serves every layer of the step.  When the pool has device
 * storage the plan's tables are copied to the device on `stream` and scratch
 * for the partial states is allocated (owned by the plan).  Calls that use a
 * plan must be ordered on one stream. */
gk_status gk_plan_build(gk_pool* pool, const gk_batch* batch, void* stream, gk_plan** out);
/* Re-plan an existing plan for the next step (same pool), reusing its host and
 * device buffers when they are large enough.  Must be called on the stream the
 * plan's earlier work was enqueued on: the new tables are copied after that work. */
gk_status gk_plan_update(gk_plan* plan, const gk_batch* batch, void* stream);
/* Frees the plan's buffers; its enqueued work must have completed. */
void gk_plan_destroy(gk_plan* plan);
gk_status gk_plan_info(const gk_plan* plan, gk_plan_summary* out);
/* The gather partition of a plan (its host copy): which tokens each CTA gathers.
 * dense = 0: the cascade suffix partition, 1: the flat one.  The counts come
 * first: *n_ctas gather CTAs and *n_segs segments.  Then, when begin and segs
 * are not NULL, begin[0 .. n_ctas] receives the offsets of each CTA's
 * segments (CTA b: [begin[b], begin[b + 1])) and segs[4 * i .. 4 * i + 3]
 * segment i: request, first token, end token (in the request's own order: the
 * dense partition counts the HOT prefix first), and the partial state it
 * writes (-1: the request's output).  Host only; GK_ERR_INVALID for a NULL
 * plan or count pointer. */
gk_status gk_plan_segments(const gk_plan* plan, int32_t dense, int32_t* n_ctas, int32_t* n_segs, int32_t* begin,
                           int32_t* segs);

/* Flat paged attention (the dense backend): each request attends its prefix
 * (read from HOT, once per request) and its COLD suffix in one online-softmax
 * pass; writes d_out and d_lse of the batch for this layer.  This is the decode
 * of "Paged KV cache", How it works step 3 (the kernel walks each sequence's
 * block table and reads its K/V in place, token slot by slot), and the
 * baseline GraniKV compares against (Section 4, the SGLang default: every
 * request re-reads the shared prefix).  A request split over several CTAs is
 * merged by GraniKV Eq. 1 (gk_plan_summary.dense_merge). */
gk_status gk_decode_dense(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch,
                          const gk_plan* plan);
/* Cascade backend: (a) per prefix group and KV head, all query rows sharing the
 * prefix are stacked into one QK^T / PV contraction on the tensor cores, read
 * once from HOT (GraniKV Section 2.3, shared-prefix matmul; Section 3.5);
 * (b) the suffix is gathered through the block table; (c) the partial states
 * are merged by log-sum-exp (GraniKV Eq. 1).  A split plan
 * (gk_plan_summary.cascade_split) runs (a) and (b) in one launch on disjoint
 * SMs, then (c); otherwise (a), (b), (c) are three launches.  Both give the
 * same bits as the three stage calls below. */
gk_status gk_decode_cascade(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch,
                            const gk_plan* plan);
/* Allocation-free dense decode.  No counterpart in the paper: it exists for
 * callers that cannot allocate device memory while serving -- an engine that
 * hands all free HBM to its KV pool at start-up, or one whose allocator is
 * owned by a framework that rejects allocations made outside it.  Same result
 * as gk_plan_build + gk_decode_dense on this batch (see those calls for the
 * arguments), but the work tables and split-K partial states live in one
 * 8 MiB array compiled into libgk (every GPU that loads the library keeps it
 * until the process exits) and no call allocates device or pinned memory.
 *  - The first call on each device looks the array's address up
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  The pool's device must be the current device
 *    (else GK_ERR_INVALID).
 *  - Each call copies its work tables from host memory that it frees on
 *    return, so on a stream that is capturing it does nothing and returns
 *    GK_ERR_UNSUPPORTED.
 *  - A batch whose tables and partial states exceed 8 MiB is refused with
 *    GK_ERR_INVALID (gk_last_error gives the bytes needed); use the plan path.
 *  - Every call reuses the same array: calls that overlap on the GPU (two
 *    streams, or two pools on one device) race and give wrong results; order
 *    them on one stream.  Nothing in the array needs to start at zero.
 *  - The pool must already have done device work (any KV write), which is when
 *    its error word is created; otherwise GK_ERR_INVALID. */
gk_status gk_decode_dense_static(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch);
/* Stages (a) and (b) of gk_decode_cascade as the plan arranges them: one split
 * launch, or the prefix then the suffix kernel.  gk_decode_cascade is exactly
 * this followed by gk_cascade_merge. */
gk_status gk_cascade_levels(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch,
                            const gk_plan* plan);
/* The three stages of gk_decode_cascade, for callers that time them or run
 * (a) and (b) on two streams: the prefix and suffix stages write disjoint
 * partial states, and the merge must follow both.  They run the plan's work
 * lists (for a split plan: prefix_ctas long items, suffix_ctas gather CTAs). */
gk_status gk_cascade_prefix(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch,
                            const gk_plan* plan);
gk_status gk_cascade_suffix(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch,
                            const gk_plan* plan);
gk_status gk_cascade_merge(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch,
                           const gk_plan* plan);

/* ---- per-step dispatch (GraniKV Section 3.6, Eq. 2) -------------------------- */

typedef struct gk_cost_model {
  double c_flat_us;               /* fixed cost of the dense backend per layer */
  double bw_flat_gbs;             /* its sustained gather bandwidth */
  double c_cascade_us;            /* fixed cost of the cascade backend per layer */
  double bw_prefix_gbs;           /* bandwidth bound of the prefix contraction (HOT reads) */
  double bw_suffix_gbs;           /* suffix gather bandwidth over every SM */
  double c_merge_us;              /* merge cost per (request, query head) */
  double prefix_tile_us;          /* one 128-key tile of a 256-row prefix work item on one SM */
  double prefix_item_us;          /* fixed cost of a prefix work item (of each wave of them) */
  double gather_sm_gbs;           /* suffix gather bandwidth one SM sustains (split plans) */
  double c_gather_us;             /* fixed cost of a separate suffix-gather launch (sequential plans) */
  double prefix_tile_split_us;    /* prefix_tile_us for an item of a split plan, which runs beside a
                                     gather that keeps HBM busy (its K/V tiles wait longer) */
  double warp_tile_us;            /* one 128-key tile of a warp-MMA prefix item alone: the part that does
                                     not grow with its rows ... */
  double warp_group_us;           /* ... plus this much per group of 16 rows (rounded up to 1, 2, 4, 8) */
  double warp_item_us;            /* fixed cost of a warp-MMA prefix item (of each wave of them) */
  double warp_split_ratio;        /* a warp item's tile beside the gather of a split plan, over alone */
  double prefix_cta_ramp_us;      /* split plans: a prefix CTA starts gathering this long after its item */
  double prefix_cta_gather_ratio; /* ... and gathers at this fraction of a gather-only CTA's rate */
  double c_merge_state_us;        /* merge cost per partial state of a request (a merge warp's round trips) */
  double prefix_item_split_us;    /* fixed cost of a tensor-core prefix item inside a split launch */
  double warp_item_split_us;      /* fixed cost of a warp-MMA prefix item inside a split launch */
  double prefix_item_crowd_us;    /* ... plus this much per prefix item of the launch (their first loads
                                     contend with each other) */
  double split_gather_ratio_tensor; /* gather rate in a split launch of tensor-core items, over gather_sm
                                     (that launch's 320-thread blocks hold the gather to fewer registers) */
  double c_gather_split_us;       /* fixed cost of the gather inside a split launch: when its gather-only
                                     CTAs start (c_gather_us is the stand-alone gather launch's) */
  double split_tensor_us;         /* what a split launch of tensor-core items costs over one of warp-MMA
                                     items (its 320-thread blocks, tensor memory, tensor maps) */
} gk_cost_model;

/* Predict both backends for the plan and pick the smaller:
 *   T_dense   = c_flat + dense_bytes / bw_flat
 *   T_cascade = c_cascade + T_levels + c_merge * B * Hq + c_merge_state * num_partials / B
 * with C = gk_plan_summary.prefix_tiles_per_item key tiles per prefix item,
 * (tile, tile_split, item) = (prefix_tile, prefix_tile_split, prefix_item) for
 * tensor-core items and, for warp-MMA items (gk_plan_summary.prefix_kernel),
 * tile = warp_tile + R * warp_group with R = gk_plan_summary.prefix_row_groups,
 * tile_split = warp_split_ratio * tile and item = warp_item; item_split =
 * (prefix_item_split or warp_item_split) + prefix_item_crowd * prefix_ctas is an
 * item's fixed cost in a split launch; and
 *   sequential plan (W = ceil(prefix_ctas / SMs) waves of prefix items):
 *     T_levels = max(prefix_bytes / bw_prefix, W * (C * tile + item))
 *                + c_gather + suffix_bytes / bw_suffix
 *   split plan (see gk_plan_summary.cascade_split; it = C * tile_split + item_split,
 *   n = prefix_ctas, A = SMs - n gather-only CTAs, G = suffix_bytes / gather_sm
 *   the gather's SM-time (gather_sm times split_gather_ratio_tensor for
 *   tensor-core items), e = prefix_cta_gather_ratio, r = prefix_cta_ramp):
 *     T_gather = (G + A * c_gather + n * e * (it + r)) / (A + n * e)
 *                when the prefix CTAs gather too (gk_plan_summary.prefix_ctas_gather),
 *              = c_gather + G / A otherwise, and at least c_gather + suffix_bytes / bw_suffix;
 *     T_levels = max(it, T_gather, (suffix_bytes + prefix_bytes) / bw_suffix)
 *   (gather-only CTAs start after c_gather, prefix CTAs r after their items,
 *   and all end together; the gather is held to HBM as a whole, and so is the launch).
 * A plan without prefix work has no prefix term, one without suffix work no
 * gather term.  GraniKV's M_eff (Eq. 2) enters through the items: a group of
 * M_eff stacked rows gives ceil(M_eff / rows per item) items per KV head and key
 * split.  The plan has already chosen the prefix kernel and the arrangement
 * with the smallest predicted time (GraniKV Section 3.6's routing between its
 * two prefix kernels, with the threshold replaced by the measured model), so
 * this call completes the three-way choice: flat, cascade over tensor-core
 * items, cascade over warp-MMA items.  Dense is chosen only when strictly
 * faster; a negative prediction (a negative c_cascade on a tiny step) counts as
 * zero.  Host only. */
gk_status gk_dispatch(const gk_pool* pool, const gk_plan* plan, gk_backend* choice, double* t_dense_us,
                      double* t_cascade_us);
gk_status gk_cost_model_set(gk_pool* pool, const gk_cost_model* cm);

/* Cascade arrangement of the plans the pool builds from now on.
 *  GK_CASCADE_AUTO (default): split when the cost model predicts it faster.
 *  GK_CASCADE_SEQUENTIAL: prefix items over every SM, then the suffix gather.
 *  GK_CASCADE_SPLIT: prefix items beside the suffix gather in one launch, with
 *    tiles_per_item 128-key tiles per item (0: the cost model's best split).
 *    A step without prefix or suffix work, or whose items would leave no SM
 *    for the gather, is planned sequentially.
 * The choice changes the work lists and the partial states, not the
 * attention computed.  Host only.  GK_ERR_INVALID for an unknown mode or a
 * negative tiles_per_item. */
typedef enum gk_cascade_mode {
  GK_CASCADE_AUTO = 0,
  GK_CASCADE_SEQUENTIAL = 1,
  GK_CASCADE_SPLIT = 2
} gk_cascade_mode;
gk_status gk_pool_set_cascade_mode(gk_pool* pool, gk_cascade_mode mode, int32_t tiles_per_item);

/* How the stand-alone gathers (the flat backend, and the suffix of a sequential
 * cascade plan) split their tokens over CTAs, in the plans the pool builds from
 * now on (a split cascade plan always gives each SM one slot of the stream).
 *  GK_PARTITION_STREAM (default): the requests' tokens as one stream cut into
 *    equal quotas (at least 64 tokens, multiples of 16) over at most one CTA per
 *    SM; a quota that crosses a request boundary yields one segment per request.
 *  GK_PARTITION_PER_REQUEST: Tangram's ahead-of-time partitioning (Algorithm 1,
 *    with requests as its head groups and their tokens as budgets): target
 *    tau = max(1, ceil(total / SMs)); request r gets S_r = max(1, ceil(n_r / tau))
 *    segments of its own tokens, the first n_r mod S_r of them one token longer,
 *    one CTA each (so up to SMs + B CTAs, in waves).
 * The choice changes the work lists and the partial states, not the attention
 * computed.  Host only.  GK_ERR_INVALID for an unknown value. */
typedef enum gk_gather_partition {
  GK_PARTITION_STREAM = 0,
  GK_PARTITION_PER_REQUEST = 1
} gk_gather_partition;
gk_status gk_pool_set_gather_partition(gk_pool* pool, gk_gather_partition partition);

/* Which kernel runs the shared-prefix level of the cascade in the plans the
 * pool builds from now on.  GraniKV Section 3.5 pairs two: the shared-prefix
 * matmul ("GKV-dense": every row sharing the prefix stacked into one
 * tensor-core contraction) and the cascade backend's level-0 kernel
 * ("GKV-cascade": a FlashAttention-style tiled online softmax that reads the
 * prefix once), and Section 3.6 routes between them on M_eff.
 *  GK_PREFIX_AUTO (default): per step, the one whose cascade the cost model
 *    predicts faster, the tensor-core items only when predicted at least 10 %
 *    faster (their predictions at small steps run low) and never when every
 *    group stacks at most 64 rows per KV head (M_eff <= 64, which a tensor-core
 *    item pads to 256).
 *  GK_PREFIX_TENSOR: tcgen05 items of 256 stacked rows (two 128-row tiles).
 *  GK_PREFIX_WARP: warp-MMA items of 128 stacked rows (8 warps x 16 rows), no
 *    tensor memory; meant for small M_eff.
 * Either kind writes the same partial states (one per request, query head and
 * key split); the arrangement (gk_pool_set_cascade_mode) applies to both.
 * Host only.  GK_ERR_INVALID for an unknown value. */
typedef enum gk_prefix_kernel {
  GK_PREFIX_AUTO = 0,
  GK_PREFIX_TENSOR = 1,
  GK_PREFIX_WARP = 2
} gk_prefix_kernel;
gk_status gk_pool_set_prefix_kernel(gk_pool* pool, gk_prefix_kernel kernel);
/* SM-aware split launches (no counterpart in the pages: they assume a uniform
 * GPU).  On GB300 some SMs gather COLD rows 5-10 % slower than others, the same
 * from launch to launch, so equal gather slots end at different times and the
 * launch waits for the slowest.  With SM speeds set, split plans size each
 * SM's slot by its speed, give the prefix items to the slowest SMs (the longest
 * item to the slowest), and the split launch's CTA on SM s takes the slot
 * planned for s (an atomic claim per launch; a slot already taken sends the CTA
 * to the next free one, so every slot is run exactly once whatever SMs the
 * CTAs land on).  The results are the same attention whichever slots run where;
 * the partial-state boundaries, and so the last bits, follow the speeds.
 *  - gk_pool_set_sm_speeds: n speeds (relative; any positive scale) for SM ids
 *    0 .. n-1, n = the device's SM count (152 for a pool without device
 *    storage, which plans as for one GB300); n = 0 clears them (plans as
 *    without).  Host only.  GK_ERR_INVALID for another n or a speed that is not
 *    positive and finite.  Plans built before keep their slots.
 *  - gk_pool_get_sm_speeds: *n = the count set (0 when none) and, when speeds is
 *    not NULL, the speeds (normalised to mean 1).
 *  - gk_sm_speeds_measure: runs the plan's gather `reps` times on `stream`,
 *    each launch alone, with each CTA's SM id and times recorded by the kernel:
 *    a split plan's own launch (gk_cascade_levels; a slot's rate counts its
 *    gather, after its item, and prefix and gather-only slots are each scaled
 *    to their own mean in the launch) or a sequential plan's stand-alone suffix
 *    gather (gk_cascade_suffix).  An SM's speed is the median over the launches
 *    of the scaled tokens per us of the slots it ran (slots with under a quarter
 *    of the largest one's tokens are left out), normalised to mean 1; SMs
 *    without a sample get 1.  Installs the speeds in the pool and, when speeds
 *    is not NULL, writes them there (dev SM count entries).  The launches write
 *    the plan's partial states (and the outputs of requests one CTA covers) and,
 *    with a fused append, the step's tokens, as the decode calls do.  Blocking;
 *    allocates and frees its own 32 bytes per CTA of device memory.
 *    GK_ERR_INVALID when the plan has no suffix segments or reps is not in
 *    1 .. 64. */
gk_status gk_pool_set_sm_speeds(gk_pool* pool, const float* speeds, int32_t n);
gk_status gk_pool_get_sm_speeds(const gk_pool* pool, float* speeds, int32_t* n);
gk_status gk_sm_speeds_measure(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch,
                               const gk_plan* plan, int32_t reps, float* speeds);
gk_status gk_cost_model_get(const gk_pool* pool, gk_cost_model* cm);
/* Re-fit the cost model on this GPU (GraniKV Section 3.6: the routing rule stays
 * and its numbers are re-fit per GPU; Appendix B.4b's sweep).  Times, with CUDA
 * events on `stream` and L2 emptied before every launch, the flat backend, the
 * suffix gather, the merge, tensor-core and warp-MMA prefix items of several
 * key-tile counts (warp items with 1, 2 and 8 groups of 16 rows), the gather
 * beside long items, and whole cascades, on layer 0 of this pool with a
 * synthetic batch of one shared prefix; fits each gk_cost_model term by least
 * squares (the flat backend's and the suffix gather's terms by relative error,
 * so that the smallest steps count as much as the largest); installs the model in the pool; and, if json_out is not
 * NULL, writes it to that file in gk_cost_model_load's format with the
 * measured points under "measured".  Blocking; a few seconds.
 *  - The pool needs device storage; its K/V contents are read as they are (the
 *    timings do not depend on the values) and never written.  Cases that do not
 *    fit its free HOT and COLD space are skipped; with at least 16384 free HOT
 *    tokens and 262144 free COLD token slots every case runs.  GK_ERR_INVALID
 *    when too few cases fit to fit every term (the model is left as it was).
 *  - HOT ranges, sequences and COLD blocks are taken from the pool's allocators
 *    and given back: afterwards the same blocks are free, though the order in
 *    which free blocks are handed out may differ.  The pool's cascade mode,
 *    prefix kernel and gather partition are restored.
 *  - The calibration's own scratch (queries, outputs, tables, 512 MiB to empty
 *    L2) is allocated with cudaMalloc and freed before returning.
 *  - The terms of the split arrangement (prefix_tile_split_us / prefix_tile_us,
 *    warp_split_ratio, prefix_item_split_us, warp_item_split_us,
 *    prefix_item_crowd_us, prefix_cta_ramp_us, gather_sm_gbs,
 *    split_gather_ratio_tensor, c_gather_split_us, split_tensor_us) and c_cascade_us are fitted
 *    to the whole cascades it times (sequential and split plans, forced and as
 *    the planner arranges them, both prefix kernels, a grid of steps with
 *    16..512-token suffixes, that grid planned again with the first fit): a
 *    coordinate search over candidate values of each term that minimises the
 *    largest plus half the mean relative error of T_cascade, the other terms
 *    held at their own fits.  c_cascade_us may come out negative
 *    (the terms timed alone each carry a launch that the cascade overlaps).
 *    prefix_cta_gather_ratio is set to 1: once it starts, a prefix CTA gathers
 *    at a gather-only CTA's rate. */
gk_status gk_calibrate(gk_pool* pool, void* stream, const char* json_out);
/* Same as gk_cost_model_set from JSON text: {"c_flat_us": .., "bw_flat_gbs": ..,
 * "c_cascade_us": .., "bw_prefix_gbs": .., "bw_suffix_gbs": .., "c_merge_us": ..,
 * "prefix_tile_us": .., "prefix_item_us": .., "gather_sm_gbs": .., "c_gather_us": ..,
 * "prefix_tile_split_us": .., "warp_tile_us": .., "warp_group_us": .., "warp_item_us": ..,
 * "warp_split_ratio": .., "prefix_cta_ramp_us": .., "prefix_cta_gather_ratio": ..,
 * "c_merge_state_us": .., "prefix_item_split_us": .., "warp_item_split_us": ..,
 * "prefix_item_crowd_us": .., "split_gather_ratio_tensor": .., "c_gather_split_us": ..,
 * "split_tensor_us": ..}.
 * Keys left out keep their current values; other keys are skipped. */
gk_status gk_cost_model_load(gk_pool* pool, const char* json);

/* ---- device error word -------------------------------------------------------- */

/* Synchronize `stream`, read and clear the pool's device error word.  *code is
 * GK_OK, GK_ERR_DEVICE_BOUNDS or GK_ERR_TIMEOUT; the return value reports
 * failures of the read itself. */
gk_status gk_device_error(gk_pool* pool, void* stream, int32_t* code);

#ifdef __cplusplus
}
#endif

#endif /* GK_H_ */
