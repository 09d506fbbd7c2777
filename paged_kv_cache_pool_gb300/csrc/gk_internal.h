// Internal declarations shared by the host runtime (.cpp) and the kernel
// launchers (.cu) of libgk.  Nothing here is part of the public ABI.
#pragma once

#include <cuda_runtime_api.h>

#include <cstdint>
#include <map>
#include <set>
#include <string>
#include <unordered_map>
#include <utility>
#include <vector>

#include "../../include/gk.h"

namespace gk {

// ---- HOT allocator (GraniKV Section 3.2, Appendix B.8b) ----------------------
struct HotAllocator {
  int64_t capacity = 0;
  int64_t top = 0;                                  // bump pointer
  std::vector<std::pair<int64_t, int64_t>> free;    // address-ordered [start, end), coalesced
  std::unordered_map<int64_t, int64_t> live;        // base -> length

  bool alloc(int64_t n, int64_t* base);
  bool release(int64_t base);
};

// HOT prefix cache (GraniKV Section 3.2): a slab per caller key, reference
// counted; a slab whose count drops to zero stays cached but evictable, and an
// allocation that does not fit evicts evictable slabs, least recently used
// first, until it does.
struct HotCacheEntry {
  int64_t base = 0, lp = 0;
  int64_t refs = 0;
  uint64_t last_use = 0;
};
struct HotCache {
  std::unordered_map<uint64_t, HotCacheEntry> entries;  // key -> slab
  std::unordered_map<int64_t, uint64_t> key_of;         // base -> key
  std::set<std::pair<uint64_t, uint64_t>> idle;         // (last use, key) of slabs with no reference
  uint64_t tick = 0;
};

// ---- COLD block manager ("Paged KV cache", How it works; Code) ---------------
struct Sequence {
  std::vector<int32_t> table;
  int64_t len = 0;
  bool alive = false;
};

struct BlockManager {
  int32_t page = 1;
  std::vector<int32_t> free_stack;   // back() is handed out next
  std::vector<int32_t> ref;
  std::vector<Sequence> seqs;
  std::vector<int32_t> free_seq_ids;
  // Prefix caching ("Paged KV cache", How it works, step 5): full blocks keyed
  // by a chained hash of their tokens.  The cache holds one reference on each
  // cached block; when the free stack is empty, take() releases the least
  // recently used cached block that only the cache still holds.
  std::unordered_map<uint64_t, int32_t> cache;        // block hash -> block
  std::unordered_map<int32_t, uint64_t> cached_hash;  // block -> its hash
  std::unordered_map<int32_t, uint64_t> cached_use;   // block -> last use
  std::set<std::pair<uint64_t, int32_t>> lru;         // (last use, block) of every cached block
  uint64_t tick = 0;

  void init(int64_t n_blocks, int32_t page_size, uint64_t seed);
  int32_t take();                    // -1 when empty and nothing is evictable
  void drop(int32_t b);
  void touch(int32_t b);             // a cached block was used now
};
// hash of a full block of page_size tokens under its parent block's hash (0 for the first block)
uint64_t block_hash(uint64_t parent, const int32_t* tokens, int32_t page_size);

// ---- geometry-dependent kernel limits ---------------------------------------
constexpr int kPrefixTileM = 128;    // stacked query rows per tensor-core tile
constexpr int kPrefixRowsPerCta = 2 * kPrefixTileM;  // two Q tiles per prefix CTA
constexpr int kPrefixTileN = 128;    // prefix keys per tile
constexpr int kPrefixWarpRows = 128; // stacked query rows per warp-MMA prefix item (8 warps x 16)
constexpr int kGatherT = 16;         // tokens per gather pipeline stage
constexpr int kMaxKvHeads = 8;

struct DeviceInfo {
  int device = -1;
  int num_sms = 152;
  bool queried = false;
};

struct Pool {
  gk_pool_config cfg{};
  bool has_device = false;
  HotAllocator hot;
  HotCache hot_cache;
  BlockManager cold;
  gk_cost_model cost{};
  gk_cascade_mode cascade_mode = GK_CASCADE_AUTO;
  int32_t cascade_tiles = 0;         // GK_CASCADE_SPLIT: tiles per item (0 = best predicted)
  gk_gather_partition gather_partition = GK_PARTITION_STREAM;  // stand-alone gathers' work split
  gk_prefix_kernel prefix_kernel = GK_PREFIX_AUTO;             // which prefix item the plans use
  std::string last_error;
  DeviceInfo dev;
  int32_t* d_error = nullptr;        // device error word (allocated on first device use)
  // SM-aware split launches: each SM's gather speed relative to the mean (empty: not
  // used), the per-slot claim words of the split launch and the launch counter that
  // tags a claim to one launch
  std::vector<float> sm_speed;
  uint32_t* d_slot_claim = nullptr;  // [dev.num_sms] (allocated on first device use)
  uint32_t split_epoch = 0;
  int32_t g() const { return cfg.num_q_heads / cfg.num_kv_heads; }
};

// ---- plan ---------------------------------------------------------------------
// Device-side records (plain structs, copied with one H2D memcpy).
struct PrefixGroupDev {
  int32_t lp;          // prefix length (keys)
  int32_t m;           // stacked rows B_g * g
  int32_t req_base;    // offset into prefix_reqs
  int32_t nsplit;      // splits over the prefix keys
  int32_t split_tiles; // key tiles (of kPrefixTileN) per split
  int32_t tmap_index;  // first of the group's 2 tensor maps: K, V (128-key box)
  int32_t pad0, pad1;
};

struct PrefixItemDev {  // one CTA of the tensor-core prefix kernel
  int32_t group;
  int32_t mblock;      // 256-row block of the stacked Q rows
  int32_t head;
  int32_t split;       // first key split of the item
  int32_t splits;      // consecutive key splits it covers (> 1 only for a one-Q-tile row block)
  int32_t pad0;
};

struct SegmentDev {     // one contiguous run of one request's tokens inside a gather CTA
  int32_t req;
  int32_t t0, t1;      // token range in the request's own order (dense: prefix then suffix)
  int32_t entry;       // partial-state index, or -1 = write the final output directly
};

struct RequestDev {
  int64_t hot_base;    // -1 = no HOT prefix
  int32_t lp;          // HOT prefix tokens (0 when none)
  int32_t slen;        // COLD tokens
  int32_t entry_cas;   // first partial entry in the cascade layout
  int32_t n_entry_cas;
  int32_t entry_dense;
  int32_t n_entry_dense;
  int32_t group;       // HOT prefix group, -1 = none
  int32_t pad0;
};

struct Plan {
  Pool* pool = nullptr;
  int32_t B = 0;
  gk_plan_summary summary{};
  // host mirrors
  std::vector<PrefixGroupDev> groups;
  std::vector<int64_t> group_hot_base;
  std::vector<int32_t> prefix_reqs;      // requests of each group, concatenated
  std::vector<PrefixItemDev> prefix_items;
  std::vector<RequestDev> reqs;
  std::vector<int32_t> suf_seg_begin;    // [suffix_ctas + 1]
  std::vector<SegmentDev> suf_segs;
  std::vector<int32_t> dense_seg_begin;  // [dense_ctas + 1]
  std::vector<SegmentDev> dense_segs;
  int32_t n_entries_cas = 0, n_entries_dense = 0;
  bool dense_needs_merge = false;
  std::vector<int64_t> group_bytes, group_flops;
  // device copies
  void* d_buf = nullptr;
  void* h_stage = nullptr;               // pinned staging of the device tables
  cudaEvent_t upload_done = nullptr;     // the last upload has left h_stage
  bool staged = false;
  size_t d_bytes = 0;
  size_t off_groups = 0, off_prefix_reqs = 0, off_prefix_items = 0, off_reqs = 0;
  size_t off_suf_begin = 0, off_suf_segs = 0, off_dense_begin = 0, off_dense_segs = 0;
  size_t off_tmaps = 0;
  float* d_part_o = nullptr;             // [entries][Hq][d]
  float* d_part_l = nullptr;             // [entries][Hq] (log2 domain)
  size_t part_entries = 0;
  bool uploaded = false;
  bool split = false;                    // cascade arrangement: prefix items and suffix gather side by side
  int32_t prefix_kind = 0;               // 0: tensor-core items (256 rows), 1: warp-MMA items (128 rows)
  // split plans sized by the pool's SM speeds: slot_of_sm[s] = the work slot (prefix
  // item and gather slot) planned for SM s; empty: CTA b takes slot b
  std::vector<int32_t> slot_of_sm;
  size_t off_slot_of_sm = 0;
};

// host half of gk_plan_build: grouping, work lists and partial-state layout (no device work)
gk_status build_host_plan(Pool* p, const gk_batch* b, Plan* pl);

// ---- cost model (plan.cpp) ----------------------------------------------------------
struct SplitTime {
  double t;       // predicted levels time of the split launch, us
  double share;   // a prefix CTA's gather tokens over a gather-only CTA's
};
SplitTime split_time(const gk_cost_model& cm, int num_sms, int64_t n_pre, double it, double S, double P,
                     bool gather, double gather_sm_gbs);
double merge_us(const gk_cost_model& cm, int32_t B, int32_t Hq, int64_t partials);
// the model's cascade and flat times for a plan (gk_dispatch's predictions)
void predict_plan(const gk_cost_model& cm, int num_sms, int32_t Hq, const Plan& pl, double* t_dense_us,
                  double* t_cascade_us);

// ---- status helpers -------------------------------------------------------------
gk_status fail(Pool* p, gk_status s, const std::string& msg);
gk_status cuda_fail(Pool* p, int err, const char* what);
gk_status ensure_device(Pool* p);

// ---- kernel launchers (.cu) --------------------------------------------------------
struct LaunchCommon {
  const gk_pool_config* cfg;
  int32_t* d_error;
  int num_sms;
  // split launches of plans with SM-indexed slots: the claim words and this launch's tag
  uint32_t* slot_claim = nullptr;
  uint32_t epoch = 0;
  // stand-alone gathers: per-CTA SM id, start and end (%globaltimer), when not null
  unsigned long long* gather_stamps = nullptr;
  // split launches: per-slot SM id, start, start of its gather and end, when not null
  unsigned long long* split_stamps = nullptr;
};

int launch_cow_copy(const LaunchCommon& lc, void* stream, int32_t layer, int32_t n_cow,
                    const int32_t* d_pairs);
int launch_scatter(const LaunchCommon& lc, void* stream, int32_t layer, int32_t n,
                   const int64_t* d_slots, const void* d_k, const void* d_v);
int launch_write_prefix(const LaunchCommon& lc, void* stream, int32_t layer, int64_t base,
                        int64_t lp, int64_t t0, int64_t n, const void* d_k, const void* d_v);

// gather attention over COLD (and HOT when dense) tokens; writes partials or outputs
int launch_gather(const LaunchCommon& lc, void* stream, int32_t layer, const gk_batch* b,
                  const Plan* plan, bool dense);
int launch_merge(const LaunchCommon& lc, void* stream, const gk_batch* b, const Plan* plan,
                 bool dense);
// the plan's prefix items as one launch (tensor-core or warp-MMA items, as planned)
int launch_prefix(const LaunchCommon& lc, void* stream, int32_t layer, const gk_batch* b,
                  const Plan* plan);
int launch_prefix_warp(const LaunchCommon& lc, void* stream, int32_t layer, const gk_batch* b,
                       const Plan* plan);
// split arrangement: the prefix items and the suffix gather of one layer in one
// launch, on disjoint SMs (the merge follows as its own launch)
int launch_cascade_split(const LaunchCommon& lc, void* stream, int32_t layer, const gk_batch* b,
                         const Plan* plan);
// resident gather CTAs per SM for the pool's geometry (no device query, so
// host-only pools plan identically)
int gather_ctas_per_sm(const gk_pool_config* cfg);
// encode the tensor maps of a plan's prefix groups into host memory (128 B each,
// 2 per group: K and V with a 128-key box for the prefix kernel)
int encode_prefix_tmaps(const gk_pool_config* cfg, const Plan* plan, std::vector<uint8_t>* out);
size_t tmap_bytes();

}  // namespace gk

struct gk_pool {
  gk::Pool impl;
};
struct gk_plan {
  gk::Plan impl;
};
