// Host runtime of libgk: pool lifetime, the HOT allocator, the COLD block
// manager and the KV-write entry points.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <new>

#include "gk_internal.h"

namespace gk {

// ---------------------------------------------------------------------------
// HOT allocator.  GraniKV Section 3.2: one contiguous range per shared prefix;
// a released range joins the free list and merges with its neighbours.
// Appendix B.8b packs first-fit.  A free range that reaches the bump pointer
// lowers it instead of staying on the list.
// ---------------------------------------------------------------------------
bool HotAllocator::alloc(int64_t n, int64_t* base) {
  for (size_t i = 0; i < free.size(); ++i) {
    int64_t a = free[i].first, b = free[i].second;
    if (b - a >= n) {
      if (b - a == n)
        free.erase(free.begin() + (ptrdiff_t)i);
      else
        free[i].first = a + n;
      live[a] = n;
      *base = a;
      return true;
    }
  }
  if (top + n > capacity) return false;
  *base = top;
  live[top] = n;
  top += n;
  return true;
}

bool HotAllocator::release(int64_t base) {
  auto it = live.find(base);
  if (it == live.end()) return false;
  int64_t a = base, b = base + it->second;
  live.erase(it);
  // neighbours: the range ending at a and the range starting at b
  auto pos = std::lower_bound(free.begin(), free.end(), std::make_pair(a, a));
  if (pos != free.end() && pos->first == b) {
    b = pos->second;
    pos = free.erase(pos);
  }
  if (pos != free.begin() && (pos - 1)->second == a) {
    --pos;
    a = pos->first;
    pos = free.erase(pos);
  }
  if (b == top)
    top = a;
  else
    free.insert(pos, {a, b});
  return true;
}

// ---------------------------------------------------------------------------
// COLD block manager.  "Paged KV cache", How it works (steps 1-4) and Code:
// a stack of free blocks, refcounts, a table per sequence, copy-on-write of a
// shared partial last block before the write.
// ---------------------------------------------------------------------------
static uint64_t splitmix64_next(uint64_t* state) {
  // splitmix64 (Steele, Lea & Flood, OOPSLA 2014)
  uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

void BlockManager::init(int64_t n_blocks, int32_t page_size, uint64_t seed) {
  page = page_size;
  std::vector<int32_t> order((size_t)n_blocks);
  for (int64_t i = 0; i < n_blocks; ++i) order[(size_t)i] = (int32_t)i;
  if (seed != 0) {
    // Fisher-Yates from the top: j = floor(u * (i + 1) / 2^64)
    uint64_t st = seed;
    for (int64_t i = n_blocks - 1; i >= 1; --i) {
      uint64_t u = splitmix64_next(&st);
      uint64_t j = (uint64_t)(((unsigned __int128)u * (unsigned __int128)(uint64_t)(i + 1)) >> 64);
      std::swap(order[(size_t)i], order[(size_t)j]);
    }
  }
  free_stack.assign(order.rbegin(), order.rend());   // pops hand out order[0], order[1], ...
  ref.assign((size_t)n_blocks, 0);
  seqs.clear();
  free_seq_ids.clear();
  cache.clear();
  cached_hash.clear();
  cached_use.clear();
  lru.clear();
  tick = 0;
}

int32_t BlockManager::take() {
  if (free_stack.empty()) {
    // evict the least recently used cached block that no sequence holds
    for (auto it = lru.begin(); it != lru.end(); ++it) {
      const int32_t b = it->second;
      if (ref[(size_t)b] != 1) continue;
      cache.erase(cached_hash[b]);
      cached_hash.erase(b);
      cached_use.erase(b);
      lru.erase(it);
      drop(b);                     // the cache's reference: the block is free now
      break;
    }
    if (free_stack.empty()) return -1;
  }
  int32_t b = free_stack.back();
  free_stack.pop_back();
  ref[(size_t)b] = 1;
  return b;
}

void BlockManager::touch(int32_t b) {
  auto it = cached_use.find(b);
  if (it == cached_use.end()) return;
  lru.erase({it->second, b});
  it->second = ++tick;
  lru.insert({it->second, b});
}

// The splitmix64 output function (Steele, Lea & Flood, OOPSLA 2014) as a mixer.
static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t block_hash(uint64_t parent, const int32_t* tokens, int32_t page_size) {
  uint64_t h = mix64(parent + 0x9E3779B97F4A7C15ull);
  for (int32_t i = 0; i < page_size; ++i) h = mix64(h ^ ((uint64_t)(uint32_t)tokens[i] * 0x9E3779B97F4A7C15ull));
  return h;
}

void BlockManager::drop(int32_t b) {
  if (--ref[(size_t)b] == 0) free_stack.push_back(b);
}

gk_status fail(Pool* p, gk_status s, const std::string& msg) {
  if (p) p->last_error = msg;
  return s;
}

gk_status cuda_fail(Pool* p, int err, const char* what) {
  std::string m = std::string(what) + ": " + cudaGetErrorString((cudaError_t)err);
  return fail(p, GK_ERR_CUDA, m);
}

gk_status ensure_device(Pool* p) {
  if (!p->has_device) return fail(p, GK_ERR_INVALID, "pool has no device storage");
  if (!p->dev.queried) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(p, e, "cudaGetDevice");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(p, e, "cudaDeviceGetAttribute");
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major * 10 + minor != 103)
      return fail(p, GK_ERR_UNSUPPORTED, "libgk is built for sm_103a (GB300) only");
    p->dev.device = dev;
    p->dev.num_sms = sms;
    p->dev.queried = true;
  }
  if (!p->d_error) {
    cudaError_t e = cudaMalloc(&p->d_error, sizeof(int32_t));
    if (e != cudaSuccess) return cuda_fail(p, e, "cudaMalloc(error word)");
    e = cudaMemset(p->d_error, 0, sizeof(int32_t));
    if (e != cudaSuccess) return cuda_fail(p, e, "cudaMemset(error word)");
  }
  if (!p->d_slot_claim) {
    const size_t bytes = sizeof(uint32_t) * (size_t)p->dev.num_sms;
    cudaError_t e = cudaMalloc(&p->d_slot_claim, bytes);
    if (e != cudaSuccess) return cuda_fail(p, e, "cudaMalloc(slot claims)");
    e = cudaMemset(p->d_slot_claim, 0, bytes);
    if (e != cudaSuccess) return cuda_fail(p, e, "cudaMemset(slot claims)");
    p->split_epoch = 0;
  }
  return GK_OK;
}

static Sequence* get_seq(Pool* p, int32_t id) {
  if (id < 0 || (size_t)id >= p->cold.seqs.size() || !p->cold.seqs[(size_t)id].alive) return nullptr;
  return &p->cold.seqs[(size_t)id];
}

static int32_t new_seq_id(Pool* p) {
  BlockManager& c = p->cold;
  if (!c.free_seq_ids.empty()) {
    int32_t id = c.free_seq_ids.back();
    c.free_seq_ids.pop_back();
    c.seqs[(size_t)id] = Sequence();
    c.seqs[(size_t)id].alive = true;
    return id;
  }
  c.seqs.emplace_back();
  c.seqs.back().alive = true;
  return (int32_t)c.seqs.size() - 1;
}

}  // namespace gk

using gk::Pool;

extern "C" {

const char* gk_status_string(gk_status s) {
  switch (s) {
    case GK_OK: return "ok";
    case GK_ERR_INVALID: return "invalid argument";
    case GK_ERR_OOM: return "COLD pool out of blocks";
    case GK_ERR_HOT_FULL: return "HOT pool has no range that fits";
    case GK_ERR_CUDA: return "CUDA error";
    case GK_ERR_DEVICE_BOUNDS: return "kernel met an out-of-range block or slot";
    case GK_ERR_TIMEOUT: return "kernel wait timed out";
    case GK_ERR_UNSUPPORTED: return "unsupported geometry";
  }
  return "unknown status";
}

gk_status gk_pool_create(const gk_pool_config* cfg, gk_pool** out) {
  if (!cfg || !out) return GK_ERR_INVALID;
  *out = nullptr;
  const gk_pool_config& c = *cfg;
  if (c.num_layers <= 0 || c.num_q_heads <= 0 || c.num_kv_heads <= 0 ||
      c.num_kv_heads > gk::kMaxKvHeads || c.num_q_heads % c.num_kv_heads != 0)
    return GK_ERR_INVALID;
  if (c.head_dim != 64 && c.head_dim != 128) return GK_ERR_UNSUPPORTED;
  int g = c.num_q_heads / c.num_kv_heads;
  bool g_ok = c.head_dim == 128 ? (g == 1 || g == 2 || g == 4 || g == 5 || g == 8) : (g == 1 || g == 2 || g == 4);
  if (!g_ok) return GK_ERR_UNSUPPORTED;
  if (c.hot_tokens < 0 || c.cold_slots < 0 || c.cold_page_size <= 0 ||
      c.cold_slots % c.cold_page_size != 0 || c.cold_slots > INT32_MAX)
    return GK_ERR_INVALID;
  bool any = c.hot_k || c.hot_v || c.cold_k || c.cold_v;
  bool all = c.hot_k && c.hot_v && c.cold_k && c.cold_v;
  if (any && !all) return GK_ERR_INVALID;
  if (all) {
    for (void* ptr : {c.hot_k, c.hot_v, c.cold_k, c.cold_v})
      if (((uintptr_t)ptr) % 256 != 0) return GK_ERR_INVALID;   // 16 B is the TMA floor; ask for 256
  }
  gk_pool* p = new (std::nothrow) gk_pool;
  if (!p) return GK_ERR_INVALID;
  Pool& P = p->impl;
  P.cfg = c;
  P.has_device = all;
  P.hot.capacity = c.hot_tokens;
  P.cold.init(c.cold_slots / c.cold_page_size, c.cold_page_size, c.seed);
  // default cost model: nominal GB300 figures until a measured one is loaded
  gk_cost_model& cm = P.cost;
  cm.c_flat_us = 6.0;
  cm.bw_flat_gbs = 5500.0;
  cm.c_cascade_us = 12.0;
  cm.bw_prefix_gbs = 5500.0;
  cm.bw_suffix_gbs = 5000.0;
  cm.c_merge_us = 0.0;
  cm.prefix_tile_us = 1.65;
  cm.prefix_item_us = 10.5;
  cm.gather_sm_gbs = 44.0;
  cm.c_gather_us = 10.0;
  cm.prefix_tile_split_us = 2.1;
  // warp-MMA prefix items: priced high until a measured model is loaded
  cm.warp_tile_us = 3.0;
  cm.warp_group_us = 1.0;
  cm.warp_item_us = 8.0;
  cm.warp_split_ratio = 1.3;
  cm.prefix_cta_ramp_us = 12.0;
  cm.prefix_cta_gather_ratio = 1.0;
  cm.c_merge_state_us = 0.0;
  cm.prefix_item_split_us = 10.5;
  cm.warp_item_split_us = 8.0;
  cm.prefix_item_crowd_us = 0.0;
  cm.split_gather_ratio_tensor = 1.0;
  cm.c_gather_split_us = 10.0;
  cm.split_tensor_us = 0.0;
  *out = p;
  return GK_OK;
}

void gk_pool_destroy(gk_pool* pool) {
  if (!pool) return;
  if (pool->impl.d_error) cudaFree(pool->impl.d_error);
  if (pool->impl.d_slot_claim) cudaFree(pool->impl.d_slot_claim);
  delete pool;
}

const char* gk_last_error(const gk_pool* pool) { return pool ? pool->impl.last_error.c_str() : ""; }

gk_status gk_prefix_alloc(gk_pool* pool, int64_t prefix_len, int64_t* hot_base) {
  if (!pool || !hot_base) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  if (prefix_len <= 0 || prefix_len > INT32_MAX)
    return gk::fail(p, GK_ERR_INVALID, "prefix_len must be in [1, 2^31)");
  if (!p->hot.alloc(prefix_len, hot_base))
    return gk::fail(p, GK_ERR_HOT_FULL, "no HOT range fits the prefix");
  return GK_OK;
}

gk_status gk_prefix_release(gk_pool* pool, int64_t hot_base) {
  if (!pool) return GK_ERR_INVALID;
  if (pool->impl.hot_cache.key_of.count(hot_base))
    return gk::fail(&pool->impl, GK_ERR_INVALID, "the prefix at this base belongs to the prefix cache (gk_prefix_unref)");
  if (!pool->impl.hot.release(hot_base))
    return gk::fail(&pool->impl, GK_ERR_INVALID, "no live prefix at this base");
  return GK_OK;
}

gk_status gk_prefix_acquire(gk_pool* pool, uint64_t key, int64_t prefix_len, int64_t* hot_base, int32_t* hit) {
  if (!pool || !hot_base || !hit) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  gk::HotCache& hc = p->hot_cache;
  if (prefix_len <= 0 || prefix_len > INT32_MAX)
    return gk::fail(p, GK_ERR_INVALID, "prefix_len must be in [1, 2^31)");
  auto it = hc.entries.find(key);
  if (it != hc.entries.end()) {
    gk::HotCacheEntry& e = it->second;
    if (e.lp != prefix_len) return gk::fail(p, GK_ERR_INVALID, "key is cached with another prefix length");
    if (e.refs == 0) hc.idle.erase({e.last_use, key});
    ++e.refs;
    e.last_use = ++hc.tick;
    *hot_base = e.base;
    *hit = 1;
    return GK_OK;
  }
  int64_t base = 0;
  while (!p->hot.alloc(prefix_len, &base)) {
    // evict the least recently used slab nobody holds, then try again
    if (hc.idle.empty()) return gk::fail(p, GK_ERR_HOT_FULL, "no HOT range fits the prefix, even after evicting idle ones");
    const uint64_t victim = hc.idle.begin()->second;
    hc.idle.erase(hc.idle.begin());
    const int64_t vb = hc.entries[victim].base;
    hc.entries.erase(victim);
    hc.key_of.erase(vb);
    p->hot.release(vb);
  }
  gk::HotCacheEntry e;
  e.base = base;
  e.lp = prefix_len;
  e.refs = 1;
  e.last_use = ++hc.tick;
  hc.entries[key] = e;
  hc.key_of[base] = key;
  *hot_base = base;
  *hit = 0;
  return GK_OK;
}

gk_status gk_prefix_unref(gk_pool* pool, uint64_t key) {
  if (!pool) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  gk::HotCache& hc = p->hot_cache;
  auto it = hc.entries.find(key);
  if (it == hc.entries.end() || it->second.refs == 0)
    return gk::fail(p, GK_ERR_INVALID, "no held prefix under this key");
  gk::HotCacheEntry& e = it->second;
  e.last_use = ++hc.tick;
  if (--e.refs == 0) hc.idle.insert({e.last_use, key});
  return GK_OK;
}

gk_status gk_hot_cache_stats(const gk_pool* pool, int64_t* cached, int64_t* idle, int64_t* idle_tokens) {
  if (!pool) return GK_ERR_INVALID;
  const gk::HotCache& hc = pool->impl.hot_cache;
  int64_t tok = 0;
  for (const auto& ik : hc.idle) tok += hc.entries.at(ik.second).lp;
  if (cached) *cached = (int64_t)hc.entries.size();
  if (idle) *idle = (int64_t)hc.idle.size();
  if (idle_tokens) *idle_tokens = tok;
  return GK_OK;
}

gk_status gk_hot_stats(const gk_pool* pool, int64_t* bump_top, int64_t* free_ranges, int64_t* free_tokens) {
  if (!pool) return GK_ERR_INVALID;
  const gk::HotAllocator& h = pool->impl.hot;
  int64_t used = 0;
  for (auto& kv : h.live) used += kv.second;
  if (bump_top) *bump_top = h.top;
  if (free_ranges) *free_ranges = (int64_t)h.free.size();
  if (free_tokens) *free_tokens = h.capacity - used;
  return GK_OK;
}

gk_status gk_seq_create(gk_pool* pool, int32_t* seq) {
  if (!pool || !seq) return GK_ERR_INVALID;
  *seq = gk::new_seq_id(&pool->impl);
  return GK_OK;
}

gk_status gk_seq_fork(gk_pool* pool, int32_t parent, int32_t* child) {
  if (!pool || !child) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  if (!gk::get_seq(p, parent)) return gk::fail(p, GK_ERR_INVALID, "unknown parent sequence");
  int32_t id = gk::new_seq_id(p);
  gk::Sequence* par = gk::get_seq(p, parent);    // the vector may have grown
  gk::Sequence* s = &p->cold.seqs[(size_t)id];
  s->table = par->table;
  s->len = par->len;
  for (int32_t b : s->table) ++p->cold.ref[(size_t)b];
  *child = id;
  return GK_OK;
}

gk_status gk_seq_create_cached(gk_pool* pool, int32_t n_tokens, const int32_t* tokens, int32_t* seq, int64_t* n_cached) {
  if (!pool || !seq || !n_cached || n_tokens < 0 || (n_tokens > 0 && !tokens)) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  gk::BlockManager& c = p->cold;
  const int32_t id = gk::new_seq_id(p);
  gk::Sequence* s = &c.seqs[(size_t)id];
  uint64_t h = 0;
  for (int64_t i = 0; (i + 1) * c.page <= n_tokens; ++i) {
    h = gk::block_hash(h, tokens + i * c.page, c.page);
    auto it = c.cache.find(h);
    if (it == c.cache.end()) break;
    s->table.push_back(it->second);
    ++c.ref[(size_t)it->second];
    c.touch(it->second);
  }
  s->len = (int64_t)s->table.size() * c.page;
  *seq = id;
  *n_cached = s->len;
  return GK_OK;
}

gk_status gk_seq_cache_blocks(gk_pool* pool, int32_t seq, int32_t n_tokens, const int32_t* tokens, int32_t* n_new) {
  if (!pool || n_tokens < 0 || (n_tokens > 0 && !tokens)) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  gk::BlockManager& c = p->cold;
  gk::Sequence* s = gk::get_seq(p, seq);
  if (!s) return gk::fail(p, GK_ERR_INVALID, "unknown sequence");
  const int64_t full = std::min<int64_t>(n_tokens, s->len) / c.page;
  int32_t added = 0;
  uint64_t h = 0;
  for (int64_t i = 0; i < full; ++i) {
    h = gk::block_hash(h, tokens + i * c.page, c.page);
    const int32_t b = s->table[(size_t)i];
    if (c.cache.count(h) || c.cached_hash.count(b)) continue;
    c.cache[h] = b;
    c.cached_hash[b] = h;
    c.cached_use[b] = ++c.tick;
    c.lru.insert({c.tick, b});
    ++c.ref[(size_t)b];          // the cache's reference
    ++added;
  }
  if (n_new) *n_new = added;
  return GK_OK;
}

gk_status gk_cold_cache_stats(const gk_pool* pool, int64_t* cached_blocks, int64_t* evictable_blocks) {
  if (!pool) return GK_ERR_INVALID;
  const gk::BlockManager& c = pool->impl.cold;
  int64_t ev = 0;
  for (const auto& kv : c.cached_hash) ev += c.ref[(size_t)kv.first] == 1 ? 1 : 0;
  if (cached_blocks) *cached_blocks = (int64_t)c.cached_hash.size();
  if (evictable_blocks) *evictable_blocks = ev;
  return GK_OK;
}

gk_status gk_seq_release(gk_pool* pool, int32_t seq) {
  if (!pool) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  gk::Sequence* s = gk::get_seq(p, seq);
  if (!s) return gk::fail(p, GK_ERR_INVALID, "unknown sequence");
  for (int32_t b : s->table) p->cold.drop(b);
  s->table.clear();
  s->len = 0;
  s->alive = false;
  p->cold.free_seq_ids.push_back(seq);
  return GK_OK;
}

gk_status gk_seq_table(const gk_pool* pool, int32_t seq, const int32_t** table, int32_t* nblocks, int64_t* len) {
  if (!pool) return GK_ERR_INVALID;
  Pool* p = const_cast<Pool*>(&pool->impl);
  gk::Sequence* s = gk::get_seq(p, seq);
  if (!s) return gk::fail(p, GK_ERR_INVALID, "unknown sequence");
  if (table) *table = s->table.data();
  if (nblocks) *nblocks = (int32_t)s->table.size();
  if (len) *len = s->len;
  return GK_OK;
}

gk_status gk_seq_append_slots(gk_pool* pool, int32_t n, const int32_t* seqs, int64_t* slot_mapping_out,
                              int32_t* n_cow, int32_t* cow_pairs_out, int32_t* n_done) {
  if (!pool || n < 0 || (n > 0 && (!seqs || !slot_mapping_out || !cow_pairs_out)) || !n_cow)
    return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  gk::BlockManager& c = p->cold;
  const int64_t P = c.page;
  *n_cow = 0;
  if (n_done) *n_done = 0;
  for (int32_t i = 0; i < n; ++i) {
    gk::Sequence* s = gk::get_seq(p, seqs[i]);
    if (!s) return gk::fail(p, GK_ERR_INVALID, "unknown sequence in append");
    int64_t off = s->len % P;
    if (off == 0) {
      int32_t b = c.take();
      if (b < 0) return gk::fail(p, GK_ERR_OOM, "COLD pool out of blocks");
      s->table.push_back(b);
    } else {
      int32_t shared = s->table.back();
      if (c.ref[(size_t)shared] > 1) {           // shared partial block: copy on write
        int32_t fresh = c.take();
        if (fresh < 0) return gk::fail(p, GK_ERR_OOM, "COLD pool out of blocks (copy-on-write)");
        c.drop(shared);
        s->table.back() = fresh;
        cow_pairs_out[2 * *n_cow] = shared;
        cow_pairs_out[2 * *n_cow + 1] = fresh;
        ++*n_cow;
      }
    }
    slot_mapping_out[i] = (int64_t)s->table.back() * P + off;
    ++s->len;
    if (n_done) *n_done = i + 1;
  }
  return GK_OK;
}

gk_status gk_seq_tables(const gk_pool* pool, int32_t n, const int32_t* seqs, int32_t max_blocks, int32_t* table_out,
                        int32_t* len_out) {
  if (!pool || n < 0 || max_blocks < 0 || (n > 0 && (!seqs || !table_out))) return GK_ERR_INVALID;
  Pool* p = const_cast<Pool*>(&pool->impl);
  for (int32_t i = 0; i < n; ++i) {
    gk::Sequence* s = gk::get_seq(p, seqs[i]);
    if (!s) return gk::fail(p, GK_ERR_INVALID, "unknown sequence");
    if ((int64_t)s->table.size() > max_blocks) return gk::fail(p, GK_ERR_INVALID, "table longer than max_blocks");
    int32_t* row = table_out + (int64_t)i * max_blocks;
    std::memcpy(row, s->table.data(), s->table.size() * sizeof(int32_t));
    std::memset(row + s->table.size(), 0, (size_t)(max_blocks - (int64_t)s->table.size()) * sizeof(int32_t));
    if (len_out) len_out[i] = (int32_t)s->len;
  }
  return GK_OK;
}

gk_status gk_cold_stats(const gk_pool* pool, int64_t* free_blocks, int64_t* total_blocks) {
  if (!pool) return GK_ERR_INVALID;
  if (free_blocks) *free_blocks = (int64_t)pool->impl.cold.free_stack.size();
  if (total_blocks) *total_blocks = (int64_t)pool->impl.cold.ref.size();
  return GK_OK;
}

gk_status gk_block_refcount(const gk_pool* pool, int32_t block, int32_t* refcount) {
  if (!pool || !refcount) return GK_ERR_INVALID;
  const gk::BlockManager& c = pool->impl.cold;
  if (block < 0 || (size_t)block >= c.ref.size()) return GK_ERR_INVALID;
  *refcount = c.ref[(size_t)block];
  return GK_OK;
}

gk_status gk_append_kv(gk_pool* pool, void* stream, int32_t layer, int32_t n, const int64_t* d_slot_mapping,
                       const void* d_k, const void* d_v, int32_t n_cow, const int32_t* d_cow_pairs) {
  if (!pool) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  if (layer < 0 || layer >= p->cfg.num_layers || n < 0 || n_cow < 0)
    return gk::fail(p, GK_ERR_INVALID, "bad layer or count");
  if ((n > 0 && (!d_slot_mapping || !d_k || !d_v)) || (n_cow > 0 && !d_cow_pairs))
    return gk::fail(p, GK_ERR_INVALID, "null device pointer");
  gk_status st = gk::ensure_device(p);
  if (st != GK_OK) return st;
  gk::LaunchCommon lc{&p->cfg, p->d_error, p->dev.num_sms};
  if (n_cow > 0) {
    int e = gk::launch_cow_copy(lc, stream, layer, n_cow, d_cow_pairs);
    if (e) return gk::cuda_fail(p, e, "copy-on-write kernel");
  }
  if (n > 0) {
    int e = gk::launch_scatter(lc, stream, layer, n, d_slot_mapping, d_k, d_v);
    if (e) return gk::cuda_fail(p, e, "reshape_and_cache kernel");
  }
  return GK_OK;
}

gk_status gk_write_prefix_kv(gk_pool* pool, void* stream, int32_t layer, int64_t hot_base, int64_t prefix_len,
                             int64_t t0, int64_t n, const void* d_k, const void* d_v) {
  if (!pool) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  auto it = p->hot.live.find(hot_base);
  if (it == p->hot.live.end() || it->second != prefix_len)
    return gk::fail(p, GK_ERR_INVALID, "no live prefix of this length at this base");
  if (layer < 0 || layer >= p->cfg.num_layers || t0 < 0 || n < 0 || t0 + n > prefix_len)
    return gk::fail(p, GK_ERR_INVALID, "token range outside the prefix");
  if (n > 0 && (!d_k || !d_v)) return gk::fail(p, GK_ERR_INVALID, "null device pointer");
  gk_status st = gk::ensure_device(p);
  if (st != GK_OK) return st;
  if (n == 0) return GK_OK;
  gk::LaunchCommon lc{&p->cfg, p->d_error, p->dev.num_sms};
  int e = gk::launch_write_prefix(lc, stream, layer, hot_base, prefix_len, t0, n, d_k, d_v);
  if (e) return gk::cuda_fail(p, e, "prefix write kernel");
  return GK_OK;
}

gk_status gk_device_error(gk_pool* pool, void* stream, int32_t* code) {
  if (!pool || !code) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  *code = GK_OK;
  if (!p->d_error) return GK_OK;
  int32_t h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, p->d_error, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return gk::cuda_fail(p, e, "reading the device error word");
  if (h != 0) {
    e = cudaMemsetAsync(p->d_error, 0, sizeof(int32_t), (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return gk::cuda_fail(p, e, "clearing the device error word");
  }
  *code = h;
  return GK_OK;
}

}  // extern "C"
