// gk_calibrate: the dispatcher's cost model measured on this GPU.
//
// GraniKV Section 3.6 keeps the routing rule and says its threshold must be
// re-fit on each GPU (Appendix B.4b fits M_sat = 1024 on A100 with a sweep).
// Here the rule is the cost model of gk_dispatch, and this call is the re-fit:
// it times the kernels with CUDA events on one layer of the caller's pool, L2
// emptied before every launch, and fits each term by least squares.
//   flat backend, several batches            -> c_flat_us + bytes / bw_flat_gbs
//   suffix gather over every SM               -> c_gather_us + bytes / bw_suffix_gbs
//     (these two by relative error: the smallest steps weigh as much as the largest)
//   merge                                     -> c_merge_us per (request, query head)
//                                                + c_merge_state_us per partial state of a request
//   tensor-core prefix items of C key tiles   -> prefix_item_us + C * prefix_tile_us
//   warp-MMA prefix items, R row groups       -> warp_item_us + C * (warp_tile_us + R * warp_group_us)
//   the gather alone on the SMs long items leave it -> gather_sm_gbs (median per SM)
// The split arrangement's own terms -- how much longer an item's tile takes
// beside a gather that keeps HBM busy (per kind of item), when and how fast a
// prefix CTA gathers after its item, when the gather-only CTAs start -- and c_cascade_us are then fitted to the
// whole cascades timed here (both arrangements, forced and as the planner
// arranges them, both kinds of item): a grid search for the smallest largest
// relative error of the predicted cascade, the other terms held at their fits.
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <cstdio>
#include <string>
#include <vector>

#include "device_common.cuh"
#include "gk_internal.h"

namespace gk {
namespace {

constexpr double kPrefixBandwidthGbs = 6000.0;   // HOT reads of a sequential plan's prefix launch
constexpr size_t kFlushBytes = 256u << 20;       // twice this is written and read between launches

// Reads a buffer far larger than L2, so that a timed launch starts from an L2
// that holds none of its inputs and no dirty lines (whose write-back it would pay).
__global__ void l2_sweep_kernel(const uint4* __restrict__ p, size_t n, uint32_t* sink) {
  uint32_t acc = 0;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const uint4 v = __ldcg(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x9E3779B9u) *sink = acc;   // keeps the loads; the buffer is zero, so never taken
}

// Queries for the timings: bf16 values in [-2, 2) from a hash of the index
// (timing does not depend on them; they only have to be finite).
__global__ void fill_queries_kernel(uint16_t* q, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    uint32_t h = (uint32_t)i * 2654435761u;
    h ^= h >> 15;
    h *= 2246822519u;
    h ^= h >> 13;
    const float v = ((float)(h & 0xFFFFu) / 65536.f - 0.5f) * 4.f;
    q[i] = (uint16_t)(__float_as_uint(v) >> 16);
  }
}

// least squares y = c0 + c1 x (the intercept may come out negative).  relative:
// each point weighted by 1 / y^2, so the fit minimises the relative error, which
// is what a choice between two predicted times at any scale depends on.
bool linfit(const std::vector<std::pair<double, double>>& pts, double* c0, double* c1, bool relative = false) {
  if (pts.size() < 2) return false;
  double n = 0, sx = 0, sy = 0, sxx = 0, sxy = 0;
  for (auto& q : pts) {
    const double w = relative ? 1.0 / (q.second * q.second) : 1.0;
    if (!std::isfinite(w)) return false;
    n += w;
    sx += w * q.first;
    sy += w * q.second;
    sxx += w * q.first * q.first;
    sxy += w * q.first * q.second;
  }
  const double den = n * sxx - sx * sx;
  if (!(std::fabs(den) > 1e-12 * n * sxx)) return false;   // all x (nearly) equal
  *c1 = (n * sxy - sx * sy) / den;
  *c0 = (sy - *c1 * sx) / n;
  return true;
}

// least squares y = a0 + a1 x1 + a2 x2 (normal equations, Cramer's rule)
bool fit3(const std::vector<std::array<double, 3>>& pts, double a[3]) {
  if (pts.size() < 3) return false;
  double M[3][3] = {}, v[3] = {};
  for (auto& q : pts) {
    const double f[3] = {1.0, q[0], q[1]};
    for (int i = 0; i < 3; ++i) {
      v[i] += f[i] * q[2];
      for (int j = 0; j < 3; ++j) M[i][j] += f[i] * f[j];
    }
  }
  auto det = [](const double m[3][3]) {
    return m[0][0] * (m[1][1] * m[2][2] - m[1][2] * m[2][1]) - m[0][1] * (m[1][0] * m[2][2] - m[1][2] * m[2][0]) +
           m[0][2] * (m[1][0] * m[2][1] - m[1][1] * m[2][0]);
  };
  const double D = det(M);
  if (std::fabs(D) < 1e-30) return false;
  for (int c = 0; c < 3; ++c) {
    double T[3][3];
    for (int i = 0; i < 3; ++i)
      for (int j = 0; j < 3; ++j) T[i][j] = j == c ? v[i] : M[i][j];
    a[c] = det(T) / D;
  }
  return true;
}

double median(std::vector<double> v) {
  if (v.empty()) return 0.0;
  std::sort(v.begin(), v.end());
  return v[v.size() / 2];
}

// One calibration run: scratch buffers on the device, timing, and the cases'
// resources taken from (and given back to) the pool's allocators.
struct Calib {
  gk_pool* pool = nullptr;
  Pool* p = nullptr;
  cudaStream_t st = nullptr;
  int32_t max_b = 0, max_blocks = 0;
  uint16_t* d_q = nullptr;
  float* d_out = nullptr;
  float* d_lse = nullptr;
  int32_t* d_table = nullptr;
  uint8_t* flush = nullptr;     // 2 * kFlushBytes: written, then the other half read
  uint32_t* sink = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  int reps = 7;
  std::string why;              // first failure

  bool cuda(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return true;
    if (why.empty()) why = std::string(what) + ": " + cudaGetErrorString(e);
    return false;
  }
  bool setup(int32_t B, int32_t blocks) {
    const gk_pool_config& c = p->cfg;
    max_b = B;
    max_blocks = blocks;
    const size_t nq = (size_t)B * c.num_q_heads * c.head_dim;
    return cuda(cudaMalloc(&d_q, nq * 2), "cudaMalloc(queries)") &&
           cuda(cudaMalloc(&d_out, nq * 4), "cudaMalloc(outputs)") &&
           cuda(cudaMalloc(&d_lse, (size_t)B * c.num_q_heads * 4), "cudaMalloc(lse)") &&
           cuda(cudaMalloc(&d_table, (size_t)B * blocks * 4), "cudaMalloc(block tables)") &&
           cuda(cudaMalloc(&flush, 2 * kFlushBytes), "cudaMalloc(L2 flush)") &&
           cuda(cudaMalloc(&sink, 4), "cudaMalloc(sink)") &&
           cuda(cudaMemsetAsync(flush, 0, 2 * kFlushBytes, st), "cudaMemsetAsync") &&
           cuda(cudaEventCreate(&e0), "cudaEventCreate") && cuda(cudaEventCreate(&e1), "cudaEventCreate") &&
           (fill_queries_kernel<<<256, 256, 0, st>>>(d_q, nq), cuda(cudaGetLastError(), "query fill"));
  }
  void teardown() {
    cudaStreamSynchronize(st);
    for (void* b : {(void*)d_q, (void*)d_out, (void*)d_lse, (void*)d_table, (void*)flush, (void*)sink})
      if (b) cudaFree(b);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
  }
  // write one half of the flush buffer and read the other: the next launch meets an L2
  // with none of its data and nothing dirty
  bool flush_l2() {
    return cuda(cudaMemsetAsync(flush, 0, kFlushBytes, st), "cudaMemsetAsync(flush)") &&
           (l2_sweep_kernel<<<4 * std::max(1, p->dev.num_sms), 512, 0, st>>>(
                reinterpret_cast<const uint4*>(flush + kFlushBytes), kFlushBytes / 16, sink),
            cuda(cudaGetLastError(), "L2 sweep"));
  }
  // median of `reps` timings (one warm-up launch first), microseconds; < 0 on failure
  template <class F>
  double time_us(F launch) {
    std::vector<double> ts;
    for (int r = 0; r <= reps; ++r) {
      if (!flush_l2()) return -1;
      if (!cuda(cudaEventRecord(e0, st), "cudaEventRecord")) return -1;
      const gk_status s = launch();
      if (s != GK_OK) {
        if (why.empty()) why = std::string("a timed call failed: ") + gk_last_error(pool);
        return -1;
      }
      if (!cuda(cudaEventRecord(e1, st), "cudaEventRecord") || !cuda(cudaEventSynchronize(e1), "cudaEventSynchronize"))
        return -1;
      float ms = 0;
      if (!cuda(cudaEventElapsedTime(&ms, e0, e1), "cudaEventElapsedTime")) return -1;
      if (r > 0) ts.push_back(ms * 1e3);
    }
    return median(ts);
  }
};

// One synthetic step: B requests share one HOT prefix of lp tokens, each with a
// COLD suffix of s tokens, reserved through the pool's own block manager.
struct Case {
  int32_t B = 0, lp = 0, s = 0;
  int64_t hot_base = -1;
  std::vector<int32_t> seqs, slen, lps;
  std::vector<int64_t> bases;
  gk_batch batch{};
  bool open = false;
};

// Suffix lengths of a case: s tokens each, or (s < 0) lengths uniform in
// 16..512 tokens (the pages' user turns) drawn from a generator seeded by -s
// (splitmix64 increments, the top bits scaled to the range).
// s >= 0: every suffix s tokens; s < 0: drawn from lo..hi (default 16..512, the
// pages' user turns) by a splitmix64 stream seeded by -s
std::vector<int32_t> suffix_lengths(int32_t B, int32_t s, int32_t lo = 16, int32_t hi = 512) {
  std::vector<int32_t> out((size_t)B, s);
  if (s >= 0) return out;
  uint64_t x = (uint64_t)(-(int64_t)s) * 0x9E3779B97F4A7C15ull;
  for (auto& v : out) {
    x += 0x9E3779B97F4A7C15ull;
    uint64_t z = x;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    v = lo + (int32_t)((z >> 32) % (uint32_t)(hi - lo + 1));
  }
  return out;
}

// false when the pool has no room for the case (it is then skipped) or on an error (c.why set)
bool open_case(Calib& c, Case& k, int32_t B, int32_t lp, int32_t s, int32_t lo = 16, int32_t hi = 512) {
  k = Case{};
  k.B = B;
  k.lp = lp;
  k.s = s;
  const std::vector<int32_t> lens = suffix_lengths(B, s, lo, hi);
  const int32_t P = c.p->cfg.cold_page_size;
  int32_t smax = 0;
  for (int32_t v : lens) smax = std::max(smax, v);
  const int32_t blocks = (smax + P - 1) / P;
  if (B > c.max_b || blocks > c.max_blocks) return false;
  if (gk_prefix_alloc(c.pool, lp, &k.hot_base) != GK_OK) return false;
  for (int32_t r = 0; r < B; ++r) {
    int32_t sq = -1;
    if (gk_seq_create(c.pool, &sq) != GK_OK) break;
    k.seqs.push_back(sq);
  }
  k.open = true;
  if ((int32_t)k.seqs.size() < B) return false;
  std::vector<int32_t> order;
  for (int32_t r = 0; r < B; ++r) order.insert(order.end(), (size_t)lens[(size_t)r], k.seqs[(size_t)r]);
  std::vector<int64_t> slots(order.size());
  std::vector<int32_t> cow(2 * order.size() + 2);
  int32_t n_cow = 0, n_done = 0;
  if (!order.empty() && gk_seq_append_slots(c.pool, (int32_t)order.size(), order.data(), slots.data(), &n_cow,
                                            cow.data(), &n_done) != GK_OK)
    return false;   // out of COLD blocks: what was appended is released with the sequences
  std::vector<int32_t> table((size_t)B * c.max_blocks);
  k.slen.assign(B, 0);
  if (gk_seq_tables(c.pool, B, k.seqs.data(), c.max_blocks, table.data(), k.slen.data()) != GK_OK) return false;
  if (!c.cuda(cudaMemcpyAsync(c.d_table, table.data(), table.size() * 4, cudaMemcpyHostToDevice, c.st),
              "cudaMemcpyAsync(block tables)") ||
      !c.cuda(cudaStreamSynchronize(c.st), "cudaStreamSynchronize"))
    return false;
  k.bases.assign(B, k.hot_base);
  k.lps.assign(B, lp);
  k.batch = gk_batch{};
  k.batch.num_requests = B;
  k.batch.max_blocks = c.max_blocks;
  k.batch.prefix_hot_base = k.bases.data();
  k.batch.prefix_len = k.lps.data();
  k.batch.suffix_len = k.slen.data();
  k.batch.d_block_table = c.d_table;
  k.batch.d_q = c.d_q;
  k.batch.d_out = c.d_out;
  k.batch.d_lse = c.d_lse;
  return true;
}

void close_case(Calib& c, Case& k) {
  if (!k.open) return;
  for (int32_t sq : k.seqs) gk_seq_release(c.pool, sq);
  if (k.hot_base >= 0) gk_prefix_release(c.pool, k.hot_base);
  k = Case{};
}

}  // namespace
}  // namespace gk

using gk::Calib;
using gk::Case;

extern "C" gk_status gk_calibrate(gk_pool* pool, void* stream, const char* json_out) {
  if (!pool) return GK_ERR_INVALID;
  gk::Pool* p = &pool->impl;
  if (!p->has_device) return gk::fail(p, GK_ERR_INVALID, "gk_calibrate needs a pool with device storage");
  gk_status st = gk::ensure_device(p);
  if (st != GK_OK) return st;
  const gk_pool_config cfg = p->cfg;
  const int32_t g = cfg.num_q_heads / cfg.num_kv_heads;
  const int num_sms = p->dev.num_sms;
  // the pool's settings are the calibration's to change; they are put back at the end
  const gk_cascade_mode mode0 = p->cascade_mode;
  const int32_t tiles0 = p->cascade_tiles;
  const gk_prefix_kernel kernel0 = p->prefix_kernel;
  const gk_gather_partition part0 = p->gather_partition;
  const gk_cost_model cost0 = p->cost;
  p->gather_partition = GK_PARTITION_STREAM;

  Calib c;
  c.pool = pool;
  c.p = p;
  c.st = (cudaStream_t)stream;
  std::vector<gk_plan*> plans;                          // kept for the residual fit
  std::vector<std::pair<gk_plan*, double>> cascades;    // (plan, measured whole cascade)
  std::vector<std::pair<double, double>> flat, suffix, tile, gather_sm;
  std::vector<std::array<double, 3>> merge;             // (B * Hq, partial states per request, us)
  std::vector<std::array<double, 3>> warp;              // (C, C * R, us)
  bool ok = c.setup(512, (2048 + cfg.cold_page_size - 1) / cfg.cold_page_size + 1);

  auto plan_for = [&](Case& k, gk_cascade_mode mode, int32_t tiles, gk_prefix_kernel kern) -> gk_plan* {
    p->cascade_mode = mode;
    p->cascade_tiles = tiles;
    p->prefix_kernel = kern;
    gk_plan* pl = nullptr;
    if (gk_plan_build(pool, &k.batch, stream, &pl) != GK_OK) {
      if (c.why.empty()) c.why = std::string("gk_plan_build: ") + gk_last_error(pool);
      return nullptr;
    }
    plans.push_back(pl);
    return pl;
  };
  auto timed = [&](auto fn) { return c.time_us(fn); };
  Case k;

  // (1) sequential plans over tensor-core items: flat, suffix gather, merge, prefix items, whole cascade
  const int32_t base_cases[6][3] = {{8, 512, 64},     {8, 2048, 256},   {32, 4096, 512},
                                    {64, 16384, 1024}, {128, 8192, 512}, {256, 4096, 1024}};
  for (auto& bc : base_cases) {
    if (!ok) break;
    if (gk::open_case(c, k, bc[0], bc[1], bc[2])) {
      gk_plan* pl = plan_for(k, GK_CASCADE_SEQUENTIAL, 0, GK_PREFIX_TENSOR);
      ok = pl != nullptr;
      gk_plan_summary sm{};
      if (ok) gk_plan_info(pl, &sm);
      double t;
      if (ok && (ok = (t = timed([&] { return gk_decode_dense(pool, stream, 0, &k.batch, pl); })) >= 0))
        flat.push_back({(double)sm.dense_bytes, t});
      if (ok && (ok = (t = timed([&] { return gk_cascade_suffix(pool, stream, 0, &k.batch, pl); })) >= 0))
        suffix.push_back({(double)sm.suffix_bytes, t});
      if (ok && (ok = (t = timed([&] { return gk_cascade_merge(pool, stream, 0, &k.batch, pl); })) >= 0))
        merge.push_back({(double)k.B * cfg.num_q_heads, (double)sm.num_partials / k.B, t});
      if (ok && sm.prefix_ctas <= num_sms &&
          (ok = (t = timed([&] { return gk_cascade_prefix(pool, stream, 0, &k.batch, pl); })) >= 0))
        tile.push_back({(double)sm.prefix_tiles_per_item, t});
      if (ok && (ok = (t = timed([&] { return gk_decode_cascade(pool, stream, 0, &k.batch, pl); })) >= 0))
        cascades.push_back({pl, t});
    } else if (!c.why.empty()) {
      ok = false;
    }
    gk::close_case(c, k);
  }
  // (2) split plans with long tensor-core items: the items alone and the whole cascade
  if (ok && gk::open_case(c, k, 64, 16384, 1024)) {
    for (int32_t C : {16, 32, 64, 128}) {
      gk_plan* pl = plan_for(k, GK_CASCADE_SPLIT, C, GK_PREFIX_TENSOR);
      if (!(ok = pl != nullptr)) break;
      gk_plan_summary sm{};
      gk_plan_info(pl, &sm);
      if (!sm.cascade_split) continue;
      double t;
      if (!(ok = (t = timed([&] { return gk_cascade_prefix(pool, stream, 0, &k.batch, pl); })) >= 0)) break;
      tile.push_back({(double)sm.prefix_tiles_per_item, t});
      if (!(ok = (t = timed([&] { return gk_decode_cascade(pool, stream, 0, &k.batch, pl); })) >= 0)) break;
      cascades.push_back({pl, t});
    }
  } else if (!c.why.empty()) {
    ok = false;
  }
  gk::close_case(c, k);
  // (3) the gather alone on the SMs that one-split items (M_eff 512 g) leave it
  if (ok && gk::open_case(c, k, 512, 16384, 128)) {
    gk_plan* pl = plan_for(k, GK_CASCADE_SPLIT, 128, GK_PREFIX_TENSOR);
    gk_plan_summary sm{};
    double t = -1;
    if ((ok = pl != nullptr)) {
      gk_plan_info(pl, &sm);
      if (sm.cascade_split && sm.suffix_ctas > sm.prefix_ctas) {
        ok = (t = timed([&] { return gk_cascade_suffix(pool, stream, 0, &k.batch, pl); })) >= 0;
        if (ok) gather_sm.push_back({(double)(sm.suffix_ctas - sm.prefix_ctas),
                                     (double)sm.suffix_bytes / (t * 1e3) / (sm.suffix_ctas - sm.prefix_ctas)});
      }
    }
  } else if (!c.why.empty()) {
    ok = false;
  }
  gk::close_case(c, k);
  // (4) warp-MMA items of 16, 32 and 128 stacked rows (R = 1, 2, 8) and C key tiles
  for (int32_t rows : {16, 32, 128}) {
    if (!ok) break;
    if (gk::open_case(c, k, (rows + g - 1) / g, 16384, 64)) {
      for (int32_t C : {8, 32, 128}) {
        gk_plan* pl = plan_for(k, GK_CASCADE_SPLIT, C, GK_PREFIX_WARP);
        if (!(ok = pl != nullptr)) break;
        gk_plan_summary sm{};
        gk_plan_info(pl, &sm);
        if (!sm.cascade_split) continue;
        double t;
        if (!(ok = (t = timed([&] { return gk_cascade_prefix(pool, stream, 0, &k.batch, pl); })) >= 0)) break;
        warp.push_back({(double)sm.prefix_tiles_per_item, (double)sm.prefix_tiles_per_item * sm.prefix_row_groups, t});
        if (!(ok = (t = timed([&] { return gk_decode_cascade(pool, stream, 0, &k.batch, pl); })) >= 0)) break;
        cascades.push_back({pl, t});
      }
    } else if (!c.why.empty()) {
      ok = false;
    }
    gk::close_case(c, k);
  }

  // (5) a grid of steps (Lp x B, suffixes of 16..512 tokens), each prefix kernel,
  //     arranged by the planner (cascade mode AUTO) and, in the first round,
  //     sequentially: the merge and the whole cascade.  The second round re-plans
  //     the grid with the fitted model, whose plans are the ones it will price.
  auto run_grid = [&](bool sequential_too) {
    for (int32_t lp : {512, 2048, 8192, 16384})
      for (int32_t B : {8, 32, 128, 512}) {
        if (!ok) return;
        if (gk::open_case(c, k, B, lp, -(lp * 1000 + B))) {
          for (gk_prefix_kernel kern : {GK_PREFIX_TENSOR, GK_PREFIX_WARP})
            for (gk_cascade_mode mode : {GK_CASCADE_AUTO, GK_CASCADE_SEQUENTIAL}) {
              if (!ok) break;
              if (mode == GK_CASCADE_SEQUENTIAL && !sequential_too) continue;
              gk_plan* pl = plan_for(k, mode, 0, kern);
              if (!(ok = pl != nullptr)) break;
              gk_plan_summary sm{};
              gk_plan_info(pl, &sm);
              double t;
              if (!(ok = (t = timed([&] { return gk_cascade_merge(pool, stream, 0, &k.batch, pl); })) >= 0)) break;
              merge.push_back({(double)k.B * cfg.num_q_heads, (double)sm.num_partials / k.B, t});
              if (!(ok = (t = timed([&] { return gk_decode_cascade(pool, stream, 0, &k.batch, pl); })) >= 0)) break;
              cascades.push_back({pl, t});
            }
        } else if (!c.why.empty()) {
          ok = false;
        }
        gk::close_case(c, k);
      }
  };
  run_grid(true);
  // (6) steps the size of whole decode layers (long suffixes, hundreds of MB each):
  //     the arrangement the planner picks for each prefix kernel and, in the
  //     first round, the sequential one and split launches of tensor-core items
  //     of 16 and 32 key tiles, so that the split terms are fitted where a
  //     step's time goes, not only on the short steps of the grid
  auto run_large = [&](bool forced_too) {
    const int32_t large_cases[3][5] = {{64, 16384, 256, 2048, 1}, {256, 4096, 64, 1024, 2}, {128, 16384, 512, 2048, 3}};
    for (auto& lc : large_cases) {
      if (!ok) return;
      if (gk::open_case(c, k, lc[0], lc[1], -(1000000 + lc[4]), lc[2], lc[3])) {
        struct Arr { gk_cascade_mode mode; int32_t tiles; gk_prefix_kernel kern; };
        const Arr arrs[] = {{GK_CASCADE_AUTO, 0, GK_PREFIX_TENSOR}, {GK_CASCADE_AUTO, 0, GK_PREFIX_WARP},
                            {GK_CASCADE_SEQUENTIAL, 0, GK_PREFIX_TENSOR}, {GK_CASCADE_SPLIT, 16, GK_PREFIX_TENSOR},
                            {GK_CASCADE_SPLIT, 32, GK_PREFIX_TENSOR}};
        for (const Arr& a : arrs) {
          if (a.mode != GK_CASCADE_AUTO && !forced_too) continue;
          gk_plan* pl = plan_for(k, a.mode, a.tiles, a.kern);
          if (!(ok = pl != nullptr)) break;
          double t;
          if (!(ok = (t = timed([&] { return gk_decode_cascade(pool, stream, 0, &k.batch, pl); })) >= 0)) break;
          cascades.push_back({pl, t});
        }
      } else if (!c.why.empty()) {
        ok = false;
      }
      gk::close_case(c, k);
    }
  };
  run_large(true);

  // ---- fits ----
  gk_cost_model cm = p->cost;
  double a0 = 0, a1 = 0;
  if (ok) {
    std::string miss;
    if (!gk::linfit(flat, &a0, &a1, true) || a1 <= 0) miss += " flat";
    else { cm.c_flat_us = std::max(0.0, a0); cm.bw_flat_gbs = 1.0 / a1 / 1e3; }
    if (!gk::linfit(suffix, &a0, &a1, true) || a1 <= 0) miss += " suffix";
    else { cm.c_gather_us = std::max(0.0, a0); cm.bw_suffix_gbs = 1.0 / a1 / 1e3; }
    double mw[3];
    if (!gk::fit3(merge, mw)) {
      miss += " merge";
    } else if (mw[1] >= 0 && mw[2] >= 0) {
      cm.c_merge_us = mw[1];
      cm.c_merge_state_us = mw[2];
    } else {
      // a negative slope: keep the term that grows with the warps alone
      std::vector<std::pair<double, double>> pts;
      for (auto& q : merge) pts.push_back({q[0], q[2]});
      cm.c_merge_us = gk::linfit(pts, &a0, &a1) ? std::max(0.0, a1) : 0.0;
      cm.c_merge_state_us = 0.0;
    }
    if (!gk::linfit(tile, &a0, &a1) || a1 <= 0) miss += " prefix-items";
    else {
      cm.prefix_item_us = std::max(0.0, a0);
      cm.prefix_tile_us = a1;
    }
    double w[3];
    if (!gk::fit3(warp, w)) miss += " warp-items";
    else {
      // a tile's part that does not grow with the rows must stay positive; if the fit
      // puts it below zero, refit with it pinned near zero (all of the tile on the rows)
      cm.warp_item_us = std::max(0.0, w[0]);
      if (w[1] > 0 && w[2] >= 0) {
        cm.warp_tile_us = w[1];
        cm.warp_group_us = w[2];
      } else {
        std::vector<std::pair<double, double>> pts;
        for (auto& q : warp) pts.push_back({q[1], q[2] - cm.warp_item_us});
        double b0, b1;
        cm.warp_tile_us = 1e-3;
        cm.warp_group_us = gk::linfit(pts, &b0, &b1) && b1 > 0 ? b1 : 1.0;
      }
    }
    std::vector<double> per_sm;
    for (auto& q : gather_sm) per_sm.push_back(q.second);
    if (per_sm.empty()) miss += " gather-per-SM";
    else cm.gather_sm_gbs = gk::median(per_sm);
    cm.bw_prefix_gbs = gk::kPrefixBandwidthGbs;
    if (!miss.empty()) {
      ok = false;
      c.why = "pool too small to calibrate (no room for the cases of:" + miss +
              "); give it at least 16384 HOT tokens and 262144 COLD token slots";
    }
  }
  // The split arrangement's terms and the cascade's fixed cost, fitted to the whole
  // cascades: tile ratio and fixed cost of an item in a split launch (each kind),
  // the cost each concurrent item adds to every item's, the prefix CTAs' gather
  // ramp and rate, the per-SM gather rate (around its own measurement), its
  // ratio in tensor-core split launches, when a split launch's gather-only
  // CTAs start (around the stand-alone gather's c_gather) and what a split
  // launch of tensor-core items costs over one of warp-MMA items.  A coordinate search over candidate
  // values of each term in turn (six passes) minimises the largest plus half the
  // mean relative error of T_cascade; for each candidate c_cascade minimises the
  // same (convex in c: ternary search).  Run on the first round's cascades, then,
  // after the grid is re-planned with that model, on all of them.
  std::vector<std::pair<double, double>> resid;   // (predicted without c_cascade, measured)
  const gk_cost_model parts = cm;                 // the terms fitted on their own
  auto fit_cascades = [&]() {
    if (!ok || cascades.empty()) return;
    const int32_t Hq = cfg.num_q_heads;
    const size_t n = cascades.size();
    std::vector<double> pred(n);
    auto score = [&](double cc) {
      double mx = 0, sum = 0;
      for (size_t i = 0; i < n; ++i) {
        const double e = std::fabs(std::max(0.0, pred[i] + cc) - cascades[i].second) / cascades[i].second;
        mx = std::max(mx, e);
        sum += e;
      }
      return mx + 0.5 * sum / n;
    };
    // the model's score with its best c_cascade (set in m)
    auto evaluate = [&](gk_cost_model& m) {
      m.c_cascade_us = 0.0;
      for (size_t i = 0; i < n; ++i) {
        double td;
        gk::predict_plan(m, num_sms, Hq, cascades[i].first->impl, &td, &pred[i]);
      }
      // no prediction below zero inside the search, so the score is convex in c
      double lo = -60.0, hi = 60.0;
      for (double q : pred) lo = std::max(lo, -q);
      for (int s2 = 0; s2 < 50; ++s2) {
        const double m1 = lo + (hi - lo) / 3, m2 = hi - (hi - lo) / 3;
        if (score(m1) <= score(m2)) hi = m2; else lo = m1;
      }
      m.c_cascade_us = 0.5 * (lo + hi);
      return score(m.c_cascade_us);
    };
    struct Term {
      double gk_cost_model::*field;
      std::vector<double> values;
    };
    std::vector<Term> terms;
    auto span = [](double base, double lo, double hi, double step) {
      std::vector<double> v;
      for (double x = lo; x <= hi + 1e-9; x += step) v.push_back(std::max(0.0, base + x));
      return v;
    };
    terms.push_back({&gk_cost_model::prefix_tile_split_us, {}});
    for (double r = 1.0; r <= 1.401; r += 0.05) terms.back().values.push_back(parts.prefix_tile_us * r);
    terms.push_back({&gk_cost_model::warp_split_ratio, span(0.0, 0.9, 1.4, 0.1)});
    terms.push_back({&gk_cost_model::prefix_item_split_us, span(parts.prefix_item_us, -4.0, 8.0, 2.0)});
    terms.push_back({&gk_cost_model::warp_item_split_us, span(parts.warp_item_us, -4.0, 8.0, 2.0)});
    terms.push_back({&gk_cost_model::prefix_item_crowd_us, span(0.0, 0.0, 0.16, 0.02)});
    // A prefix CTA gathers with the same code on the same kind of SM as a
    // gather-only CTA: the model gives it the same rate (ratio 1) and fits only
    // when it starts.  (Per-CTA %globaltimer timelines of split launches show
    // prefix CTAs gathering at 0.94-1.0 of a gather-only CTA's rate; the fitted
    // start is a later one than the timelines show, as it also carries what the
    // model leaves out of a prefix CTA's short gathers.)
    terms.push_back({&gk_cost_model::prefix_cta_ramp_us, span(0.0, 0.0, 40.0, 2.0)});
    terms.push_back({&gk_cost_model::gather_sm_gbs, {}});
    for (double r = 0.8; r <= 1.301; r += 0.1) terms.back().values.push_back(parts.gather_sm_gbs * r);
    terms.push_back({&gk_cost_model::split_gather_ratio_tensor, span(0.0, 0.5, 1.0, 0.1)});
    terms.push_back({&gk_cost_model::c_gather_split_us, span(parts.c_gather_us, -4.0, 24.0, 2.0)});
    terms.push_back({&gk_cost_model::split_tensor_us, span(0.0, 0.0, 12.0, 1.0)});
    // start from the middle of each range
    gk_cost_model best = parts;
    best.prefix_cta_gather_ratio = 1.0;
    for (auto& t : terms) best.*(t.field) = t.values[t.values.size() / 2];
    double best_s = evaluate(best);
    for (int pass = 0; pass < 6; ++pass)
      for (auto& t : terms)
        for (double v : t.values) {
          gk_cost_model m = best;
          m.*(t.field) = v;
          const double sc = evaluate(m);
          if (sc < best_s - 1e-12) {
            best_s = sc;
            best = m;
          }
        }
    cm = best;
  };
  fit_cascades();
  if (ok) {
    p->cost = cm;          // the second round plans with the fitted model
    run_grid(false);
    run_large(false);
    fit_cascades();
  }
  if (ok) {
    gk_cost_model m0 = cm;
    m0.c_cascade_us = 0.0;
    for (auto& pc : cascades) {
      double td, tc;
      gk::predict_plan(m0, num_sms, cfg.num_q_heads, pc.first->impl, &td, &tc);
      resid.push_back({tc, pc.second});
    }
  }
  std::vector<gk_plan_summary> cas_plans;        // the timed cascades' plans, for the JSON
  for (auto& pc : cascades) cas_plans.push_back(pc.first->impl.summary);
  for (gk_plan* pl : plans) gk_plan_destroy(pl);   // after the stream's work (timed calls synchronised)
  c.teardown();
  p->cascade_mode = mode0;
  p->cascade_tiles = tiles0;
  p->prefix_kernel = kernel0;
  p->gather_partition = part0;
  if (!ok) {
    p->cost = cost0;   // the model in force before the call is kept on failure
    return gk::fail(p, c.why.find("pool too small") == 0 ? GK_ERR_INVALID : GK_ERR_CUDA, "gk_calibrate: " + c.why);
  }
  st = gk_cost_model_set(pool, &cm);
  if (st != GK_OK) return st;
  if (json_out) {
    FILE* f = std::fopen(json_out, "w");
    if (!f) return gk::fail(p, GK_ERR_INVALID, std::string("gk_calibrate: cannot write ") + json_out);
    auto pts = [&](const char* name, const std::vector<std::pair<double, double>>& v, bool last) {
      std::fprintf(f, "  \"%s\": [", name);
      for (size_t i = 0; i < v.size(); ++i) std::fprintf(f, "%s[%.6g, %.6g]", i ? ", " : "", v[i].first, v[i].second);
      std::fprintf(f, "]%s\n", last ? "" : ",");
    };
    std::fprintf(f, "{\n");
    const std::pair<const char*, double> terms[] = {
        {"c_flat_us", cm.c_flat_us},         {"bw_flat_gbs", cm.bw_flat_gbs},
        {"c_cascade_us", cm.c_cascade_us},   {"bw_prefix_gbs", cm.bw_prefix_gbs},
        {"bw_suffix_gbs", cm.bw_suffix_gbs}, {"c_merge_us", cm.c_merge_us},
        {"prefix_tile_us", cm.prefix_tile_us}, {"prefix_item_us", cm.prefix_item_us},
        {"gather_sm_gbs", cm.gather_sm_gbs}, {"c_gather_us", cm.c_gather_us},
        {"prefix_tile_split_us", cm.prefix_tile_split_us}, {"warp_tile_us", cm.warp_tile_us},
        {"warp_group_us", cm.warp_group_us}, {"warp_item_us", cm.warp_item_us},
        {"warp_split_ratio", cm.warp_split_ratio}, {"prefix_cta_ramp_us", cm.prefix_cta_ramp_us},
        {"prefix_cta_gather_ratio", cm.prefix_cta_gather_ratio}, {"c_merge_state_us", cm.c_merge_state_us},
        {"prefix_item_split_us", cm.prefix_item_split_us}, {"warp_item_split_us", cm.warp_item_split_us},
        {"prefix_item_crowd_us", cm.prefix_item_crowd_us},
        {"split_gather_ratio_tensor", cm.split_gather_ratio_tensor}, {"c_gather_split_us", cm.c_gather_split_us},
        {"split_tensor_us", cm.split_tensor_us}};
    for (auto& t : terms) std::fprintf(f, " \"%s\": %.17g,\n", t.first, t.second);
    std::fprintf(f, " \"geometry\": {\"num_q_heads\": %d, \"num_kv_heads\": %d, \"head_dim\": %d, \"sms\": %d},\n",
                 cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim, num_sms);
    std::fprintf(f, " \"measured\": {\n");
    pts("flat (dense bytes, us)", flat, false);
    pts("suffix (suffix bytes, us)", suffix, false);
    std::fprintf(f, "  \"merge (requests x query heads, partial states per request, us)\": [");
    for (size_t i = 0; i < merge.size(); ++i)
      std::fprintf(f, "%s[%.6g, %.6g, %.6g]", i ? ", " : "", merge[i][0], merge[i][1], merge[i][2]);
    std::fprintf(f, "],\n");
    pts("prefix items (tiles per item, us)", tile, false);
    std::fprintf(f, "  \"warp items (tiles per item, tiles x row groups, us)\": [");
    for (size_t i = 0; i < warp.size(); ++i)
      std::fprintf(f, "%s[%.6g, %.6g, %.6g]", i ? ", " : "", warp[i][0], warp[i][1], warp[i][2]);
    std::fprintf(f, "],\n");
    pts("gather per SM (SMs, GB/s per SM)", gather_sm, false);
    pts("cascade (predicted without c_cascade, measured us)", resid, false);
    // each timed cascade's plan, so that the model can be refitted from this file alone
    std::fprintf(f, "  \"cascade plans (split, prefix CTAs gather, warp items, tiles per item, prefix CTAs, "
                    "row groups, suffix bytes, prefix bytes, partial states, requests, measured us)\": [");
    for (size_t i = 0; i < cascades.size(); ++i) {
      const gk_plan_summary& q = cas_plans[i];
      std::fprintf(f, "%s[%d, %d, %d, %d, %d, %d, %lld, %lld, %d, %d, %.6g]", i ? ", " : "", q.cascade_split,
                   q.prefix_ctas_gather, q.prefix_kernel == GK_PREFIX_WARP ? 1 : 0, q.prefix_tiles_per_item,
                   q.prefix_ctas, q.prefix_row_groups, (long long)q.suffix_bytes, (long long)q.prefix_bytes,
                   q.num_partials, q.num_requests, cascades[i].second);
    }
    std::fprintf(f, "]\n");
    std::fprintf(f, " }\n}\n");
    const bool werr = std::ferror(f) != 0;
    std::fclose(f);
    if (werr) return gk::fail(p, GK_ERR_INVALID, std::string("gk_calibrate: writing ") + json_out + " failed");
  }
  return GK_OK;
}

// Per-SM gather speeds, taken where the plan runs its gather: a split plan's
// own launch (each slot's SM id, start, end of its item and end of its gather,
// recorded by the kernel; a slot's rate counts its gather only, and prefix and
// gather-only slots are each scaled to their own mean in the launch, since a
// gather that starts beside running items sees another HBM than one that
// starts after them), or a sequential plan's stand-alone suffix gather (each
// CTA's SM id, start and end).  Each launch alone.
extern "C" gk_status gk_sm_speeds_measure(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch,
                                          const gk_plan* plan, int32_t reps, float* speeds) {
  if (!pool || !batch || !plan) return GK_ERR_INVALID;
  gk::Pool* p = &pool->impl;
  if (reps < 1 || reps > 64) return gk::fail(p, GK_ERR_INVALID, "reps must be in 1 .. 64");
  gk_status st = gk::ensure_device(p);
  if (st != GK_OK) return st;
  const gk::Plan& pl = plan->impl;
  if (pl.pool != p) return gk::fail(p, GK_ERR_INVALID, "plan belongs to another pool");
  if (layer < 0 || layer >= p->cfg.num_layers) return gk::fail(p, GK_ERR_INVALID, "layer out of range");
  if (!pl.uploaded || !pl.d_buf) return gk::fail(p, GK_ERR_INVALID, "plan has no device tables");
  const int gctas = pl.summary.suffix_ctas;
  if (gctas <= 0 || pl.suf_segs.empty() || (int)pl.suf_seg_begin.size() != gctas + 1)
    return gk::fail(p, GK_ERR_INVALID, "the plan has no suffix segments");
  const bool split = pl.split;
  const int n_pre = split ? (int)pl.prefix_items.size() : 0;
  const int ctas = split ? std::max(n_pre, gctas) : gctas;
  const int words = split ? 4 : 3;
  std::vector<int64_t> tok((size_t)ctas, 0);
  int64_t tmax = 0;
  for (int b = 0; b < gctas; ++b) {
    for (int32_t i = pl.suf_seg_begin[(size_t)b]; i < pl.suf_seg_begin[(size_t)b + 1]; ++i)
      tok[(size_t)b] += pl.suf_segs[(size_t)i].t1 - pl.suf_segs[(size_t)i].t0;
    tmax = std::max(tmax, tok[(size_t)b]);
  }
  const size_t bytes = sizeof(unsigned long long) * words * (size_t)ctas;
  unsigned long long* d_st = nullptr;
  cudaError_t e = cudaMalloc(&d_st, bytes);
  if (e != cudaSuccess) return gk::cuda_fail(p, e, "cudaMalloc(timeline stamps)");
  std::vector<unsigned long long> h((size_t)words * ctas);
  const int n_sm = p->dev.num_sms;
  std::vector<std::vector<double>> rates((size_t)n_sm);
  cudaStream_t s = (cudaStream_t)stream;
  for (int r = 0; r < reps && st == GK_OK; ++r) {
    if ((e = cudaMemsetAsync(d_st, 0, bytes, s)) != cudaSuccess) {
      st = gk::cuda_fail(p, e, "cudaMemsetAsync(timeline stamps)");
      break;
    }
    gk::LaunchCommon lc{&p->cfg, p->d_error, n_sm};
    int le;
    if (split) {
      lc.split_stamps = d_st;
      if (!pl.slot_of_sm.empty()) {
        if (++p->split_epoch == 0) {
          if ((e = cudaMemsetAsync(p->d_slot_claim, 0, sizeof(uint32_t) * (size_t)n_sm, s)) != cudaSuccess) {
            st = gk::cuda_fail(p, e, "cudaMemsetAsync(slot claims)");
            break;
          }
          ++p->split_epoch;
        }
        lc.slot_claim = p->d_slot_claim;
        lc.epoch = p->split_epoch;
      }
      le = gk::launch_cascade_split(lc, stream, layer, batch, &pl);
    } else {
      lc.gather_stamps = d_st;
      le = gk::launch_gather(lc, stream, layer, batch, &pl, false);
    }
    if (le) {
      st = gk::cuda_fail(p, le, split ? "split cascade kernel" : "suffix gather kernel");
      break;
    }
    if ((e = cudaMemcpyAsync(h.data(), d_st, bytes, cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess) {
      st = gk::cuda_fail(p, e, "reading the timeline stamps");
      break;
    }
    // this launch's rates, each role scaled to its own mean
    std::vector<std::pair<int, double>> got[2];
    for (int b = 0; b < ctas; ++b) {
      const unsigned long long* w = &h[(size_t)words * b];
      const unsigned long long sm = w[0], t0 = split ? w[2] : w[1], t1 = split ? w[3] : w[2];
      if (sm >= (unsigned long long)n_sm || t1 <= t0 || 4 * tok[(size_t)b] < tmax) continue;
      got[b < n_pre ? 1 : 0].push_back({(int)sm, (double)tok[(size_t)b] / ((double)(t1 - t0) * 1e-3)});
    }
    for (auto& role : got) {
      double mean = 0.0;
      for (auto& x : role) mean += x.second;
      if (role.empty() || mean <= 0.0) continue;
      mean /= (double)role.size();
      for (auto& x : role) rates[(size_t)x.first].push_back(x.second / mean);
    }
  }
  cudaFree(d_st);
  if (st != GK_OK) return st;
  std::vector<float> v((size_t)n_sm, 1.0f);
  int have = 0;
  for (int sm = 0; sm < n_sm; ++sm)
    if (!rates[(size_t)sm].empty()) {
      v[(size_t)sm] = (float)gk::median(rates[(size_t)sm]);
      ++have;
    }
  if (have == 0) return gk::fail(p, GK_ERR_INVALID, "no CTA of the plan's gather gave a speed");
  st = gk_pool_set_sm_speeds(pool, v.data(), n_sm);
  if (st != GK_OK) return st;
  if (speeds) gk_pool_get_sm_speeds(pool, speeds, &have);
  return GK_OK;
}
