// Gather attention (suffix kernel and flat/dense backend) and the LSE merge.
//
// Suffix kernel (GraniKV Section 3.3 / 3.5, cascade level 1): each request's
// COLD tokens are gathered through its block table ("Paged KV cache", How it
// works step 3: slot = table[t / P] * P + t % P) and attended with an online
// softmax.  Dense backend: the same kernel walks a request's whole context,
// its HOT prefix (contiguous per KV head, re-read for every request) then its
// COLD suffix, the flat paged decode the pages compare against.
//
// Work split: the plan cuts the concatenated token stream of all requests into
// one equal quota per resident CTA (persistent grid); a quota that spans a
// request boundary yields one segment per request.  Each segment produces a
// partial (O, LSE) state or, when it covers a whole request, the final output.
//
// CTA layout: warps 0..Hkv-1 are consumers (warp h = KV head h, its g query
// heads), warp Hkv is the producer.  The producer moves T tokens per stage
// into shared memory with bulk async copies (the TMA engine; one 16-byte
// aligned copy per COLD token row of Hkv*d bf16, or per HOT head run of T*d)
// and signals an mbarrier; consumers read 16-byte vectors from shared memory,
// reduce q.k across the lanes of a token with warp shuffles and keep a
// running max / sum (online softmax) in registers.
#include <cfloat>

#include "device_common.cuh"
#include "gk_internal.h"

namespace gk {
namespace {

constexpr int kT = 8;       // tokens per stage
constexpr int kStages = 3;  // pipeline depth

struct GatherParams {
  const uint16_t* hot_k;
  const uint16_t* hot_v;
  const uint16_t* cold_k;
  const uint16_t* cold_v;
  int64_t cold_slots;
  int64_t n_blocks;
  int32_t L, Hkv, Hq, page;
  int32_t layer;
  int32_t dense;
  const int32_t* block_table;
  int32_t max_blocks;
  const uint16_t* q;
  float* out;
  float* lse;
  float* part_o;
  float* part_l;
  const RequestDev* reqs;
  const int32_t* seg_begin;
  const SegmentDev* segs;
  int32_t* err;
  float q_scale;  // log2(e) / sqrt(d): scores come out in the log2 domain
};

__host__ __device__ constexpr size_t stage_bytes(int hkv, int d) { return (size_t)kT * hkv * d * 2; }

template <int D, int G>
__global__ void __launch_bounds__(32 * (kMaxKvHeads + 1), (G <= 4 ? 2 : 1)) gather_kernel(const GatherParams p) {
  constexpr int LPT = D / 8;     // lanes per token row (one 16-byte vector each)
  constexpr int TPI = 32 / LPT;  // token rows per warp-wide vector load
  constexpr int R = kT / TPI;    // rows per lane per stage
  static_assert(kT % TPI == 0, "stage must hold whole warp loads");

  extern __shared__ __align__(1024) uint8_t smem[];
  const int Hkv = p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t sb = stage_bytes(Hkv, D);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kStages * sb);
  const uint32_t smem0 = smem_u32(smem);
  auto k_stage = [&](int s) { return smem0 + (uint32_t)(2 * s * sb); };
  auto v_stage = [&](int s) { return smem0 + (uint32_t)((2 * s + 1) * sb); };
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[kStages + s]); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), Hkv);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int seg0 = p.seg_begin[blockIdx.x], seg1 = p.seg_begin[blockIdx.x + 1];
  const int64_t layer_rows = (int64_t)p.layer * p.cold_slots;

  if (warp == Hkv) {
    // ------------------------------- producer -------------------------------
    int k = 0;
    bool ok = true;
    for (int sg = seg0; sg < seg1 && ok; ++sg) {
      const SegmentDev seg = p.segs[sg];
      const RequestDev rq = p.reqs[seg.req];
      const int lp = p.dense ? rq.lp : 0;
      const int32_t* table = p.block_table + (int64_t)seg.req * p.max_blocks;
      for (int t = seg.t0; t < seg.t1;) {
        int n = min(kT, seg.t1 - t);
        if (t < lp) n = min(n, lp - t);
        const int s = k % kStages;
        const int round = k / kStages;
        if (round > 0 && !mbar_wait(empty_bar(s), (round - 1) & 1, p.err)) {
          ok = false;
          break;
        }
        const uint16_t *src_k = nullptr, *src_v = nullptr;
        uint32_t dst_off = 0, unit_bytes;
        bool issue;
        if (t < lp) {
          // HOT: one run of n tokens per head; slab layout [L][Hkv][Lp][d]
          unit_bytes = (uint32_t)n * D * 2;
          issue = lane < Hkv;
          if (issue) {
            int64_t row = rq.hot_base * (int64_t)p.L * Hkv + ((int64_t)p.layer * Hkv + lane) * lp + t;
            src_k = p.hot_k + row * D;
            src_v = p.hot_v + row * D;
            dst_off = (uint32_t)lane * kT * D * 2;
          }
        } else {
          // COLD: one row of Hkv*d per token, through the block table
          unit_bytes = (uint32_t)Hkv * D * 2;
          issue = false;
          if (lane < n) {
            int64_t tt = (int64_t)(t - lp) + lane;
            int32_t blk = table[tt / p.page];
            if (blk >= 0 && blk < p.n_blocks) {
              int64_t slot = (int64_t)blk * p.page + tt % p.page;
              src_k = p.cold_k + (layer_rows + slot) * Hkv * D;
              src_v = p.cold_v + (layer_rows + slot) * Hkv * D;
              dst_off = (uint32_t)lane * Hkv * D * 2;
              issue = true;
            } else {
              report_error(p.err, kErrBounds);
            }
          }
        }
        const unsigned mask = __ballot_sync(0xffffffffu, issue);
        if (lane == 0) mbar_arrive_expect_tx(full_bar(s), (uint32_t)__popc(mask) * unit_bytes * 2);
        __syncwarp();
        if (issue) {
          bulk_g2s(k_stage(s) + dst_off, src_k, unit_bytes, full_bar(s));
          bulk_g2s(v_stage(s) + dst_off, src_v, unit_bytes, full_bar(s));
        }
        t += n;
        ++k;
      }
    }
    if (!ok) {
      // an abort: let copies already in flight land before the CTA exits
      for (int j = max(0, k - kStages); j < k; ++j) mbar_wait(full_bar(j % kStages), (j / kStages) & 1, nullptr);
    }
    return;
  }
  if (warp > Hkv) return;

  // ------------------------------- consumers --------------------------------
  const int h = warp;
  const int sub = lane % LPT;  // 8-dim slice [8*sub, 8*sub+8)
  const int grp = lane / LPT;  // token row within a warp load
  int k = 0;
  for (int sg = seg0; sg < seg1; ++sg) {
    const SegmentDev seg = p.segs[sg];
    const RequestDev rq = p.reqs[seg.req];
    const int lp = p.dense ? rq.lp : 0;

    float qf[G][8];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const uint4 w = *reinterpret_cast<const uint4*>(p.q + ((int64_t)seg.req * p.Hq + h * G + j) * D + sub * 8);
      qf[j][0] = bf_lo(w.x) * p.q_scale; qf[j][1] = bf_hi(w.x) * p.q_scale;
      qf[j][2] = bf_lo(w.y) * p.q_scale; qf[j][3] = bf_hi(w.y) * p.q_scale;
      qf[j][4] = bf_lo(w.z) * p.q_scale; qf[j][5] = bf_hi(w.z) * p.q_scale;
      qf[j][6] = bf_lo(w.w) * p.q_scale; qf[j][7] = bf_hi(w.w) * p.q_scale;
    }
    float m[G], ls[G], acc[G][8];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      m[j] = -INFINITY;
      ls[j] = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
    }

    bool ok = true;
    for (int t = seg.t0; t < seg.t1;) {
      int n = min(kT, seg.t1 - t);
      if (t < lp) n = min(n, lp - t);
      const int s = k % kStages;
      if (!mbar_wait(full_bar(s), (k / kStages) & 1, p.err)) {
        ok = false;
        break;
      }
      const bool hot = t < lp;
      const uint32_t tok_stride = hot ? D * 2 : (uint32_t)Hkv * D * 2;
      const uint32_t head_off = hot ? (uint32_t)h * kT * D * 2 : (uint32_t)h * D * 2;
      const uint32_t kb = k_stage(s) + head_off + sub * 16;
      const uint32_t vb = v_stage(s) + head_off + sub * 16;

      float sc[R][G];
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const uint4 w = lds128(kb + (uint32_t)(i * TPI + grp) * tok_stride);
        float kf[8] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y), bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w)};
#pragma unroll
        for (int j = 0; j < G; ++j) {
          float a = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) a = fmaf(qf[j][e], kf[e], a);
          sc[i][j] = a;
        }
      }
#pragma unroll
      for (int off = LPT / 2; off >= 1; off >>= 1)
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
          for (int j = 0; j < G; ++j) sc[i][j] += __shfl_xor_sync(0xffffffffu, sc[i][j], off);

      float alpha[G];
#pragma unroll
      for (int j = 0; j < G; ++j) {
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < R; ++i) {
          if (i * TPI + grp >= n) sc[i][j] = -INFINITY;
          mx = fmaxf(mx, sc[i][j]);
        }
#pragma unroll
        for (int off = LPT; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float mn = fmaxf(m[j], mx);
        alpha[j] = ex2(m[j] - mn);
        m[j] = mn;
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i) {
          sc[i][j] = ex2(sc[i][j] - mn);
          sum += sc[i][j];
        }
        ls[j] = ls[j] * alpha[j] + sum;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j][e] *= alpha[j];
      }
#pragma unroll
      for (int i = 0; i < R; ++i) {
        uint4 w = lds128(vb + (uint32_t)(i * TPI + grp) * tok_stride);
        if (i * TPI + grp >= n) w = make_uint4(0, 0, 0, 0);
        float vf[8] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y), bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w)};
#pragma unroll
        for (int j = 0; j < G; ++j)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[j][e] = fmaf(sc[i][j], vf[e], acc[j][e]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));
      t += n;
      ++k;
    }
    if (!ok) return;

    // combine the token rows of the warp (lanes with the same 8-dim slice)
#pragma unroll
    for (int off = LPT; off < 32; off <<= 1)
#pragma unroll
      for (int j = 0; j < G; ++j) {
        ls[j] += __shfl_xor_sync(0xffffffffu, ls[j], off);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j][e] += __shfl_xor_sync(0xffffffffu, acc[j][e], off);
      }
    if (grp == 0) {
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const float inv = 1.f / ls[j];
        const float lse2 = m[j] + __log2f(ls[j]);
        const int qh = h * G + j;
        float4 o0 = make_float4(acc[j][0] * inv, acc[j][1] * inv, acc[j][2] * inv, acc[j][3] * inv);
        float4 o1 = make_float4(acc[j][4] * inv, acc[j][5] * inv, acc[j][6] * inv, acc[j][7] * inv);
        float* dst;
        if (seg.entry >= 0) {
          dst = p.part_o + ((int64_t)seg.entry * p.Hq + qh) * D + sub * 8;
          if (sub == 0) p.part_l[(int64_t)seg.entry * p.Hq + qh] = lse2;
        } else {
          dst = p.out + ((int64_t)seg.req * p.Hq + qh) * D + sub * 8;
          if (sub == 0 && p.lse) p.lse[(int64_t)seg.req * p.Hq + qh] = lse2 * kLn2;
        }
        reinterpret_cast<float4*>(dst)[0] = o0;
        reinterpret_cast<float4*>(dst)[1] = o1;
      }
    }
  }
}

// LSE merge (GraniKV Eq. 1, applied to any number of partial states): for each
// request and query head, O = sum_e 2^(l_e - m) O_e / sum_e 2^(l_e - m),
// LSE = (m + log2 sum_e 2^(l_e - m)) * ln 2, with m = max_e l_e (log2 domain).
// One warp per (request, query head): lanes first reduce the max over the
// entries' LSEs, then each lane accumulates its 4-float slice of d.
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_l,
                                                    const RequestDev* __restrict__ reqs, int32_t B, int32_t dense,
                                                    int32_t Hq, int32_t D, float* __restrict__ out,
                                                    float* __restrict__ lse) {
  const int gw = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= B * Hq) return;
  const int r = gw / Hq, qh = gw % Hq;
  const RequestDev rq = reqs[r];
  const int e0 = dense ? rq.entry_dense : rq.entry_cas;
  const int ne = dense ? rq.n_entry_dense : rq.n_entry_cas;
  if (ne < 0) return;  // written directly by its only segment
  float mx = -INFINITY;
  for (int e = lane; e < ne; e += 32) mx = fmaxf(mx, part_l[(int64_t)(e0 + e) * Hq + qh]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  const int vecs = D / 4;  // 16 or 32 float4 per row
  float z = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  if (mx != -INFINITY && lane < vecs) {
#pragma unroll 4
    for (int e = 0; e < ne; ++e) {
      const float w = ex2(part_l[(int64_t)(e0 + e) * Hq + qh] - mx);
      const float4 pe = reinterpret_cast<const float4*>(part_o + ((int64_t)(e0 + e) * Hq + qh) * D)[lane];
      o.x = fmaf(w, pe.x, o.x);
      o.y = fmaf(w, pe.y, o.y);
      o.z = fmaf(w, pe.z, o.z);
      o.w = fmaf(w, pe.w, o.w);
      z += w;
    }
    const float inv = 1.f / z;
    o.x *= inv; o.y *= inv; o.z *= inv; o.w *= inv;
  }
  if (lane < vecs) reinterpret_cast<float4*>(out + ((int64_t)r * Hq + qh) * D)[lane] = o;
  if (lane == 0 && lse) lse[(int64_t)r * Hq + qh] = mx == -INFINITY ? -INFINITY : (mx + __log2f(z)) * kLn2;
}

template <int D, int G>
int launch_gather_t(const GatherParams& gp, int ctas, cudaStream_t st) {
  const size_t smem = 2 * kStages * stage_bytes(gp.Hkv, D) + 2 * kStages * sizeof(uint64_t);
  auto kern = gather_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  kern<<<ctas, 32 * (gp.Hkv + 1), smem, st>>>(gp);
  return (int)cudaGetLastError();
}

}  // namespace

int gather_ctas_per_sm(const gk_pool_config* cfg) {
  const size_t smem = 2 * kStages * stage_bytes(cfg->num_kv_heads, cfg->head_dim) + 1024;
  int by_smem = (int)((227 * 1024) / (smem + 1024));
  int threads = 32 * (cfg->num_kv_heads + 1);
  int by_threads = 2048 / threads;
  int g = cfg->num_q_heads / cfg->num_kv_heads;
  int by_regs = g <= 4 ? 2 : 1;   // register footprint grows with the query heads per warp
  int n = by_smem < by_threads ? by_smem : by_threads;
  n = n < by_regs ? n : by_regs;
  return n < 1 ? 1 : n;
}

int launch_gather(const LaunchCommon& lc, void* stream, int32_t layer, const gk_batch* b, const Plan* pl,
                  bool dense) {
  const gk_pool_config& c = *lc.cfg;
  GatherParams gp{};
  gp.hot_k = (const uint16_t*)c.hot_k;
  gp.hot_v = (const uint16_t*)c.hot_v;
  gp.cold_k = (const uint16_t*)c.cold_k;
  gp.cold_v = (const uint16_t*)c.cold_v;
  gp.cold_slots = c.cold_slots;
  gp.n_blocks = c.cold_slots / c.cold_page_size;
  gp.L = c.num_layers;
  gp.Hkv = c.num_kv_heads;
  gp.Hq = c.num_q_heads;
  gp.page = c.cold_page_size;
  gp.layer = layer;
  gp.dense = dense ? 1 : 0;
  gp.block_table = b->d_block_table;
  gp.max_blocks = b->max_blocks;
  gp.q = (const uint16_t*)b->d_q;
  gp.out = b->d_out;
  gp.lse = b->d_lse;
  gp.part_o = pl->d_part_o;
  gp.part_l = pl->d_part_l;
  const uint8_t* base = (const uint8_t*)pl->d_buf;
  gp.reqs = (const RequestDev*)(base + pl->off_reqs);
  gp.seg_begin = (const int32_t*)(base + (dense ? pl->off_dense_begin : pl->off_suf_begin));
  gp.segs = (const SegmentDev*)(base + (dense ? pl->off_dense_segs : pl->off_suf_segs));
  gp.err = lc.d_error;
  gp.q_scale = kLog2e / sqrtf((float)c.head_dim);
  const int ctas = dense ? pl->summary.dense_ctas : pl->summary.suffix_ctas;
  if (ctas <= 0) return 0;
  const int g = c.num_q_heads / c.num_kv_heads;
  cudaStream_t st = (cudaStream_t)stream;
  if (c.head_dim == 128) {
    switch (g) {
      case 1: return launch_gather_t<128, 1>(gp, ctas, st);
      case 2: return launch_gather_t<128, 2>(gp, ctas, st);
      case 4: return launch_gather_t<128, 4>(gp, ctas, st);
      case 5: return launch_gather_t<128, 5>(gp, ctas, st);
      case 8: return launch_gather_t<128, 8>(gp, ctas, st);
    }
  } else if (c.head_dim == 64) {
    switch (g) {
      case 1: return launch_gather_t<64, 1>(gp, ctas, st);
      case 2: return launch_gather_t<64, 2>(gp, ctas, st);
      case 4: return launch_gather_t<64, 4>(gp, ctas, st);
    }
  }
  return (int)cudaErrorInvalidValue;
}

int launch_merge(const LaunchCommon& lc, void* stream, const gk_batch* b, const Plan* pl, bool dense) {
  const gk_pool_config& c = *lc.cfg;
  const uint8_t* base = (const uint8_t*)pl->d_buf;
  const int64_t warps = (int64_t)pl->B * c.num_q_heads;
  const int blocks = (int)((warps + 7) / 8);
  merge_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(pl->d_part_o, pl->d_part_l,
                                                         (const RequestDev*)(base + pl->off_reqs), pl->B,
                                                         dense ? 1 : 0, c.num_q_heads, c.head_dim, b->d_out, b->d_lse);
  return (int)cudaGetLastError();
}

}  // namespace gk
