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
// CTA layout: warps 0..Hkv-1 are consumers (warp h = KV head h and its g query
// heads), warp Hkv is the producer.  The producer stages 16 tokens at a time in
// shared memory with the TMA engine: one 16-byte aligned bulk copy per COLD
// token (its Hkv*d row of K, and of V), rows placed 16 bytes apart modulo 128
// so that eight consecutive tokens fall in eight different bank groups; HOT
// runs (dense backend) arrive as 128-byte-swizzled tensor tiles.  Consumers
// load 8x8 tiles with ldmatrix and run the two small per-head products on the
// warp-level tensor-core MMA (m16n8k16, bf16 in, fp32 accumulate):
//   S^T[16 tok x 8] = K[16 tok x d] . Q_h^T[d x 8]   (the g query heads, padded to 8)
//   O^T[d x 8]     += V^T[d x 16 tok] . P^T[16 tok x 8]
// with the online softmax (running max, rescale, sum) on the S^T fragments and
// warp shuffles across the lanes that hold one head.  P^T is re-packed into
// the B-operand layout with movmatrix.  The K/V rows do not form any operand
// layout the 5th-generation MMA reads from shared memory (they are 256-byte
// runs at a 2 KB stride), and this product is 2*g flops per byte: the kernel
// is bound by HBM, the MMA only keeps the issue slots free for it.
#include <cfloat>

#include "device_common.cuh"
#include "gk_internal.h"

namespace gk {
namespace {

constexpr int kT = kGatherT;  // tokens per stage (one m16 / k16 MMA step)
constexpr int kStages = 3;    // pipeline depth

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
  const uint8_t* tmaps;
  int32_t* err;
  float q_scale;  // log2(e) / sqrt(d): scores come out in the log2 domain
};

// shared-memory geometry of one K (or V) stage
__host__ __device__ constexpr uint32_t cold_row_bytes(int hkv, int d) { return (uint32_t)hkv * d * 2 + 16; }
__host__ __device__ constexpr uint32_t half_stage_bytes(int hkv, int d) {
  // max of the COLD rows (kT x row) and the HOT tiles (hkv x d/64 regions of kT x 128 B), 1 KB aligned
  uint32_t cold = (uint32_t)kT * cold_row_bytes(hkv, d);
  uint32_t hot = (uint32_t)hkv * (d / 64) * kT * 128;
  uint32_t m = cold > hot ? cold : hot;
  return (m + 1023u) & ~1023u;
}
__host__ __device__ constexpr size_t gather_smem_bytes(int hkv, int d) {
  return 1024 + 2 * kStages * (size_t)half_stage_bytes(hkv, d) + 2 * kStages * 8;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// D = A(16x16, row) . B(16x8, col) + D ; bf16 in, fp32 accumulate
__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int D, int G>
__global__ void __launch_bounds__(32 * (kMaxKvHeads + 1), 1) gather_kernel(const GatherParams p) {
  constexpr int KSTEPS = D / 16;  // k16 steps of the QK product, m16 tiles of the PV product
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const int Hkv = p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t hs = half_stage_bytes(Hkv, D);
  const uint32_t rs = cold_row_bytes(Hkv, D);
  auto k_stage = [&](int s) { return base + (uint32_t)(2 * s) * hs; };
  auto v_stage = [&](int s) { return base + (uint32_t)(2 * s + 1) * hs; };
  const uint32_t bars = base + 2 * kStages * hs;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };

  griddep_launch_dependents();
  // Zero the stages once: a partial stage leaves rows past its tokens untouched,
  // and those rows must hold finite values (they meet P = 0 in the MMA).
  for (uint32_t off = threadIdx.x * 16; off < 2 * kStages * hs; off += blockDim.x * 16)
    sts128(base + off, make_uint4(0, 0, 0, 0));
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), Hkv);
    }
    fence_mbar_init();
  }
  fence_async_shared();
  __syncthreads();
  griddep_wait();   // queries, pool rows and the partial-state buffer are written upstream

  const int seg0 = p.seg_begin[blockIdx.x], seg1 = p.seg_begin[blockIdx.x + 1];
  const int64_t layer_rows = (int64_t)p.layer * p.cold_slots;

  if (warp == Hkv) {
    // ------------------------------- producer -------------------------------
    // Stages are visited in the consumers' order.  The block ids of the next
    // stage are loaded while this stage's buffer is awaited, so the table
    // lookup never sits between a free buffer and its copies.
    struct SegState {
      SegmentDev seg;
      int lp;
      int64_t hot_base;
      const int32_t* table;
      const uint8_t* tm;
    };
    auto seg_state = [&](int sg) {
      SegState st;
      st.seg = p.segs[sg];
      const RequestDev rq = p.reqs[st.seg.req];
      st.lp = p.dense ? rq.lp : 0;
      st.hot_base = rq.hot_base;
      st.table = p.block_table + (int64_t)st.seg.req * p.max_blocks;
      st.tm = rq.group >= 0 ? p.tmaps + (size_t)(4 * rq.group + 2) * 128 : nullptr;
      return st;
    };
    auto stage_len = [&](const SegState& st, int t) {
      int n = min(kT, st.seg.t1 - t);
      if (t < st.lp) n = min(n, st.lp - t);
      return n;
    };
    auto block_id = [&](const SegState& st, int t, int n) -> int32_t {
      if (t < st.lp || lane >= n) return -1;
      return st.table[((int64_t)(t - st.lp) + lane) / p.page];
    };
    int k = 0;
    bool ok = seg0 < seg1;
    SegState cur{};
    int t = 0, sg = seg0;
    int32_t blk = -1;
    if (ok) {
      cur = seg_state(sg);
      t = cur.seg.t0;
      blk = block_id(cur, t, stage_len(cur, t));
      if (cur.lp > 0 && lane == 0) {
        tmap_acquire(cur.tm);
        tmap_acquire(cur.tm + 128);
      }
    }
    while (ok) {
      const int n = stage_len(cur, t);
      // next stage position and its block ids (prefetch)
      SegState nxt = cur;
      int t_next = t + n, sg_next = sg;
      bool has_next = true;
      if (t_next >= cur.seg.t1) {
        sg_next = sg + 1;
        has_next = sg_next < seg1;
        if (has_next) {
          nxt = seg_state(sg_next);
          t_next = nxt.seg.t0;
        }
      }
      const int32_t blk_next = has_next ? block_id(nxt, t_next, stage_len(nxt, t_next)) : -1;

      const int s = k % kStages;
      const int round = k / kStages;
      if (round > 0 && !mbar_wait(empty_bar(s), (round - 1) & 1, p.err)) {
        ok = false;
        break;
      }
      if (t < cur.lp) {
        // HOT: per head, D/64 swizzled boxes of 16 keys x 64 dims (zeros past Lp)
        if (lane == 0) {
          const uint32_t bytes = (uint32_t)Hkv * (D / 64) * kT * 128;
          mbar_arrive_expect_tx(full_bar(s), 2 * bytes);
          for (int h = 0; h < Hkv; ++h)
            for (int x = 0; x < D / 64; ++x) {
              const uint32_t off = (uint32_t)(h * (D / 64) + x) * kT * 128;
              tma_load_3d(k_stage(s) + off, cur.tm, x * 64, t, p.layer * Hkv + h, full_bar(s));
              tma_load_3d(v_stage(s) + off, cur.tm + 128, x * 64, t, p.layer * Hkv + h, full_bar(s));
            }
        }
      } else {
        // COLD: one bulk copy per token row of Hkv*d through the block table
        bool issue = false;
        const uint16_t *src_k = nullptr, *src_v = nullptr;
        if (lane < n) {
          if (blk >= 0 && blk < p.n_blocks) {
            const int64_t slot = (int64_t)blk * p.page + ((int64_t)(t - cur.lp) + lane) % p.page;
            src_k = p.cold_k + (layer_rows + slot) * Hkv * D;
            src_v = p.cold_v + (layer_rows + slot) * Hkv * D;
            issue = true;
          } else {
            report_error(p.err, kErrBounds);
          }
        }
        const unsigned mask = __ballot_sync(0xffffffffu, issue);
        const uint32_t row = (uint32_t)Hkv * D * 2;
        if (lane == 0) mbar_arrive_expect_tx(full_bar(s), (uint32_t)__popc(mask) * row * 2);
        __syncwarp();
        if (issue) {
          bulk_g2s(k_stage(s) + lane * rs, src_k, row, full_bar(s));
          bulk_g2s(v_stage(s) + lane * rs, src_v, row, full_bar(s));
        }
      }
      __syncwarp();
      ++k;
      if (!has_next) break;
      if (sg_next != sg && nxt.lp > 0 && lane == 0) {
        tmap_acquire(nxt.tm);
        tmap_acquire(nxt.tm + 128);
      }
      cur = nxt;
      sg = sg_next;
      t = t_next;
      blk = blk_next;
    }
    if (!ok) {
      for (int j = max(0, k - kStages); j < k; ++j) mbar_wait(full_bar(j % kStages), (j / kStages) & 1, nullptr);
    }
    return;
  }

  // ------------------------------- consumers --------------------------------
  const int h = warp;
  const int gq = lane >> 2;  // fragment row group
  const int tq = lane & 3;   // fragment column pair
  const int mi = lane >> 3, mj = lane & 7;  // ldmatrix: matrix index, row within it
  int k = 0;
  for (int sg = seg0; sg < seg1; ++sg) {
    const SegmentDev seg = p.segs[sg];
    const int lp = p.dense ? p.reqs[seg.req].lp : 0;

    // Q_h^T as the B operand: b[kk][0] = (d 16kk+2tq, +1; head gq), b[kk][1] = (d +8, +9; head gq)
    uint32_t qb[KSTEPS][2];
    {
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + ((int64_t)seg.req * p.Hq + h * G + min(gq, G - 1)) * D);
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        qb[kk][0] = gq < G ? qrow[kk * 8 + tq] : 0u;
        qb[kk][1] = gq < G ? qrow[kk * 8 + 4 + tq] : 0u;
      }
    }
    float o[KSTEPS][4];
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2tq and 2tq+1

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
      // address of 16-byte chunk c of token row tok of head h in a stage
      auto chunk_addr = [&](uint32_t stage, int tok, int c) -> uint32_t {
        if (hot)
          return stage + (uint32_t)(h * (D / 64) + (c >> 3)) * kT * 128 + tok * 128 + ((((c & 7) ^ (tok & 7))) << 4);
        return stage + (uint32_t)tok * rs + (uint32_t)h * D * 2 + c * 16;
      };
      // S^T = K Q_h^T
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(chunk_addr(k_stage(s), mj + 8 * (mi & 1), 2 * kk + (mi >> 1)), a0, a1, a2, a3);
        mma16816(sc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
      }
      // online softmax over the 16 tokens (rows gq and gq+8) for heads 2tq, 2tq+1
      const bool v_lo = gq < n, v_hi = gq + 8 < n;
      const float s00 = v_lo ? sc[0] * p.q_scale : -INFINITY;
      const float s01 = v_lo ? sc[1] * p.q_scale : -INFINITY;
      const float s10 = v_hi ? sc[2] * p.q_scale : -INFINITY;
      const float s11 = v_hi ? sc[3] * p.q_scale : -INFINITY;
      float x0 = fmaxf(s00, s10), x1 = fmaxf(s01, s11);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
      }
      const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
      if (__any_sync(0xffffffffu, n0 != m0 || n1 != m1)) {
        const float a0 = ex2(m0 - n0), a1 = ex2(m1 - n1);
        l0 *= a0;
        l1 *= a1;
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt) {
          o[mt][0] *= a0; o[mt][1] *= a1; o[mt][2] *= a0; o[mt][3] *= a1;
        }
        m0 = n0;
        m1 = n1;
      }
      const float p00 = ex2(s00 - m0), p01 = ex2(s01 - m1), p10 = ex2(s10 - m0), p11 = ex2(s11 - m1);
      l0 += p00 + p10;
      l1 += p01 + p11;
      // P^T (16 tok x 8 heads) -> B operand of the PV product
      const uint32_t pb0 = movm_t(pack_bf16x2(p00, p01));
      const uint32_t pb1 = movm_t(pack_bf16x2(p10, p11));
      // O^T += V^T P^T
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(chunk_addr(v_stage(s), mj + 8 * (mi >> 1), 2 * mt + (mi & 1)), a0, a1, a2, a3);
        mma16816(o[mt], a0, a1, a2, a3, pb0, pb1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));
      t += n;
      ++k;
    }
    if (!ok) return;

    // finish: the row sums live on the 8 lanes that share tq
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    const float i0 = 1.f / l0, i1 = 1.f / l1;
    const int hh0 = 2 * tq, hh1 = 2 * tq + 1;
    float* dst;
    float* dl;
    int64_t row0;
    if (seg.entry >= 0) {
      row0 = (int64_t)seg.entry * p.Hq + h * G;
      dst = p.part_o;
      dl = p.part_l;
    } else {
      row0 = (int64_t)seg.req * p.Hq + h * G;
      dst = p.out;
      dl = p.lse;
    }
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) {
      const int d0 = mt * 16 + gq;
      if (hh0 < G) {
        dst[(row0 + hh0) * D + d0] = o[mt][0] * i0;
        dst[(row0 + hh0) * D + d0 + 8] = o[mt][2] * i0;
      }
      if (hh1 < G) {
        dst[(row0 + hh1) * D + d0] = o[mt][1] * i1;
        dst[(row0 + hh1) * D + d0 + 8] = o[mt][3] * i1;
      }
    }
    if (gq == 0 && dl) {
      const float f = seg.entry >= 0 ? 1.f : kLn2;   // partials keep log2, outputs are natural log
      if (hh0 < G) dl[row0 + hh0] = (m0 + __log2f(l0)) * f;
      if (hh1 < G) dl[row0 + hh1] = (m1 + __log2f(l1)) * f;
    }
  }
}

// LSE merge (GraniKV Eq. 1, applied to any number of partial states): for each
// request and query head, O = sum_e 2^(l_e - m) O_e / sum_e 2^(l_e - m),
// LSE = (m + log2 sum_e 2^(l_e - m)) * ln 2, with m = max_e l_e (log2 domain).
// One warp per (request, query head).  Lane e holds entry e's LSE and weight
// (entries beyond 32 are folded in a second round); the d-wide rows are then
// read 16 entries at a time with every load in flight before any is used.
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_l,
                                                    const RequestDev* __restrict__ reqs, int32_t B, int32_t dense,
                                                    int32_t Hq, int32_t D, float* __restrict__ out,
                                                    float* __restrict__ lse) {
  griddep_launch_dependents();
  const int gw = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= B * Hq) return;
  const int r = gw / Hq, qh = gw % Hq;
  const RequestDev rq = reqs[r];
  griddep_wait();
  const int e0 = dense ? rq.entry_dense : rq.entry_cas;
  const int ne = dense ? rq.n_entry_dense : rq.n_entry_cas;
  if (ne < 0) return;  // written directly by its only segment
  float mx = -INFINITY;
  for (int e = lane; e < ne; e += 32) mx = fmaxf(mx, part_l[(int64_t)(e0 + e) * Hq + qh]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  const int vecs = D / 4;  // float4 per row: 16 or 32
  const bool has = lane < vecs;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  float z = 0.f;
  if (mx != -INFINITY) {
    for (int eb = 0; eb < ne; eb += 32) {
      const int e = eb + lane;
      const float w = e < ne ? ex2(part_l[(int64_t)(e0 + e) * Hq + qh] - mx) : 0.f;
      float wz = w;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) wz += __shfl_xor_sync(0xffffffffu, wz, off);
      z += wz;
      const int nb = min(32, ne - eb);
      for (int c0 = 0; c0 < nb; c0 += 16) {
        float4 v[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          v[k] = (has && c0 + k < nb)
                     ? reinterpret_cast<const float4*>(part_o + ((int64_t)(e0 + eb + c0 + k) * Hq + qh) * D)[lane]
                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float wk = __shfl_sync(0xffffffffu, w, (c0 + k) & 31);
          o.x = fmaf(wk, v[k].x, o.x);
          o.y = fmaf(wk, v[k].y, o.y);
          o.z = fmaf(wk, v[k].z, o.z);
          o.w = fmaf(wk, v[k].w, o.w);
        }
      }
    }
    const float inv = 1.f / z;
    o.x *= inv; o.y *= inv; o.z *= inv; o.w *= inv;
  }
  if (has) reinterpret_cast<float4*>(out + ((int64_t)r * Hq + qh) * D)[lane] = o;
  if (lane == 0 && lse) lse[(int64_t)r * Hq + qh] = mx == -INFINITY ? -INFINITY : (mx + __log2f(z)) * kLn2;
}

template <int D, int G>
int launch_gather_t(const GatherParams& gp, int ctas, cudaStream_t st) {
  const size_t smem = gather_smem_bytes(gp.Hkv, D);
  auto kern = gather_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  e = launch_pdl(kern, dim3(ctas), dim3(32 * (gp.Hkv + 1)), smem, st, gp);
  return (int)e;
}

}  // namespace

int gather_ctas_per_sm(const gk_pool_config* cfg) {
  const size_t smem = gather_smem_bytes(cfg->num_kv_heads, cfg->head_dim);
  int by_smem = (int)((228 * 1024) / (smem + 1024));
  int n = by_smem < 4 ? by_smem : 4;
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
  gp.tmaps = base + pl->off_tmaps;
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
  return (int)launch_pdl(merge_kernel, dim3(blocks), dim3(256), 0, (cudaStream_t)stream, pl->d_part_o,
                         pl->d_part_l, (const RequestDev*)(base + pl->off_reqs), pl->B, dense ? 1 : 0,
                         c.num_q_heads, c.head_dim, b->d_out, b->d_lse);
}

}  // namespace gk
