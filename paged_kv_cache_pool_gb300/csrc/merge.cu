// LSE merge kernel: combines the partial states (prefix splits and suffix
// segments of the cascade, or the segments of a request the flat backend split)
// into each request's output and log-sum-exp.
#include <algorithm>
#include <cmath>

#include "device_common.cuh"
#include "gk_internal.h"

namespace gk {
namespace {

// LSE merge (GraniKV Eq. 1, applied to any number of partial states): for each
// request and query head, O = sum_e 2^(l_e - m) O_e / sum_e 2^(l_e - m),
// LSE = (m + log2 sum_e 2^(l_e - m)) * ln 2, with m = max_e l_e (log2 domain).
// One warp per (request, query head): entries [e0, e0 + ne).  Lane e holds
// entry e's LSE and weight (entries beyond 32 are folded in a second round);
// the d-wide rows are read ROWS entries per round trip, every load of a round
// in flight before any is used: 8 (128 registers, two 256-thread blocks per
// SM) or 4 (64 registers, four blocks per SM); the launch picks the variant
// with fewer (round trips x waves of warps).  Partial states come from other
// CTAs, so they are read at L2 (ld.global.cg).
template <int ROWS>
__device__ __forceinline__ void merge_head(const float* part_o, const float* part_l, int e0, int ne, int r, int qh,
                                           int Hq, int D, float* out, float* lse) {
  const int lane = threadIdx.x & 31;
  const int vecs = D / 4;  // float4 per row: 16 or 32
  const bool has = lane < vecs;
  // rows c .. c + N - 1 of the block of 32 partial states starting at eb (nb of them valid)
  auto load_rows = [&](auto& v, int eb, int c, int nb) {
    constexpr int N = sizeof(v) / sizeof(float4);
#pragma unroll
    for (int k = 0; k < N; ++k)
      v[k] = (has && c + k < nb)
                 ? __ldcg(reinterpret_cast<const float4*>(part_o + ((int64_t)(e0 + eb + c + k) * Hq + qh) * D) + lane)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  // The LSE of the first 32 partial states and the O rows of the first ROWS are
  // requested together: the rows do not depend on the weights, so a request
  // with few partial states waits for one round trip to L2, not two.
  const float l0 = lane < ne ? __ldcg(part_l + (int64_t)(e0 + lane) * Hq + qh) : -INFINITY;
  float4 v0[ROWS];
  load_rows(v0, 0, 0, min(32, ne));
  float mx = l0;
  for (int e = lane + 32; e < ne; e += 32) mx = fmaxf(mx, __ldcg(part_l + (int64_t)(e0 + e) * Hq + qh));
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  float z = 0.f;
  if (mx != -INFINITY) {
    // a state of weight 0 (LSE -inf: an empty state, whose O row may never have
    // been written) contributes nothing, whatever its row holds
    auto accumulate = [&](const auto& v, float w, int c) {
      constexpr int N = sizeof(v) / sizeof(float4);
#pragma unroll
      for (int k = 0; k < N; ++k) {
        const float wk = __shfl_sync(0xffffffffu, w, (c + k) & 31);
        if (wk != 0.f) {
          o.x = fmaf(wk, v[k].x, o.x);
          o.y = fmaf(wk, v[k].y, o.y);
          o.z = fmaf(wk, v[k].z, o.z);
          o.w = fmaf(wk, v[k].w, o.w);
        }
      }
    };
    for (int eb = 0; eb < ne; eb += 32) {
      const int e = eb + lane;
      const float le = eb == 0 ? l0 : (e < ne ? __ldcg(part_l + (int64_t)(e0 + e) * Hq + qh) : -INFINITY);
      const float w = e < ne ? ex2(le - mx) : 0.f;
      float wz = w;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) wz += __shfl_xor_sync(0xffffffffu, wz, off);
      z += wz;
      const int nb = min(32, ne - eb);
      int c = 0;
      if (eb == 0) {
        accumulate(v0, w, 0);
        c = ROWS;
      }
      for (; c < nb; c += ROWS) {
        float4 v[ROWS];
        load_rows(v, eb, c, nb);
        accumulate(v, w, c);
      }
    }
    const float inv = 1.f / z;
    o.x *= inv; o.y *= inv; o.z *= inv; o.w *= inv;
  }
  if (has) reinterpret_cast<float4*>(out + ((int64_t)r * Hq + qh) * D)[lane] = o;
  if (lane == 0 && lse) lse[(int64_t)r * Hq + qh] = mx == -INFINITY ? -INFINITY : (mx + __log2f(z)) * kLn2;
}

template <int ROWS>
__global__ void __launch_bounds__(256, ROWS == 4 ? 4 : 2) merge_kernel(const float* part_o, const float* part_l,
                                                                     const RequestDev* __restrict__ reqs, int32_t B,
                                                                     int32_t dense, int32_t Hq, int32_t D,
                                                                     float* __restrict__ out, float* __restrict__ lse) {
  griddep_launch_dependents();
  const int gw = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  if (gw >= B * Hq) return;
  const int r = gw / Hq, qh = gw % Hq;
  const RequestDev rq = reqs[r];
  griddep_wait();
  const int e0 = dense ? rq.entry_dense : rq.entry_cas;
  const int ne = dense ? rq.n_entry_dense : rq.n_entry_cas;
  if (ne < 0) return;  // written directly by its only segment
  merge_head<ROWS>(part_o, part_l, e0, ne, r, qh, Hq, D, out, lse);
}

}  // namespace

int launch_merge(const LaunchCommon& lc, void* stream, const gk_batch* b, const Plan* pl, bool dense) {
  const gk_pool_config& c = *lc.cfg;
  const uint8_t* base = (const uint8_t*)pl->d_buf;
  const int64_t warps = (int64_t)pl->B * c.num_q_heads;
  const int blocks = (int)((warps + 7) / 8);
  // Latency-bound: each warp waits ceil(partial states / ROWS) round trips, and
  // warps run in waves of (SMs x resident warps); take the variant with the
  // smaller product (the 8-row one on a tie).
  const double avg = (double)(dense ? pl->n_entries_dense : pl->n_entries_cas) / std::max(1, pl->B);
  auto cost = [&](int rows, int warps_per_sm) {
    const int64_t wave = (int64_t)std::max(1, lc.num_sms) * warps_per_sm;
    return std::ceil(avg / rows) * (double)((warps + wave - 1) / wave);
  };
  const bool four = cost(4, 32) < cost(8, 16);
  return (int)launch_pdl(four ? merge_kernel<4> : merge_kernel<8>, dim3(blocks), dim3(256), 0, (cudaStream_t)stream,
                         pl->d_part_o, pl->d_part_l, (const RequestDev*)(base + pl->off_reqs), pl->B, dense ? 1 : 0,
                         c.num_q_heads, c.head_dim, b->d_out, b->d_lse);
}

}  // namespace gk
