// Body of the small-M_eff cascade prefix kernel: the shared-prefix attention of
// GraniKV Section 3.5's cascade backend ("GKV-cascade"), in which the level-0
// kernel over the shared prefix is a FlashAttention-style tiled online softmax
// that reads each prefix K/V tile once per step.  The pages pair it with the
// fat shared-prefix matmul for the regime where the stacked rows M_eff =
// B_g * g are few (Section 3.6, Appendix B.4b): there the tensor-core item's
// fixed costs (tensor-memory allocation, a single issuing thread, the S -> P
// round trip through tensor memory per key tile, a 128-row tile of which a
// quarter is used) outweigh its throughput.
//
// One work item = up to 128 stacked rows x one KV head x one split of the
// prefix keys.  The item's rows form nrg groups of 16 (nrg <= 8); each group
// gets kw = 8 / pow2ceil(nrg) warps, and warp (group r, slice k) takes keys
// [k * 128 / kw, (k + 1) * 128 / kw) of every 128-key tile, so a few rows still
// keep all 8 warps busy (flash-decoding inside the CTA).  Lane 0 of warp 0
// also loads each 128-key K and V tile once with TMA through the prefix
// group's tensor maps (the same 128-byte swizzled [128 keys x 64] regions the
// tensor-core item reads; keys past Lp read as zeros), two stages deep, and
// every warp reads its slice from shared memory with ldmatrix.  Per chunk of
// CK keys (16, 32 or 64) a warp runs on the warp-level MMA (m16n8k16, bf16 in,
// fp32 accumulate):
//   S[16 x CK]  = Q_r[16 x d] . K^T         (Q_r staged in shared memory once)
//   P = 2^(S * log2e / sqrt(d) - m)           (online softmax, in registers)
//   O[16 x d]  += P[16 x CK] . V[CK x d]     (P re-packed from the S fragments)
// At the end the slices of a row group are combined by GraniKV Eq. 1 through
// shared memory (m = max of the slices' maxima, each slice weighted by
// 2^(m_k - m)).
// The running maximum is only raised (and O rescaled) when a row's maximum
// grows by more than 2^8, as in the tensor-core item; sum and output always
// use the same maximum.  The item writes each row's partial state (O
// normalised, LSE in log2) like the tensor-core item, so the merge (GraniKV
// Eq. 1) is unchanged.
#pragma once
#include <cuda.h>

#include "device_common.cuh"
#include "gk_internal.h"
#include "prefix_body.cuh"

namespace gk {
namespace prefix_warp {

constexpr int kRows = kPrefixWarpRows;   // stacked rows per item: 8 warps x 16
constexpr int kComputeWarps = kRows / 16;
constexpr int kThreads = 32 * kComputeWarps;   // 256: the block of a warp-item launch
constexpr int kProducerThread = 0;             // lane 0 of warp 0 also issues the TMA loads
constexpr int BN = kPrefixTileN;         // keys per K/V tile (the tensor maps' box)
constexpr int kChunk = 64;               // keys per online-softmax step
constexpr int NST = 2;                   // K/V pipeline depth
constexpr uint32_t kRegion = BN * 128;   // [128 keys x 64 bf16] swizzled region

template <int D>
struct Layout {
  static constexpr uint32_t kTile = (D / 64) * kRegion;   // one K or V tile
  static constexpr uint32_t kStage = 2 * kTile;            // K then V
  static constexpr uint32_t kQ = NST * kStage;             // the item's 128 query rows, same layout
  static constexpr uint32_t kData = kQ + kTile;
  // after the tiles, a key slice's state: O [16][D + 4] fp32 (padded rows), then (m, l) per row
  static constexpr uint32_t kStateRow = (D + 4) * 4;
  static constexpr uint32_t kState = 16 * kStateRow + 16 * 8;
  static_assert(kComputeWarps * kState <= kQ, "slice states fit in the K/V stages");
};

// barrier slots in the control block (the abort flag is the tensor-core item's)
enum : int { B_FULL = 0, B_EMPTY = NST, B_COUNT = 2 * NST };
static_assert(B_COUNT * 8 <= (int)prefix::kCtlTmemSlot, "warp item barriers overlap the control fields");

// shared address of 16-byte chunk c (0 .. D/8 - 1) of key row r of a tile stored
// as D/64 regions of 128-byte swizzled rows (chunk c & 7 of row r sits at
// (c & 7) ^ (r & 7); the regions are 1024-byte aligned)
__device__ __forceinline__ uint32_t swz(uint32_t tile, int r, int c) {
  return tile + (uint32_t)(c >> 3) * kRegion + (uint32_t)r * 128u + ((uint32_t)((c & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
// D(16x8) += A(16x16, row-major) . B(16x8, column-major); bf16 in, fp32 accumulate
__device__ __forceinline__ void mma(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}


// Bounded wait on the item's barriers; gives up when another thread of the CTA
// has (abort flag) or after kWaitLimitNs (and then records GK_ERR_TIMEOUT).
__device__ __forceinline__ bool wait_item(uint32_t bar, uint32_t parity, int32_t* err, volatile int* abort_flag) {
  return prefix::wait_or_abort(bar, parity, err, abort_flag);
}

// One chunk of CK keys (starting at key kc of the staged tile, nvalid keys of
// the tile inside the prefix) for the 16 rows at qrow0 of the staged queries:
// scores, online softmax with the lazy maximum, and O += P V.
template <int D, int CK>
__device__ __forceinline__ void chunk_step(uint32_t ks, uint32_t vs, uint32_t qs, int qrow0, int kc, int nvalid,
                                           float scale_log2, float (&o)[D / 8][4], float (&m_used)[2], float (&l)[2]) {
  constexpr int KS = D / 16, NT = D / 8, NS = CK / 8;
  const int lane = threadIdx.x & 31, tq = lane & 3;
  const int mi = lane >> 3, mr = lane & 7;   // ldmatrix: matrix index, row within it
  // S = Q K^T: NS n8 tiles of keys, the k16 steps two at a time
  float s[NS][4];
#pragma unroll
  for (int n = 0; n < NS; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < KS; kk += 2) {
    // A fragments of k16 steps kk and kk + 1: (rows 0-7 | 8-15) x (d 0-7 | 8-15)
    uint32_t qa[2][4];
#pragma unroll
    for (int t = 0; t < 2; ++t)
      ldsm4(swz(qs, qrow0 + mr + 8 * (mi & 1), 2 * (kk + t) + (mi >> 1)), qa[t][0], qa[t][1], qa[t][2], qa[t][3]);
#pragma unroll
    for (int n = 0; n < NS; ++n) {
      uint32_t b0, b1, b2, b3;
      ldsm4(swz(ks, kc + 8 * n + mr, 2 * kk + mi), b0, b1, b2, b3);
      mma(s[n], qa[0], b0, b1);
      mma(s[n], qa[1], b2, b3);
    }
  }
  // scale to the log2 domain, mask keys past the prefix, row maxima (rows gq, gq + 8)
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int n = 0; n < NS; ++n) {
    const int c = kc + 8 * n + 2 * tq;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float v = (c + (e & 1)) < nvalid ? s[n][e] * scale_log2 : -INFINITY;
      s[n][e] = v;
      mx[e >> 1] = fmaxf(mx[e >> 1], v);
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
    mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
  }
  if (__any_sync(0xffffffffu, mx[0] > m_used[0] + 8.0f || mx[1] > m_used[1] + 8.0f)) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float m_new = fmaxf(m_used[i], mx[i]);
      // a row seen for the first time has nothing to rescale (O and l are zero)
      const float f = m_used[i] == -INFINITY ? 1.f : ex2(m_used[i] - m_new);
      l[i] *= f;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][2 * i] *= f;
        o[n][2 * i + 1] *= f;
      }
      m_used[i] = m_new;
    }
  }
  // P = 2^(s - m), packed as the A operand of P V (k16 step kk2 = n8 tiles 2kk2, 2kk2 + 1)
  const float mu[2] = {m_used[0] == -INFINITY ? 0.f : m_used[0], m_used[1] == -INFINITY ? 0.f : m_used[1]};
  uint32_t pa[CK / 16][4];
#pragma unroll
  for (int n = 0; n < NS; ++n) {
    const float p0 = ex2(s[n][0] - mu[0]), p1 = ex2(s[n][1] - mu[0]);
    const float p2 = ex2(s[n][2] - mu[1]), p3 = ex2(s[n][3] - mu[1]);
    l[0] += p0 + p1;
    l[1] += p2 + p3;
    pa[n >> 1][(n & 1) * 2] = pack_bf16x2(p0, p1);
    pa[n >> 1][(n & 1) * 2 + 1] = pack_bf16x2(p2, p3);
  }
  // O += P V: V^T fragments by transposing loads, two n8 tiles of d at a time
#pragma unroll
  for (int kk2 = 0; kk2 < CK / 16; ++kk2) {
#pragma unroll
    for (int n = 0; n < NT; n += 2) {
      uint32_t b0, b1, b2, b3;
      ldsm4t(swz(vs, kc + 16 * kk2 + 8 * (mi & 1) + mr, n + (mi >> 1)), b0, b1, b2, b3);
      mma(o[n], pa[kk2], b0, b1);
      mma(o[n + 1], pa[kk2], b2, b3);
    }
  }
}

// named barrier over the item's active warps (n threads, a multiple of 32)
__device__ __forceinline__ void active_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// One work item (group, 128-row block, KV head, key split) on the first 256
// threads of the CTA (any further threads only pass the CTA-wide barriers).
// `base` is the 1024-byte aligned data area (Layout<D>::kData bytes), `ctl`
// the control block (prefix::kCtlBytes, generic pointer ctl_ptr) whose abort
// flag is zero on entry.  The barriers are initialised here and invalidated
// before returning.  The item executes griddepcontrol.wait itself after its
// reads of the plan's tables.  Returns false (on every thread) when a wait
// timed out; then no partial state of the item is written.
template <int D>
__device__ __forceinline__ bool warp_item(const prefix::PrefixParams& p, const PrefixItemDev it, uint32_t base,
                                          uint32_t ctl, uint8_t* ctl_ptr) {
  using Lay = Layout<D>;
  constexpr int NT = D / 8;    // n8 tiles of O
  auto bar = [&](int i) { return ctl + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctl_ptr + prefix::kCtlFlag);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PrefixGroupDev gr = p.groups[it.group];
  const int ntiles_all = (gr.lp + BN - 1) / BN;
  const int tile0 = it.split * gr.split_tiles;
  const int ntiles = min(gr.split_tiles, ntiles_all - tile0);
  const int key0 = tile0 * BN;
  const int row0 = it.mblock * kRows;
  // row groups of 16 rows with any valid row, key slices per group, warps in use
  const int nrg = max(0, min(kComputeWarps, (gr.m - row0 + 15) / 16));
  const int kw = nrg >= 5 ? 1 : (nrg >= 3 ? 2 : (nrg == 2 ? 4 : 8));
  const int nact = nrg * kw;
  const int rg = warp / kw, kslice = warp % kw, kpw = BN / kw;
  const void* tmK = p.tmaps + (size_t)gr.tmap_index * 128;
  const void* tmV = p.tmaps + (size_t)(gr.tmap_index + 1) * 128;
  const int zc = p.layer * p.Hkv + it.head;
  const bool compute = warp < nact && ntiles > 0;
  const int gq = lane >> 2, tq = lane & 3;   // fragment row group, column pair

  // the partial-state rows of this thread's fragment rows gq and gq + 8 (slice 0 stores them)
  int64_t dst[2] = {-1, -1};
  if (compute && kslice == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int grow = row0 + rg * 16 + gq + 8 * i;
      if (grow < gr.m) {
        const int req = p.prefix_reqs[gr.req_base + grow / p.G];
        dst[i] = ((int64_t)p.reqs[req].entry_cas + it.split) * p.Hq + it.head * p.G + grow % p.G;
      }
    }
  }
  if (threadIdx.x == kProducerThread) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), (uint32_t)max(nact, 1));
    }
    fence_mbar_init();
    if (ntiles > 0) {
      tmap_acquire(tmK);
      tmap_acquire(tmV);
    }
  }
  // The first K/V stages read only the HOT pool, which no kernel that may still
  // be running writes (the slab write lets the next kernel start only once it
  // has finished): they start before the dependency wait.  The plan's tables are
  // never written by a step's kernels; the queries and the partial states wait
  // for the kernel before.
  int issued = 0;
  if (threadIdx.x == kProducerThread && nact > 0) {
    for (int j = 0; j < NST && j < ntiles; ++j) {
      mbar_arrive_expect_tx(bar(B_FULL + j), Lay::kStage);
      for (int h = 0; h < D / 64; ++h) {
        tma_load_3d(base + j * Lay::kStage + h * kRegion, tmK, h * 64, key0 + j * BN, zc, bar(B_FULL + j));
        tma_load_3d(base + j * Lay::kStage + Lay::kTile + h * kRegion, tmV, h * 64, key0 + j * BN, zc,
                    bar(B_FULL + j));
      }
      issued = j + 1;
    }
  }
  griddep_wait();
  // Row group w's 16 query rows into shared memory by warp w (128-byte swizzled
  // like the K tiles, so the ldmatrix reads of the A fragments are conflict
  // free); rows past M_eff are zero.
  const uint32_t qs = base + Lay::kQ;
  if (warp < nrg && ntiles > 0) {
    constexpr int CPR = D / 8;   // 16-byte chunks per row
    for (int c = lane; c < 16 * CPR; c += 32) {
      const int r = c / CPR, ch = c % CPR;
      const int grow = row0 + warp * 16 + r;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (grow < gr.m) {
        const int req = p.prefix_reqs[gr.req_base + grow / p.G];
        const int qh = it.head * p.G + grow % p.G;
        v = reinterpret_cast<const uint4*>(p.q + ((int64_t)req * p.Hq + qh) * D)[ch];
      }
      sts128(swz(qs, warp * 16 + r, ch), v);
    }
  }
  __syncthreads();   // barriers initialised and queries staged before anyone uses them

  if (compute) {
    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_used[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    bool ok = true;
    const int k0 = kslice * kpw;   // this warp's keys of every tile: [k0, k0 + kpw)
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % NST;
      // warp-uniform: a lane that gave up takes its whole warp out of the loop
      if (!__all_sync(0xffffffffu, wait_item(bar(B_FULL + st), (j / NST) & 1, p.err, abort_flag))) {
        ok = false;
        break;
      }
      const uint32_t ks = base + st * Lay::kStage, vs = ks + Lay::kTile;
      const int nvalid = gr.lp - (key0 + j * BN);   // keys of this tile inside the prefix
      if (kw <= 2) {
#pragma unroll 1
        for (int kc = k0; kc < k0 + kpw && kc < nvalid; kc += 64)
          chunk_step<D, 64>(ks, vs, qs, rg * 16, kc, nvalid, p.scale_log2, o, m_used, l);
      } else if (kw == 4) {
        if (k0 < nvalid) chunk_step<D, 32>(ks, vs, qs, rg * 16, k0, nvalid, p.scale_log2, o, m_used, l);
      } else {
        if (k0 < nvalid) chunk_step<D, 16>(ks, vs, qs, rg * 16, k0, nvalid, p.scale_log2, o, m_used, l);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_EMPTY + st));   // this warp is done with the stage
      if (threadIdx.x == kProducerThread && j + NST < ntiles) {
        // refill the stage with tile j + NST once every active warp has released it
        if (wait_item(bar(B_EMPTY + st), (j / NST) & 1, p.err, abort_flag)) {
          mbar_arrive_expect_tx(bar(B_FULL + st), Lay::kStage);
          for (int h = 0; h < D / 64; ++h) {
            tma_load_3d(base + st * Lay::kStage + h * kRegion, tmK, h * 64, key0 + (j + NST) * BN, zc,
                        bar(B_FULL + st));
            tma_load_3d(base + st * Lay::kStage + Lay::kTile + h * kRegion, tmV, h * 64, key0 + (j + NST) * BN, zc,
                        bar(B_FULL + st));
          }
          issued = j + NST + 1;
        }
      }
      __syncwarp();
    }
    if (threadIdx.x == kProducerThread && *abort_flag) {
      // the loads already issued land before shared memory goes away
      for (int q = max(0, issued - NST); q < issued; ++q) mbar_wait(bar(B_FULL + q % NST), (q / NST) & 1, nullptr);
    }
    // row sums live on the 4 lanes of a quad
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      l[i] += __shfl_xor_sync(0xffffffffu, l[i], 1);
      l[i] += __shfl_xor_sync(0xffffffffu, l[i], 2);
    }
    if (kw > 1) {
      // Combine the key slices of each row group (GraniKV Eq. 1) through shared
      // memory.  Every active warp passes both barriers, also after an abort
      // (every wait above is bounded), so they always complete; after the
      // first, no tile is read any more and no load is in flight.
      active_sync(1, nact * 32);
      ok = *abort_flag == 0;
      if (ok && kslice != 0) {
        const uint32_t st_o = base + (uint32_t)warp * Lay::kState;
        const uint32_t st_ml = st_o + 16 * Lay::kStateRow;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint32_t row = st_o + (uint32_t)(gq + 8 * i) * Lay::kStateRow;
#pragma unroll
          for (int n = 0; n < NT; ++n)
            asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(row + (8 * n + 2 * tq) * 4), "f"(o[n][2 * i]),
                         "f"(o[n][2 * i + 1]) : "memory");
          if (tq == 0)
            asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(st_ml + (gq + 8 * i) * 8), "f"(m_used[i]), "f"(l[i])
                         : "memory");
        }
      }
      active_sync(2, nact * 32);
      if (ok && kslice == 0) {
        for (int k = 1; k < kw; ++k) {
          const uint32_t st_o = base + (uint32_t)(warp + k) * Lay::kState;
          const uint32_t st_ml = st_o + 16 * Lay::kStateRow;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            float m2, l2;
            asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(m2), "=f"(l2) : "r"(st_ml + (gq + 8 * i) * 8));
            const float mm = fmaxf(m_used[i], m2);
            const float f1 = m_used[i] == -INFINITY ? 0.f : ex2(m_used[i] - mm);
            const float f2 = m2 == -INFINITY ? 0.f : ex2(m2 - mm);
            l[i] = l[i] * f1 + l2 * f2;
            const uint32_t row = st_o + (uint32_t)(gq + 8 * i) * Lay::kStateRow;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              float a, b;
              asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(a), "=f"(b) : "r"(row + (8 * n + 2 * tq) * 4));
              o[n][2 * i] = o[n][2 * i] * f1 + a * f2;
              o[n][2 * i + 1] = o[n][2 * i + 1] * f1 + b * f2;
            }
            m_used[i] = mm;
          }
        }
      }
    }
    if (ok && kslice == 0) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (dst[i] < 0) continue;
        const float inv = 1.f / l[i];
        float* row = p.part_o + dst[i] * D;
#pragma unroll
        for (int n = 0; n < NT; ++n)
          *reinterpret_cast<float2*>(row + 8 * n + 2 * tq) = make_float2(o[n][2 * i] * inv, o[n][2 * i + 1] * inv);
        if (tq == 0) p.part_l[dst[i]] = m_used[i] + __log2f(l[i]);
      }
    }
  }
  // the staging area is rewritten by the next user of the shared memory (generic stores, or TMA)
  fence_async_shared();
  __syncthreads();
  const bool ok_all = *abort_flag == 0;
  if (threadIdx.x == kProducerThread)
    for (int i = 0; i < B_COUNT; ++i) mbar_inval(bar(i));
  return ok_all;
}

}  // namespace prefix_warp
}  // namespace gk
