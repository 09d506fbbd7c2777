// Body of the cascade prefix contraction on 5th-generation tensor cores, shared by
// the stand-alone prefix kernel and the fused per-layer cascade kernel.
//
// GraniKV Section 2.3 ("Shared-prefix matmul") and Section 3.5 (dense backend):
// all query rows that share a prefix -- every request of the group times its
// g = Hq/Hkv query heads of one KV head -- are stacked into one matrix Q
// [M = B_g * g, d], so prefix attention is a dense contraction
// O_p = softmax(Q K_p^T / sqrt(d)) V_p against the contiguous [Lp, d] slab of
// (layer, KV head), read once per step instead of once per request.
//
// One work item = 256 stacked rows (two 128-row Q tiles) x one KV head x one
// split of the prefix keys (the plan balances splits over the SMs).  For each tile of
// 128 keys the tensor core computes S_i = Q_i K^T into tensor memory (TMEM),
// softmax warpgroup i turns S_i into P_i = 2^(S_i*log2e/sqrt(d) - m) (bf16,
// written back over S_i in TMEM), and O_i += P_i V accumulates in TMEM with P_i
// as the TMEM-resident A operand.  The single MMA thread issues, per key tile j,
//     PV_0(j), S_0(j+1), PV_1(j), S_1(j+1)
// so each softmax warpgroup has the other tile's two MMA groups to hide behind.
// tcgen05.mma instructions from one thread complete in issue order, so
// observing S_i(j) also proves PV_i(j-1) has finished with P_i and O_i.  Tiles
// of 128 keys keep every MMA at 64 tensor cycles or more: issuing one costs the
// issuing thread about 50 cycles, so narrower tiles leave the tensor core
// waiting on the issue loop.  The running max m is only raised (and O_i
// rescaled in TMEM) when a row's max grows by more than 2^8; the row sum and
// the output always use the same m, so the result is exact up to rounding.
// Each item emits a partial state (O normalised, LSE in log2) per row; the merge
// combines the splits with the suffix states by GraniKV Eq. 1.
// An item whose rows fit one Q tile (a group's last, partly filled row block)
// has no second tile to hide its softmax behind; it double-buffers S instead:
// S(j+2) goes into the buffer P(j) leaves, issued right after PV(j), so the
// softmax of tile j+1 overlaps PV(j) and S(j+2).  There observing S(j) only
// proves PV(j-2) finished, so a rescale of O at tile j first waits for PV(j-1)
// (a barrier committed after every PV).  Such an item may also cover several
// consecutive key splits of its group (the planner gives it about twice the
// keys of a full item, as its tiles cost about half): it writes its state to
// the first split's entry and marks the others empty (LSE -inf).
//
// Warp roles (320 threads): warp 0 issues TMA loads (K and V tiles, two
// stages each), warp 1 owns tensor memory and issues every MMA from one thread,
// warps 2-5 and 6-9 are the softmax warpgroups of Q tiles 0 and 1 (they also
// stage Q and write the partial outputs).
//
// Shared-memory operand layout: every [rows x 64] bf16 region is the 128-byte
// swizzled K-major layout (8-row x 128-byte atoms, 16-byte chunk c of row r
// stored at chunk c ^ (r mod 8)), written by TMA for K and V and by the threads
// for Q.  V is consumed as the MN-major B operand (N = d), K and Q as K-major
// operands.
#pragma once
#include <cuda.h>

#include "device_common.cuh"
#include "gk_internal.h"

namespace gk {
namespace prefix {

constexpr int BM = kPrefixTileM;   // 128 rows per Q tile
constexpr int BN = kPrefixTileN;   // 128 keys per K/V tile
constexpr int NST = 2;             // K and V pipeline depth
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kRegionQ = BM * 128;   // [128 rows x 64 bf16] swizzled region
constexpr uint32_t kRegionKV = BN * 128;  // [128 keys x 64 bf16] swizzled region
constexpr int kThreads = 320;          // warp roles below; warps past the tenth (a larger
constexpr int kRoleWarps = kThreads / 32;  // block shared with another role) stay idle

struct PrefixParams {
  const PrefixGroupDev* groups;
  const int32_t* prefix_reqs;
  const PrefixItemDev* items;
  const RequestDev* reqs;
  const uint8_t* tmaps;
  const uint16_t* q;
  float* part_o;
  float* part_l;
  int32_t Hkv, Hq, G, layer;
  int32_t* err;
  float scale_log2;  // log2(e) / sqrt(d)
};

// barrier slots
enum : int {
  B_QFULL = 0,
  B_KFULL = 1,                // NST
  B_KEMPTY = B_KFULL + NST,   // NST
  B_VFULL = B_KEMPTY + NST,   // NST
  B_VEMPTY = B_VFULL + NST,   // NST
  B_SFULL = B_VEMPTY + NST,   // one per Q tile
  B_PFULL = B_SFULL + 2,      // one per Q tile
  B_OFINAL = B_PFULL + 2,
  B_ODONE = B_OFINAL + 1,     // single-tile items: one phase per PV product
  B_COUNT = B_ODONE + 1
};

template <int D>
struct Layout {
  static constexpr uint32_t kTile = BN * D * 2;      // one K or V tile
  static constexpr uint32_t kQTile = BM * D * 2;     // one Q tile
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + 2 * kQTile;
  static constexpr uint32_t kV = kK + NST * kTile;
  static constexpr uint32_t kData = kV + NST * kTile;   // Q, K and V staging
  static_assert(2 * BM * (D * 4 + 16) + 2 * BM * 8 <= kData, "epilogue staging must fit in the Q/K/V area");
};

// Control block (placed after the data area by the kernel that runs the items):
// the barriers, the tensor-memory address and the CTA's abort flag.
constexpr uint32_t kCtlTmemSlot = B_COUNT * 8;
constexpr uint32_t kCtlFlag = kCtlTmemSlot + 4;
constexpr uint32_t kCtlBytes = 128;
static_assert(kCtlFlag + 4 <= kCtlBytes, "prefix control block");

// tcgen05 shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// instruction descriptor, kind::f16: bf16 A and B, fp32 D, M = 128
__host__ __device__ constexpr uint32_t idesc(int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(BM >> 4) << 24);
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t id,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(id), "r"(accumulate));
}

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, int32_t* err, volatile int* abort_flag) {
  for (int i = 0; i < 64; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      report_error(err, kErrTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

// One work item (group, 256-row block, KV head, key split) on all 320 threads
// of the CTA.  `base` is the 1024-byte aligned data area (Layout<D>::kData
// bytes), `ctl` the control block (kCtlBytes, generic pointer ctl_ptr) whose
// abort flag is zero on entry; `tmem` holds 512 allocated columns.  The
// barriers are initialised here and invalidated before returning, so items can
// run back to back.  The item executes griddepcontrol.wait itself, after the
// reads of the plan's tables and the barrier set-up (callers do not wait for
// the previous kernel before calling it).  Returns false (on every thread) when
// a wait timed out.
template <int D>
__device__ __forceinline__ bool prefix_item(const PrefixParams& p, const PrefixItemDev it, uint32_t base, uint32_t ctl,
                                            uint8_t* ctl_ptr, uint32_t tmem) {
  using Lay = Layout<D>;
  const uint32_t sQ = base + Lay::kQ, sK = base + Lay::kK, sV = base + Lay::kV;
  auto bar = [&](int i) { return ctl + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctl_ptr + kCtlFlag);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PrefixGroupDev gr = p.groups[it.group];
  const int ntiles_all = (gr.lp + BN - 1) / BN;
  const int tile0 = it.split * gr.split_tiles;
  const int ntiles = min(gr.split_tiles * it.splits, ntiles_all - tile0);
  const int key0 = tile0 * BN;
  const int row0 = it.mblock * kPrefixRowsPerCta;
  const bool two = row0 + BM < gr.m;  // does Q tile 1 hold any row?  If not, S is double-buffered
  const void* tmK = p.tmaps + (size_t)gr.tmap_index * 128;
  const void* tmV = p.tmaps + (size_t)(gr.tmap_index + 1) * 128;
  const int zc = p.layer * p.Hkv + it.head;

  const int qi_ = (warp - 2) >> 2;
  const int row_ = (warp & 3) * 32 + lane;
  const int grow_ = row0 + qi_ * BM + row_;
  const bool softmax_warp = warp >= 2 && warp < kRoleWarps;
  const bool row_valid_ = softmax_warp && grow_ < gr.m;
  int req_ = 0, qh_ = 0;
  int64_t entry_ = -1;  // the row's partial-state slot
  if (row_valid_) {
    req_ = p.prefix_reqs[gr.req_base + grow_ / p.G];
    qh_ = it.head * p.G + grow_ % p.G;
    entry_ = (int64_t)p.reqs[req_].entry_cas + it.split;
  }
  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 256);
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_PFULL + i), 128);
    }
    mbar_init(bar(B_OFINAL), 1);
    mbar_init(bar(B_ODONE), 1);
    fence_mbar_init();
    if (ntiles > 0) {
      tmap_acquire(tmK);
      tmap_acquire(tmV);
      // The first K/V tiles need nothing but the barriers and the HOT pool, which no
      // kernel that may still be running writes (the slab write lets the next
      // kernel start only once it has finished): start them now, while the kernel
      // before this one finishes.
      for (int j = 0; j < NST && j < ntiles; ++j) {
        mbar_arrive_expect_tx(bar(B_KFULL + j), Lay::kTile);
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(sK + j * Lay::kTile + h * kRegionKV, tmK, h * 64, key0 + j * BN, zc, bar(B_KFULL + j));
        mbar_arrive_expect_tx(bar(B_VFULL + j), Lay::kTile);
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(sV + j * Lay::kTile + h * kRegionKV, tmV, h * 64, key0 + j * BN, zc, bar(B_VFULL + j));
      }
    }
  }
  // Everything above reads only the plan's tables, which the kernels of a step
  // never write, and the HOT pool, so it runs while the kernel before this one
  // finishes.  The queries and the partial states (the previous merge reads
  // them) wait for it.
  griddep_wait();
  // softmax threads fetch their Q row now, so the global-load latency overlaps the set-up
  uint4 qrow[D / 8];
  if (softmax_warp) {
    const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)req_ * p.Hq + qh_) * D);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) qrow[c] = row_valid_ ? src[c] : make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  tc_fence_after();
  // columns: S of Q tile i at i*128 (P is written over it); O of Q tile i at 256 + i*128
  auto tS = [&](int i) { return tmem + (uint32_t)(i * 128); };
  auto tO = [&](int i) { return tmem + 256u + (uint32_t)i * 128u; };

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0 && ntiles > 0) {
      int issued = 2 * min(NST, ntiles);   // the first stages, issued before the dependency wait
      for (int j = NST; j < ntiles; ++j) {
        const int st = j % NST, r = j / NST;
        if (!wait_or_abort(bar(B_KEMPTY + st), (r - 1) & 1, p.err, abort_flag)) break;
        mbar_arrive_expect_tx(bar(B_KFULL + st), Lay::kTile);
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(sK + st * Lay::kTile + h * kRegionKV, tmK, h * 64, key0 + j * BN, zc, bar(B_KFULL + st));
        issued = 2 * j + 1;
        if (!wait_or_abort(bar(B_VEMPTY + st), (r - 1) & 1, p.err, abort_flag)) break;
        mbar_arrive_expect_tx(bar(B_VFULL + st), Lay::kTile);
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(sV + st * Lay::kTile + h * kRegionKV, tmV, h * 64, key0 + j * BN, zc, bar(B_VFULL + st));
        issued = 2 * j + 2;
      }
      if (*abort_flag) {
        // let the loads already issued land before shared memory goes away
        for (int q = max(0, issued - 2 * NST); q < issued; ++q) {
          const int j = q / 2;
          mbar_wait(bar((q % 2 == 0 ? B_KFULL : B_VFULL) + j % NST), (j / NST) & 1, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t kIdQK = idesc(BN, false);
      constexpr uint32_t kIdPV = idesc(D, true);
      const int nq = two ? 2 : 1;
      // Descriptors are built once; an operand at a byte offset is the base
      // descriptor plus offset/16 in the start-address field.
      const uint64_t dQ = sdesc(sQ, 16, 1024), dK = sdesc(sK, 16, 1024), dV = sdesc(sV, kRegionKV, 1024);
      const uint32_t bar0 = ctl;
      const uint32_t tS0 = tmem, tO0 = tmem + 256u;
      bool ok = wait_or_abort(bar0 + 8u * B_QFULL, 0, p.err, abort_flag) &&
                wait_or_abort(bar0 + 8u * B_KFULL, 0, p.err, abort_flag);
      // S = Q_i K^T for key tile jt (K stage kst) into TMEM columns dst
      auto issue_s = [&](uint32_t dst, int i, int kst) {
        const uint64_t a0 = dQ + ((uint32_t)i * Lay::kQTile >> 4);
        const uint64_t bk = dK + ((uint32_t)kst * Lay::kTile >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma_ss(dst, a0 + (((kk / 4) * kRegionQ + (kk % 4) * 32) >> 4),
                    bk + (((kk / 4) * kRegionKV + (kk % 4) * 32) >> 4), kIdQK, kk > 0 ? 1u : 0u);
      };
      // O_i += P (TMEM columns sbuf) V (V stage vst), accumulating from the first product on
      auto issue_pv = [&](uint32_t sbuf, uint32_t dO, int vst, bool first) {
        const uint64_t bv = dV + ((uint32_t)vst * Lay::kTile >> 4);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          tc_mma_ts(dO, sbuf + kk * 8, bv + ((kk * 2048) >> 4), kIdPV, (!first || kk > 0) ? 1u : 0u);
      };
      if (ok) {
        tc_fence_after();
        for (int i = 0; i < nq; ++i) {
          issue_s(tS0 + (uint32_t)i * 128u, i, 0);
          tc_commit(bar0 + 8u * (B_SFULL + i));
        }
        tc_commit(bar0 + 8u * B_KEMPTY);
        if (!two && ntiles > 1) {
          // single tile: S(1) into the second buffer
          ok = wait_or_abort(bar0 + 8u * (B_KFULL + 1), 0, p.err, abort_flag);
          if (ok) {
            tc_fence_after();
            issue_s(tS0 + 128u, 0, 1);
            tc_commit(bar0 + 8u * (B_SFULL + 1));
            tc_commit(bar0 + 8u * (B_KEMPTY + 1));
          }
        }
      }
      if (two) {
        // PV_0(j), S_0(j+1), PV_1(j), S_1(j+1)
        for (int j = 0; ok && j < ntiles; ++j) {
          const int st = j % NST;
          const int jn = j + 1;
          const bool more = jn < ntiles;
          const int stn = jn % NST;
          if (!wait_or_abort(bar0 + 8u * (B_VFULL + st), (j / NST) & 1, p.err, abort_flag)) { ok = false; break; }
          for (int i = 0; i < nq; ++i) {
            if (!wait_or_abort(bar0 + 8u * (B_PFULL + i), j & 1, p.err, abort_flag)) { ok = false; break; }
            tc_fence_after();
            // O_i += P_i(j) V_j with P_i(j) as the TMEM A operand ...
            const uint32_t sbuf = tS0 + (uint32_t)i * 128u;
            issue_pv(sbuf, tO0 + (uint32_t)i * 128u, st, j == 0);
            // ... then S_i(j+1) over it (in-order completion)
            if (more) {
              if (i == 0 && !wait_or_abort(bar0 + 8u * (B_KFULL + stn), (jn / NST) & 1, p.err, abort_flag)) { ok = false; break; }
              issue_s(sbuf, i, stn);
              tc_commit(bar0 + 8u * (B_SFULL + i));
            }
          }
          if (!ok) break;
          tc_commit(bar0 + 8u * (B_VEMPTY + st));
          if (more) tc_commit(bar0 + 8u * (B_KEMPTY + stn));
        }
      } else {
        // one Q tile, S in two buffers: PV(j) from buffer j & 1, then S(j+2) into it
        for (int j = 0; ok && j < ntiles; ++j) {
          const int st = j % NST;
          const int b = j & 1;
          if (!wait_or_abort(bar0 + 8u * (B_VFULL + st), (j / NST) & 1, p.err, abort_flag)) { ok = false; break; }
          if (!wait_or_abort(bar0 + 8u * (B_PFULL + b), (j >> 1) & 1, p.err, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sbuf = tS0 + (uint32_t)b * 128u;
          issue_pv(sbuf, tO0, st, j == 0);
          tc_commit(bar0 + 8u * (B_VEMPTY + st));
          tc_commit(bar0 + 8u * B_ODONE);
          const int jn = j + 2;
          if (jn < ntiles) {
            const int stn = jn % NST;
            if (!wait_or_abort(bar0 + 8u * (B_KFULL + stn), (jn / NST) & 1, p.err, abort_flag)) { ok = false; break; }
            issue_s(sbuf, 0, stn);
            tc_commit(bar0 + 8u * (B_SFULL + b));
            tc_commit(bar0 + 8u * (B_KEMPTY + stn));
          }
        }
      }
      // every MMA issued above has finished before the epilogue reads O and TMEM is released
      tc_commit(bar0 + 8u * B_OFINAL);
    }
  } else if (softmax_warp) {
    // ---------------------- softmax / correction / epilogue ---------------------
    const int qi = qi_;                      // Q tile of this warpgroup
    const int wq = warp & 3;                 // TMEM sub-partition of this warp
    const int row = row_;                    // tile row = TMEM lane
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const bool row_valid = row_valid_;
    const int req = req_, qh = qh_;
    {
      const uint32_t qbase = sQ + qi * Lay::kQTile;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const int cc = c & 7;
        sts128(qbase + (c >> 3) * kRegionQ + row * 128 + ((cc ^ (row & 7)) << 4), qrow[c]);
      }
      fence_async_shared();
      mbar_arrive(bar(B_QFULL));
    }
    const bool active = ntiles > 0 && (qi == 0 || two);
    float m_used = -INFINITY, l = 0.f;
    bool ok = active;
    for (int j = 0; ok && j < ntiles; ++j) {
      // S buffer of this tile: the Q tile's own, or (one Q tile) alternating
      const int sb = two ? qi : (j & 1);
      const uint32_t sph = two ? (uint32_t)(j & 1) : (uint32_t)((j >> 1) & 1);
      // warp-uniform: a lane that gave up takes its whole warp out of the loop
      if (!__all_sync(0xffffffffu, wait_or_abort(bar(B_SFULL + sb), sph, p.err, abort_flag))) { ok = false; break; }
      tc_fence_after();
      float s[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(tS(sb) + c * 32 + lane_off, s + c * 32);
      tc_wait_ld();
      const int nvalid = gr.lp - (key0 + j * BN);
      if (nvalid < BN) {
#pragma unroll
        for (int c = 0; c < BN; ++c) s[c] = c < nvalid ? s[c] : -INFINITY;
      }
      // row max: eight independent chains of 3-input max
      float mx8[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) mx8[c] = s[c];
#pragma unroll
      for (int c = 8; c + 16 <= BN; c += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = fmax3(mx8[k], s[c + k], s[c + 8 + k]);
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(mx8[k], s[BN - 8 + k]);
      float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
      mx *= p.scale_log2;
      if (__any_sync(0xffffffffu, mx > m_used + 8.0f)) {
        const float m_new = fmaxf(m_used, mx);
        if (j > 0) {
          // two Q tiles: S(j) completed after PV(j-1), so O holds keys 0..j-1 scaled by
          // 2^-m_used; one Q tile: S(j) only follows PV(j-2), so wait for PV(j-1)
          if (!two) {
            if (!__all_sync(0xffffffffu, wait_or_abort(bar(B_ODONE), (uint32_t)((j - 1) & 1), p.err, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const float f = ex2(m_used - m_new);
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(tO(qi) + c * 32 + lane_off, o);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= f;
            tmem_st32(tO(qi) + c * 32 + lane_off, o);
          }
          l *= f;
        }
        m_used = m_new;
      }
      // P = 2^(s*scale - m), every exponential on MUFU: the softmax is bound by
      // issue on the FMA pipe (scale, max, sum, pack), not by MUFU, so moving
      // exponentials to a polynomial on the FMA pipe measured slower
      const uint64_t sc2 = f2pack(p.scale_log2, p.scale_log2), nm2 = f2pack(-m_used, -m_used);
      uint32_t pk[BN / 2];
      uint64_t sum4[4] = {0, 0, 0, 0};
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) {
        float xa, xb;
        f2unpack(ffma2(f2pack(s[2 * c], s[2 * c + 1]), sc2, nm2), xa, xb);
        const float a = ex2(xa), b2 = ex2(xb);
        sum4[c & 3] = fadd2(sum4[c & 3], f2pack(a, b2));
        pk[c] = pack_bf16x2(a, b2);
      }
      {
        float s0, s1, s2, s3;
        f2unpack(fadd2(sum4[0], sum4[1]), s0, s1);
        f2unpack(fadd2(sum4[2], sum4[3]), s2, s3);
        l += (s0 + s1) + (s2 + s3);
      }
      // P over S in TMEM (packed bf16 pairs, key 2c in the low half of column c)
#pragma unroll
      for (int c = 0; c < BN / 64; ++c) tmem_st32(tS(sb) + c * 32 + lane_off, reinterpret_cast<const float*>(pk + c * 32));
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + sb));
    }
    if (ok && wait_or_abort(bar(B_OFINAL), 0, p.err, abort_flag)) {
      // Every MMA has finished, so the Q/K/V staging area is free: each thread
      // parks its normalised O row there, then each warp stores whole rows
      // (one coalesced d*4-byte store per row) to its partial-state slot.
      tc_fence_after();
      constexpr uint32_t kRowBytes = D * 4 + 16;          // padded: conflict-free row writes
      const uint32_t stage = sQ + (uint32_t)qi * BM * kRowBytes;
      // destination of each row, looked up once by the row's own thread
      const uint32_t dst_tab = sQ + 2u * BM * kRowBytes + (uint32_t)qi * BM * 8;
      {
        float* dst = nullptr;
        if (row_valid) {
          dst = p.part_o + (entry_ * p.Hq + qh) * D;
          p.part_l[entry_ * p.Hq + qh] = m_used + __log2f(l);
          // the further key splits this item covered hold empty states (weight 0)
          for (int k = 1; k < it.splits; ++k) p.part_l[(entry_ + k) * p.Hq + qh] = -INFINITY;
        }
        asm volatile("st.shared.u64 [%0], %1;" ::"r"(dst_tab + row * 8), "l"((uint64_t)dst) : "memory");
      }
      const float inv = 1.f / l;
      // two 32-column loads per wait
#pragma unroll 1
      for (int c = 0; c < D / 32; c += 2) {
        float o[64];
        tmem_ld32(tO(qi) + c * 32 + lane_off, o);
        tmem_ld32(tO(qi) + (c + 1) * 32 + lane_off, o + 32);
        tc_wait_ld();
#pragma unroll
        for (int e = 0; e < 64; e += 4)
          sts128(stage + row * kRowBytes + (c * 32 + e) * 4,
                 make_uint4(__float_as_uint(o[e] * inv), __float_as_uint(o[e + 1] * inv),
                            __float_as_uint(o[e + 2] * inv), __float_as_uint(o[e + 3] * inv)));
      }
      asm volatile("bar.sync %0, 128;" ::"r"(1 + qi) : "memory");
      // rows of this warp's 32-row slice; D/4 lanes cover a row
      constexpr int kLanesPerRow = D / 4;
      constexpr int kRowsPerPass = 32 / kLanesPerRow;
      const int sub = lane % kLanesPerRow;
#pragma unroll 4
      for (int r0 = 0; r0 < 32; r0 += kRowsPerPass) {
        const int rr = wq * 32 + r0 + lane / kLanesPerRow;
        uint64_t dst;
        asm volatile("ld.shared.u64 %0, [%1];" : "=l"(dst) : "r"(dst_tab + rr * 8));
        if (dst) {
          const uint4 v = lds128(stage + rr * kRowBytes + sub * 16);
          reinterpret_cast<uint4*>(dst)[sub] = v;
        }
      }
    } else if (!active) {
      // an idle warpgroup (single-tile CTA) waits for the MMAs before TMEM is released
      if (ntiles > 0) wait_or_abort(bar(B_OFINAL), 0, p.err, abort_flag);
    }
    tc_fence_before();
  }
  // Drain order on every path, aborted or not: the TMA producer has waited for
  // its own loads in flight (above); here thread 0 waits for the MMA thread's
  // final commit, which arrives once every tcgen05.mma it issued has completed
  // (it commits even after an abort, with or without MMAs issued).  Only then
  // are the barriers invalidated and, by the caller, tensor memory released.
  // Softmax warps that gave up skip their own wait for it, so this one is
  // needed; on the normal path the phase has already completed.  The MMA
  // thread's waits are bounded, so its commit comes; this wait is bounded too.
  if (threadIdx.x == 0 && ntiles > 0) mbar_wait(bar(B_OFINAL), 0, nullptr);
  // the staging area is rewritten by the next user of the shared memory through TMA
  fence_async_shared();
  __syncthreads();
  const bool ok_all = *abort_flag == 0;
  if (threadIdx.x == 0)
    for (int i = 0; i < B_COUNT; ++i) mbar_inval(bar(i));
  return ok_all;
}


}  // namespace prefix

// kernel arguments of the prefix contraction for one layer of a planned batch
int fill_prefix_params(const LaunchCommon& lc, int32_t layer, const gk_batch* b, const Plan* pl,
                       prefix::PrefixParams* out);

}  // namespace gk
