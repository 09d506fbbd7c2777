// Cascade prefix kernel: the shared-prefix contraction on 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory), fed by TMA from the HOT pool.
//
// GraniKV Section 2.3 ("Shared-prefix matmul") and Section 3.5 (dense backend):
// all query rows that share a prefix -- every request of the group times its
// g = Hq/Hkv query heads of one KV head -- are stacked into one matrix Q
// [M = B_g * g, d], so prefix attention is a dense contraction
// O_p = softmax(Q K_p^T / sqrt(d)) V_p against the contiguous [Lp, d] slab of
// (layer, KV head), read once per step instead of once per request.
//
// One CTA = 256 stacked rows (two 128-row Q tiles) x one KV head x one split of
// the prefix keys (the plan balances splits over the SMs).  For each tile of
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
// Each CTA emits a partial state (O normalised, LSE in log2) per row; the merge
// kernel combines the splits with the suffix states by GraniKV Eq. 1.
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
#include <cuda.h>

#include <cstring>

#include "device_common.cuh"
#include "gk_internal.h"

namespace gk {
namespace {

constexpr int BM = kPrefixTileM;   // 128 rows per Q tile
constexpr int BN = kPrefixTileN;   // 128 keys per K/V tile
constexpr int NST = 2;             // K and V pipeline depth
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kRegionQ = BM * 128;   // [128 rows x 64 bf16] swizzled region
constexpr uint32_t kRegionKV = BN * 128;  // [128 keys x 64 bf16] swizzled region
constexpr int kThreads = 320;

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
  B_COUNT = B_OFINAL + 1
};

template <int D>
struct Layout {
  static constexpr uint32_t kTile = BN * D * 2;      // one K or V tile
  static constexpr uint32_t kQTile = BM * D * 2;     // one Q tile
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + 2 * kQTile;
  static constexpr uint32_t kV = kK + NST * kTile;
  static constexpr uint32_t kBars = kV + NST * kTile;
  static constexpr uint32_t kTmemSlot = kBars + B_COUNT * 8;
  static constexpr uint32_t kFlag = kTmemSlot + 4;
  static constexpr uint32_t kBytes = kFlag + 4;
  // slack to align the base to 1024; at least 120 KB so that one CTA (and one
  // 512-column tensor-memory allocation) is resident per SM
  static constexpr size_t kDynamic = kBytes + 1024 > 120 * 1024 ? kBytes + 1024 : 120 * 1024;
  static_assert(2 * BM * (D * 4 + 16) + 2 * BM * 8 <= kBars, "epilogue staging must fit in the Q/K/V area");
};

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

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefix_kernel(const PrefixParams p) {
  using Lay = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + Lay::kQ, sK = base + Lay::kK, sV = base + Lay::kV;
  auto bar = [&](int i) { return base + Lay::kBars + 8u * (uint32_t)i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + Lay::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kFlag);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PrefixItemDev it = p.items[blockIdx.x];
  const PrefixGroupDev gr = p.groups[it.group];
  const int ntiles_all = (gr.lp + BN - 1) / BN;
  const int tile0 = it.split * gr.split_tiles;
  const int ntiles = min(gr.split_tiles, ntiles_all - tile0);
  const int key0 = tile0 * BN;
  const int row0 = it.mblock * kPrefixRowsPerCta;
  const bool two = row0 + BM < gr.m;  // does Q tile 1 hold any row?
  const void* tmK = p.tmaps + (size_t)gr.tmap_index * 128;
  const void* tmV = p.tmaps + (size_t)(gr.tmap_index + 1) * 128;
  const int zc = p.layer * p.Hkv + it.head;

  griddep_launch_dependents();
  // plan tables and the HOT pool are not written by the kernels of a decode
  // step; the queries and the partial-state buffer may be, so wait for them
  griddep_wait();
  // softmax threads fetch their Q row now, so the global-load latency overlaps the set-up
  const int qi_ = (warp - 2) >> 2;
  const int row_ = (warp & 3) * 32 + lane;
  const int grow_ = row0 + qi_ * BM + row_;
  const bool row_valid_ = warp >= 2 && grow_ < gr.m;
  int req_ = 0, qh_ = 0;
  if (row_valid_) {
    req_ = p.prefix_reqs[gr.req_base + grow_ / p.G];
    qh_ = it.head * p.G + grow_ % p.G;
  }
  uint4 qrow[D / 8];
  if (warp >= 2) {
    const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)req_ * p.Hq + qh_) * D);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) qrow[c] = row_valid_ ? src[c] : make_uint4(0, 0, 0, 0);
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
    *abort_flag = 0;
    fence_mbar_init();
    // the first K/V tiles need nothing but the barriers: start them now so their
    // latency overlaps the tensor-memory allocation and the Q staging
    if (ntiles > 0) {
      tmap_acquire(tmK);
      tmap_acquire(tmV);
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
  if (warp == 1) {
    tmem_alloc(base + Lay::kTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // columns: S of Q tile i at i*128 (P is written over it); O of Q tile i at 256 + i*128
  auto tS = [&](int i) { return tmem + (uint32_t)(i * 128); };
  auto tO = [&](int i) { return tmem + 256u + (uint32_t)i * 128u; };

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0 && ntiles > NST) {
      int issued = 2 * NST;
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
      const uint32_t bar0 = base + Lay::kBars;
      const uint32_t tS0 = tmem, tO0 = tmem + 256u;
      bool ok = wait_or_abort(bar0 + 8u * B_QFULL, 0, p.err, abort_flag) &&
                wait_or_abort(bar0 + 8u * B_KFULL, 0, p.err, abort_flag);
      if (ok) {
        tc_fence_after();
        for (int i = 0; i < nq; ++i) {
          const uint64_t a0 = dQ + ((uint32_t)i * Lay::kQTile >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc_mma_ss(tS0 + (uint32_t)i * 128u, a0 + (((kk / 4) * kRegionQ + (kk % 4) * 32) >> 4),
                      dK + (((kk / 4) * kRegionKV + (kk % 4) * 32) >> 4), kIdQK, kk > 0 ? 1u : 0u);
          tc_commit(bar0 + 8u * (B_SFULL + i));
        }
        tc_commit(bar0 + 8u * B_KEMPTY);
      }
      for (int j = 0; ok && j < ntiles; ++j) {
        const int st = j % NST;
        const int jn = j + 1;
        const bool more = jn < ntiles;
        const int stn = jn % NST;
        if (!wait_or_abort(bar0 + 8u * (B_VFULL + st), (j / NST) & 1, p.err, abort_flag)) { ok = false; break; }
        const uint64_t bv = dV + ((uint32_t)st * Lay::kTile >> 4);
        const uint64_t bk = dK + ((uint32_t)stn * Lay::kTile >> 4);
        for (int i = 0; i < nq; ++i) {
          if (!wait_or_abort(bar0 + 8u * (B_PFULL + i), j & 1, p.err, abort_flag)) { ok = false; break; }
          tc_fence_after();
          // O_i += P_i(j) V_j with P_i(j) as the TMEM A operand ...
          const uint32_t sbuf = tS0 + (uint32_t)i * 128u;
          const uint32_t dO = tO0 + (uint32_t)i * 128u;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            tc_mma_ts(dO, sbuf + kk * 8, bv + ((kk * 2048) >> 4), kIdPV, (j > 0 || kk > 0) ? 1u : 0u);
          // ... then S_i(j+1) over it (in-order completion)
          if (more) {
            if (i == 0 && !wait_or_abort(bar0 + 8u * (B_KFULL + stn), (jn / NST) & 1, p.err, abort_flag)) { ok = false; break; }
            const uint64_t a0 = dQ + ((uint32_t)i * Lay::kQTile >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              tc_mma_ss(sbuf, a0 + (((kk / 4) * kRegionQ + (kk % 4) * 32) >> 4),
                        bk + (((kk / 4) * kRegionKV + (kk % 4) * 32) >> 4), kIdQK, kk > 0 ? 1u : 0u);
            tc_commit(bar0 + 8u * (B_SFULL + i));
          }
        }
        if (!ok) break;
        tc_commit(bar0 + 8u * (B_VEMPTY + st));
        if (more) tc_commit(bar0 + 8u * (B_KEMPTY + stn));
      }
      // every MMA issued above has finished before the epilogue reads O and TMEM is released
      tc_commit(bar0 + 8u * B_OFINAL);
    }
  } else {
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
      if (!wait_or_abort(bar(B_SFULL + qi), j & 1, p.err, abort_flag)) { ok = false; break; }
      tc_fence_after();
      float s[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(tS(qi) + c * 32 + lane_off, s + c * 32);
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
          // S(j) completed after PV(j-1): O holds keys 0..j-1 scaled by 2^-m_used
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
      // P = 2^(s*scale - m): three pairs in four on MUFU, one on the FMA pipe
      const uint64_t sc2 = f2pack(p.scale_log2, p.scale_log2), nm2 = f2pack(-m_used, -m_used);
      uint32_t pk[BN / 2];
      uint64_t sum4[4] = {0, 0, 0, 0};
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) {
        float xa, xb, a, b2;
        f2unpack(ffma2(f2pack(s[2 * c], s[2 * c + 1]), sc2, nm2), xa, xb);
        if ((c & 3) == 3) {
          exp2_poly_pair(xa, xb, a, b2);
        } else {
          a = ex2(xa);
          b2 = ex2(xb);
        }
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
      for (int c = 0; c < BN / 64; ++c) tmem_st32(tS(qi) + c * 32 + lane_off, reinterpret_cast<const float*>(pk + c * 32));
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + qi));
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
          const int64_t entry = (int64_t)p.reqs[req].entry_cas + it.split;
          dst = p.part_o + (entry * p.Hq + qh) * D;
          p.part_l[entry * p.Hq + qh] = m_used + __log2f(l);
        }
        asm volatile("st.shared.u64 [%0], %1;" ::"r"(dst_tab + row * 8), "l"((uint64_t)dst) : "memory");
      }
      const float inv = 1.f / l;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(tO(qi) + c * 32 + lane_off, o);
        tc_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          sts128(stage + row * kRowBytes + (c * 32 + e) * 4,
                 make_uint4(__float_as_uint(o[e] * inv), __float_as_uint(o[e + 1] * inv),
                            __float_as_uint(o[e + 2] * inv), __float_as_uint(o[e + 3] * inv)));
      }
      asm volatile("bar.sync %0, 128;" ::"r"(1 + qi) : "memory");
      // rows of this warp's 32-row slice; D/4 lanes cover a row
      constexpr int kLanesPerRow = D / 4;
      constexpr int kRowsPerPass = 32 / kLanesPerRow;
      const int sub = lane % kLanesPerRow;
#pragma unroll 1
      for (int r0 = 0; r0 < 32; r0 += kRowsPerPass) {
        const int rr = wq * 32 + r0 + lane / kLanesPerRow;
        uint64_t dst;
        asm volatile("ld.shared.u64 %0, [%1];" : "=l"(dst) : "r"(dst_tab + rr * 8));
        if (dst) {
          const uint4 v = lds128(stage + rr * kRowBytes + sub * 16);
          reinterpret_cast<uint4*>(dst)[sub] = v;
        }
      }
    } else if (!active && warp >= 2) {
      // an idle warpgroup (single-tile CTA) waits for the MMAs before TMEM is released
      if (ntiles > 0) wait_or_abort(bar(B_OFINAL), 0, p.err, abort_flag);
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)f;
  }
  return fn;
}

template <int D>
int launch_prefix_t(const PrefixParams& pp, int ctas, cudaStream_t st) {
  auto kern = prefix_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Layout<D>::kDynamic);
  if (e != cudaSuccess) return (int)e;
  e = launch_pdl(kern, dim3(ctas), dim3(kThreads), Layout<D>::kDynamic, st, pp);
  return (int)e;
}

}  // namespace

size_t tmap_bytes() { return sizeof(CUtensorMap); }

// Four 3D maps per prefix group over its slab: dims (d, Lp, L*Hkv), 128-byte
// swizzle, keys past Lp read as zeros; K and V with a (64, 128, 1) box for the
// prefix kernel, then K and V with a (64, 16, 1) box for the dense gather.
int encode_prefix_tmaps(const gk_pool_config* cfg, const Plan* pl, std::vector<uint8_t>* out) {
  out->assign(pl->groups.size() * 4 * sizeof(CUtensorMap), 0);
  if (pl->groups.empty()) return 0;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return 1;
  const int D = cfg->head_dim;
  for (size_t gi = 0; gi < pl->groups.size(); ++gi) {
    const int64_t lp = pl->groups[gi].lp;
    const int64_t slab = pl->group_hot_base[gi] * cfg->num_layers * cfg->num_kv_heads * D;
    for (int m = 0; m < 4; ++m) {
      const int kv = m & 1;
      uint16_t* basep = (uint16_t*)(kv == 0 ? cfg->hot_k : cfg->hot_v) + slab;
      cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)lp, (cuuint64_t)cfg->num_layers * cfg->num_kv_heads};
      cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)lp * D * 2};
      cuuint32_t box[3] = {64, (cuuint32_t)(m < 2 ? BN : kGatherT), 1};
      cuuint32_t estr[3] = {1, 1, 1};
      CUtensorMap tm;
      CUresult r = enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, basep, dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return 2;
      std::memcpy(out->data() + (gi * 4 + m) * sizeof(CUtensorMap), &tm, sizeof(CUtensorMap));
    }
  }
  return 0;
}

int launch_prefix(const LaunchCommon& lc, void* stream, int32_t layer, const gk_batch* b, const Plan* pl) {
  const gk_pool_config& c = *lc.cfg;
  const uint8_t* base = (const uint8_t*)pl->d_buf;
  PrefixParams pp{};
  pp.groups = (const PrefixGroupDev*)(base + pl->off_groups);
  pp.prefix_reqs = (const int32_t*)(base + pl->off_prefix_reqs);
  pp.items = (const PrefixItemDev*)(base + pl->off_prefix_items);
  pp.reqs = (const RequestDev*)(base + pl->off_reqs);
  pp.tmaps = base + pl->off_tmaps;
  pp.q = (const uint16_t*)b->d_q;
  pp.part_o = pl->d_part_o;
  pp.part_l = pl->d_part_l;
  pp.Hkv = c.num_kv_heads;
  pp.Hq = c.num_q_heads;
  pp.G = c.num_q_heads / c.num_kv_heads;
  pp.layer = layer;
  pp.err = lc.d_error;
  pp.scale_log2 = kLog2e / sqrtf((float)c.head_dim);
  const int ctas = (int)pl->prefix_items.size();
  if (ctas == 0) return 0;
  if (c.head_dim == 128) return launch_prefix_t<128>(pp, ctas, (cudaStream_t)stream);
  if (c.head_dim == 64) return launch_prefix_t<64>(pp, ctas, (cudaStream_t)stream);
  return (int)cudaErrorInvalidValue;
}

}  // namespace gk
