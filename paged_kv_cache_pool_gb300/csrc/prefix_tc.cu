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
// One CTA = one 128-row tile of Q x one KV head x one split of the prefix keys
// (the plan balances splits over the SMs).  The CTA walks its split in tiles of
// 128 keys: S = Q K^T (tcgen05.mma, bf16 in, fp32 accumulate, S in TMEM),
// softmax warps read S rows from TMEM, write P = 2^(S*log2e/sqrt(d) - m) as bf16
// into shared memory, and O += P V accumulates in TMEM.  The running max m is
// only moved (and O rescaled in TMEM) when a row's max grows by more than 2^8,
// so most tiles skip the rescale; the sum and the output use the same m, which
// keeps the result exact up to rounding.  Each CTA emits a partial state
// (O normalised, LSE in log2) per row; the merge kernel combines the splits with
// the suffix states by GraniKV Eq. 1.
//
// Warp roles (192 threads): warp 0 issues TMA loads (K and V tiles, double
// buffered), warp 1 owns tensor memory and issues the MMAs from one thread,
// warps 2-5 stage Q, run the softmax and write the partial outputs.
//
// Shared-memory operand layout: every [rows x 64] bf16 region is the 128-byte
// swizzled K-major layout (8-row x 128-byte atoms, 16-byte chunk c of row r
// stored at chunk c ^ (r mod 8)), written by TMA for K and V and by the threads
// for Q and P.  V is consumed as the MN-major B operand (N = d), K and P/Q as
// K-major operands.
#include <cuda.h>

#include <cstring>

#include "device_common.cuh"
#include "gk_internal.h"

namespace gk {
namespace {

constexpr int BM = kPrefixTileM;   // 128 stacked rows
constexpr int BN = kPrefixTileN;   // 128 keys
constexpr int NSTK = 2, NSTV = 2;  // K and V pipeline depth
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kRegion = BM * 128;  // one [128 rows x 64 bf16] swizzled region = 16 KB

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
  B_KFULL = 1,                 // NSTK
  B_KEMPTY = B_KFULL + NSTK,   // NSTK
  B_VFULL = B_KEMPTY + NSTK,   // NSTV
  B_VEMPTY = B_VFULL + NSTV,   // NSTV
  B_SFULL = B_VEMPTY + NSTV,   // 2
  B_SEMPTY = B_SFULL + 2,      // 2
  B_PFULL = B_SEMPTY + 2,
  B_PVDONE = B_PFULL + 1,
  B_DRAIN = B_PVDONE + 1,
  B_COUNT = B_DRAIN + 1
};

template <int D>
struct Layout {
  static constexpr uint32_t kTile = BN * D * 2;  // one K or V tile (= Q tile bytes)
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + BM * D * 2;
  static constexpr uint32_t kV = kK + NSTK * kTile;
  static constexpr uint32_t kP = kV + NSTV * kTile;
  static constexpr uint32_t kBars = kP + BM * BN * 2;
  static constexpr uint32_t kTmemSlot = kBars + B_COUNT * 8;
  static constexpr uint32_t kFlag = kTmemSlot + 4;
  static constexpr uint32_t kBytes = kFlag + 4;
  // slack to align the base to 1024; at least 120 KB so that one CTA (and one
  // 512-column tensor-memory allocation) is resident per SM
  static constexpr size_t kDynamic = kBytes + 1024 > 120 * 1024 ? kBytes + 1024 : 120 * 1024;
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
__global__ void __launch_bounds__(192, 1) prefix_kernel(const PrefixParams p) {
  using Lay = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + Lay::kQ, sK = base + Lay::kK, sV = base + Lay::kV, sP = base + Lay::kP;
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

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 128);
    for (int s = 0; s < NSTK; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
    }
    for (int s = 0; s < NSTV; ++s) {
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_SEMPTY + s), 128);
    }
    mbar_init(bar(B_PFULL), 128);
    mbar_init(bar(B_PVDONE), 1);
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(base + Lay::kTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 2 * BN;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0 && ntiles > 0) {
      const void* tmK = p.tmaps + (size_t)gr.tmap_index * 128;
      const void* tmV = p.tmaps + (size_t)(gr.tmap_index + 1) * 128;
      tmap_acquire(tmK);
      tmap_acquire(tmV);
      const int z = p.layer * p.Hkv + it.head;
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int sk = j % NSTK, rk = j / NSTK;
        if (rk > 0 && !wait_or_abort(bar(B_KEMPTY + sk), (rk - 1) & 1, p.err, abort_flag)) break;
        mbar_arrive_expect_tx(bar(B_KFULL + sk), Lay::kTile);
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(sK + sk * Lay::kTile + h * kRegion, tmK, h * 64, key0 + j * BN, z, bar(B_KFULL + sk));
        const int sv = j % NSTV, rv = j / NSTV;
        if (rv > 0 && !wait_or_abort(bar(B_VEMPTY + sv), (rv - 1) & 1, p.err, abort_flag)) {
          issued = 2 * j + 1;
          break;
        }
        mbar_arrive_expect_tx(bar(B_VFULL + sv), Lay::kTile);
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(sV + sv * Lay::kTile + h * kRegion, tmV, h * 64, key0 + j * BN, z, bar(B_VFULL + sv));
        issued = 2 * j + 2;
      }
      if (*abort_flag) {
        // let the loads already issued land before shared memory goes away
        for (int q = max(0, issued - 2 * NSTK); q < issued; ++q) {
          const int j = q / 2;
          if (q % 2 == 0) mbar_wait(bar(B_KFULL + j % NSTK), (j / NSTK) & 1, nullptr);
          else mbar_wait(bar(B_VFULL + j % NSTV), (j / NSTV) & 1, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t kIdQK = idesc(BN, false);
      constexpr uint32_t kIdPV = idesc(D, true);
      bool ok = wait_or_abort(bar(B_QFULL), 0, p.err, abort_flag);
      auto issue_pv = [&](int i) -> bool {
        if (!wait_or_abort(bar(B_PFULL), i & 1, p.err, abort_flag)) return false;
        const int sv = i % NSTV;
        if (!wait_or_abort(bar(B_VFULL + sv), (i / NSTV) & 1, p.err, abort_flag)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t a = sdesc(sP + (kk / 4) * kRegion + (kk % 4) * 32, 16, 1024);
          const uint64_t b = sdesc(sV + sv * Lay::kTile + kk * 2048, kRegion, 1024);
          tc_mma_ss(tO, a, b, kIdPV, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(B_PVDONE));
        tc_commit(bar(B_VEMPTY + sv));
        return true;
      };
      for (int j = 0; ok && j < ntiles; ++j) {
        const int sk = j % NSTK, sb = j & 1;
        if (!wait_or_abort(bar(B_KFULL + sk), (j / NSTK) & 1, p.err, abort_flag)) { ok = false; break; }
        if (j >= 2 && !wait_or_abort(bar(B_SEMPTY + sb), ((j - 2) >> 1) & 1, p.err, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t a = sdesc(sQ + (kk / 4) * kRegion + (kk % 4) * 32, 16, 1024);
          const uint64_t b = sdesc(sK + sk * Lay::kTile + (kk / 4) * kRegion + (kk % 4) * 32, 16, 1024);
          tc_mma_ss(tS + sb * BN, a, b, kIdQK, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(B_SFULL + sb));
        tc_commit(bar(B_KEMPTY + sk));
        if (j >= 1 && !issue_pv(j - 1)) ok = false;
      }
      if (ok) issue_pv(ntiles - 1);
      // every MMA issued above has finished before tensor memory is released
      tc_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, nullptr);
    }
  } else {
    // ---------------------- softmax / correction / epilogue ---------------------
    const int wq = warp & 3;                // TMEM sub-partition of this warp
    const int row = wq * 32 + lane;         // tile row = TMEM lane
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int grow = it.mtile * BM + row;   // stacked row within the group
    const bool row_valid = grow < gr.m;
    int req = 0, qh = 0;
    if (row_valid) {
      req = p.prefix_reqs[gr.req_base + grow / p.G];
      qh = it.head * p.G + grow % p.G;
    }
    // stage Q (zero rows pad the tile)
    {
      const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)req * p.Hq + qh) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        uint4 v = row_valid ? src[c] : make_uint4(0, 0, 0, 0);
        const int cc = c & 7;
        sts128(sQ + (c >> 3) * kRegion + row * 128 + ((cc ^ (row & 7)) << 4), v);
      }
      fence_async_shared();
      mbar_arrive(bar(B_QFULL));
    }
    float m_used = -INFINITY, l = 0.f;
    bool ok = ntiles > 0;
    for (int j = 0; ok && j < ntiles; ++j) {
      const int sb = j & 1;
      if (!wait_or_abort(bar(B_SFULL + sb), (j >> 1) & 1, p.err, abort_flag)) { ok = false; break; }
      tc_fence_after();
      float s[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(tS + sb * BN + c * 32 + lane_off, s + c * 32);
      tc_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(B_SEMPTY + sb));

      const int nvalid = min(BN, gr.lp - (key0 + j * BN));
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BN; ++c) {
        s[c] = c < nvalid ? s[c] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, s[c]);
      }
      bool pv_waited = false;
      const bool need = mx > m_used + 8.0f;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = fmaxf(m_used, mx);
        if (j > 0) {
          // O holds tiles 0..j-1 scaled by 2^-m_used: wait for PV(j-1), then rescale in TMEM
          if (!wait_or_abort(bar(B_PVDONE), (j - 1) & 1, p.err, abort_flag)) { ok = false; break; }
          pv_waited = true;
          tc_fence_after();
          const float f = ex2(m_used - m_new);
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(tO + c * 32 + lane_off, o);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= f;
            tmem_st32(tO + c * 32 + lane_off, o);
          }
          tc_wait_st();
          l *= f;
        }
        m_used = m_new;
      }
      uint32_t pk[BN / 2];
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) {
        const float a = ex2(s[2 * c] - m_used), b = ex2(s[2 * c + 1] - m_used);
        sum += a + b;
        pk[c] = pack_bf16x2(a, b);
      }
      l += sum;
      if (!pv_waited && j > 0) {
        // the P buffer is free once PV(j-1) has read it
        if (!wait_or_abort(bar(B_PVDONE), (j - 1) & 1, p.err, abort_flag)) { ok = false; break; }
      }
#pragma unroll
      for (int c = 0; c < BN / 8; ++c) {
        const int cc = c & 7;
        sts128(sP + (c >> 3) * kRegion + row * 128 + ((cc ^ (row & 7)) << 4),
               make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
      }
      fence_async_shared();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL));
    }
    if (ok && wait_or_abort(bar(B_PVDONE), (ntiles - 1) & 1, p.err, abort_flag)) {
      tc_fence_after();
      const float inv = 1.f / l;
      const float lse2 = m_used + __log2f(l);
      const int64_t entry = row_valid ? (int64_t)p.reqs[req].entry_cas + it.split : 0;
      float* dst = p.part_o + (entry * p.Hq + qh) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(tO + c * 32 + lane_off, o);
        tc_wait_ld();
        if (row_valid) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + c * 32 + e) = make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv, o[e + 3] * inv);
        }
      }
      if (row_valid) p.part_l[entry * p.Hq + qh] = lse2;
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
  kern<<<ctas, 192, Layout<D>::kDynamic, st>>>(pp);
  return (int)cudaGetLastError();
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
