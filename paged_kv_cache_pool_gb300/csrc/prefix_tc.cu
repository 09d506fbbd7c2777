// Stand-alone cascade prefix kernel (GraniKV Section 2.3, the shared-prefix
// matmul; the body is in prefix_body.cuh): one launch of the tensor-core
// contraction over every prefix group's work items, writing partial states.
// Also encodes the per-group tensor maps both prefix paths and the dense
// gather read through.
#include <cuda.h>

#include <cstring>

#include "prefix_body.cuh"

namespace gk {
using namespace prefix;
namespace {

// dynamic shared memory: alignment slack, data area, control block; at least
// 120 KB so that one CTA (and one 512-column tensor-memory allocation) is
// resident per SM
template <int D>
constexpr size_t kernel_smem() {
  const size_t b = 1024 + Layout<D>::kData + kCtlBytes;
  return b > 120 * 1024 ? b : 120 * 1024;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefix_kernel(const PrefixParams p, int n_items) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t ctl = base + Layout<D>::kData;
  uint8_t* ctl_ptr = smem_raw + (ctl - raw);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctl_ptr + kCtlTmemSlot);
  const int warp = threadIdx.x >> 5;

  griddep_launch_dependents();
  if (threadIdx.x == 0) *reinterpret_cast<volatile int*>(ctl_ptr + kCtlFlag) = 0;
  if (warp == 1) {
    tmem_alloc(ctl + kCtlTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // one item per CTA: a loop over items here costs the softmax warps registers.
  // The item waits for the kernel before this one itself, after its table reads.
  if ((int)blockIdx.x < n_items) prefix_item<D>(p, p.items[blockIdx.x], base, ctl, ctl_ptr, tmem);
  else griddep_wait();
  __syncthreads();
  if (warp == 1) {
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
int launch_prefix_t(const PrefixParams& pp, int n_items, int ctas, cudaStream_t st) {
  auto kern = prefix_kernel<D>;
  const size_t smem = kernel_smem<D>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  e = launch_pdl(kern, dim3(ctas), dim3(kThreads), smem, st, pp, n_items);
  return (int)e;
}

}  // namespace

size_t tmap_bytes() { return sizeof(CUtensorMap); }

// Two 3D maps per prefix group over its slab: dims (d, Lp, L*Hkv), 128-byte
// swizzle, keys past Lp read as zeros; K and V with a (64, 128, 1) box.
int encode_prefix_tmaps(const gk_pool_config* cfg, const Plan* pl, std::vector<uint8_t>* out) {
  out->assign(pl->groups.size() * 2 * sizeof(CUtensorMap), 0);
  if (pl->groups.empty()) return 0;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return 1;
  const int D = cfg->head_dim;
  for (size_t gi = 0; gi < pl->groups.size(); ++gi) {
    const int64_t lp = pl->groups[gi].lp;
    const int64_t slab = pl->group_hot_base[gi] * cfg->num_layers * cfg->num_kv_heads * D;
    for (int m = 0; m < 2; ++m) {
      const int kv = m & 1;
      uint16_t* basep = (uint16_t*)(kv == 0 ? cfg->hot_k : cfg->hot_v) + slab;
      cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)lp, (cuuint64_t)cfg->num_layers * cfg->num_kv_heads};
      cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)lp * D * 2};
      cuuint32_t box[3] = {64, (cuuint32_t)BN, 1};
      cuuint32_t estr[3] = {1, 1, 1};
      CUtensorMap tm;
      CUresult r = enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, basep, dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return 2;
      std::memcpy(out->data() + (gi * 2 + m) * sizeof(CUtensorMap), &tm, sizeof(CUtensorMap));
    }
  }
  return 0;
}

int fill_prefix_params(const LaunchCommon& lc, int32_t layer, const gk_batch* b, const Plan* pl, PrefixParams* out) {
  const gk_pool_config& c = *lc.cfg;
  const uint8_t* base = (const uint8_t*)pl->d_buf;
  PrefixParams& pp = *out;
  pp = PrefixParams{};
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
  return 0;
}

int launch_prefix(const LaunchCommon& lc, void* stream, int32_t layer, const gk_batch* b, const Plan* pl) {
  if (pl->prefix_kind == 1) return launch_prefix_warp(lc, stream, layer, b, pl);
  const gk_pool_config& c = *lc.cfg;
  PrefixParams pp;
  fill_prefix_params(lc, layer, b, pl, &pp);
  const int n_items = (int)pl->prefix_items.size();
  if (n_items == 0) return 0;
  if (c.head_dim == 128) return launch_prefix_t<128>(pp, n_items, n_items, (cudaStream_t)stream);
  if (c.head_dim == 64) return launch_prefix_t<64>(pp, n_items, n_items, (cudaStream_t)stream);
  return (int)cudaErrorInvalidValue;
}

}  // namespace gk
