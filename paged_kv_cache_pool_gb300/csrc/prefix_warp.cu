// Stand-alone launch of the warp-MMA prefix items (GraniKV Section 3.5, the
// cascade backend's level-0 kernel; the body is in prefix_warp_body.cuh): one
// CTA per item over every prefix group of the plan, writing partial states.
// A split plan runs the same items inside the split cascade launch instead.
#include "prefix_warp_body.cuh"

namespace gk {
using namespace prefix_warp;
namespace {

template <int D>
constexpr size_t warp_kernel_smem() {
  return 1024 + Layout<D>::kData + prefix::kCtlBytes;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefix_warp_kernel(const prefix::PrefixParams p, int n_items) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t ctl = base + Layout<D>::kData;
  uint8_t* ctl_ptr = smem_raw + (ctl - raw);
  griddep_launch_dependents();
  if (threadIdx.x == 0) *reinterpret_cast<volatile int*>(ctl_ptr + prefix::kCtlFlag) = 0;
  __syncthreads();
  // the item waits for the kernel before this one itself, after its table reads
  if ((int)blockIdx.x < n_items) warp_item<D>(p, p.items[blockIdx.x], base, ctl, ctl_ptr);
  else griddep_wait();
}

template <int D>
int launch_t(const prefix::PrefixParams& pp, int n_items, cudaStream_t st) {
  auto kern = prefix_warp_kernel<D>;
  const size_t smem = warp_kernel_smem<D>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  return (int)launch_pdl(kern, dim3(n_items), dim3(kThreads), smem, st, pp, n_items);
}

}  // namespace

int launch_prefix_warp(const LaunchCommon& lc, void* stream, int32_t layer, const gk_batch* b, const Plan* pl) {
  const gk_pool_config& c = *lc.cfg;
  prefix::PrefixParams pp;
  fill_prefix_params(lc, layer, b, pl, &pp);
  const int n_items = (int)pl->prefix_items.size();
  if (n_items == 0) return 0;
  if (c.head_dim == 128) return launch_t<128>(pp, n_items, (cudaStream_t)stream);
  if (c.head_dim == 64) return launch_t<64>(pp, n_items, (cudaStream_t)stream);
  return (int)cudaErrorInvalidValue;
}

}  // namespace gk
