// KV writes: reshape_and_cache into COLD slots, copy-on-write block copies,
// and the HOT prefix-slab write.  Pure data movement with 16-byte vectors.
//
// "Paged KV cache", How it works: step 1 writes each token's K/V through the
// slot mapping (reshape_and_cache); step 2 copies a shared partial block before
// a sequence writes into it (copy-on-write).  Copies run first, in their own
// launch, so a write into a freshly copied block can never be overwritten.
#include "device_common.cuh"
#include "gk_internal.h"

namespace gk {
namespace {

// One CTA per copy-on-write pair: copy the P slots of block src to block dst (K and V).
__global__ void cow_copy_kernel(uint4* __restrict__ cold_k, uint4* __restrict__ cold_v, int64_t layer_vecs,
                                int64_t block_vecs, int64_t n_blocks, const int32_t* __restrict__ pairs,
                                int32_t* err) {
  griddep_launch_dependents();
  griddep_wait();
  int32_t src = pairs[2 * blockIdx.x], dst = pairs[2 * blockIdx.x + 1];
  if (src < 0 || dst < 0 || src >= n_blocks || dst >= n_blocks) {
    if (threadIdx.x == 0) report_error(err, kErrBounds);
    return;
  }
  const uint4* ks = cold_k + layer_vecs + (int64_t)src * block_vecs;
  const uint4* vs = cold_v + layer_vecs + (int64_t)src * block_vecs;
  uint4* kd = cold_k + layer_vecs + (int64_t)dst * block_vecs;
  uint4* vd = cold_v + layer_vecs + (int64_t)dst * block_vecs;
  for (int64_t i = threadIdx.x; i < block_vecs; i += blockDim.x) {
    kd[i] = ks[i];
    vd[i] = vs[i];
  }
}

// One warp per token: K and V rows [Hkv][d] (row_vecs 16-byte vectors each) to its slot.
__global__ void scatter_kernel(uint4* __restrict__ cold_k, uint4* __restrict__ cold_v, int64_t layer_vecs,
                               int32_t row_vecs, int64_t cold_slots, int32_t n, const int64_t* __restrict__ slots,
                               const uint4* __restrict__ k, const uint4* __restrict__ v, int32_t* err) {
  griddep_launch_dependents();
  griddep_wait();
  int32_t tok = (int32_t)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  int lane = threadIdx.x & 31;
  if (tok >= n) return;
  int64_t slot = slots[tok];
  if (slot < 0 || slot >= cold_slots) {
    if (lane == 0) report_error(err, kErrBounds);
    return;
  }
  uint4* kd = cold_k + layer_vecs + slot * row_vecs;
  uint4* vd = cold_v + layer_vecs + slot * row_vecs;
  const uint4* ks = k + (int64_t)tok * row_vecs;
  const uint4* vs = v + (int64_t)tok * row_vecs;
  for (int i = lane; i < row_vecs; i += 32) {
    kd[i] = ks[i];
    vd[i] = vs[i];
  }
}

// Prefix tokens [t0, t0+n) of one layer: input [n][Hkv][d] -> slab [Hkv][Lp][d] at (layer).
__global__ void hot_slab_write_kernel(uint4* __restrict__ hot_k, uint4* __restrict__ hot_v, int64_t slab_vecs,
                                    int32_t hkv, int32_t d_vecs, int64_t lp, int64_t t0, int64_t n,
                                    const uint4* __restrict__ k, const uint4* __restrict__ v) {
  // No early trigger: the kernel after this one starts only once every slab write
  // has finished, so the prefix items may fetch HOT tiles before their own
  // dependency wait (no kernel of a later launch can then overlap a slab write).
  griddep_wait();
  int64_t total = n * hkv * d_vecs;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t e = i % d_vecs;
    int64_t h = (i / d_vecs) % hkv;
    int64_t t = i / ((int64_t)d_vecs * hkv);
    int64_t dst = slab_vecs + (h * lp + t0 + t) * d_vecs + e;
    hot_k[dst] = k[i];
    hot_v[dst] = v[i];
  }
}

}  // namespace

int launch_cow_copy(const LaunchCommon& lc, void* stream, int32_t layer, int32_t n_cow, const int32_t* d_pairs) {
  const gk_pool_config& c = *lc.cfg;
  int64_t row_vecs = (int64_t)c.num_kv_heads * c.head_dim / 8;
  int64_t layer_vecs = (int64_t)layer * c.cold_slots * row_vecs;
  int64_t block_vecs = (int64_t)c.cold_page_size * row_vecs;
  return (int)launch_pdl(cow_copy_kernel, dim3(n_cow), dim3(256), 0, (cudaStream_t)stream, (uint4*)c.cold_k,
                         (uint4*)c.cold_v, layer_vecs, block_vecs, (int64_t)(c.cold_slots / c.cold_page_size),
                         d_pairs, lc.d_error);
}

int launch_scatter(const LaunchCommon& lc, void* stream, int32_t layer, int32_t n, const int64_t* d_slots,
                   const void* d_k, const void* d_v) {
  const gk_pool_config& c = *lc.cfg;
  int32_t row_vecs = c.num_kv_heads * c.head_dim / 8;
  int64_t layer_vecs = (int64_t)layer * c.cold_slots * row_vecs;
  int warps_per_block = 8;
  int blocks = (n + warps_per_block - 1) / warps_per_block;
  return (int)launch_pdl(scatter_kernel, dim3(blocks), dim3(32 * warps_per_block), 0, (cudaStream_t)stream,
                         (uint4*)c.cold_k, (uint4*)c.cold_v, layer_vecs, row_vecs, (int64_t)c.cold_slots, n, d_slots,
                         (const uint4*)d_k, (const uint4*)d_v, lc.d_error);
}

int launch_write_prefix(const LaunchCommon& lc, void* stream, int32_t layer, int64_t base, int64_t lp, int64_t t0,
                        int64_t n, const void* d_k, const void* d_v) {
  const gk_pool_config& c = *lc.cfg;
  int32_t d_vecs = c.head_dim / 8;
  // slab of (base, layer): element offset (base*L*Hkv + layer*Hkv*Lp) * d
  int64_t slab_vecs = (base * c.num_layers * c.num_kv_heads + (int64_t)layer * c.num_kv_heads * lp) * d_vecs;
  int64_t total = n * c.num_kv_heads * d_vecs;
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)lc.num_sms * 16) blocks = (int64_t)lc.num_sms * 16;
  return (int)launch_pdl(hot_slab_write_kernel, dim3((unsigned)blocks), dim3(256), 0, (cudaStream_t)stream,
                         (uint4*)c.hot_k, (uint4*)c.hot_v, slab_vecs, (int32_t)c.num_kv_heads, d_vecs, lp, t0, n,
                         (const uint4*)d_k, (const uint4*)d_v);
}

}  // namespace gk
