// Stand-alone gather attention kernel (suffix level of the cascade, flat
// backend); the body is in gather_body.cuh.
#include "gather_body.cuh"

namespace gk {
using namespace gather;
namespace {

struct GatherLaunch {
  GatherParams p;
  unsigned long long* stamps;  // per CTA: SM id, start, end of its gather (%globaltimer), or null
};

template <int D, int G, bool DENSE>
__global__ void __launch_bounds__(kGatherThreads, 1) gather_kernel(const GatherLaunch g) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const int b = blockIdx.x;
  if (g.stamps && threadIdx.x == 0) {
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    g.stamps[3 * b] = smid;
    g.stamps[3 * b + 1] = globaltimer_ns();
  }
  griddep_launch_dependents();
  gather_segments<D, G, DENSE>(g.p, base, b);
  if (g.stamps && (threadIdx.x & 31) == 0) atomicMax(&g.stamps[3 * b + 2], (unsigned long long)globaltimer_ns());
}

template <int D, int G>
int launch_gather_t(const GatherLaunch& gl, int ctas, cudaStream_t st) {
  const GatherParams& gp = gl.p;
  const size_t smem = gather_smem_bytes(gp.Hkv, D, gp.nst);
  auto kern = gp.dense ? gather_kernel<D, G, true> : gather_kernel<D, G, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  e = launch_pdl(kern, dim3(ctas), dim3(32 * gp.Hkv), smem, st, gl);
  return (int)e;
}

}  // namespace

// One gather CTA per SM: its Hkv warps and rings as deep as the SM's shared
// memory allows (single_cta_stages).
int gather_ctas_per_sm(const gk_pool_config*) { return 1; }

int fill_gather_params(const LaunchCommon& lc, int32_t layer, const gk_batch* b, const Plan* pl, bool dense,
                       GatherParams* out) {
  const gk_pool_config& c = *lc.cfg;
  GatherParams& gp = *out;
  gp = GatherParams{};
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
  gp.page_shift = -1;
  for (int sh = 0; sh < 31; ++sh)
    if ((1 << sh) == c.cold_page_size) gp.page_shift = sh;
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
  gp.nst = single_cta_stages(c.num_kv_heads, c.head_dim);
  gp.new_k = (const uint16_t*)b->d_new_k;
  gp.new_v = (const uint16_t*)b->d_new_v;
  return 0;
}

int launch_gather(const LaunchCommon& lc, void* stream, int32_t layer, const gk_batch* b, const Plan* pl,
                  bool dense) {
  const gk_pool_config& c = *lc.cfg;
  GatherLaunch gp;
  if (int e = fill_gather_params(lc, layer, b, pl, dense, &gp.p)) return e;
  gp.stamps = lc.gather_stamps;
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

}  // namespace gk
