// Split cascade launch: the prefix contraction and the suffix gather of one
// layer (GraniKV Section 3.3, the two levels of the cascade) in one launch,
// one CTA per SM.
//
// The prefix level is a dense contraction on the tensor cores that reads each
// prefix K/V tile once; the suffix level is a gather bound by HBM.  Run one
// after the other, every SM first waits on tensor-core work with HBM half
// idle, then streams with the tensor cores idle, and each launch pays its own
// ramp and tail.  Here CTA b < n_pre first runs prefix work item b (the plan
// makes items long: few key splits), then every CTA gathers its slot of the
// suffix partition; a prefix CTA's slot is cut to the time its item leaves,
// so that all CTAs are predicted to finish together while the tensor-core
// items overlap the other SMs' HBM stream.  Both levels write partial states;
// the merge (GraniKV Eq. 1) follows as its own launch.
#include "gather_body.cuh"
#include "prefix_body.cuh"
#include "prefix_warp_body.cuh"

namespace gk {
namespace {

struct SplitParams {
  prefix::PrefixParams pp;
  gather::GatherParams gp;
  int32_t n_pre;        // CTAs [0, n_pre) first run prefix item b
  int32_t n_gather;     // CTAs [0, n_gather) gather suffix slot b
  uint32_t data_bytes;  // shared data area: max of the prefix and gather layouts
  // SM-indexed slots (plans sized by the pool's SM speeds), else null: the CTA on SM s
  // takes slot slot_of_sm[s] (its prefix item, if the slot has one, and its gather
  // slot), claimed in slot_claim with this launch's tag; a slot already taken this
  // launch sends the CTA to the next free one
  const int32_t* slot_of_sm;
  uint32_t* slot_claim;
  uint32_t epoch;
  int32_t n_slots;
  unsigned long long* stamps;  // per slot: SM id, start, gather start, end (%globaltimer), or null
};

// The slot of the calling CTA (thread 0): its SM's planned slot if free this launch,
// else the next free one.  Every CTA claims exactly one of the n_slots slots, which
// the launch has as many CTAs as (atomic claims, no waiting); an SM that runs two
// CTAs one after the other gives the second another SM's slot.
__device__ __forceinline__ int claim_slot(const SplitParams& f) {
  unsigned smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  const int n = f.n_slots;
  int want = smid < (unsigned)n ? f.slot_of_sm[smid] : (int)(smid % (unsigned)n);
  if (want < 0 || want >= n) want = 0;
  for (int k = 0; k < n; ++k) {
    int t = want + k;
    if (t >= n) t -= n;
    if (atomicMax(&f.slot_claim[t], f.epoch) < f.epoch) return t;
  }
  return (int)blockIdx.x;  // unreachable: n CTAs claim n slots
}

constexpr uint32_t kSplitCtlBytes = prefix::kCtlBytes;
static_assert(1024 + kSplitCtlBytes <= gather::kSoleCtaReserve, "control area exceeds the gather reserve");

template <int D>
size_t split_data_bytes(int hkv) {
  const size_t g = gather::gather_data_bytes(hkv, D, gather::single_cta_stages(hkv, D));
  static_assert(prefix_warp::Layout<D>::kData <= prefix::Layout<D>::kData, "warp items fit the prefix layout");
  return g > prefix::Layout<D>::kData ? g : prefix::Layout<D>::kData;
}

// the block serves both roles: the prefix body's warps and the gather's
constexpr int kSplitThreads = prefix::kThreads > gather::kGatherThreads ? prefix::kThreads : gather::kGatherThreads;
static_assert(32 * kMaxKvHeads <= kSplitThreads && 32 * kMaxKvHeads <= prefix_warp::kThreads,
              "a gather CTA needs a warp per KV head");

// WARP: the prefix items are warp-MMA items (no tensor memory), else tensor-core
// items; two instantiations, so that neither path's registers constrain the other
// (warp items and the gather need 256 threads, which leaves each thread up to
// 255 registers; tensor-core items need 320)
template <int D, int G, bool WARP>
__global__ void __launch_bounds__(WARP ? prefix_warp::kThreads : kSplitThreads, 1)
    cascade_split_kernel(const SplitParams f) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t ctl = base + f.data_bytes;
  uint8_t* ctl_ptr = smem_raw + (ctl - raw);
  __shared__ int s_slot;
  int b = blockIdx.x;
  if (f.slot_of_sm) {
    if (threadIdx.x == 0) s_slot = claim_slot(f);
    __syncthreads();
    b = s_slot;
  }
  if (f.stamps && threadIdx.x == 0) {
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    f.stamps[4 * b] = smid;
    f.stamps[4 * b + 1] = globaltimer_ns();
  }

  griddep_launch_dependents();
  if (WARP && b < f.n_pre) {
    if (threadIdx.x == 0) *reinterpret_cast<volatile int*>(ctl_ptr + prefix::kCtlFlag) = 0;
    __syncthreads();
    // the item waits for the kernel before this one itself, after its table reads
    if (!prefix_warp::warp_item<D>(f.pp, f.pp.items[b], base, ctl, ctl_ptr)) return;  // same on every thread
  } else if (!WARP && b < f.n_pre) {
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctl_ptr + prefix::kCtlTmemSlot);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) *reinterpret_cast<volatile int*>(ctl_ptr + prefix::kCtlFlag) = 0;
    if (warp == 1) {
      tmem_alloc(ctl + prefix::kCtlTmemSlot, prefix::kTmemCols);
      tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the item waits for the kernel before this one itself, after its table reads
    const bool ok = prefix::prefix_item<D>(f.pp, f.pp.items[b], base, ctl, ctl_ptr, tmem);
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, prefix::kTmemCols);
    }
    if (!ok) return;  // same value on every thread
  }
  if (f.stamps && threadIdx.x == 0) f.stamps[4 * b + 2] = globaltimer_ns();
  // the item's staging area is free: the gather re-initialises the shared memory
  if (b < f.n_gather) gather::gather_segments<D, G, false>(f.gp, base, b);
  if (f.stamps && (threadIdx.x & 31) == 0) atomicMax(&f.stamps[4 * b + 3], (unsigned long long)globaltimer_ns());
}

template <int D, int G>
int launch_split_t(const SplitParams& fp, int ctas, cudaStream_t st, bool warp_items) {
  const size_t smem = 1024 + fp.data_bytes + kSplitCtlBytes;
  auto kern = warp_items ? cascade_split_kernel<D, G, true> : cascade_split_kernel<D, G, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  return (int)launch_pdl(kern, dim3(ctas), dim3(warp_items ? prefix_warp::kThreads : kSplitThreads), smem, st, fp);
}

}  // namespace

int launch_cascade_split(const LaunchCommon& lc, void* stream, int32_t layer, const gk_batch* b, const Plan* pl) {
  const gk_pool_config& c = *lc.cfg;
  SplitParams fp{};
  fill_prefix_params(lc, layer, b, pl, &fp.pp);
  if (int e = fill_gather_params(lc, layer, b, pl, false, &fp.gp)) return e;
  fp.n_pre = (int32_t)pl->prefix_items.size();
  const bool wi = pl->prefix_kind == 1;
  fp.n_gather = pl->summary.suffix_ctas;
  fp.stamps = lc.split_stamps;
  const int ctas = std::max(fp.n_pre, fp.n_gather);
  if (ctas == 0) return 0;
  if (!pl->slot_of_sm.empty()) {
    if (!lc.slot_claim || (int)pl->slot_of_sm.size() != ctas) return (int)cudaErrorInvalidValue;
    fp.slot_of_sm = (const int32_t*)((const uint8_t*)pl->d_buf + pl->off_slot_of_sm);
    fp.slot_claim = lc.slot_claim;
    fp.epoch = lc.epoch;
    fp.n_slots = ctas;
  }
  const int g = c.num_q_heads / c.num_kv_heads;
  cudaStream_t st = (cudaStream_t)stream;
  if (c.head_dim == 128) {
    fp.data_bytes = (uint32_t)split_data_bytes<128>(c.num_kv_heads);
    switch (g) {
      case 1: return launch_split_t<128, 1>(fp, ctas, st, wi);
      case 2: return launch_split_t<128, 2>(fp, ctas, st, wi);
      case 4: return launch_split_t<128, 4>(fp, ctas, st, wi);
      case 5: return launch_split_t<128, 5>(fp, ctas, st, wi);
      case 8: return launch_split_t<128, 8>(fp, ctas, st, wi);
    }
  } else if (c.head_dim == 64) {
    fp.data_bytes = (uint32_t)split_data_bytes<64>(c.num_kv_heads);
    switch (g) {
      case 1: return launch_split_t<64, 1>(fp, ctas, st, wi);
      case 2: return launch_split_t<64, 2>(fp, ctas, st, wi);
      case 4: return launch_split_t<64, 4>(fp, ctas, st, wi);
    }
  }
  return (int)cudaErrorInvalidValue;
}

}  // namespace gk
