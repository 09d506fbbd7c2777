// gk_decode_dense_static: the dense (flat) decode with its scratch in a fixed
// device array instead of memory allocated by the library or the caller.
//
// Who needs this: a serving engine that reserves all free HBM for its KV pool
// when it starts ("Paged KV cache", Implementation notes: allocate the whole
// pool up front and give the rest of the GPU to KV blocks), or any caller whose
// allocator is owned by a framework that fails or forbids allocations made
// behind its back.  Such callers cannot let a decode call grow device memory
// in the middle of serving.  gk_plan_build allocates device tables and partial
// states; this entry point instead keeps both in one statically sized array
// that is part of the loaded library image.
#include <atomic>
#include <cstring>

#include "device_common.cuh"
#include "gk_internal.h"

namespace gk {
namespace {

// The scratch: work tables and split-K partial states of one call.
// Every GPU that loads libgk holds these bytes until the process exits.
constexpr size_t kStaticScratchBytes = 8u << 20;
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
// device address of g_static_scratch, per device; host threads making their
// first call at the same time may both look it up and store the same value
std::atomic<uint8_t*> g_scratch_ptr[kMaxDevices] = {};

// Once per device, with that device current: host code names the array only
// through its symbol, so the device address comes from cudaGetSymbolAddress.
// The current device must be the pool's: another device's copy of the array
// would be a peer address the kernels must not touch.
gk_status scratch_address(Pool* p, uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(p, e, "cudaGetDevice");
  if (dev != p->dev.device)
    return fail(p, GK_ERR_INVALID, "the current device is not the pool's device (make the pool's device current)");
  if (dev < 0 || dev >= kMaxDevices) return fail(p, GK_ERR_UNSUPPORTED, "device ordinal beyond the static scratch table");
  uint8_t* ptr = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!ptr) {
    void* sym = nullptr;
    e = cudaGetSymbolAddress(&sym, g_static_scratch);
    if (e != cudaSuccess || !sym) return cuda_fail(p, e, "cudaGetSymbolAddress(static scratch)");
    ptr = (uint8_t*)sym;
    g_scratch_ptr[dev].store(ptr, std::memory_order_release);
  }
  *out = ptr;
  return GK_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace
}  // namespace gk

using gk::Plan;
using gk::Pool;

extern "C" gk_status gk_decode_dense_static(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch) {
  if (!pool || !batch) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  if (!p->has_device) return gk::fail(p, GK_ERR_INVALID, "pool has no device storage");
  if (layer < 0 || layer >= p->cfg.num_layers) return gk::fail(p, GK_ERR_INVALID, "layer out of range");
  if (batch->num_requests > 0 && (!batch->d_q || !batch->d_out || !batch->d_block_table))
    return gk::fail(p, GK_ERR_INVALID, "batch device pointers missing");
  if ((batch->d_new_k == nullptr) != (batch->d_new_v == nullptr))
    return gk::fail(p, GK_ERR_INVALID, "fused append needs both d_new_k and d_new_v");
  // the pool's error word is allocated when the pool first touches the device;
  // this call does not allocate it
  if (!p->d_error || !p->dev.queried)
    return gk::fail(p, GK_ERR_INVALID, "pool has not been used on the device yet (write its KV first)");
  // The work tables are copied from host memory that is freed on return; a
  // capturing stream would record that copy, so it is refused before any work.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t ce = cudaStreamIsCapturing((cudaStream_t)stream, &cap);
  if (ce != cudaSuccess) return gk::cuda_fail(p, ce, "cudaStreamIsCapturing");
  if (cap != cudaStreamCaptureStatusNone)
    return gk::fail(p, GK_ERR_UNSUPPORTED, "gk_decode_dense_static cannot run on a capturing stream");
  uint8_t* scratch = nullptr;
  gk_status st = gk::scratch_address(p, &scratch);
  if (st != GK_OK) return st;

  Plan pl;
  st = gk::build_host_plan(p, batch, &pl);
  if (st != GK_OK) return st;
  if (pl.B == 0) return GK_OK;

  // lay out the device tables and partial states inside the scratch
  const gk_pool_config& c = p->cfg;
  size_t off = 0;
  auto region = [&](size_t bytes, size_t align) {
    size_t o = gk::align_up(off, align);
    off = o + bytes;
    return o;
  };
  // the dense gather reads no tensor maps (only the prefix contraction does)
  pl.off_reqs = region(pl.reqs.size() * sizeof(gk::RequestDev), 16);
  pl.off_dense_begin = region(pl.dense_seg_begin.size() * sizeof(int32_t), 16);
  pl.off_dense_segs = region(pl.dense_segs.size() * sizeof(gk::SegmentDev), 16);
  pl.off_tmaps = 0;
  const size_t table_bytes = off;
  const size_t entries = (size_t)(pl.n_entries_dense > 0 ? pl.n_entries_dense : 0);
  const size_t po = region(entries * c.num_q_heads * c.head_dim * sizeof(float), 256);
  const size_t pll = region(entries * c.num_q_heads * sizeof(float), 256);
  if (off > gk::kStaticScratchBytes) {
    std::string m = "batch needs " + std::to_string(off) + " bytes of scratch; gk_decode_dense_static holds at most " +
                    std::to_string(gk::kStaticScratchBytes) + " (use gk_plan_build + gk_decode_dense)";
    return gk::fail(p, GK_ERR_INVALID, m);
  }
  // Everything the kernels read from the scratch is written here first; the
  // partial states are fully written before the merge reads them, so nothing
  // needs clearing.  Pageable copies: the host arrays may be freed on return.
  std::vector<uint8_t> host(table_bytes, 0);
  auto put = [&](size_t o, const void* src, size_t bytes) { if (bytes) std::memcpy(host.data() + o, src, bytes); };
  put(pl.off_reqs, pl.reqs.data(), pl.reqs.size() * sizeof(gk::RequestDev));
  put(pl.off_dense_begin, pl.dense_seg_begin.data(), pl.dense_seg_begin.size() * sizeof(int32_t));
  put(pl.off_dense_segs, pl.dense_segs.data(), pl.dense_segs.size() * sizeof(gk::SegmentDev));
  cudaError_t e = cudaMemcpyAsync(scratch, host.data(), table_bytes, cudaMemcpyHostToDevice, (cudaStream_t)stream);
  if (e != cudaSuccess) return gk::cuda_fail(p, e, "copying the work tables into the static scratch");
  pl.d_buf = scratch;
  pl.d_part_o = (float*)(scratch + po);
  pl.d_part_l = (float*)(scratch + pll);
  pl.part_entries = entries;
  pl.uploaded = true;

  gk::LaunchCommon lc{&p->cfg, p->d_error, p->dev.num_sms};
  int err;
  if (!pl.dense_segs.empty() && (err = gk::launch_gather(lc, stream, layer, batch, &pl, true)))
    return gk::cuda_fail(p, err, "dense gather kernel");
  if (pl.dense_needs_merge && (err = gk::launch_merge(lc, stream, batch, &pl, true)))
    return gk::cuda_fail(p, err, "merge kernel");
  // keep `host` alive until the pageable copy has been staged (it has, on return of cudaMemcpyAsync)
  return GK_OK;
}
