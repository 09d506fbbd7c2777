// Body of the gather attention (suffix kernel, flat backend), shared by the
// stand-alone kernel and the split cascade kernel.  The merge of the partial
// states is in merge.cu.
//
// Suffix kernel (GraniKV Section 3.3 / 3.5, cascade level 1): each request's
// COLD tokens are gathered through its block table ("Paged KV cache", How it
// works step 3: slot = table[t / P] * P + t % P) and attended with an online
// softmax.  Dense backend: the same kernel walks a request's whole context,
// its HOT prefix (contiguous per KV head, re-read for every request) then its
// COLD suffix, the flat paged decode the pages compare against.
//
// Work split: the plan cuts the concatenated token stream of all requests into
// one equal quota per CTA (one CTA per SM); a quota that spans a request
// boundary yields one segment per request.  Each segment produces a partial
// (O, LSE) state or, when it covers a whole request, the final output.
//
// CTA layout: warp h is KV head h and its g query heads, and it moves its own
// data.  A COLD token's row is Hkv*d contiguous bf16 in the pool; warp h
// copies only its head's d-wide slice of K and of V (256 bytes at d = 128)
// with 16-byte cp.async, 16 tokens per stage, into a private ring of stages in
// shared memory, nst - 1 stages ahead of its compute.  Many warps each with a
// few stages in flight keep more bytes moving per SM than one copy engine fed
// 2 KB rows, and no warp ever waits for another.  The warp loads 8x8 tiles
// with ldmatrix and runs the two small per-head products on the warp-level
// tensor-core MMA (m16n8k16, bf16 in, fp32 accumulate):
//   S^T[16 tok x 8] = K[16 tok x d] . Q_h^T[d x 8]   (the g query heads, padded to 8)
//   O^T[d x 8]     += V^T[d x 16 tok] . P^T[16 tok x 8]
// with the online softmax (running max, rescale, sum) on the S^T fragments and
// warp shuffles across the lanes that hold one head.  P^T is re-packed into
// the B-operand layout with movmatrix.  The product is 2*g flops per byte, so
// the kernel is bound by HBM; the MMA only keeps the issue slots free for the
// copies.
#pragma once
#include <cfloat>

#include "device_common.cuh"
#include "gk_internal.h"

namespace gk {
namespace gather {

constexpr int kT = kGatherT;  // tokens per stage (one m16 / k16 MMA step)
constexpr int kMaxStages = 16;  // ring depth cap (the rings take what shared memory the SM has)
constexpr int kGatherThreads = 32 * kMaxKvHeads;  // block size of the stand-alone kernel (warps = Hkv)

struct GatherParams {
  const uint16_t* hot_k;
  const uint16_t* hot_v;
  const uint16_t* cold_k;
  const uint16_t* cold_v;
  int64_t cold_slots;
  int64_t n_blocks;
  int32_t L, Hkv, Hq, page;
  int32_t page_shift;  // log2(page) when page is a power of two, else -1
  int32_t layer;
  int32_t dense;
  const int32_t* block_table;
  int32_t max_blocks;
  const uint16_t* q;
  float* out;
  float* lse;
  float* part_o;
  float* part_l;
  const RequestDev* reqs;
  const int32_t* seg_begin;
  const SegmentDev* segs;
  const uint8_t* tmaps;
  int32_t* err;
  float q_scale;  // log2(e) / sqrt(d): scores come out in the log2 domain
  int32_t nst;    // pipeline stages (<= kMaxStages)
  // fused append (else null): this layer's new token of every request, [B][Hkv][d];
  // a request's last COLD token is read from here and written into the pool
  const uint16_t* new_k;
  const uint16_t* new_v;
};

// Shared memory: each consumer warp owns a ring of nst stages; a stage holds
// its head's slices of kT tokens, K then V, one token row (d bf16) every
// slice_row_bytes -- 16 bytes more than the row, so that the eight rows an
// ldmatrix reads fall in eight different 16-byte bank groups.
__host__ __device__ constexpr uint32_t slice_row_bytes(int d) { return (uint32_t)d * 2 + 16; }
__host__ __device__ constexpr uint32_t warp_stage_bytes(int d) { return 2u * kT * slice_row_bytes(d); }
// each warp also keeps, per ring stage, which of its tokens was appended this
// step (fused append) and that token's pool offset
constexpr uint32_t kFreshRecBytes = 16;
// and a ring of nst + 1 slots of the block ids of a stage's tokens (kT int32),
// filled by cp.async nst + 1 stages ahead of the stage's copies
constexpr uint32_t kTabSlotBytes = kT * 4;
// and, for the whole CTA, its first kSegCache segment descriptors with the
// request fields the gather needs (req, t0, t1, entry, slen, lp, hot_base)
constexpr int kSegCache = 16;
constexpr uint32_t kSegRecBytes = 32;
__host__ __device__ constexpr size_t gather_rings_bytes(int hkv, int d, int nst) {
  return (size_t)hkv * nst * warp_stage_bytes(d) + (size_t)hkv * kMaxStages * kFreshRecBytes +
         (size_t)hkv * (nst + 1) * kTabSlotBytes;
}
__host__ __device__ constexpr size_t gather_data_bytes(int hkv, int d, int nst) {
  return gather_rings_bytes(hkv, d, nst) + (size_t)kSegCache * kSegRecBytes;
}
__host__ __device__ constexpr size_t gather_smem_bytes(int hkv, int d, int nst) {
  return 1024 + gather_data_bytes(hkv, d, nst);
}
// opt-in dynamic shared memory of one CTA, and what a CTA that has the SM to
// itself keeps outside the rings (alignment slack, control blocks)
constexpr size_t kSmemPerCtaMax = 232448;
constexpr size_t kSoleCtaReserve = 1024 + 3072;
// ring depth when the gather CTA has the SM (and its shared memory) to itself
__host__ __device__ constexpr int single_cta_stages(int hkv, int d) {
  const int n = (int)((kSmemPerCtaMax - kSoleCtaReserve - (size_t)kSegCache * kSegRecBytes -
                       (size_t)hkv * (kMaxStages * kFreshRecBytes + kTabSlotBytes)) /
                      ((size_t)hkv * (warp_stage_bytes(d) + kTabSlotBytes)));
  return n > kMaxStages ? kMaxStages : n;
}

// wait until at most n (0..kMaxStages-1) of this thread's cp.async groups are pending
__device__ __forceinline__ void cp_async_wait_pending(int n) {
  switch (n) {
#define GK_WAIT_CASE(i) \
  case i:               \
    asm volatile("cp.async.wait_group %0;" ::"n"(i) : "memory"); \
    break;
    GK_WAIT_CASE(0) GK_WAIT_CASE(1) GK_WAIT_CASE(2) GK_WAIT_CASE(3) GK_WAIT_CASE(4) GK_WAIT_CASE(5)
    GK_WAIT_CASE(6) GK_WAIT_CASE(7) GK_WAIT_CASE(8) GK_WAIT_CASE(9) GK_WAIT_CASE(10) GK_WAIT_CASE(11)
    GK_WAIT_CASE(12) GK_WAIT_CASE(13) GK_WAIT_CASE(14)
#undef GK_WAIT_CASE
    default:
      asm volatile("cp.async.wait_group 15;" ::: "memory");
  }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// D = A(16x16, row) . B(16x8, col) + D ; bf16 in, fp32 accumulate
__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The gather work of CTA `cta` (its segments of the plan's partition) on the
// calling CTA.  Warp h < Hkv is KV head h and its g query heads; further warps
// return at once.  Each warp streams its own data: it copies its head's K and
// V slices of the stage nst-1 ahead into its ring with 16-byte cp.async (one
// commit group per stage), waits for the oldest group, and computes on it, so
// no warp waits for another.  The block ids of a stage are read (cp.async,
// into shared memory) nst + 1 stages before its copies.  `base` (16-byte
// aligned) holds gather_data_bytes(Hkv, D, p.nst).  All threads of the CTA
// call it.
template <int D, int G, bool DENSE>
__device__ __forceinline__ void gather_segments(const GatherParams& p, uint32_t base, int cta) {
  constexpr int KSTEPS = D / 16;       // k16 steps of the QK product, m16 tiles of the PV product
  constexpr uint32_t SR = slice_row_bytes(D);
  constexpr uint32_t WS = warp_stage_bytes(D);
  constexpr int CPT = D / 8;           // 16-byte chunks per token slice
  constexpr int CPL = kT * CPT / 32;   // chunks per lane per stage and tensor
  const int Hkv = p.Hkv;
  const int nst = p.nst;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Zero the rings once: a partial stage leaves rows past its tokens untouched,
  // and those rows must hold finite values (they meet P = 0 in the MMA).
  for (uint32_t off = threadIdx.x * 16; off < (uint32_t)gather_rings_bytes(Hkv, D, nst); off += blockDim.x * 16)
    sts128(base + off, make_uint4(0, 0, 0, 0));
  // The CTA's segment descriptors and their requests' fields, read once into
  // shared memory: a segment change then costs no round trip to memory.  The
  // plan's tables are never written by the kernels of a step, so this runs
  // before the dependency wait, while the kernel before this one finishes.
  const int seg0 = p.seg_begin[cta], seg1 = p.seg_begin[cta + 1];
  const uint32_t segc = base + (uint32_t)gather_rings_bytes(Hkv, D, nst);
  for (int i = threadIdx.x; i < min(seg1 - seg0, kSegCache); i += blockDim.x) {
    const SegmentDev sd = p.segs[seg0 + i];
    const RequestDev& rq = p.reqs[sd.req];
    const int64_t hb = rq.hot_base;
    sts128(segc + i * kSegRecBytes, make_uint4((uint32_t)sd.req, (uint32_t)sd.t0, (uint32_t)sd.t1, (uint32_t)sd.entry));
    sts128(segc + i * kSegRecBytes + 16, make_uint4((uint32_t)rq.slen, (uint32_t)rq.lp, (uint32_t)hb, (uint32_t)(hb >> 32)));
  }
  __syncthreads();
  griddep_wait();   // queries, pool rows and the partial-state buffer are written upstream
  if (warp >= Hkv) return;

  const int h = warp;
  const uint32_t ring = base + (uint32_t)h * nst * WS;
  // per ring stage, 16 bytes: index in the stage of the request's appended token
  // (-1: none) and its pool offset (elements, head h; the same for K and V)
  const uint32_t recs = base + (uint32_t)Hkv * nst * WS + (uint32_t)h * kMaxStages * kFreshRecBytes;
  const bool fused_append = p.new_k != nullptr;
  const int64_t layer_rows = (int64_t)p.layer * p.cold_slots;
  // head h's slice of pool row 0 of this layer; row r's slice is Hkv * D elements further per row
  const uint16_t* const ck_h = p.cold_k + (layer_rows * Hkv + h) * D;
  const uint16_t* const cv_h = p.cold_v + (layer_rows * Hkv + h) * D;
  // segment sg's descriptor and its request's fields (shared-memory copy when cached)
  struct SegInfo {
    int req, t0, t1, entry, slen, lp;
    int64_t hot_base;
  };
  auto seg_info = [&](int sg) {
    SegInfo si;
    if (sg - seg0 < kSegCache) {
      const uint4 a = lds128(segc + (sg - seg0) * kSegRecBytes);
      const uint4 b = lds128(segc + (sg - seg0) * kSegRecBytes + 16);
      si.req = (int)a.x; si.t0 = (int)a.y; si.t1 = (int)a.z; si.entry = (int)a.w;
      si.slen = (int)b.x; si.lp = (int)b.y;
      si.hot_base = (int64_t)(((uint64_t)b.w << 32) | b.z);
    } else {
      const SegmentDev sd = p.segs[sg];
      const RequestDev rq = p.reqs[sd.req];
      si.req = sd.req; si.t0 = sd.t0; si.t1 = sd.t1; si.entry = sd.entry;
      si.slen = rq.slen; si.lp = rq.lp; si.hot_base = rq.hot_base;
    }
    return si;
  };

  // ---- block-id lookups nst + 1 stages ahead of the copies ----
  // A stage's copies need its tokens' block ids, and a table read is a round
  // trip to memory (the table does not stay in L2 under the KV stream).  A
  // lookup cursor runs nst + 1 stages ahead of the copy cursor and has each
  // lane cp.async its token's block id into the warp's ring of id slots; the
  // ids travel in the cp.async groups of the stages copied in between, so a
  // stage's ids have landed (its group waited for) before the stage is copied,
  // and no register ever holds an id whose load is still in flight (a register
  // queue of ids stalls the warp when it shifts).
  struct Cursor {
    int sg, t, t1, lp, req, slen;
    const int32_t* table;
    int64_t hot_row0;  // element offset of the (layer, head h) rows of the request's HOT prefix
  };
  const uint32_t tabs = base + (uint32_t)Hkv * nst * WS + (uint32_t)Hkv * kMaxStages * kFreshRecBytes +
                        (uint32_t)h * (nst + 1) * kTabSlotBytes;
  auto cursor_at = [&](int sg) {
    Cursor c{};
    c.sg = sg;
    if (sg < seg1) {
      const SegInfo si = seg_info(sg);
      c.t = si.t0;
      c.t1 = si.t1;
      c.req = si.req;
      c.slen = si.slen;
      c.lp = DENSE ? si.lp : 0;
      c.table = p.block_table + (int64_t)si.req * p.max_blocks;
      if (DENSE && c.lp > 0) c.hot_row0 = si.hot_base * p.L * Hkv * D + ((int64_t)p.layer * Hkv + h) * c.lp * D;
    }
    return c;
  };
  auto stage_len = [&](const Cursor& c) {
    int n = min(kT, c.t1 - c.t);
    if (DENSE && c.t < c.lp) n = min(n, c.lp - c.t);
    return n;
  };
  auto advance = [&](const Cursor& c) {
    if (c.sg >= seg1) return c;
    Cursor r = c;
    r.t += stage_len(c);
    return r.t < r.t1 ? r : cursor_at(c.sg + 1);
  };
  // the lookup cursor: read the block ids of its stage into id slot lslot, move on
  Cursor lk = cursor_at(seg0);
  int lslot = 0;
  auto lookup = [&]() {
    if (lk.sg < seg1) {
      const int n = stage_len(lk);
      if (!(DENSE && lk.t < lk.lp) && lane < n) {
        const int ti = lk.t - lk.lp + lane;
        const int32_t* src = lk.table + (p.page_shift >= 0 ? ti >> p.page_shift : ti / p.page);
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(tabs + (uint32_t)lslot * kTabSlotBytes + lane * 4),
                     "l"(src) : "memory");
      }
      lk = advance(lk);
    }
    if (++lslot == nst + 1) lslot = 0;
  };
  // the copy cursor: issue its stage's copies into ring slot islot, move on
  Cursor cc = lk;
  int islot = 0, cidslot = 0;  // ring slot and id slot of the next stage copied
  auto copy_stage = [&]() {
    const uint32_t kdst = ring + (uint32_t)islot * WS, vdst = kdst + kT * SR;
    const uint32_t rec = recs + (uint32_t)islot * kFreshRecBytes;
    const int n = cc.sg < seg1 ? stage_len(cc) : 0;
    if (n > 0 && DENSE && cc.t < cc.lp) {
      // HOT: the stage's rows of this head are contiguous
      const int64_t row0 = cc.hot_row0 + (int64_t)cc.t * D;
      for (int ci = lane; ci < n * CPT; ci += 32) {
        const uint32_t o = (uint32_t)(ci / CPT) * SR + (ci % CPT) * 16;
        cp_async16(kdst + o, p.hot_k + row0 + ci * 8);
        cp_async16(vdst + o, p.hot_v + row0 + ci * 8);
      }
      if (lane == 0) sts128(rec, make_uint4(0xffffffffu, 0u, 0u, 0u));
    } else if (n > 0) {
      // COLD: lane i < n turns its token's block id into its pool row (slot;
      // the pool holds fewer than 2^31 slots)
      const int tt0 = cc.t - cc.lp;
      int32_t row = -1;
      if (lane < n) {
        int32_t blk;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(blk) : "r"(tabs + (uint32_t)cidslot * kTabSlotBytes + lane * 4));
        const int ti = tt0 + lane;
        const int in_page = p.page_shift >= 0 ? ti & (p.page - 1) : ti % p.page;
        if (blk >= 0 && blk < p.n_blocks)
          row = blk * p.page + in_page;
        else
          report_error(p.err, kErrBounds);
      }
      // the appended token comes from the new-token arrays (copied after the
      // loop, which keeps the loop free of branches); its pool slot is written
      // once the stage lands (see the compute loop)
      const int fi = cc.slen - 1 - tt0;
      const int fresh = fused_append && fi >= 0 && fi < n ? fi : -1;
      int64_t fresh_off = -1;
      if (fresh >= 0) {
        const int32_t fr = __shfl_sync(0xffffffffu, row, fresh);
        if (fr >= 0) fresh_off = ((layer_rows + fr) * Hkv + h) * D;
        if (lane == fresh) row = -1;
      }
      if (lane == 0)
        sts128(rec, make_uint4((uint32_t)(fresh_off >= 0 ? fresh : -1), (uint32_t)fresh_off,
                               (uint32_t)(fresh_off >> 32), 0u));
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int ci = lane + 32 * j, tok = ci / CPT, ch = ci % CPT;
        const int32_t r = __shfl_sync(0xffffffffu, row, tok);
        if (tok < n && r >= 0) {
          const uint32_t o = (uint32_t)tok * SR + ch * 16;
          const int64_t src = (int64_t)r * (Hkv * D) + ch * 8;
          cp_async16(kdst + o, ck_h + src);
          cp_async16(vdst + o, cv_h + src);
        }
      }
      if (fresh_off >= 0 && lane < CPT) {
        const int64_t fs = ((int64_t)cc.req * Hkv + h) * D + lane * 8;
        const uint32_t o = (uint32_t)fresh * SR + lane * 16;
        cp_async16(kdst + o, p.new_k + fs);
        cp_async16(vdst + o, p.new_v + fs);
      }
    } else if (lane == 0) {
      sts128(rec, make_uint4(0xffffffffu, 0u, 0u, 0u));
    }
    cp_async_commit();
    cc = advance(cc);
    if (++islot == nst) islot = 0;
    if (++cidslot == nst + 1) cidslot = 0;
  };
  // one stage copied, one looked up: the ids read here join the next stage's group
  auto issue_next = [&]() {
    copy_stage();
    lookup();
  };
  // Q_h^T of a segment as the B operand: b[kk][0] = (d 16kk+2tq, +1; head gq),
  // b[kk][1] = (d +8, +9; head gq).  Each segment's rows are loaded one segment
  // ahead (the first ones here, before the prologue's waits).
  const int gq = lane >> 2;  // fragment row group
  const int tq = lane & 3;   // fragment column pair
  uint32_t qn[KSTEPS][2];
  auto load_q = [&](int req) {
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + ((int64_t)req * p.Hq + h * G + min(gq, G - 1)) * D);
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      qn[kk][0] = gq < G ? qrow[kk * 8 + tq] : 0u;
      qn[kk][1] = gq < G ? qrow[kk * 8 + 4 + tq] : 0u;
    }
  };
  if (seg0 < seg1) load_q(seg_info(seg0).req);
  // the first nst + 1 stages' ids in a group of their own, waited for once
  for (int i = 0; i < nst + 1; ++i) lookup();
  cp_async_commit();
  cp_async_wait_pending(0);
  __syncwarp();
  for (int i = 0; i < nst - 1; ++i) issue_next();

  // ---- compute, segment by segment ----
  const int mi = lane >> 3, mj = lane & 7;  // ldmatrix: matrix index, row within it
  int cslot = 0;  // ring slot of the stage computed next
  for (int sg = seg0; sg < seg1; ++sg) {
    const SegInfo seg = seg_info(sg);
    const int lp = DENSE ? seg.lp : 0;
    uint32_t qb[KSTEPS][2];
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      qb[kk][0] = qn[kk][0];
      qb[kk][1] = qn[kk][1];
    }
    if (sg + 1 < seg1) load_q(seg_info(sg + 1).req);
    float o[KSTEPS][4];
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2tq and 2tq+1

    for (int t = seg.t0; t < seg.t1;) {
      int n = min(kT, seg.t1 - t);
      if (DENSE && t < lp) n = min(n, lp - t);
      issue_next();                  // stage k + nst - 1
      cp_async_wait_pending(nst - 1);  // stage k has landed (this lane's copies) ...
      __syncwarp();                  // ... and every lane's
      const uint32_t ks = ring + (uint32_t)cslot * WS, vs = ks + kT * SR;
      if (fused_append) {
        // the request's appended token is in this stage: put head h's rows into the pool
        const uint4 rec = lds128(recs + (uint32_t)cslot * kFreshRecBytes);
        const int ft = (int)rec.x;
        if (ft >= 0 && lane < CPT) {
          const int64_t off = (int64_t)(((uint64_t)rec.z << 32) | rec.y);
          uint16_t* pk = const_cast<uint16_t*>(p.cold_k) + off;
          uint16_t* pv = const_cast<uint16_t*>(p.cold_v) + off;
          reinterpret_cast<uint4*>(pk)[lane] = lds128(ks + (uint32_t)ft * SR + lane * 16);
          reinterpret_cast<uint4*>(pv)[lane] = lds128(vs + (uint32_t)ft * SR + lane * 16);
        }
      }
      // address of 16-byte chunk c of token row tok in a slice
      auto chunk_addr = [&](uint32_t slice, int tok, int c) -> uint32_t { return slice + (uint32_t)tok * SR + c * 16; };
      // S^T = K Q_h^T, the even and odd k16 steps in two accumulators (two
      // MMA dependency chains of half the length)
      float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < KSTEPS; kk += 2) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(chunk_addr(ks, mj + 8 * (mi & 1), 2 * kk + (mi >> 1)), a0, a1, a2, a3);
        ldsm_x4(chunk_addr(ks, mj + 8 * (mi & 1), 2 * (kk + 1) + (mi >> 1)), b0, b1, b2, b3);
        mma16816(sc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
        mma16816(sd, b0, b1, b2, b3, qb[kk + 1][0], qb[kk + 1][1]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) sc[i] += sd[i];
      // online softmax over the 16 tokens (rows gq and gq+8) for heads 2tq, 2tq+1
      const bool v_lo = gq < n, v_hi = gq + 8 < n;
      const float s00 = v_lo ? sc[0] * p.q_scale : -INFINITY;
      const float s01 = v_lo ? sc[1] * p.q_scale : -INFINITY;
      const float s10 = v_hi ? sc[2] * p.q_scale : -INFINITY;
      const float s11 = v_hi ? sc[3] * p.q_scale : -INFINITY;
      float x0 = fmaxf(s00, s10), x1 = fmaxf(s01, s11);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
      }
      const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
      if (__any_sync(0xffffffffu, n0 != m0 || n1 != m1)) {
        const float a0 = ex2(m0 - n0), a1 = ex2(m1 - n1);
        l0 *= a0;
        l1 *= a1;
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt) {
          o[mt][0] *= a0; o[mt][1] *= a1; o[mt][2] *= a0; o[mt][3] *= a1;
        }
        m0 = n0;
        m1 = n1;
      }
      const float p00 = ex2(s00 - m0), p01 = ex2(s01 - m1), p10 = ex2(s10 - m0), p11 = ex2(s11 - m1);
      l0 += p00 + p10;
      l1 += p01 + p11;
      // P^T (16 tok x 8 heads) -> B operand of the PV product
      const uint32_t pb0 = movm_t(pack_bf16x2(p00, p01));
      const uint32_t pb1 = movm_t(pack_bf16x2(p10, p11));
      // O^T += V^T P^T
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(chunk_addr(vs, mj + 8 * (mi >> 1), 2 * mt + (mi & 1)), a0, a1, a2, a3);
        mma16816(o[mt], a0, a1, a2, a3, pb0, pb1);
      }
      __syncwarp();                  // every lane has read the stage before it is refilled
      t += n;
      if (++cslot == nst) cslot = 0;
    }

    // finish: the row sums live on the 8 lanes that share tq
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    const float i0 = 1.f / l0, i1 = 1.f / l1;
    const int hh0 = 2 * tq, hh1 = 2 * tq + 1;
    float* dst;
    float* dl;
    int64_t row0;
    if (seg.entry >= 0) {
      row0 = (int64_t)seg.entry * p.Hq + h * G;
      dst = p.part_o;
      dl = p.part_l;
    } else {
      row0 = (int64_t)seg.req * p.Hq + h * G;
      dst = p.out;
      dl = p.lse;
    }
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) {
      const int d0 = mt * 16 + gq;
      if (hh0 < G) {
        dst[(row0 + hh0) * D + d0] = o[mt][0] * i0;
        dst[(row0 + hh0) * D + d0 + 8] = o[mt][2] * i0;
      }
      if (hh1 < G) {
        dst[(row0 + hh1) * D + d0] = o[mt][1] * i1;
        dst[(row0 + hh1) * D + d0 + 8] = o[mt][3] * i1;
      }
    }
    if (gq == 0 && dl) {
      const float f = seg.entry >= 0 ? 1.f : kLn2;   // partials keep log2, outputs are natural log
      if (hh0 < G) dl[row0 + hh0] = (m0 + __log2f(l0)) * f;
      if (hh1 < G) dl[row0 + hh1] = (m1 + __log2f(l1)) * f;
    }
  }
  cp_async_wait_pending(0);
}

}  // namespace gather

// kernel arguments of the gather for one layer of a planned batch (dense: the
// flat backend's partition, else the cascade suffix partition)
int fill_gather_params(const LaunchCommon& lc, int32_t layer, const gk_batch* b, const Plan* pl, bool dense,
                       gather::GatherParams* out);

}  // namespace gk
