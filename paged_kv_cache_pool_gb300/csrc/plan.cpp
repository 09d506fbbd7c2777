// Per-step planner, dispatcher and the decode entry points of libgk.
//
// One plan per decode step, reused by every layer (the plan depends only on
// which requests share which prefix and on the context lengths).
#include <cuda_runtime.h>

#include <algorithm>
#include <cctype>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <unordered_map>

#include "gk_internal.h"

namespace gk {

namespace {

constexpr int kGatherQuantum = 16;        // gather CTAs get token quotas in multiples of this
constexpr int kMinGatherQuota = 64;
// A split plan's prefix CTAs keep at least this share of a gather-only CTA's
// suffix: an item that leaves its CTA nothing to gather ends late beside a
// gather that keeps HBM busy, and then the other SMs wait for it.
constexpr double kMinPrefixShare = 0.15;
// The split search prices each item this much longer than the model: per-CTA
// timelines of split launches put item ends up to about 15 % from the fitted
// item time.
constexpr double kSplitItemMargin = 1.15;
// GK_PREFIX_AUTO keeps tensor-core items only when their cascade is predicted
// faster than the warp-MMA items' by this factor, and never for a step whose
// groups stack at most kWarpOnlyMeff rows per KV head: a tensor-core item pads
// them to 256 rows, and on the GB300 sweep the warp-MMA items won every such
// step the model would have given to tensor-core items.
constexpr double kTensorAutoEdge = 0.9;
constexpr int32_t kWarpOnlyMeff = 64;

}  // namespace

// Split launch (one CTA per SM): CTAs [0, n_pre) first run a prefix item of `it`
// us, and the suffix (S bytes; W = S / gather_sm SM-us at a gather-only CTA's
// rate, gather_sm_gbs for the launch's kind of item) is spread over the CTAs so
// that all end together.  Gather-only CTAs start after c_gather_split (the split
// launch's own fixed cost, fitted apart from the stand-alone gather's c_gather);
// a prefix CTA starts prefix_cta_ramp after its item and gathers at
// prefix_cta_gather_ratio of that rate.  With gather = false only the
// gather-only CTAs gather.  The gather as a whole takes at least c_gather_split +
// S / bw_suffix, and the launch at least (S + P) / bw_suffix (HBM).  share = a
// prefix CTA's tokens over a gather-only CTA's.
SplitTime split_time(const gk_cost_model& cm, int num_sms, int64_t n_pre, double it, double S, double P,
                     bool gather, double gather_sm_gbs) {
  SplitTime r{std::max(it, (S + P) / (cm.bw_suffix_gbs * 1e3)), 0.0};
  if (S <= 0.0) return r;
  const double cg = cm.c_gather_split_us, ramp = cm.prefix_cta_ramp_us, e = cm.prefix_cta_gather_ratio;
  const double W = S / (gather_sm_gbs * 1e3);
  const double n = (double)n_pre, a = (double)(num_sms - n_pre);
  double T;
  if (gather && n > 0 && e > 0) {
    T = (W + a * cg + n * e * (it + ramp)) / (a + n * e);
    const double busy = T - cg;
    r.share = busy > 0 ? std::max(0.0, e * (T - it - ramp) / busy) : 0.0;
  } else {
    T = a > 0 ? cg + W / a : 1e300;
  }
  T = std::max(T, cg + S / (cm.bw_suffix_gbs * 1e3));
  r.t = std::max(r.t, T);
  return r;
}

// Gather weights of the CTAs (slots) of a split launch, one prefix item time per
// prefix slot (it[b], slot b < it.size(); none when the prefix CTAs do not
// gather) and one relative gather speed per slot (v[b]: the speed of the SM the
// slot is planned on, 1 without SM speeds).  Items of different lengths leave
// their CTAs different times to gather, and SMs gather at different speeds.
// Slot b starts gathering at s_b = max(c_gather_split, it[b] + prefix_cta_ramp),
// at prefix_cta_gather_ratio (e) of the rate; gather-only slots at c =
// c_gather_split.  The common end T is the one at which the slots together gather
// W = S / gather_sm SM-us:
//   sum_gather-only v_x (T - c) + sum_b e v_b max(0, T - s_b) = W
// (increasing in T: bisection).  Weight = a slot's tokens over those of a
// gather-only slot of speed 1.
std::vector<double> split_weights(const gk_cost_model& cm, int num_sms, const std::vector<double>& it, double S,
                                  double gather_sm_gbs, const std::vector<double>& v, bool prefix_gathers) {
  std::vector<double> w((size_t)num_sms, 1.0);
  const double c = cm.c_gather_split_us, e = cm.prefix_cta_gather_ratio;
  const double W = S / (gather_sm_gbs * 1e3);
  const size_t n_pre = std::min(it.size(), w.size());
  std::vector<double> start(w.size(), c), rate(w.size(), 1.0);
  for (size_t x = 0; x < w.size(); ++x) rate[x] = x < v.size() ? v[x] : 1.0;
  for (size_t b = 0; b < n_pre; ++b) {
    start[b] = std::max(c, it[b] + cm.prefix_cta_ramp_us);
    rate[b] *= prefix_gathers ? e : 0.0;
  }
  auto capacity = [&](double T) {
    double cap = 0.0;
    for (size_t x = 0; x < w.size(); ++x) cap += rate[x] * std::max(0.0, T - start[x]);
    return cap;
  };
  double lo = c, hi = c + 1.0;
  while (capacity(hi) < W && hi < 1e12) hi = c + 2.0 * (hi - c);
  for (int i = 0; i < 100; ++i) {
    const double mid = 0.5 * (lo + hi);
    (capacity(mid) < W ? lo : hi) = mid;
  }
  const double full = std::max(hi - c, 1e-9);
  for (size_t x = 0; x < w.size(); ++x) w[x] = rate[x] * std::max(0.0, hi - start[x]) / full;
  return w;
}

double merge_us(const gk_cost_model& cm, int32_t B, int32_t Hq, int64_t partials) {
  if (B <= 0) return 0.0;
  return cm.c_merge_us * (double)B * Hq + cm.c_merge_state_us * (double)partials / B;
}

namespace {

template <class T>
size_t append_region(size_t* off, size_t count, size_t align = 16) {
  size_t o = (*off + align - 1) / align * align;
  *off = o + count * sizeof(T);
  return o;
}

// Split the concatenated token stream of all requests (lengths n[r]) into CTA
// quotas; each CTA's slice becomes one segment per request it touches.
void partition_tokens(const std::vector<int64_t>& n, int64_t max_ctas, std::vector<int32_t>* begin,
                      std::vector<SegmentDev>* segs) {
  begin->clear();
  segs->clear();
  int64_t total = 0;
  for (int64_t x : n) total += x;
  begin->push_back(0);
  if (total == 0) return;
  int64_t quota = (total + max_ctas - 1) / max_ctas;
  quota = std::max<int64_t>(quota, kMinGatherQuota);
  quota = (quota + kGatherQuantum - 1) / kGatherQuantum * kGatherQuantum;
  int64_t left = quota;
  for (size_t r = 0; r < n.size(); ++r) {
    int64_t t = 0;
    while (t < n[r]) {
      int64_t take = std::min(left, n[r] - t);
      segs->push_back(SegmentDev{(int32_t)r, (int32_t)t, (int32_t)(t + take), -1});
      t += take;
      left -= take;
      if (left == 0) {
        begin->push_back((int32_t)segs->size());
        left = quota;
      }
    }
  }
  if (begin->back() != (int32_t)segs->size()) begin->push_back((int32_t)segs->size());
}

// Tangram's ahead-of-time work partitioning (Algorithm 1) with requests in the
// place of its head groups and their token counts as budgets: the per-split
// target is tau = max(1, ceil(total / ctas)), request r takes
// S_r = max(1, ceil(n_r / tau)) splits, and each split is one CTA's single
// segment; the first n_r mod S_r splits are one token longer.
void partition_per_request(const std::vector<int64_t>& n, int64_t ctas, std::vector<int32_t>* begin,
                           std::vector<SegmentDev>* segs) {
  begin->clear();
  segs->clear();
  begin->push_back(0);
  int64_t total = 0;
  for (int64_t x : n) total += x;
  if (total == 0) return;
  const int64_t tau = std::max<int64_t>(1, (total + ctas - 1) / ctas);
  for (size_t r = 0; r < n.size(); ++r) {
    if (n[r] == 0) continue;
    const int64_t splits = std::max<int64_t>(1, (n[r] + tau - 1) / tau);
    const int64_t base = n[r] / splits, extra = n[r] % splits;
    int64_t t = 0;
    for (int64_t i = 0; i < splits; ++i) {
      const int64_t len = base + (i < extra ? 1 : 0);
      segs->push_back(SegmentDev{(int32_t)r, (int32_t)t, (int32_t)(t + len), -1});
      t += len;
      begin->push_back((int32_t)segs->size());
    }
  }
}

// As partition_tokens, over exactly w.size() CTA slots: slot b's quota is the
// share w[b] / sum(w) of the tokens, its end rounded to a multiple of
// kGatherQuantum (the last slot takes the rest); a slot may be empty.
void partition_tokens_weighted(const std::vector<int64_t>& n, const std::vector<double>& w,
                               std::vector<int32_t>* begin, std::vector<SegmentDev>* segs) {
  begin->clear();
  segs->clear();
  int64_t total = 0;
  for (int64_t x : n) total += x;
  begin->push_back(0);
  if (total == 0) return;
  double wsum = 0.0;
  for (double x : w) wsum += x;
  // end of each slot in the concatenated token stream
  std::vector<int64_t> ends(w.size());
  double acc = 0.0;
  for (size_t b = 0; b < w.size(); ++b) {
    acc += w[b];
    int64_t e = (int64_t)((double)total * acc / wsum + 0.5);
    e = (e + kGatherQuantum / 2) / kGatherQuantum * kGatherQuantum;
    e = std::min(total, std::max(e, b ? ends[b - 1] : (int64_t)0));
    ends[b] = b + 1 == w.size() ? total : e;
  }
  size_t slot = 0;
  int64_t pos = 0;   // tokens of the stream already placed
  while (slot < w.size() && ends[slot] == 0) {
    begin->push_back(0);
    ++slot;
  }
  for (size_t r = 0; r < n.size(); ++r) {
    int64_t t = 0;
    while (t < n[r]) {
      const int64_t take = std::min(ends[slot] - pos, n[r] - t);
      segs->push_back(SegmentDev{(int32_t)r, (int32_t)t, (int32_t)(t + take), -1});
      t += take;
      pos += take;
      while (slot < w.size() && pos == ends[slot]) {
        begin->push_back((int32_t)segs->size());
        ++slot;
      }
    }
  }
  while (begin->size() < w.size() + 1) begin->push_back((int32_t)segs->size());
}

// 16-row groups of the fullest warp-MMA item of a step, rounded up to 1, 2, 4 or
// 8: a group of M stacked rows fills items of kPrefixWarpRows rows, the last
// one with M mod kPrefixWarpRows
int32_t warp_row_groups(const Pool*, const std::vector<std::vector<int32_t>>& members, int32_t g) {
  int32_t rows = 0;
  for (const auto& m : members) rows = std::max(rows, std::min<int32_t>((int32_t)m.size() * g, kPrefixWarpRows));
  const int32_t groups = (rows + 15) / 16;
  int32_t r = 1;
  while (r < groups) r *= 2;
  return rows > 0 ? r : 0;
}

}  // namespace

namespace {

// The host plan with prefix items of one kind (GK_PREFIX_TENSOR or GK_PREFIX_WARP).
gk_status build_host_plan_kind(Pool* p, const gk_batch* b, Plan* pl, gk_prefix_kernel kind) {
  const gk_pool_config& c = p->cfg;
  const int32_t B = b->num_requests;
  const int32_t Hkv = c.num_kv_heads, Hq = c.num_q_heads, d = c.head_dim, g = Hq / Hkv;
  const int64_t P = c.cold_page_size;
  if (B < 0) return fail(p, GK_ERR_INVALID, "num_requests < 0");
  if (B > 0 && (!b->prefix_hot_base || !b->prefix_len || !b->suffix_len))
    return fail(p, GK_ERR_INVALID, "batch host arrays missing");
  pl->pool = p;
  pl->B = B;
  pl->groups.clear();
  pl->group_hot_base.clear();
  pl->prefix_reqs.clear();
  pl->prefix_items.clear();
  pl->reqs.assign((size_t)B, RequestDev{});
  pl->group_bytes.clear();
  pl->group_flops.clear();

  // ---- validate and group by HOT prefix (stable: first appearance) -------------
  std::unordered_map<int64_t, int32_t> gid;
  std::vector<std::vector<int32_t>> members;
  for (int32_t r = 0; r < B; ++r) {
    int64_t base = b->prefix_hot_base[r];
    int32_t lp = b->prefix_len[r], s = b->suffix_len[r];
    if (s < 0) return fail(p, GK_ERR_INVALID, "negative suffix length");
    if ((int64_t)s > (int64_t)b->max_blocks * P)
      return fail(p, GK_ERR_INVALID, "suffix longer than the block-table row");
    RequestDev& rq = pl->reqs[(size_t)r];
    rq.hot_base = base;
    rq.slen = s;
    if (base < 0) {
      if (lp != 0) return fail(p, GK_ERR_INVALID, "prefix_len must be 0 without a HOT prefix");
      rq.hot_base = -1;
      rq.lp = 0;
      rq.group = -1;
      continue;
    }
    auto it = p->hot.live.find(base);
    if (it == p->hot.live.end() || it->second != lp)
      return fail(p, GK_ERR_INVALID, "request names a HOT prefix that is not live with that length");
    rq.lp = lp;
    auto f = gid.find(base);
    int32_t grp;
    if (f == gid.end()) {
      grp = (int32_t)members.size();
      gid[base] = grp;
      members.emplace_back();
      pl->group_hot_base.push_back(base);
    } else {
      grp = f->second;
    }
    members[(size_t)grp].push_back(r);
    rq.group = grp;
  }

  // ---- prefix contraction work: kind of item, arrangement, keys per item ---------
  const int num_sms = p->dev.num_sms;
  const int32_t G = (int32_t)members.size();
  std::vector<int32_t> ntiles((size_t)G);
  int32_t max_ntiles = 1;
  for (int32_t gi = 0; gi < G; ++gi) {
    int32_t lp = pl->reqs[(size_t)members[(size_t)gi][0]].lp;
    ntiles[(size_t)gi] = (lp + kPrefixTileN - 1) / kPrefixTileN;
    max_ntiles = std::max(max_ntiles, ntiles[(size_t)gi]);
  }
  const gk_cost_model& cm = p->cost;
  const int64_t kv_tok = 2LL * Hkv * d * 2;
  int64_t suffix_tokens = 0;
  for (int32_t r = 0; r < B; ++r) suffix_tokens += pl->reqs[(size_t)r].slen;
  const double S = (double)suffix_tokens * (double)kv_tok;
  double prefix_bytes = 0.0;
  for (int32_t gi = 0; gi < G; ++gi)
    prefix_bytes += (double)pl->reqs[(size_t)members[(size_t)gi][0]].lp * (double)kv_tok;

  // One kind of prefix item: `rows` stacked rows per item, its cost-model terms.
  // Sequential arrangement: every SM takes prefix items (waves of them), then
  // every SM gathers.  Keys per split: the fewest that minimise the waves times
  // the time of one item alone (C * tile + item).
  // Split arrangement: one launch in which CTA b < n_pre first runs one prefix
  // item of C key tiles, and every CTA (one per SM) gathers a slot of the
  // suffix, a prefix CTA's slot cut to the time its item leaves.  Predicted
  //   item'(C)  = C * tile_split + item_split
  //   T_split   = split_time(): the later of the items and the gather spread over
  //               the CTAs (gather-only ones from the start, prefix CTAs after their
  //               items when their share is worth it), held to HBM,
  // against the sequential arrangement's W waves of c_seq-tile items then the
  // gather as a second launch:
  //   T_seq = max(prefix_bytes / bw_prefix, W * item(c_seq)) + c_gather + S / bw_suffix.
  // The split is taken when some C is predicted faster than the sequential
  // arrangement; among equal predictions the fewest items (fewest partials)
  // win, and the chosen item count is then spread evenly over the key tiles.
  // Prefix CTAs whose share would fall below kMinPrefixShare of a gather-only
  // CTA's gather nothing; then the gather needs an SM of its own.
  struct KindPlan {
    int32_t rows = 0;
    std::vector<int32_t> mtiles;
    std::vector<uint8_t> single;   // the group's last row block fills one Q tile at most
    double tile = 0, tile_split = 0, item = 0, item_split = 0;
    bool split = false;
    int32_t c = 0;              // key tiles per item
    double t_levels = 0;        // predicted levels time of the chosen arrangement
    double prefix_cta_share = 1.0;
  };
  auto plan_kind = [&](int32_t rows, double tile, double tile_split, double item, double item_split) {
    KindPlan k;
    k.rows = rows;
    k.tile = tile;
    k.tile_split = tile_split;
    k.item = item;
    k.item_split = item_split;
    k.mtiles.resize((size_t)G);
    k.single.assign((size_t)G, 0);
    for (int32_t gi = 0; gi < G; ++gi) {
      const int32_t m = (int32_t)members[(size_t)gi].size() * g;
      k.mtiles[(size_t)gi] = (m + rows - 1) / rows;
      // a tensor-core row block with one Q tile's rows runs its tiles at about
      // twice the rate: in a sequential plan its items take two key splits each;
      // in a split plan one, and its CTA then gathers the longer for it
      k.single[(size_t)gi] = rows == kPrefixRowsPerCta && m % rows != 0 && m % rows <= kPrefixTileM;
    }
    // items of a plan with C tiles per split; `paired`: a one-Q-tile block's items
    // take two splits each (sequential plans)
    auto count_items = [&](int32_t C, bool paired) {
      int64_t units = 0;
      for (int32_t gi = 0; gi < G; ++gi) {
        const int64_t ns = (ntiles[(size_t)gi] + C - 1) / C;
        const int64_t one = paired ? k.single[(size_t)gi] : 0;
        units += ((int64_t)k.mtiles[(size_t)gi] - one) * Hkv * ns + one * Hkv * ((ns + 1) / 2);
      }
      return units;
    };
    auto n_items = [&](int32_t C) { return count_items(C, true); };
    auto n_split_items = [&](int32_t C) { return count_items(C, false); };
    int32_t c_seq = max_ntiles;
    {
      double best_cost = 1e300;
      for (int32_t C = 1; G > 0 && C <= max_ntiles; ++C) {
        const double cost = (double)((n_items(C) + num_sms - 1) / num_sms) * (C * tile + item);
        if (cost < best_cost - 1e-9) {
          best_cost = cost;
          c_seq = C;
        }
      }
    }
    double t_seq = S / (cm.bw_suffix_gbs * 1e3) + cm.c_gather_us;
    if (G > 0) {
      const double waves = (double)((n_items(c_seq) + num_sms - 1) / num_sms);
      t_seq += std::max(prefix_bytes / (cm.bw_prefix_gbs * 1e3), waves * (std::min(c_seq, max_ntiles) * tile + item));
    }
    auto item_us = [&](int32_t C) { return C * tile_split + item_split + cm.prefix_item_crowd_us * n_split_items(C); };
    // the split launch for items of C tiles: the prefix CTAs gather a share when it
    // reaches kMinPrefixShare of a gather-only CTA's, else only the others gather
    const double gsm = rows == kPrefixRowsPerCta ? cm.gather_sm_gbs * cm.split_gather_ratio_tensor : cm.gather_sm_gbs;
    auto split_of = [&](int32_t C, bool* gather, double margin = 1.0) {
      const double it = margin * item_us(C);
      SplitTime st = split_time(cm, num_sms, n_split_items(C), it, S, prefix_bytes, true, gsm);
      *gather = st.share >= kMinPrefixShare;
      if (!*gather) st = split_time(cm, num_sms, n_split_items(C), it, S, prefix_bytes, false, gsm);
      if (rows == kPrefixRowsPerCta) st.t += cm.split_tensor_us;
      return st;
    };
    int32_t c_split = 0;
    double t_split = 1e300;
    const bool can_split = G > 0 && suffix_tokens > 0 && p->cascade_mode != GK_CASCADE_SEQUENTIAL;
    if (can_split && p->cascade_mode == GK_CASCADE_SPLIT && p->cascade_tiles > 0) {
      const int32_t C = std::min(p->cascade_tiles, max_ntiles);
      if (n_split_items(C) <= num_sms) {
        bool gth;
        c_split = C;
        t_split = split_of(C, &gth).t;
      }
    } else {
      // items priced kSplitItemMargin long: beside the gather an item's time is
      // the model's least certain term, and an item that outlasts the gather
      // holds the whole launch
      double t_best = 1e300;
      for (int32_t C = max_ntiles; can_split && C >= 1; --C) {
        if (n_split_items(C) > num_sms) break;  // items only grow as C shrinks
        bool gth;
        const double t = split_of(C, &gth, kSplitItemMargin).t;
        // the gather needs an SM of its own unless the prefix CTAs take part
        if (!gth && n_split_items(C) >= num_sms) continue;
        if (t < t_best - 1e-9) {
          t_best = t;
          c_split = C;
        }
      }
      bool gth;
      if (c_split > 0) t_split = split_of(c_split, &gth).t;
    }
    // balance the chosen split: the fewest tiles per item that gives as many items
    while (c_split > 1 && n_split_items(c_split - 1) == n_split_items(c_split)) --c_split;
    k.split = c_split > 0 && (p->cascade_mode == GK_CASCADE_SPLIT || t_split < t_seq);
    k.c = k.split ? c_split : c_seq;
    k.t_levels = k.split ? t_split : t_seq;
    if (k.split) {
      bool gth;
      const SplitTime st = split_of(c_split, &gth);
      k.t_levels = st.t;
      k.prefix_cta_share = gth ? st.share : 0.0;
    }
    return k;
  };
  // Warp items: a tile costs warp_tile + R * warp_group, R the 16-row groups of the
  // fullest item rounded up to a power of two (its warps split the keys 8 / R ways).
  const int32_t warp_groups = warp_row_groups(p, members, g);
  const double warp_tile = cm.warp_tile_us + warp_groups * cm.warp_group_us;
  const KindPlan kp = kind == GK_PREFIX_WARP
                          ? plan_kind(kPrefixWarpRows, warp_tile, warp_tile * cm.warp_split_ratio, cm.warp_item_us,
                                      cm.warp_item_split_us)
                          : plan_kind(kPrefixRowsPerCta, cm.prefix_tile_us, cm.prefix_tile_split_us, cm.prefix_item_us,
                                      cm.prefix_item_split_us);
  pl->prefix_kind = kp.rows == kPrefixWarpRows ? 1 : 0;
  pl->split = kp.split;
  const int32_t best_c = kp.c;
  const std::vector<int32_t>& mtiles = kp.mtiles;
  const std::vector<uint8_t>& single = kp.single;
  const double prefix_cta_share = kp.prefix_cta_share;
  int32_t max_m = 0;
  int64_t pre_bytes = 0, pre_flops = 0;
  for (int32_t gi = 0; gi < G; ++gi) {
    PrefixGroupDev gd{};
    gd.lp = pl->reqs[(size_t)members[(size_t)gi][0]].lp;
    gd.m = (int32_t)members[(size_t)gi].size() * g;
    gd.req_base = (int32_t)pl->prefix_reqs.size();
    gd.split_tiles = best_c;
    gd.nsplit = (ntiles[(size_t)gi] + best_c - 1) / best_c;
    gd.tmap_index = 2 * gi;
    for (int32_t r : members[(size_t)gi]) pl->prefix_reqs.push_back(r);
    pl->groups.push_back(gd);
    max_m = std::max(max_m, gd.m);
    int64_t gb = (int64_t)gd.lp * 2 * Hkv * d * 2;
    int64_t gf = 4LL * (int64_t)members[(size_t)gi].size() * Hq * gd.lp * d;
    pl->group_bytes.push_back(gb);
    pl->group_flops.push_back(gf);
    pre_bytes += gb;
    pre_flops += gf;
  }
  // CTA order: longest items first (a one-Q-tile block's tiles count half); within a
  // length, (group, split, head, row block) so CTAs reading the same K/V tiles run
  // side by side.  In a sequential plan a one-Q-tile row block's items cover two
  // consecutive splits (the second's entry is left empty).
  struct Item { PrefixItemDev it; int32_t tiles; bool half; };
  std::vector<Item> items;
  for (int32_t gi = 0; gi < G; ++gi) {
    const PrefixGroupDev& gd = pl->groups[(size_t)gi];
    const int32_t last = mtiles[(size_t)gi] - 1;
    for (int32_t s = 0; s < gd.nsplit; ++s) {
      for (int32_t h = 0; h < Hkv; ++h)
        for (int32_t mt = 0; mt <= last; ++mt) {
          const bool half = single[(size_t)gi] && mt == last;
          const bool pair = half && !pl->split;
          if (pair && s % 2 != 0) continue;
          const int32_t n = pair ? std::min(2, gd.nsplit - s) : 1;
          const int32_t t0 = s * gd.split_tiles;
          const int32_t t1 = std::min(ntiles[(size_t)gi], t0 + n * gd.split_tiles);
          items.push_back({PrefixItemDev{gi, mt, h, s, n, 0}, t1 - t0, half});
        }
    }
  }
  std::stable_sort(items.begin(), items.end(), [](const Item& a, const Item& b2) {
    return (a.half ? a.tiles : 2 * a.tiles) > (b2.half ? b2.tiles : 2 * b2.tiles);
  });
  for (auto& it : items) pl->prefix_items.push_back(it.it);

  // ---- gather work: cascade suffix and dense (flat) ------------------------------
  // Gather CTAs own an SM each; a split plan leaves the gather the SMs its
  // prefix items do not take.
  int64_t max_ctas = (int64_t)num_sms * std::max(1, gather_ctas_per_sm(&c));
  std::vector<int64_t> n_suf((size_t)B), n_dense((size_t)B);
  int64_t suf_tokens = 0, dense_tokens = 0;
  for (int32_t r = 0; r < B; ++r) {
    n_suf[(size_t)r] = pl->reqs[(size_t)r].slen;
    n_dense[(size_t)r] = (int64_t)pl->reqs[(size_t)r].lp + pl->reqs[(size_t)r].slen;
    suf_tokens += n_suf[(size_t)r];
    dense_tokens += n_dense[(size_t)r];
  }
  pl->slot_of_sm.clear();
  if (pl->split) {
    // one slot per SM; a prefix CTA's slot is sized to the time its own item
    // leaves it (a one-Q-tile block's item runs its tiles at about twice the rate).
    // With the pool's SM speeds the slots are planned per SM: the slowest SMs
    // take the prefix items (the longest on the slowest), and every slot's
    // gather follows its SM's speed.
    std::vector<double> v((size_t)num_sms, 1.0);
    if ((int)p->sm_speed.size() == num_sms) {
      std::vector<int32_t> order((size_t)num_sms);
      for (int32_t s = 0; s < num_sms; ++s) order[(size_t)s] = s;
      std::stable_sort(order.begin(), order.end(),
                       [&](int32_t a, int32_t b2) { return p->sm_speed[(size_t)a] < p->sm_speed[(size_t)b2]; });
      pl->slot_of_sm.assign((size_t)num_sms, 0);
      for (int32_t k = 0; k < num_sms; ++k) {
        pl->slot_of_sm[(size_t)order[(size_t)k]] = k;
        v[(size_t)k] = p->sm_speed[(size_t)order[(size_t)k]];
      }
    }
    std::vector<double> it;
    const double crowd = cm.prefix_item_crowd_us * (double)items.size();
    for (const Item& x : items) it.push_back((x.half ? 0.5 : 1.0) * x.tiles * kp.tile_split + kp.item_split + crowd);
    const double gsm = kp.rows == kPrefixRowsPerCta ? cm.gather_sm_gbs * cm.split_gather_ratio_tensor
                                                    : cm.gather_sm_gbs;
    const std::vector<double> w = split_weights(cm, num_sms, it, (double)S, gsm, v, prefix_cta_share > 0.0);
    partition_tokens_weighted(n_suf, w, &pl->suf_seg_begin, &pl->suf_segs);
  } else {
    if (p->gather_partition == GK_PARTITION_PER_REQUEST)
      partition_per_request(n_suf, num_sms, &pl->suf_seg_begin, &pl->suf_segs);
    else
      partition_tokens(n_suf, num_sms, &pl->suf_seg_begin, &pl->suf_segs);
  }
  if (p->gather_partition == GK_PARTITION_PER_REQUEST)
    partition_per_request(n_dense, max_ctas, &pl->dense_seg_begin, &pl->dense_segs);
  else
    partition_tokens(n_dense, max_ctas, &pl->dense_seg_begin, &pl->dense_segs);

  // ---- partial-state entries ----------------------------------------------------
  // cascade: request r owns [entry_cas, entry_cas + n_entry_cas): its prefix
  // splits first, then its suffix segments.
  std::vector<int32_t> nseg_suf((size_t)B, 0), nseg_dense((size_t)B, 0);
  for (auto& sgm : pl->suf_segs) ++nseg_suf[(size_t)sgm.req];
  for (auto& sgm : pl->dense_segs) ++nseg_dense[(size_t)sgm.req];
  int32_t e = 0;
  std::vector<int32_t> prefix_splits((size_t)B, 0);
  for (int32_t gi = 0; gi < G; ++gi)
    for (int32_t r : members[(size_t)gi]) prefix_splits[(size_t)r] = pl->groups[(size_t)gi].nsplit;
  for (int32_t r = 0; r < B; ++r) {
    RequestDev& rq = pl->reqs[(size_t)r];
    rq.entry_cas = e;
    rq.n_entry_cas = prefix_splits[(size_t)r] + nseg_suf[(size_t)r];
    e += rq.n_entry_cas;
  }
  pl->n_entries_cas = e;
  std::vector<int32_t> next((size_t)B);
  for (int32_t r = 0; r < B; ++r) next[(size_t)r] = pl->reqs[(size_t)r].entry_cas + prefix_splits[(size_t)r];
  for (auto& sgm : pl->suf_segs) sgm.entry = next[(size_t)sgm.req]++;
  // dense: a request covered by one segment writes its output directly
  e = 0;
  pl->dense_needs_merge = false;
  for (int32_t r = 0; r < B; ++r) {
    RequestDev& rq = pl->reqs[(size_t)r];
    rq.entry_dense = e;
    if (nseg_dense[(size_t)r] == 1) {
      rq.n_entry_dense = -1;
    } else {
      rq.n_entry_dense = nseg_dense[(size_t)r];
      e += nseg_dense[(size_t)r];
      pl->dense_needs_merge = true;
    }
  }
  pl->n_entries_dense = e;
  for (int32_t r = 0; r < B; ++r) next[(size_t)r] = pl->reqs[(size_t)r].entry_dense;
  for (auto& sgm : pl->dense_segs)
    sgm.entry = pl->reqs[(size_t)sgm.req].n_entry_dense < 0 ? -1 : next[(size_t)sgm.req]++;

  gk_plan_summary& sm = pl->summary;
  sm = gk_plan_summary{};
  sm.num_requests = B;
  sm.num_groups = G;
  sm.max_m_eff = max_m;
  sm.prefix_ctas = (int32_t)pl->prefix_items.size();
  sm.suffix_ctas = (int32_t)pl->suf_seg_begin.size() - 1;
  sm.dense_ctas = (int32_t)pl->dense_seg_begin.size() - 1;
  sm.num_partials = pl->n_entries_cas;
  sm.dense_merge = pl->dense_needs_merge ? 1 : 0;
  sm.prefix_bytes = pre_bytes;
  sm.prefix_flops = pre_flops;
  sm.suffix_bytes = suf_tokens * 2 * Hkv * d * 2;
  sm.dense_bytes = dense_tokens * 2 * Hkv * d * 2;
  sm.cascade_split = pl->split ? 1 : 0;
  sm.prefix_tiles_per_item = 0;
  for (int32_t gi = 0; gi < G; ++gi) sm.prefix_tiles_per_item = std::max(sm.prefix_tiles_per_item, std::min(best_c, ntiles[(size_t)gi]));
  sm.prefix_kernel = pl->prefix_kind ? GK_PREFIX_WARP : GK_PREFIX_TENSOR;
  sm.prefix_rows_per_item = kp.rows;
  sm.prefix_row_groups = pl->prefix_kind && G > 0 ? warp_groups : 0;
  sm.prefix_ctas_gather = pl->split && prefix_cta_share > 0.0 ? 1 : 0;
  sm.sm_slots = pl->slot_of_sm.empty() ? 0 : 1;
  return GK_OK;
}

}  // namespace

// GK_PREFIX_AUTO plans the step with each kind of prefix item and keeps the one
// whose whole cascade (levels and merge) the cost model predicts faster:
// GraniKV Section 3.6's routing between its two prefix kernels, with the
// measured model in place of the M_sat threshold.  The tensor-core items must
// be predicted kTensorAutoEdge faster: on GB300 the model's times for their
// cascade at small steps came out up to a quarter under the measured ones, the
// warp-MMA items' within a fifth.  Steps of at most kWarpOnlyMeff stacked rows
// per head take the warp-MMA items (the pages' M_eff routing between the two).
gk_status build_host_plan(Pool* p, const gk_batch* b, Plan* pl) {
  if (p->prefix_kernel != GK_PREFIX_AUTO) return build_host_plan_kind(p, b, pl, p->prefix_kernel);
  gk_status st = build_host_plan_kind(p, b, pl, GK_PREFIX_TENSOR);
  if (st != GK_OK || pl->summary.num_groups == 0) return st;
  Plan w;   // host fields only: no device buffers are made here
  st = build_host_plan_kind(p, b, &w, GK_PREFIX_WARP);
  if (st != GK_OK) return st;
  const int32_t Hq = p->cfg.num_q_heads;
  double td, t_tensor, t_warp;
  predict_plan(p->cost, p->dev.num_sms, Hq, *pl, &td, &t_tensor);
  predict_plan(p->cost, p->dev.num_sms, Hq, w, &td, &t_warp);
  if (pl->summary.max_m_eff <= kWarpOnlyMeff || !(t_tensor < kTensorAutoEdge * t_warp)) {
    pl->summary = w.summary;
    pl->groups.swap(w.groups);
    pl->group_hot_base.swap(w.group_hot_base);
    pl->prefix_reqs.swap(w.prefix_reqs);
    pl->prefix_items.swap(w.prefix_items);
    pl->reqs.swap(w.reqs);
    pl->suf_seg_begin.swap(w.suf_seg_begin);
    pl->suf_segs.swap(w.suf_segs);
    pl->dense_seg_begin.swap(w.dense_seg_begin);
    pl->dense_segs.swap(w.dense_segs);
    pl->n_entries_cas = w.n_entries_cas;
    pl->n_entries_dense = w.n_entries_dense;
    pl->dense_needs_merge = w.dense_needs_merge;
    pl->group_bytes.swap(w.group_bytes);
    pl->group_flops.swap(w.group_flops);
    pl->split = w.split;
    pl->prefix_kind = w.prefix_kind;
    pl->slot_of_sm.swap(w.slot_of_sm);
  }
  return GK_OK;
}

static gk_status upload_plan(Pool* p, Plan* pl, void* stream) {
  const gk_pool_config& c = p->cfg;
  size_t off = 0;
  pl->off_groups = append_region<PrefixGroupDev>(&off, pl->groups.size());
  pl->off_prefix_reqs = append_region<int32_t>(&off, pl->prefix_reqs.size());
  pl->off_prefix_items = append_region<PrefixItemDev>(&off, pl->prefix_items.size());
  pl->off_reqs = append_region<RequestDev>(&off, pl->reqs.size());
  pl->off_suf_begin = append_region<int32_t>(&off, pl->suf_seg_begin.size());
  pl->off_suf_segs = append_region<SegmentDev>(&off, pl->suf_segs.size());
  pl->off_dense_begin = append_region<int32_t>(&off, pl->dense_seg_begin.size());
  pl->off_dense_segs = append_region<SegmentDev>(&off, pl->dense_segs.size());
  pl->off_slot_of_sm = append_region<int32_t>(&off, pl->slot_of_sm.size());
  std::vector<uint8_t> tmaps;
  int te = encode_prefix_tmaps(&c, pl, &tmaps);
  if (te) return fail(p, GK_ERR_CUDA, "encoding the prefix tensor maps failed");
  pl->off_tmaps = append_region<uint8_t>(&off, tmaps.size(), 128);
  size_t need = std::max<size_t>(off, 256);

  cudaError_t e;
  if (need > pl->d_bytes) {
    if (pl->d_buf) {
      e = cudaStreamSynchronize((cudaStream_t)stream);
      if (e != cudaSuccess) return cuda_fail(p, e, "cudaStreamSynchronize");
      cudaFree(pl->d_buf);
      cudaFreeHost(pl->h_stage);
      pl->d_buf = nullptr;
      pl->h_stage = nullptr;
    }
    size_t cap = need + need / 2;
    e = cudaMalloc(&pl->d_buf, cap);
    if (e != cudaSuccess) return cuda_fail(p, e, "cudaMalloc(plan)");
    e = cudaHostAlloc(&pl->h_stage, cap, cudaHostAllocDefault);
    if (e != cudaSuccess) return cuda_fail(p, e, "cudaHostAlloc(plan staging)");
    pl->d_bytes = cap;
  } else if (pl->staged) {
    // the previous upload must have left the staging buffer before it is rewritten
    e = cudaEventSynchronize(pl->upload_done);
    if (e != cudaSuccess) return cuda_fail(p, e, "cudaEventSynchronize");
  }
  uint8_t* h = (uint8_t*)pl->h_stage;
  auto put = [&](size_t o, const void* src, size_t bytes) { if (bytes) std::memcpy(h + o, src, bytes); };
  put(pl->off_groups, pl->groups.data(), pl->groups.size() * sizeof(PrefixGroupDev));
  put(pl->off_prefix_reqs, pl->prefix_reqs.data(), pl->prefix_reqs.size() * sizeof(int32_t));
  put(pl->off_prefix_items, pl->prefix_items.data(), pl->prefix_items.size() * sizeof(PrefixItemDev));
  put(pl->off_reqs, pl->reqs.data(), pl->reqs.size() * sizeof(RequestDev));
  put(pl->off_suf_begin, pl->suf_seg_begin.data(), pl->suf_seg_begin.size() * sizeof(int32_t));
  put(pl->off_suf_segs, pl->suf_segs.data(), pl->suf_segs.size() * sizeof(SegmentDev));
  put(pl->off_dense_begin, pl->dense_seg_begin.data(), pl->dense_seg_begin.size() * sizeof(int32_t));
  put(pl->off_dense_segs, pl->dense_segs.data(), pl->dense_segs.size() * sizeof(SegmentDev));
  put(pl->off_slot_of_sm, pl->slot_of_sm.data(), pl->slot_of_sm.size() * sizeof(int32_t));
  put(pl->off_tmaps, tmaps.data(), tmaps.size());
  e = cudaMemcpyAsync(pl->d_buf, h, off, cudaMemcpyHostToDevice, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(p, e, "plan upload");
  if (!pl->upload_done) {
    e = cudaEventCreateWithFlags(&pl->upload_done, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(p, e, "cudaEventCreate");
  }
  e = cudaEventRecord(pl->upload_done, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(p, e, "cudaEventRecord");
  pl->staged = true;

  size_t entries = (size_t)std::max(pl->n_entries_cas, pl->n_entries_dense);
  if (entries > pl->part_entries) {
    if (pl->d_part_o) {
      e = cudaStreamSynchronize((cudaStream_t)stream);
      if (e != cudaSuccess) return cuda_fail(p, e, "cudaStreamSynchronize");
      cudaFree(pl->d_part_o);
      cudaFree(pl->d_part_l);
      pl->d_part_o = pl->d_part_l = nullptr;
    }
    size_t cap = entries + entries / 4 + 16;
    e = cudaMalloc(&pl->d_part_o, cap * (size_t)c.num_q_heads * c.head_dim * sizeof(float));
    if (e != cudaSuccess) return cuda_fail(p, e, "cudaMalloc(partial outputs)");
    e = cudaMalloc(&pl->d_part_l, cap * (size_t)c.num_q_heads * sizeof(float));
    if (e != cudaSuccess) return cuda_fail(p, e, "cudaMalloc(partial lse)");
    pl->part_entries = cap;
  }
  pl->uploaded = true;
  return GK_OK;
}

static gk_status plan_for(Pool* p, Plan* pl, const gk_batch* b, void* stream) {
  if (p->has_device) {
    gk_status st = ensure_device(p);
    if (st != GK_OK) return st;
  }
  gk_status st = build_host_plan(p, b, pl);
  if (st != GK_OK) return st;
  if (p->has_device) return upload_plan(p, pl, stream);
  return GK_OK;
}

static void free_plan_buffers(Plan* pl) {
  if (pl->d_buf) cudaFree(pl->d_buf);
  if (pl->h_stage) cudaFreeHost(pl->h_stage);
  if (pl->d_part_o) cudaFree(pl->d_part_o);
  if (pl->d_part_l) cudaFree(pl->d_part_l);
  if (pl->upload_done) cudaEventDestroy(pl->upload_done);
  pl->d_buf = pl->h_stage = nullptr;
  pl->d_part_o = pl->d_part_l = nullptr;
  pl->upload_done = nullptr;
}

// ---- cost model ----------------------------------------------------------------
static bool valid_cost_model(const gk_cost_model& cm) {
  if (!(cm.bw_flat_gbs > 0 && cm.bw_prefix_gbs > 0 && cm.bw_suffix_gbs > 0)) return false;
  if (!(cm.prefix_tile_us > 0 && cm.prefix_tile_split_us > 0 && cm.prefix_item_us >= 0 && cm.gather_sm_gbs > 0))
    return false;
  if (!(cm.warp_tile_us > 0 && cm.warp_group_us >= 0 && cm.warp_item_us >= 0 && cm.warp_split_ratio > 0))
    return false;
  if (!(cm.c_flat_us >= 0 && std::isfinite(cm.c_cascade_us) && cm.c_merge_us >= 0 && cm.c_gather_us >= 0))
    return false;
  if (!(cm.prefix_cta_ramp_us >= 0 && cm.prefix_cta_gather_ratio > 0 && cm.prefix_cta_gather_ratio <= 1 &&
        cm.c_merge_state_us >= 0 && cm.prefix_item_split_us >= 0 && cm.warp_item_split_us >= 0 &&
        cm.prefix_item_crowd_us >= 0 && cm.split_gather_ratio_tensor > 0 && cm.c_gather_split_us >= 0 &&
        cm.split_tensor_us >= 0))
    return false;
  return true;
}

// Minimal JSON reader for the cost-model object (numbers and one array of pairs).
struct JsonReader {
  const char* s;
  bool ok = true;
  void ws() { while (*s && std::isspace((unsigned char)*s)) ++s; }
  bool eat(char ch) { ws(); if (*s == ch) { ++s; return true; } return false; }
  bool str(std::string* out) {
    ws();
    if (*s != '"') return false;
    ++s;
    out->clear();
    while (*s && *s != '"') out->push_back(*s++);
    if (*s != '"') return false;
    ++s;
    return true;
  }
  bool num(double* v) {
    ws();
    char* end = nullptr;
    *v = std::strtod(s, &end);
    if (end == s) return false;
    s = end;
    return true;
  }
  // skip any value (number, string, literal, array, object) of a key we do not use
  bool skip() {
    ws();
    if (*s == '"') {
      std::string t;
      return str(&t);
    }
    if (*s == '[' || *s == '{') {
      const char open = *s, close = (*s == '[') ? ']' : '}';
      ++s;
      ws();
      if (*s == close) { ++s; return true; }
      while (true) {
        if (open == '{') {
          std::string k;
          if (!str(&k) || !eat(':')) return false;
        }
        if (!skip()) return false;
        ws();
        if (*s == ',') { ++s; continue; }
        if (*s == close) { ++s; return true; }
        return false;
      }
    }
    double v;
    if (num(&v)) return true;
    for (const char* lit : {"true", "false", "null"}) {
      size_t n = std::strlen(lit);
      if (std::strncmp(s, lit, n) == 0) { s += n; return true; }
    }
    return false;
  }
};

}  // namespace gk

namespace gk {

void predict_plan(const gk_cost_model& cm, int num_sms, int32_t Hq, const Plan& pl, double* t_dense_us,
                  double* t_cascade_us) {
  const gk_plan_summary& sm = pl.summary;
  *t_dense_us = cm.c_flat_us + (double)sm.dense_bytes / (cm.bw_flat_gbs * 1e3);
  double t_levels = 0.0;
  const bool warp = pl.prefix_kind == 1;
  const double wtile = cm.warp_tile_us + sm.prefix_row_groups * cm.warp_group_us;
  const double tile = warp ? wtile : cm.prefix_tile_us;
  const double tile_split = warp ? wtile * cm.warp_split_ratio : cm.prefix_tile_split_us;
  const double item_fixed = warp ? cm.warp_item_us : cm.prefix_item_us;
  const double item_split = warp ? cm.warp_item_split_us : cm.prefix_item_split_us;
  if (pl.split) {
    const double it =
        sm.prefix_ctas > 0 ? sm.prefix_tiles_per_item * tile_split + item_split + cm.prefix_item_crowd_us * sm.prefix_ctas
                           : 0.0;
    const double gsm = warp ? cm.gather_sm_gbs : cm.gather_sm_gbs * cm.split_gather_ratio_tensor;
    t_levels = split_time(cm, num_sms, sm.prefix_ctas, it, (double)sm.suffix_bytes, (double)sm.prefix_bytes,
                          sm.prefix_ctas_gather != 0, gsm).t;
    if (!warp) t_levels += cm.split_tensor_us;
  } else {
    if (sm.prefix_ctas > 0) {
      const double item = sm.prefix_tiles_per_item * tile + item_fixed;
      const double waves = (double)((sm.prefix_ctas + num_sms - 1) / num_sms);
      t_levels = std::max((double)sm.prefix_bytes / (cm.bw_prefix_gbs * 1e3), waves * item);
    }
    if (sm.suffix_bytes > 0) t_levels += cm.c_gather_us + (double)sm.suffix_bytes / (cm.bw_suffix_gbs * 1e3);
  }
  *t_cascade_us = std::max(0.0, cm.c_cascade_us + t_levels + merge_us(cm, pl.B, Hq, sm.num_partials));
}

}  // namespace gk

using gk::Plan;
using gk::Pool;

extern "C" {

gk_status gk_plan_build(gk_pool* pool, const gk_batch* batch, void* stream, gk_plan** out) {
  if (!pool || !batch || !out) return GK_ERR_INVALID;
  *out = nullptr;
  gk_plan* pl = new (std::nothrow) gk_plan;
  if (!pl) return GK_ERR_INVALID;
  gk_status st = gk::plan_for(&pool->impl, &pl->impl, batch, stream);
  if (st != GK_OK) {
    gk::free_plan_buffers(&pl->impl);
    delete pl;
    return st;
  }
  *out = pl;
  return GK_OK;
}

gk_status gk_plan_update(gk_plan* plan, const gk_batch* batch, void* stream) {
  if (!plan || !batch || !plan->impl.pool) return GK_ERR_INVALID;
  plan->impl.uploaded = false;
  return gk::plan_for(plan->impl.pool, &plan->impl, batch, stream);
}

void gk_plan_destroy(gk_plan* plan) {
  if (!plan) return;
  gk::free_plan_buffers(&plan->impl);
  delete plan;
}

gk_status gk_plan_info(const gk_plan* plan, gk_plan_summary* out) {
  if (!plan || !out) return GK_ERR_INVALID;
  *out = plan->impl.summary;
  return GK_OK;
}

gk_status gk_plan_segments(const gk_plan* plan, int32_t dense, int32_t* n_ctas, int32_t* n_segs, int32_t* begin,
                           int32_t* segs) {
  if (!plan || !n_ctas || !n_segs) return GK_ERR_INVALID;
  const Plan& pl = plan->impl;
  const std::vector<int32_t>& bg = dense ? pl.dense_seg_begin : pl.suf_seg_begin;
  const std::vector<gk::SegmentDev>& sg = dense ? pl.dense_segs : pl.suf_segs;
  *n_ctas = bg.empty() ? 0 : (int32_t)bg.size() - 1;
  *n_segs = (int32_t)sg.size();
  if (begin) std::copy(bg.begin(), bg.end(), begin);
  if (segs)
    for (size_t i = 0; i < sg.size(); ++i) {
      segs[4 * i] = sg[i].req;
      segs[4 * i + 1] = sg[i].t0;
      segs[4 * i + 2] = sg[i].t1;
      segs[4 * i + 3] = sg[i].entry;
    }
  return GK_OK;
}

gk_status gk_dispatch(const gk_pool* pool, const gk_plan* plan, gk_backend* choice, double* t_dense_us,
                      double* t_cascade_us) {
  if (!pool || !plan || !choice) return GK_ERR_INVALID;
  double t_flat, t_cas;
  gk::predict_plan(pool->impl.cost, pool->impl.dev.num_sms, pool->impl.cfg.num_q_heads, plan->impl, &t_flat, &t_cas);
  *choice = t_flat < t_cas ? GK_BACKEND_DENSE : GK_BACKEND_CASCADE;
  if (t_dense_us) *t_dense_us = t_flat;
  if (t_cascade_us) *t_cascade_us = t_cas;
  return GK_OK;
}

gk_status gk_pool_set_cascade_mode(gk_pool* pool, gk_cascade_mode mode, int32_t tiles_per_item) {
  if (!pool) return GK_ERR_INVALID;
  if (mode != GK_CASCADE_AUTO && mode != GK_CASCADE_SEQUENTIAL && mode != GK_CASCADE_SPLIT)
    return gk::fail(&pool->impl, GK_ERR_INVALID, "unknown cascade mode");
  if (tiles_per_item < 0) return gk::fail(&pool->impl, GK_ERR_INVALID, "tiles_per_item < 0");
  pool->impl.cascade_mode = mode;
  pool->impl.cascade_tiles = tiles_per_item;
  return GK_OK;
}

gk_status gk_pool_set_gather_partition(gk_pool* pool, gk_gather_partition partition) {
  if (!pool) return GK_ERR_INVALID;
  if (partition != GK_PARTITION_STREAM && partition != GK_PARTITION_PER_REQUEST)
    return gk::fail(&pool->impl, GK_ERR_INVALID, "unknown gather partition");
  pool->impl.gather_partition = partition;
  return GK_OK;
}

gk_status gk_pool_set_prefix_kernel(gk_pool* pool, gk_prefix_kernel kernel) {
  if (!pool) return GK_ERR_INVALID;
  if (kernel != GK_PREFIX_AUTO && kernel != GK_PREFIX_TENSOR && kernel != GK_PREFIX_WARP)
    return gk::fail(&pool->impl, GK_ERR_INVALID, "unknown prefix kernel");
  pool->impl.prefix_kernel = kernel;
  return GK_OK;
}

gk_status gk_pool_set_sm_speeds(gk_pool* pool, const float* speeds, int32_t n) {
  if (!pool) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  if (n == 0) {
    p->sm_speed.clear();
    return GK_OK;
  }
  if (p->has_device) {
    gk_status st = gk::ensure_device(p);   // the device's SM count
    if (st != GK_OK) return st;
  }
  if (!speeds || n != p->dev.num_sms) return gk::fail(p, GK_ERR_INVALID, "one speed per SM of the device");
  double sum = 0.0;
  for (int32_t s = 0; s < n; ++s) {
    if (!(std::isfinite(speeds[s]) && speeds[s] > 0.0f)) return gk::fail(p, GK_ERR_INVALID, "SM speeds must be positive");
    sum += speeds[s];
  }
  p->sm_speed.assign((size_t)n, 1.0f);
  for (int32_t s = 0; s < n; ++s) p->sm_speed[(size_t)s] = (float)(speeds[s] * n / sum);
  return GK_OK;
}

gk_status gk_pool_get_sm_speeds(const gk_pool* pool, float* speeds, int32_t* n) {
  if (!pool || !n) return GK_ERR_INVALID;
  const Pool* p = &pool->impl;
  *n = (int32_t)p->sm_speed.size();
  if (speeds) std::copy(p->sm_speed.begin(), p->sm_speed.end(), speeds);
  return GK_OK;
}

gk_status gk_cost_model_set(gk_pool* pool, const gk_cost_model* cm) {
  if (!pool || !cm) return GK_ERR_INVALID;
  if (!gk::valid_cost_model(*cm)) return gk::fail(&pool->impl, GK_ERR_INVALID, "invalid cost model");
  pool->impl.cost = *cm;
  return GK_OK;
}

gk_status gk_cost_model_get(const gk_pool* pool, gk_cost_model* cm) {
  if (!pool || !cm) return GK_ERR_INVALID;
  *cm = pool->impl.cost;
  return GK_OK;
}

gk_status gk_cost_model_load(gk_pool* pool, const char* json) {
  if (!pool || !json) return GK_ERR_INVALID;
  gk_cost_model cm = pool->impl.cost;
  gk::JsonReader rd{json};
  auto bad = [&](const char* why) { return gk::fail(&pool->impl, GK_ERR_INVALID, std::string("cost model JSON: ") + why); };
  if (!rd.eat('{')) return bad("expected an object");
  bool first = true;
  while (true) {
    if (rd.eat('}')) break;
    if (!first && !rd.eat(',')) return bad("expected ','");
    first = false;
    std::string key;
    if (!rd.str(&key)) return bad("expected a key");
    if (!rd.eat(':')) return bad("expected ':'");
    static const char* kNumeric[] = {"c_flat_us",      "bw_flat_gbs",    "c_cascade_us",  "bw_prefix_gbs",
                                     "bw_suffix_gbs",  "c_merge_us",     "prefix_tile_us", "prefix_item_us",
                                     "gather_sm_gbs",  "c_gather_us",    "prefix_tile_split_us",
                                     "warp_tile_us",   "warp_group_us",  "warp_item_us",
                                     "warp_split_ratio", "prefix_cta_ramp_us", "prefix_cta_gather_ratio",
                                     "c_merge_state_us", "prefix_item_split_us", "warp_item_split_us",
                                     "prefix_item_crowd_us", "split_gather_ratio_tensor", "c_gather_split_us",
                                     "split_tensor_us"};
    bool known = false;
    for (const char* k : kNumeric) known = known || key == k;
    if (!known) {
      if (!rd.skip()) return bad("malformed value");
      continue;
    }
    double v;
    if (!rd.num(&v)) return bad("values must be numbers");
    if (key == "c_flat_us") cm.c_flat_us = v;
    else if (key == "bw_flat_gbs") cm.bw_flat_gbs = v;
    else if (key == "c_cascade_us") cm.c_cascade_us = v;
    else if (key == "bw_prefix_gbs") cm.bw_prefix_gbs = v;
    else if (key == "bw_suffix_gbs") cm.bw_suffix_gbs = v;
    else if (key == "c_merge_us") cm.c_merge_us = v;
    else if (key == "prefix_tile_us") cm.prefix_tile_us = v;
    else if (key == "prefix_item_us") cm.prefix_item_us = v;
    else if (key == "gather_sm_gbs") cm.gather_sm_gbs = v;
    else if (key == "c_gather_us") cm.c_gather_us = v;
    else if (key == "prefix_tile_split_us") cm.prefix_tile_split_us = v;
    else if (key == "warp_tile_us") cm.warp_tile_us = v;
    else if (key == "warp_group_us") cm.warp_group_us = v;
    else if (key == "warp_item_us") cm.warp_item_us = v;
    else if (key == "warp_split_ratio") cm.warp_split_ratio = v;
    else if (key == "prefix_cta_ramp_us") cm.prefix_cta_ramp_us = v;
    else if (key == "prefix_cta_gather_ratio") cm.prefix_cta_gather_ratio = v;
    else if (key == "c_merge_state_us") cm.c_merge_state_us = v;
    else if (key == "prefix_item_split_us") cm.prefix_item_split_us = v;
    else if (key == "warp_item_split_us") cm.warp_item_split_us = v;
    else if (key == "prefix_item_crowd_us") cm.prefix_item_crowd_us = v;
    else if (key == "split_gather_ratio_tensor") cm.split_gather_ratio_tensor = v;
    else if (key == "c_gather_split_us") cm.c_gather_split_us = v;
    else if (key == "split_tensor_us") cm.split_tensor_us = v;
  }
  return gk_cost_model_set(pool, &cm);
}

static gk_status check_decode(Pool* p, int32_t layer, const gk_batch* b, const Plan* pl) {
  if (layer < 0 || layer >= p->cfg.num_layers) return gk::fail(p, GK_ERR_INVALID, "layer out of range");
  if (pl->pool != p) return gk::fail(p, GK_ERR_INVALID, "plan belongs to another pool");
  if (!pl->uploaded) return gk::fail(p, GK_ERR_INVALID, "plan has no device tables");
  if (b->num_requests != pl->B) return gk::fail(p, GK_ERR_INVALID, "batch size differs from the plan");
  if (pl->B > 0 && (!b->d_q || !b->d_out || !b->d_block_table))
    return gk::fail(p, GK_ERR_INVALID, "batch device pointers missing");
  if ((b->d_new_k == nullptr) != (b->d_new_v == nullptr))
    return gk::fail(p, GK_ERR_INVALID, "fused append needs both d_new_k and d_new_v");
  return gk::ensure_device(p);
}

gk_status gk_cascade_prefix(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch, const gk_plan* plan) {
  if (!pool || !batch || !plan) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  const Plan* pl = &plan->impl;
  gk_status st = check_decode(p, layer, batch, pl);
  if (st != GK_OK) return st;
  if (pl->prefix_items.empty()) return GK_OK;
  gk::LaunchCommon lc{&p->cfg, p->d_error, p->dev.num_sms};
  int e = gk::launch_prefix(lc, stream, layer, batch, pl);
  return e ? gk::cuda_fail(p, e, "cascade prefix kernel") : GK_OK;
}

gk_status gk_cascade_suffix(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch, const gk_plan* plan) {
  if (!pool || !batch || !plan) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  const Plan* pl = &plan->impl;
  gk_status st = check_decode(p, layer, batch, pl);
  if (st != GK_OK) return st;
  if (pl->suf_segs.empty()) return GK_OK;
  gk::LaunchCommon lc{&p->cfg, p->d_error, p->dev.num_sms};
  int e = gk::launch_gather(lc, stream, layer, batch, pl, false);
  return e ? gk::cuda_fail(p, e, "suffix gather kernel") : GK_OK;
}

gk_status gk_cascade_merge(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch, const gk_plan* plan) {
  if (!pool || !batch || !plan) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  const Plan* pl = &plan->impl;
  gk_status st = check_decode(p, layer, batch, pl);
  if (st != GK_OK) return st;
  if (pl->B == 0) return GK_OK;
  gk::LaunchCommon lc{&p->cfg, p->d_error, p->dev.num_sms};
  int e = gk::launch_merge(lc, stream, batch, pl, false);
  return e ? gk::cuda_fail(p, e, "merge kernel") : GK_OK;
}

gk_status gk_cascade_levels(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch, const gk_plan* plan) {
  if (!pool || !batch || !plan) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  const Plan* pl = &plan->impl;
  gk_status st = check_decode(p, layer, batch, pl);
  if (st != GK_OK) return st;
  if (pl->B == 0) return GK_OK;
  if (!pl->split) {
    st = gk_cascade_prefix(pool, stream, layer, batch, plan);
    return st == GK_OK ? gk_cascade_suffix(pool, stream, layer, batch, plan) : st;
  }
  gk::LaunchCommon lc{&p->cfg, p->d_error, p->dev.num_sms};
  if (!pl->slot_of_sm.empty()) {
    // a new tag per launch; when the counter wraps, the claim words are cleared
    if (!p->d_slot_claim) return gk::fail(p, GK_ERR_INVALID, "pool has no slot-claim words");
    if (++p->split_epoch == 0) {
      cudaError_t ce = cudaMemsetAsync(p->d_slot_claim, 0, sizeof(uint32_t) * (size_t)p->dev.num_sms,
                                       (cudaStream_t)stream);
      if (ce != cudaSuccess) return gk::cuda_fail(p, ce, "cudaMemsetAsync(slot claims)");
      ++p->split_epoch;
    }
    lc.slot_claim = p->d_slot_claim;
    lc.epoch = p->split_epoch;
  }
  int e = gk::launch_cascade_split(lc, stream, layer, batch, pl);
  return e ? gk::cuda_fail(p, e, "split cascade kernel") : GK_OK;
}

gk_status gk_decode_cascade(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch, const gk_plan* plan) {
  gk_status st = gk_cascade_levels(pool, stream, layer, batch, plan);
  return st == GK_OK ? gk_cascade_merge(pool, stream, layer, batch, plan) : st;
}

gk_status gk_decode_dense(gk_pool* pool, void* stream, int32_t layer, const gk_batch* batch, const gk_plan* plan) {
  if (!pool || !batch || !plan) return GK_ERR_INVALID;
  Pool* p = &pool->impl;
  const Plan* pl = &plan->impl;
  gk_status st = check_decode(p, layer, batch, pl);
  if (st != GK_OK) return st;
  if (pl->B == 0) return GK_OK;
  gk::LaunchCommon lc{&p->cfg, p->d_error, p->dev.num_sms};
  int e;
  if (!pl->dense_segs.empty() && (e = gk::launch_gather(lc, stream, layer, batch, pl, true)))
    return gk::cuda_fail(p, e, "dense gather kernel");
  if (pl->dense_needs_merge && (e = gk::launch_merge(lc, stream, batch, pl, true)))
    return gk::cuda_fail(p, e, "merge kernel");
  return GK_OK;
}

}  // extern "C"
