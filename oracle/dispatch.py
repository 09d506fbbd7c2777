"""ORACLE (test infrastructure): the per-step backend choice and cascade arrangement.

GraniKV Section 3.6, Eq. 2: M_eff(step) = B_step * n_q/kv, the M dimension of the
stacked shared-prefix contraction.  The pages route on M_eff >= M_sat with an
A100 threshold (M_sat = 1024, Appendix B.4b / Table 16) and state that the
number must be re-fit per GPU while the rule stays.  Here the rule is a
measured cost model evaluated on the step's plan; the backend with the smaller
predicted time runs (flat wins only when strictly faster):

  T_flat    = c_flat + bytes_flat / bw_flat
  T_cascade = c_cascade + T_levels + c_merge * B * Hq
  item(C)   = C * prefix_tile + prefix_item        (one prefix work item of C key tiles, alone)
  item'(C)  = C * prefix_tile_split + prefix_item  (the same beside a gather that keeps HBM busy)
  T_levels  = max(bytes_pre / bw_prefix, W * item(C)) + c_gather
              + bytes_suffix / bw_suffix                          (sequential plan)
            = max(item'(C), (bytes_suffix / gather_sm + n_pre * item'(C)) / SMs,
                  (bytes_suffix + bytes_pre) / bw_suffix)          (split plan)

Work items: a group of M_eff stacked rows and Lp keys contributes ceil(M/256)
row blocks x Hkv heads x ceil(ceil(Lp/128)/C) items, so M_eff enters through the
item count.  A sequential plan runs them in W = ceil(items/SMs) waves over every
SM, with C the smallest value minimising W * item(C); then the gather runs over every SM
as its own launch.  A split plan is one launch with a CTA per SM: CTA b < n_pre
first runs prefix item b, and every CTA gathers a slot of the suffix, a prefix
CTA's slot cut to the time its item leaves (the middle term spreads the
gather's SM-time and the items over all SMs; the last is HBM).  The planner
takes the C with the smallest split prediction (the largest C among equal
ones, i.e. the fewest items), among those with no more items than SMs whose
prefix CTAs keep a gather share of at least MIN_PREFIX_SHARE (share =
max(0, T - item'(C) - c_gather) / T; a forced split with no such C takes the
best prediction), then
lowers C to the smallest value giving as many items (balanced items), and
splits when that beats the sequential T_levels.  A sequential plan's gather
partition cuts the suffix tokens into quotas of ceil(total/n) rounded up to 64
and then to a multiple of 16, so it may use fewer CTAs than SMs; a split
plan's has one slot per SM.

Times are in microseconds, bandwidths in GB/s (1 GB/s = 1e3 bytes per us).

Parity of the choice itself is unpinned by the pages (their threshold is
specific to the A100); Eq. 2 and the formula are pinned by closed forms.
"""
from __future__ import annotations


def m_eff(batch_requests: int, q_per_kv: int) -> int:
    return batch_requests * q_per_kv


def features(prefix_lens, suffix_lens, group_of, Hq, Hkv, d):
    """Plan features of one step.  group_of[r] = HOT prefix group of request r, -1 = none."""
    kv_tok = 2 * Hkv * d * 2
    g = Hq // Hkv
    groups = {}
    for r, grp in enumerate(group_of):
        if grp >= 0:
            groups.setdefault(grp, []).append(r)
    pre = []
    for grp, members in groups.items():
        lp = prefix_lens[members[0]]
        pre.append(dict(M=m_eff(len(members), g), bytes=lp * kv_tok,
                        flops=4 * len(members) * Hq * lp * d, lp=lp))
    return dict(
        bytes_flat=sum(p + s for p, s in zip(prefix_lens, suffix_lens)) * kv_tok,
        bytes_suffix=sum(suffix_lens) * kv_tok,
        prefix=pre, B=len(group_of), Hq=Hq, Hkv=Hkv, suffix_tokens=sum(suffix_lens))


def gather_ctas(tokens, n):
    """CTAs the gather partition of `tokens` over at most n CTAs uses."""
    if tokens == 0:
        return 0
    quota = max(-(-tokens // n), 64)
    quota = -(-quota // 16) * 16
    return -(-tokens // quota)


def _tiles(f):
    return [-(-p["M"] // 256) for p in f["prefix"]], [-(-p["lp"] // 128) for p in f["prefix"]]


def n_items(f, C):
    mtiles, ntiles = _tiles(f)
    return sum(m * f["Hkv"] * -(-n // C) for m, n in zip(mtiles, ntiles))


def sequential_tiles(cm, f, num_sms):
    """Key tiles per item of a sequential plan: the smallest C minimising
    waves * (C * prefix_tile_us + prefix_item_us), an item's time alone."""
    _, ntiles = _tiles(f)
    best, best_c = None, max(ntiles)
    for C in range(1, max(ntiles) + 1):
        cost = -(-n_items(f, C) // num_sms) * item_us(cm, C)
        if best is None or cost < best - 1e-9:
            best, best_c = cost, C
    return best_c


def item_us(cm, C, split=False):
    """A prefix item of C key tiles: alone (sequential plans) or beside the gather (split plans)."""
    return C * cm["prefix_tile_split_us" if split else "prefix_tile_us"] + cm["prefix_item_us"]


def sequential_levels(cm, f, C, num_sms):
    t = cm["c_gather_us"] + f["bytes_suffix"] / (cm["bw_suffix_gbs"] * 1e3)
    if f["prefix"]:
        waves = -(-n_items(f, C) // num_sms)
        t += max(sum(p["bytes"] for p in f["prefix"]) / (cm["bw_prefix_gbs"] * 1e3), waves * item_us(cm, C))
    return t


# a split C qualifies only if its prefix CTAs keep this share of a gather-only CTA's suffix
MIN_PREFIX_SHARE = 0.15


def prefix_share(cm, C, T):
    """Gather share of a prefix CTA (relative to a gather-only CTA) for items of C tiles, launch T."""
    return max(0.0, T - item_us(cm, C, split=True) - cm["c_gather_us"]) / T


def split_levels(cm, f, C, n_pre, num_sms):
    it = item_us(cm, C, split=True)
    bytes_pre = sum(p["bytes"] for p in f["prefix"])
    bal = (f["bytes_suffix"] / (cm["gather_sm_gbs"] * 1e3) + n_pre * it) / num_sms
    return max(it, bal, (f["bytes_suffix"] + bytes_pre) / (cm["bw_suffix_gbs"] * 1e3))


def arrangement(cm, f, num_sms):
    """-> dict(split, C, n_pre, n_gather): the planner's choice for the step."""
    if not f["prefix"]:
        return dict(split=False, C=None, n_pre=0, n_gather=gather_ctas(f["suffix_tokens"], num_sms))
    c_seq = sequential_tiles(cm, f, num_sms)
    seq = dict(split=False, C=c_seq, n_pre=n_items(f, c_seq), n_gather=gather_ctas(f["suffix_tokens"], num_sms))
    if f["suffix_tokens"] == 0:
        return seq
    best, best_c = None, None
    for C in range(max(_tiles(f)[1]), 0, -1):
        items = n_items(f, C)
        if items > num_sms:
            break
        t = split_levels(cm, f, C, items, num_sms)
        if prefix_share(cm, C, t) < MIN_PREFIX_SHARE:
            continue
        if best is None or t < best - 1e-9:
            best, best_c = t, C
    if best is None or not best < sequential_levels(cm, f, c_seq, num_sms):
        return seq
    n_pre = n_items(f, best_c)
    while best_c > 1 and n_items(f, best_c - 1) == n_pre:
        best_c -= 1
    return dict(split=True, C=best_c, n_pre=n_pre, n_gather=num_sms)


def predict(cm, f, num_sms=152):
    t_flat = cm["c_flat_us"] + f["bytes_flat"] / (cm["bw_flat_gbs"] * 1e3)
    a = arrangement(cm, f, num_sms)
    if a["split"]:
        t_levels = split_levels(cm, f, a["C"], a["n_pre"], num_sms)
    else:
        t_levels = sequential_levels(cm, f, a["C"], num_sms)
    t_cas = cm["c_cascade_us"] + t_levels + cm["c_merge_us"] * f["B"] * f["Hq"]
    return t_flat, t_cas


def choose(cm, f, num_sms=152):
    t_flat, t_cas = predict(cm, f, num_sms)
    return ("dense" if t_flat < t_cas else "cascade"), t_flat, t_cas


def aot_splits(budgets, n_cta):
    """Tangram, Algorithm 1 (AOT workload partitioning), for one layer, with requests
    in the place of its head groups and their token counts as the budgets:
    Omega = sum of the budgets; tau = max(1, ceil(Omega / N_CTA)); each group's
    split factor S_i = max(1, ceil(Phi_i / tau)).  A request with no tokens has
    nothing to split and gets no split (the algorithm's max(1, .) would give it an
    empty one).  -> list of split factors (0 for empty requests)."""
    omega = sum(budgets)
    if omega == 0:
        return [0] * len(budgets)
    tau = max(1, -(-omega // n_cta))
    return [max(1, -(-phi // tau)) if phi > 0 else 0 for phi in budgets]


def aot_segments(budgets, n_cta):
    """The segments of each request's tokens under aot_splits: S_r pieces, the first
    n_r mod S_r of them one token longer -> [(request, t0, t1)] in request order."""
    out = []
    for r, (n, s) in enumerate(zip(budgets, aot_splits(budgets, n_cta))):
        t = 0
        for i in range(s):
            ln = n // s + (1 if i < n % s else 0)
            out.append((r, t, t + ln))
            t += ln
    return out
