"""ORACLE (test infrastructure): the dispatcher's cost formula and work decomposition.

GraniKV Section 3.6, Eq. 2: M_eff(step) = B_step * n_q/kv, the M dimension of the
stacked shared-prefix contraction.  The pages route on M_eff >= M_sat with an
A100 threshold (M_sat = 1024, Appendix B.4b / Table 16) and state that the
number must be re-fit per GPU while the rule stays.  Here the rule is a
measured cost model evaluated on the step's plan; the backend with the smaller
predicted time runs (flat wins only when strictly faster):

  T_flat    = c_flat + bytes_flat / bw_flat
  T_cascade = max(0, c_cascade + T_levels + c_merge * B * Hq + c_merge_state * partials / B)
  item(C)   = C * tile + item_fixed          (one prefix work item of C key tiles, alone)
  item'(C)  = C * tile_split + item_split + crowd * n_pre
                                             (the same inside a split launch, beside a gather
                                              that keeps HBM busy, among n_pre items whose first
                                              loads contend)
  T_levels  = max(bytes_pre / bw_prefix, W * item(C)) + c_gather
              + bytes_suffix / bw_suffix                          (sequential plan, W waves)
            = max(item'(C), T_gather, (bytes_suffix + bytes_pre) / bw_suffix)
              + split_tensor (a split launch of tensor-core items)        (split plan)
  T_gather  = (G + A * c_gs + n * e * (item'(C) + r)) / (A + n * e)   (prefix CTAs gather too)
            = c_gs + G / A                                        (only the other CTAs gather)
              and at least c_gs + bytes_suffix / bw_suffix        (the gather held to HBM)
with n = n_pre prefix CTAs, A = SMs - n gather-only CTAs, G = bytes_suffix /
gather_sm the gather's SM-time (gather_sm times split_gather_ratio_tensor in a
split launch of tensor-core items), r = prefix_cta_ramp_us and e =
prefix_cta_gather_ratio: gather-only CTAs start after c_gs = c_gather_split_us (the
split launch's own fixed cost; c_gather_us is the stand-alone gather launch's), a
prefix CTA r after its item and at e of their rate, and all end together.  A step without
suffix tokens has no gather term (and no c_gather in the sequential plan).

with (tile, tile_split, item_fixed, item_split) the terms of the plan's prefix
kernel: tensor-core items (prefix_tile_us, prefix_tile_split_us, prefix_item_us,
prefix_item_split_us; 256 stacked rows per item) or warp-MMA items (tile =
warp_tile_us + R * warp_group_us, tile_split = warp_split_ratio * tile,
warp_item_us, warp_item_split_us; 128 rows per item), the two prefix kernels
Section 3.5 pairs, and crowd = prefix_item_crowd_us.  R = the 16-row groups of the
fullest warp item, rounded up to 1, 2, 4 or 8.

Work decomposition (fixed by the kernels' tiling, not a heuristic): a group of
M_eff stacked rows and Lp keys contributes ceil(M_eff / rows) row blocks x Hkv
heads x ceil(ceil(Lp / 128) / C) key splits.  Each (row block, head, split) is
one item, except that in a sequential plan a tensor-core row block holding at
most one 128-row Q tile (M_eff mod 256 in 1..128, the group's last block) runs
its tiles at about twice the rate and so takes two consecutive splits per item:
ceil(splits / 2) items.  (A split plan gives such a block one split per item and
its CTA a longer share of the gather instead.)

Parity unpinned: which arrangement a plan takes (split or sequential, the key
tiles per item C, the prefix kernel, whether its prefix CTAs also gather) is
the planner's search over this model,
and the pages fix none of it (their threshold is specific to the A100).  This
oracle does not restate that search; it evaluates the formula above for the
arrangement a plan reports, and the choice itself is held to measurement on
the GPU (the dispatcher's pick against the faster backend's measured time, and
each prediction against the measured layer time).

Times are in microseconds, bandwidths in GB/s (1 GB/s = 1e3 bytes per us).
"""
from __future__ import annotations

ROWS = {"tensor": 256, "warp": 128}
KEY_TILE = 128
Q_TILE = 128        # rows of one tensor-core Q tile (two per tensor-core row block)


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


def _ceil(a, b):
    return -(-a // b)


def n_items(f, C, kind="tensor", paired=True):
    """Prefix work items of a plan with C key tiles per split: every (row block, KV head,
    key split) of every group once; with `paired` (sequential plans) a one-Q-tile
    tensor-core block's splits two at a time."""
    rows = ROWS[kind]
    total = 0
    for p in f["prefix"]:
        blocks = _ceil(p["M"], rows)
        splits = _ceil(_ceil(p["lp"], KEY_TILE), C)
        one = 1 if paired and kind == "tensor" and 0 < p["M"] % rows <= Q_TILE else 0
        total += (blocks - one) * f["Hkv"] * splits + one * f["Hkv"] * _ceil(splits, 2)
    return total


def gather_ctas(tokens, n):
    """CTAs the stream partition of `tokens` over at most n CTAs uses: quotas of
    ceil(tokens / n), at least 64 tokens, rounded up to a multiple of 16."""
    if tokens == 0:
        return 0
    quota = max(_ceil(tokens, n), 64)
    quota = _ceil(quota, 16) * 16
    return _ceil(tokens, quota)


def warp_row_groups(f):
    """R of a step: 16-row groups of its fullest warp item (min(M_eff, 128) rows of the
    largest group), rounded up to a power of two; 0 without prefix work."""
    rows = max([min(p["M"], ROWS["warp"]) for p in f["prefix"]], default=0)
    if rows == 0:
        return 0
    r = 1
    while r < _ceil(rows, 16):
        r *= 2
    return r


def _terms(cm, kind, R=0):
    if kind == "warp":
        tile = cm["warp_tile_us"] + R * cm["warp_group_us"]
        return tile, tile * cm["warp_split_ratio"], cm["warp_item_us"], cm["warp_item_split_us"]
    return cm["prefix_tile_us"], cm["prefix_tile_split_us"], cm["prefix_item_us"], cm["prefix_item_split_us"]


def item_us(cm, C, split=False, kind="tensor", R=0):
    """A prefix item of C key tiles: alone (sequential plans) or inside a split launch."""
    tile, tile_split, fixed, fixed_split = _terms(cm, kind, R)
    return C * tile_split + fixed_split if split else C * tile + fixed


def sequential_levels(cm, f, C, n_pre, num_sms, kind="tensor", R=0):
    t = cm["c_gather_us"] + f["bytes_suffix"] / (cm["bw_suffix_gbs"] * 1e3) if f["bytes_suffix"] else 0.0
    if f["prefix"] and n_pre:
        waves = -(-n_pre // num_sms)
        t += max(sum(p["bytes"] for p in f["prefix"]) / (cm["bw_prefix_gbs"] * 1e3),
                 waves * item_us(cm, C, kind=kind, R=R))
    return t


def split_levels(cm, f, C, n_pre, num_sms, kind="tensor", R=0, gather=True):
    it = item_us(cm, C, split=True, kind=kind, R=R) + cm["prefix_item_crowd_us"] * n_pre if n_pre else 0.0
    bytes_pre = sum(p["bytes"] for p in f["prefix"])
    t = max(it, (f["bytes_suffix"] + bytes_pre) / (cm["bw_suffix_gbs"] * 1e3))
    if f["bytes_suffix"] == 0:
        return t
    rate = cm["gather_sm_gbs"] * (cm["split_gather_ratio_tensor"] if kind == "tensor" else 1.0)
    G = f["bytes_suffix"] / (rate * 1e3)
    A = num_sms - n_pre
    e, r, cg = cm["prefix_cta_gather_ratio"], cm["prefix_cta_ramp_us"], cm["c_gather_split_us"]
    if gather and n_pre:
        t_gather = (G + A * cg + n_pre * e * (it + r)) / (A + n_pre * e)
    else:
        t_gather = cg + G / A
    t = max(t, t_gather, cg + f["bytes_suffix"] / (cm["bw_suffix_gbs"] * 1e3))
    return t + (cm["split_tensor_us"] if kind == "tensor" else 0.0)


def predict(cm, f, plan, num_sms=152):
    """(T_flat, T_cascade) for the arrangement a plan reports: plan = dict(split, C, n_pre,
    kind, gather, partials); a warp plan's R comes from the step (warp_row_groups)."""
    t_flat = cm["c_flat_us"] + f["bytes_flat"] / (cm["bw_flat_gbs"] * 1e3)
    R = warp_row_groups(f) if plan["kind"] == "warp" else 0
    if plan["split"]:
        t_levels = split_levels(cm, f, plan["C"], plan["n_pre"], num_sms, plan["kind"], R, plan["gather"])
    else:
        t_levels = sequential_levels(cm, f, plan["C"], plan["n_pre"], num_sms, plan["kind"], R)
    merge = cm["c_merge_us"] * f["B"] * f["Hq"]
    if f["B"]:
        merge += cm["c_merge_state_us"] * plan["partials"] / f["B"]
    t_cas = max(0.0, cm["c_cascade_us"] + t_levels + merge)
    return t_flat, t_cas


def choose(t_flat, t_cas):
    """The backend the rule picks from the two predictions (flat only when strictly faster)."""
    return "dense" if t_flat < t_cas else "cascade"


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
