"""ORACLE (test infrastructure): the per-step backend choice.

GraniKV Section 3.6, Eq. 2: M_eff(step) = B_step * n_q/kv, the M dimension of the
stacked shared-prefix contraction.  The pages route on M_eff >= M_sat with an
A100 threshold (M_sat = 1024, Appendix B.4b / Table 16) and state that the
number must be re-fit per GPU while the rule stays.  Here the rule is a
measured cost model evaluated on the step's plan; the backend with the smaller
predicted time runs (flat wins only when strictly faster):

  T_flat    = c_flat + bytes_flat / bw_flat
  T_cascade = c_cascade + sum_g max(bytes_pre_g / bw_prefix, flops_pre_g / TC(M_eff_g))
              + bytes_suffix / bw_suffix + c_merge * B * Hq
  TC(M)     = piecewise-linear through the calibrated (M, TFLOP/s) points,
              proportional to M below the first point, flat above the last.

Times are in microseconds, bandwidths in GB/s (1 GB/s = 1e3 bytes per us),
tensor throughput in TFLOP/s (1e6 flop per us).

Parity of the choice itself is unpinned by the pages (their threshold is
specific to the A100); Eq. 2 and the formula are pinned by closed forms.
"""
from __future__ import annotations


def m_eff(batch_requests: int, q_per_kv: int) -> int:
    return batch_requests * q_per_kv


def tc_at(points, M):
    pts = sorted((float(m), float(t)) for m, t in points)
    if M <= pts[0][0]:
        return pts[0][1] * M / pts[0][0]
    for (m0, t0), (m1, t1) in zip(pts, pts[1:]):
        if M <= m1:
            return t0 + (t1 - t0) * (M - m0) / (m1 - m0)
    return pts[-1][1]


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
                        flops=4 * len(members) * Hq * lp * d))
    return dict(
        bytes_flat=sum(p + s for p, s in zip(prefix_lens, suffix_lens)) * kv_tok,
        bytes_suffix=sum(suffix_lens) * kv_tok,
        prefix=pre, B=len(group_of), Hq=Hq)


def predict(cm, f):
    t_flat = cm["c_flat_us"] + f["bytes_flat"] / (cm["bw_flat_gbs"] * 1e3)
    t_pre = 0.0
    for p in f["prefix"]:
        t_pre += max(p["bytes"] / (cm["bw_prefix_gbs"] * 1e3),
                     p["flops"] / (tc_at(cm["tc_points"], p["M"]) * 1e6))
    t_cas = (cm["c_cascade_us"] + t_pre + f["bytes_suffix"] / (cm["bw_suffix_gbs"] * 1e3)
             + cm["c_merge_us"] * f["B"] * f["Hq"])
    return t_flat, t_cas


def choose(cm, f):
    t_flat, t_cas = predict(cm, f)
    return ("dense" if t_flat < t_cas else "cascade"), t_flat, t_cas
