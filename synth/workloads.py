"""The five synthetic decode workloads (shapes, lengths and seeds), as plain data.

Shapes follow the multi-agent setups of "GraniKV: Asymmetric Granularity
KV-Cache Paging for Multi-Agent Systems with Long Shared Prefix" (Section 4.2,
Table 3; Llama-3.1-8B, Qwen-2.5-14B and Qwen-2.5-32B attention geometry).  The
pages evaluate on ShareGPT-V3 turns; these seeded draws stand in for them.

Lengths are drawn from one splitmix64 stream per workload (stream key
(seed, KIND_LENGTHS)): uniform integers include both ends, log-uniform lengths
are round(exp(U(ln lo, ln hi))).
"""
from __future__ import annotations

from dataclasses import dataclass, field

from .gen import KIND_LENGTHS, SplitMix64, log_uniform_int, stream_key


@dataclass
class Request:
    prefix: int        # index into Workload.prefix_lens; -1 = no HOT prefix
    suffix_len: int    # suffix tokens cached before step 0
    source: int        # suffix stream id (the parent sequence when forked)


@dataclass
class Workload:
    name: str
    seed: int
    L: int
    Hq: int
    Hkv: int
    d: int
    page_size: int
    prefix_lens: list
    requests: list
    steps: int = 0                 # decode steps that append a token before attention
    fork_children: int = 0         # >0: requests are forked from parents at step 0
    parents: list = field(default_factory=list)   # suffix lengths of fork parents
    q_log2_scale: int = 0          # 3 gives the "peaked" variant (Q x 8)
    extra_steps: int = 0           # COLD headroom for bench steps beyond `steps`

    @property
    def B(self) -> int:
        return len(self.requests)

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    def hot_tokens(self) -> int:
        return max(1, sum(self.prefix_lens))

    def cold_slots(self, page_size: int = 0) -> int:
        P = page_size or self.page_size
        total_steps = self.steps + self.extra_steps
        if self.fork_children:
            blocks = sum(-(-s // P) for s in self.parents)
        else:
            blocks = sum(-(-r.suffix_len // P) for r in self.requests)
        blocks += self.B * (-(-total_steps // P) + 2) if total_steps else 0
        blocks = int(blocks * 1.02) + 8
        return blocks * P

    def prefix_len(self, r: int) -> int:
        p = self.requests[r].prefix
        return self.prefix_lens[p] if p >= 0 else 0

    def context_len(self, r: int, appended: int = 0) -> int:
        """Tokens request r attends after `appended` decode-step appends."""
        return self.prefix_len(r) + self.requests[r].suffix_len + appended


def _geometry(name):
    return {
        "llama8b": dict(Hq=32, Hkv=8, d=128),
        "qwen14b": dict(Hq=40, Hkv=8, d=128),
        "qwen32b": dict(Hq=40, Hkv=8, d=128),
    }[name]


def config(n: int, **overrides) -> Workload:
    """Workload n in 1..5; keyword overrides shrink or vary it (tests use them for small cases)."""
    seed = n
    rng = SplitMix64(stream_key(seed, KIND_LENGTHS))
    if n == 1:
        reqs = [Request(0, rng.uniform_int(1, 48), i) for i in range(4)]
        w = Workload("tiny_1L_hq4_hkv2_d64_lp64_b4", seed, 1, 4, 2, 64, 1, [64], reqs)
    elif n == 2:
        B = overrides.pop("B", 64)
        lp = overrides.pop("Lp", 16384)
        lo, hi = overrides.pop("suffix_range", (256, 2048))
        reqs = [Request(0, rng.uniform_int(lo, hi), i) for i in range(B)]
        w = Workload(f"llama8b_32L_lp{lp}_b{B}_s{lo}-{hi}", seed, 32, **_geometry("llama8b"),
                     page_size=1, prefix_lens=[lp], requests=reqs)
    elif n == 3:
        B = overrides.pop("B", 256)
        lp = overrides.pop("Lp", 4096)
        lo, hi = overrides.pop("suffix_range", (64, 1024))
        reqs = [Request(0, rng.uniform_int(lo, hi), i) for i in range(B)]
        w = Workload(f"llama8b_32L_lp{lp}_b{B}_s{lo}-{hi}", seed, 32, **_geometry("llama8b"),
                     page_size=1, prefix_lens=[lp], requests=reqs)
    elif n == 4:
        n_prefix = overrides.pop("n_prefix", 8)
        lp_lo, lp_hi = overrides.pop("lp_range", (2048, 16384))
        bg_lo, bg_hi = overrides.pop("bg_range", (16, 64))
        s_lo, s_hi = overrides.pop("suffix_range", (128, 4096))
        lps = [log_uniform_int(rng, lp_lo, lp_hi) for _ in range(n_prefix)]
        reqs = []
        for p in range(n_prefix):
            for _ in range(rng.uniform_int(bg_lo, bg_hi)):
                reqs.append(Request(p, rng.uniform_int(s_lo, s_hi), 0))
        # interleave the groups in batch order (seeded Fisher-Yates on the request list)
        for i in range(len(reqs) - 1, 0, -1):
            j = (rng.next() * (i + 1)) >> 64
            reqs[i], reqs[j] = reqs[j], reqs[i]
        for i, r in enumerate(reqs):
            r.source = i
        w = Workload(f"qwen14b_48L_{n_prefix}prefix_b{len(reqs)}", seed, 48, **_geometry("qwen14b"),
                     page_size=1, prefix_lens=lps, requests=reqs)
    elif n == 5:
        n_parent = overrides.pop("n_parent", 32)
        children = overrides.pop("children", 4)
        lp = overrides.pop("Lp", 16384)
        s_lo, s_hi = overrides.pop("suffix_range", (512, 2048))
        steps = overrides.pop("steps", 32)
        parents = [rng.uniform_int(s_lo, s_hi) for _ in range(n_parent)]
        reqs = [Request(0, parents[p], p) for p in range(n_parent) for _ in range(children)]
        w = Workload(f"qwen32b_64L_lp{lp}_b{len(reqs)}_fork{children}_steps{steps}", seed, 64,
                     **_geometry("qwen32b"), page_size=16, prefix_lens=[lp], requests=reqs,
                     steps=steps, fork_children=children, parents=parents)
    else:
        raise ValueError(f"no workload {n}")
    for k, v in overrides.items():
        if not hasattr(w, k):
            raise TypeError(f"unknown override {k}")
        setattr(w, k, v)
    return w
