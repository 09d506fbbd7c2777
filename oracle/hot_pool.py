"""ORACLE (test infrastructure): GraniKV's HOT pool allocator.

GraniKV Section 3.2: a contiguous allocator over a reserved region, one range of
Lp token slots per shared prefix; a released range returns to a free list and
merges with adjacent free ranges, and later allocations reuse freed ranges.
Appendix B.8b packs prefixes first-fit.  Reading taken where the two differ:
first fit over the address-ordered, coalesced free list, else advance the bump
pointer; a free range that ends at the bump pointer lowers it instead.
Units are tokens: a prefix at base b owns tokens [b, b + Lp).
"""
from __future__ import annotations


class HotFull(Exception):
    pass


class HotPool:
    def __init__(self, capacity: int):
        self.capacity = capacity
        self.top = 0
        self.free = []          # address-ordered list of [start, end)
        self.live = {}          # base -> length

    def alloc(self, n: int) -> int:
        if n <= 0:
            raise ValueError("prefix length must be positive")
        for i, (a, b) in enumerate(self.free):
            if b - a >= n:
                if b - a == n:
                    del self.free[i]
                else:
                    self.free[i] = (a + n, b)
                self.live[a] = n
                return a
        if self.top + n > self.capacity:
            raise HotFull(n)
        base = self.top
        self.top += n
        self.live[base] = n
        return base

    def release(self, base: int) -> None:
        n = self.live.pop(base)
        a, b = base, base + n
        merged = []
        for (x, y) in self.free:
            if y == a:
                a = x
            elif x == b:
                b = y
            else:
                merged.append((x, y))
        if b == self.top:
            self.top = a
        else:
            merged.append((a, b))
        self.free = sorted(merged)

    def free_tokens(self) -> int:
        return self.capacity - sum(self.live.values())
