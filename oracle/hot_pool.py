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


class HotPrefixCache:
    """GraniKV Section 3.2's life cycle of a HOT slab: each shared prefix (named by
    a caller key) holds one slab and a count of the requests using it; at zero the
    slab is evictable but still cached, so a later request for the same prefix
    finds its K/V in place.  An allocation that does not fit evicts evictable
    slabs, the one unused for longest first, returning each range to the free
    list (where it merges with its neighbours), until it fits.

    Uses are numbered: every acquire and every release of a reference is a use,
    and "unused for longest" is the evictable slab with the smallest number."""

    def __init__(self, pool: HotPool):
        self.pool = pool
        self.slabs = {}       # key -> dict(base, lp, refs, used)
        self.clock = 0

    def _use(self):
        self.clock += 1
        return self.clock

    def acquire(self, key: int, lp: int):
        """-> (base, hit)."""
        slab = self.slabs.get(key)
        if slab is not None:
            if slab["lp"] != lp:
                raise ValueError("key cached with another length")
            slab["refs"] += 1
            slab["used"] = self._use()
            return slab["base"], True
        while True:
            try:
                base = self.pool.alloc(lp)
                break
            except HotFull:
                idle = [(s["used"], k) for k, s in self.slabs.items() if s["refs"] == 0]
                if not idle:
                    raise
                _, victim = min(idle)
                self.pool.release(self.slabs.pop(victim)["base"])
        self.slabs[key] = dict(base=base, lp=lp, refs=1, used=self._use())
        return base, False

    def unref(self, key: int) -> None:
        slab = self.slabs[key]
        if slab["refs"] == 0:
            raise ValueError("no reference held")
        slab["refs"] -= 1
        slab["used"] = self._use()

    def stats(self):
        idle = [s for s in self.slabs.values() if s["refs"] == 0]
        return len(self.slabs), len(idle), sum(s["lp"] for s in idle)
