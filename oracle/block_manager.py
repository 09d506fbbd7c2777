"""ORACLE (test infrastructure): the refcounted copy-on-write block pool.

Restated from "Paged KV cache" (How it works, steps 1-4; Code: BlockPool / Seq):
* a free list used as a stack; a block popped from it gets refcount 1, and a
  block whose refcount drops to zero is pushed back (most recently freed is
  reused first);
* append(seq): the next token goes at offset off = len mod P of the last block.
  When off == 0 a new block is taken.  Otherwise, when the last block is held by
  more than one sequence, the sequence takes a fresh block, drops its reference
  to the shared one and reports the (shared, fresh) pair as a block copy the GPU
  must do before writing (copy-on-write).  The token's slot is
  last_block * P + off.  Running out of blocks returns None and changes nothing;
* fork(seq): the child shares every block (refcount + 1), nothing is copied;
* release(seq): every block loses one reference; the sequence becomes empty.

* prefix caching (step 5): a full block is keyed by a hash of its parent
  block's key and its P token ids; a new request whose leading blocks' keys are
  cached starts with those blocks (each gains a reference) instead of writing
  them again.  The cache itself holds one reference on each cached block, so the
  block survives the requests that used it; when the free list is empty, a
  block is taken by first dropping the cache's reference on the cached block
  that no request holds and that was used longest ago (creating a request from
  the cache and caching a block count as uses).

Initial free order: with seed 0, pops hand out blocks 0, 1, 2, ...  With a
nonzero seed, pops hand out a Fisher-Yates permutation of 0..n-1 driven by
splitmix64 (Steele, Lea & Flood 2014) seeded with the seed: for i = n-1 down to
1, j = floor(next() * (i + 1) / 2^64), swap a[i] and a[j].  The generator is
implemented here from its published definition, independently of the library.
"""
from __future__ import annotations

_M64 = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15


def _splitmix64_stream(seed: int):
    state = seed & _M64
    while True:
        state = (state + _GOLDEN) & _M64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
        yield z ^ (z >> 31)


def initial_order(n: int, seed: int) -> list:
    """Order in which a fresh pool hands out its blocks."""
    order = list(range(n))
    if seed == 0:
        return order
    gen = _splitmix64_stream(seed)
    for i in range(n - 1, 0, -1):
        j = (next(gen) * (i + 1)) >> 64
        order[i], order[j] = order[j], order[i]
    return order


def _mix(z: int) -> int:
    """The output function of splitmix64 applied to z (64-bit)."""
    z &= _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def block_key(parent: int, tokens) -> int:
    """Key of a full block: h = mix(parent + G), then h = mix(h XOR t * G) for each
    token id t (as an unsigned 32-bit value), G = 0x9E3779B97F4A7C15, 64-bit."""
    h = _mix(parent + _GOLDEN)
    for t in tokens:
        h = _mix(h ^ (((t & 0xFFFFFFFF) * _GOLDEN) & _M64))
    return h


def slot_of(table, page_size: int, t: int) -> int:
    """Physical slot of logical token t: table[t // P] * P + t % P."""
    return table[t // page_size] * page_size + t % page_size


class Seq:
    def __init__(self, table=None, length=0):
        self.table = list(table or [])
        self.len = length


class BlockPool:
    def __init__(self, n_blocks: int, page_size: int = 16, seed: int = 0):
        self.n = n_blocks
        self.P = page_size
        order = initial_order(n_blocks, seed)
        self.free = order[::-1]           # stack: the end is popped first
        self.ref = [0] * n_blocks
        self.cache = {}                   # block key -> block
        self.cached = {}                  # block -> [key, last use]
        self.clock = 0

    def num_free(self) -> int:
        return len(self.free)

    def _use(self):
        self.clock += 1
        return self.clock

    def _take(self):
        if not self.free:
            held_by_cache_only = [(u, b) for b, (k, u) in self.cached.items() if self.ref[b] == 1]
            if held_by_cache_only:
                _, b = min(held_by_cache_only)
                key, _ = self.cached.pop(b)
                del self.cache[key]
                self._drop(b)
        if not self.free:
            return None
        b = self.free.pop()
        self.ref[b] = 1
        return b

    def _drop(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    def append(self, s: Seq):
        """Reserve the slot of s's next token -> (slot, cow or None), or None when out of blocks."""
        off = s.len % self.P
        cow = None
        if off == 0:
            b = self._take()
            if b is None:
                return None
            s.table.append(b)
        else:
            shared = s.table[-1]
            if self.ref[shared] > 1:
                fresh = self._take()
                if fresh is None:
                    return None
                self._drop(shared)
                s.table[-1] = fresh
                cow = (shared, fresh)
        slot = s.table[-1] * self.P + off
        s.len += 1
        return slot, cow

    def fork(self, s: Seq) -> Seq:
        for b in s.table:
            self.ref[b] += 1
        return Seq(s.table, s.len)

    def release(self, s: Seq) -> None:
        for b in s.table:
            self._drop(b)
        s.table = []
        s.len = 0

    def create_cached(self, tokens):
        """A new request over the longest cached chain of tokens' leading full blocks -> (Seq, tokens reused)."""
        s = Seq()
        key = 0
        for i in range(len(tokens) // self.P):
            key = block_key(key, tokens[i * self.P:(i + 1) * self.P])
            if key not in self.cache:
                break
            b = self.cache[key]
            self.ref[b] += 1
            self.cached[b][1] = self._use()
            s.table.append(b)
        s.len = len(s.table) * self.P
        return s, s.len

    def cache_blocks(self, s: Seq, tokens) -> int:
        """Cache s's full blocks covering tokens (up to s.len); keys already cached and
        blocks cached under another key are left alone -> blocks added."""
        added = 0
        key = 0
        for i in range(min(len(tokens), s.len) // self.P):
            key = block_key(key, tokens[i * self.P:(i + 1) * self.P])
            b = s.table[i]
            if key in self.cache or b in self.cached:
                continue
            self.cache[key] = b
            self.cached[b] = [key, self._use()]
            self.ref[b] += 1
            added += 1
        return added

    def cache_stats(self):
        return len(self.cached), sum(1 for b in self.cached if self.ref[b] == 1)
