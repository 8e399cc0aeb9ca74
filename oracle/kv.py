"""Orca-style K/V reservation pool (oracle).

[0h-n0] "スケジューラのアルゴリズム" (scheduler algorithm): when a request is
admitted, K/V space for its maximum length is reserved up front so that it can
never run out of memory mid-generation, and the space is returned when the
request finishes ([houmin] 3.1.1 "算法": K/V is released as soon as the
request's generation ends).  [0h-n0] "実装のポイント" (implementation notes):
the pool is allocated once at start-up, never with per-request device
allocations.

The pages do not say how a reservation is placed inside the pool.  The reading
taken: a token-granular pool of ``kv_slots`` tokens; a reservation is one
contiguous range placed first-fit at the lowest free address; a free merges
with its free neighbours.  This makes every offset deterministic.
"""

from __future__ import annotations


class KVPool:
    def __init__(self, kv_slots: int):
        if kv_slots <= 0:
            raise ValueError("kv_slots must be positive")
        self.kv_slots = int(kv_slots)
        self.free_list = [(0, self.kv_slots)]  # (offset, length), sorted by offset, never adjacent
        self.owned = {}  # rid -> (offset, length)

    def alloc(self, rid: int, n_tokens: int):
        """Reserve ``n_tokens`` contiguous slots for ``rid``; offset or None if full."""
        if n_tokens <= 0 or rid in self.owned:
            raise ValueError("bad reservation")
        for i, (off, length) in enumerate(self.free_list):
            if length >= n_tokens:
                if length == n_tokens:
                    del self.free_list[i]
                else:
                    self.free_list[i] = (off + n_tokens, length - n_tokens)
                self.owned[rid] = (off, n_tokens)
                return off
        return None

    def free(self, rid: int) -> None:
        off, length = self.owned.pop(rid)
        # insert, keeping the list sorted, then merge with the neighbours
        pos = 0
        while pos < len(self.free_list) and self.free_list[pos][0] < off:
            pos += 1
        self.free_list.insert(pos, (off, length))
        if pos + 1 < len(self.free_list):
            o, l = self.free_list[pos]
            o2, l2 = self.free_list[pos + 1]
            if o + l == o2:
                self.free_list[pos] = (o, l + l2)
                del self.free_list[pos + 1]
        if pos > 0:
            o0, l0 = self.free_list[pos - 1]
            o, l = self.free_list[pos]
            if o0 + l0 == o:
                self.free_list[pos - 1] = (o0, l0 + l)
                del self.free_list[pos]

    def used(self) -> int:
        return sum(l for _, l in self.owned.values())

    def reservation(self, rid: int):
        return self.owned.get(rid)
