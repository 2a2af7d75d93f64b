"""Prefix cache as a hash chain over blocks (oracle).

Test infrastructure (see ``oracle/__init__``).  Restates, in my own code, the
tutorial page "LLM 推理服务引擎深度拆解", section 4.2 (hash chain: each block's
hash covers the parent block's hash, the block's token ids and an extra
string) and section 4.3 (lookup / insert with least-recently-used eviction,
hit and miss counts):

- key(block i) = first 32 hex digits of sha256(parent + tokens + extra), with
  parent = key of block i-1 or "ROOT", tokens = the ids in decimal joined by
  ",", the three strings hashed one after the other;
- only full blocks are keyed; lookup walks the prompt's keys, counts the
  leading ones found in the table as hit tokens (block_size each) and touches
  them; a lookup with any hit counts as a hit, else as a miss;
- insert gives each key it does not hold the matching block id, evicting the
  least recently used key first when the table is full, and touches every
  key of the chain.

Reading adopted where the page's listing and text disagree: the listing's
lookup stops building the chain at the first miss, so an insert after it
could add one new block per request, while the text describes caching whole
prompts and reports hit rates above 90% after the first turns.  Here lookup
returns the keys of all full blocks (hits still end at the first miss), so
one insert caches the whole prompt.
"""
from __future__ import annotations

import hashlib


def block_key(parent: str | None, tokens, extra: str = "") -> str:
    h = hashlib.sha256()
    h.update((parent if parent is not None else "ROOT").encode())
    h.update(",".join(str(int(t)) for t in tokens).encode())
    h.update(extra.encode())
    return h.hexdigest()[:32]


class PrefixCache:
    def __init__(self, capacity_blocks: int, block_size: int):
        self.capacity = capacity_blocks
        self.block_size = block_size
        self.table: dict[str, int] = {}
        self.recency: list[str] = []      # least recently used first
        self.hits = 0
        self.misses = 0

    def _touch(self, key: str) -> None:
        if key in self.recency:
            self.recency.remove(key)
        self.recency.append(key)

    def lookup(self, token_ids, extra: str = ""):
        """(hit tokens, keys of every full block, block ids of the hits)."""
        S = self.block_size
        keys, hit_blocks = [], []
        parent = None
        prefix = True
        for start in range(0, len(token_ids) - S + 1, S):
            key = block_key(parent, token_ids[start:start + S], extra)
            keys.append(key)
            if prefix and key in self.table:
                hit_blocks.append(self.table[key])
                self._touch(key)
            else:
                prefix = False
            parent = key
        hit = len(hit_blocks) * S
        if hit:
            self.hits += 1
        else:
            self.misses += 1
        return hit, keys, hit_blocks

    def insert(self, keys, block_ids):
        """Returns the block ids of evicted entries."""
        evicted = []
        for key, bid in zip(keys, block_ids):
            if key not in self.table:
                if len(self.table) >= self.capacity:
                    victim = self.recency.pop(0)
                    if victim in self.table:
                        evicted.append(self.table.pop(victim))
                self.table[key] = bid
            self._touch(key)
        return evicted

    @property
    def hit_rate(self) -> float:
        total = self.hits + self.misses
        return self.hits / total if total else 0.0
