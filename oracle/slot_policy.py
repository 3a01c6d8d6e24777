"""Slot-pool policy oracle: LFU + recency eviction (TEST INFRASTRUCTURE ONLY).

The Swiftlet pages (Swiftlet README "How it works" and "Relation to TurboFieldfare")
cache hot routed experts in a bounded pool of slots and evict by "LFU plus
recency"; they do not spell the rule out.  The reading written here:

  * the pool of a layer has n_slots slots; a table maps expert id -> slot
    (-1 = not resident);
  * one lookup is one (layer, step): a global clock advances by one per
    lookup; the experts needed by that lookup are served in the order given;
  * a resident needed expert is a hit: freq += 1, last_use = clock;
  * a missing expert takes the lowest-numbered empty slot if one exists,
    otherwise evicts, among resident experts NOT needed by this lookup, the one
    with the smallest freq, then the oldest last_use, then the lowest slot id;
    the filled slot starts at freq = 1, last_use = clock;
  * a lookup whose distinct needed experts exceed n_slots cannot be served.

Two more victim rules, for policy studies (the pages name only the first):
  * "lru": the smallest last_use, then the lowest slot id;
  * "lfu": the smallest freq, then the lowest slot id.
Use counts and last_use are kept the same way under every rule.

Plain Python, one slot at a time; independent of the C++ policy in the
library.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple


class PoolExhausted(RuntimeError):
    pass


# victim order of each rule: the candidate slot with the smallest key is evicted
_KEYS = {
    "lfu_recency": lambda fr, la, j: (fr[j], la[j], j),
    "lru": lambda fr, la, j: (la[j], j),
    "lfu": lambda fr, la, j: (fr[j], j),
}


class SlotPolicy:
    def __init__(self, n_layers: int, n_experts: int, n_slots: int, rule: str = "lfu_recency"):
        if rule not in _KEYS:
            raise ValueError(f"unknown rule {rule!r}")
        self.key = _KEYS[rule]
        self.n_layers, self.n_experts, self.n_slots = n_layers, n_experts, n_slots
        self.table = [[-1] * n_experts for _ in range(n_layers)]
        self.owner = [[-1] * n_slots for _ in range(n_layers)]
        self.freq = [[0] * n_slots for _ in range(n_layers)]
        self.last = [[0] * n_slots for _ in range(n_layers)]
        self.clock = 0
        self.hits = self.misses = self.evictions = 0

    def lookup(self, layer: int, needed: Sequence[int]) -> Tuple[List[int], List[Tuple[int, int]]]:
        """Serve one lookup.  Returns (slot of each needed expert, [(expert,
        slot) filled by this lookup]).  Repeated ids in `needed` are served once."""
        uniq = []
        for e in needed:
            if e not in uniq:
                uniq.append(int(e))
        if len(uniq) > self.n_slots:
            raise PoolExhausted(f"{len(uniq)} experts needed, {self.n_slots} slots")
        self.clock += 1
        tab, own, fr, la = self.table[layer], self.owner[layer], self.freq[layer], self.last[layer]
        missing = []
        for e in uniq:
            s = tab[e]
            if s >= 0:
                fr[s] += 1
                la[s] = self.clock
                self.hits += 1
            else:
                missing.append(e)
        fills = []
        for e in missing:
            empty = [s for s in range(self.n_slots) if own[s] < 0]
            if empty:
                s = empty[0]
            else:
                cands = [s for s in range(self.n_slots) if own[s] not in uniq]
                s = min(cands, key=lambda j: self.key(fr, la, j))
                tab[own[s]] = -1
                self.evictions += 1
            own[s] = e
            tab[e] = s
            fr[s] = 1
            la[s] = self.clock
            self.misses += 1
            fills.append((e, s))
        return [tab[e] for e in needed], fills
