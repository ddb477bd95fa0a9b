"""Oracle of the shared LRU expert-slot cache (TEST INFRASTRUCTURE ONLY).

The pages fix the policy's shape: the GPU cache holds complete (layer, expert) entries
identified by one logical mapping, recency is shared across layers and tokens, and the
cache follows routing instead of being fixed at load time (FreeToken RTX 4090, section
"how the MoE memory hierarchy works"; FreeToken benchmark, section "how FreeToken serves
large MoE models"); its capacity can be rebuilt at scheduler safe points without
reloading the host pool (FreeToken vram, elastic-cache paragraph; FreeToken benchmark,
"elastic cache").  They leave the granularity, order and tie rules open; the readings
implemented here:

* One forward call of layer l touches S = the distinct experts routed in that call.
* A global counter ``tick`` starts at 0; every stamp is ``++tick``; a free slot has stamp 0.
* Within a call: first the hits, in ascending expert id, get fresh stamps; then the
  misses, in ascending expert id, each take the lowest-numbered free slot, or else evict
  the slot with the smallest (stamp, slot id) among slots whose stamp is <= the tick at
  the start of the call (so nothing touched in this call is evicted), and get a fresh
  stamp and a fill record (slot, layer, expert).
* |S| > n_slots: the call fails (capacity) and changes nothing.
* Prewarm at pool load: entries (l, e) in lexicographic order take slots
  0 .. min(n_slots, L*E) - 1 with stamps 1 .. n; tick = n.
* Resize to n_new: the min(n_new, occupied) entries with the largest stamps survive, moved
  to slots 0 .. m-1 in descending stamp order, keeping their stamps; tick is unchanged.
"""
from __future__ import annotations

import numpy as np

OK = 0
ERR_CAPACITY = 5


class SlotCacheSim:
    """Slot-level simulator: the state the GPU keeps, field for field."""

    def __init__(self, L: int, E: int, n_slots: int, entry_bytes: int = 0,
                 prewarm: bool = True):
        self.L, self.E, self.n_slots, self.entry_bytes = L, E, n_slots, entry_bytes
        self.table = np.full((L, E), -1, dtype=np.int64)      # (layer, expert) -> slot
        self.owner = np.full(n_slots, -1, dtype=np.int64)     # slot -> layer*E + expert
        self.stamp = np.zeros(n_slots, dtype=np.int64)        # 0 = free
        self.tick = 0
        self.hits = self.misses = self.evictions = self.resizes = 0
        self.fills_total = 0
        if prewarm:
            n = min(n_slots, L * E)
            for key in range(n):
                self.table[key // E, key % E] = key
                self.owner[key] = key
                self.stamp[key] = key + 1
            self.tick = n

    # -- one forward call ---------------------------------------------------------
    def access(self, layer: int, experts):
        """Touch the distinct ``experts`` of one call of ``layer``.

        Returns (status, hit_experts, fills) with fills = [(slot, layer, expert,
        evicted_key or -1)] in processing order.
        """
        S = sorted(set(int(e) for e in experts))
        if len(S) > self.n_slots:
            return ERR_CAPACITY, [], []
        t0 = self.tick
        hit_e = [e for e in S if self.table[layer, e] >= 0]
        miss_e = [e for e in S if self.table[layer, e] < 0]
        for e in hit_e:
            self.tick += 1
            self.stamp[self.table[layer, e]] = self.tick
        fills = []
        for e in miss_e:
            free = np.nonzero(self.owner < 0)[0]
            evicted = -1
            if free.size:
                s = int(free[0])
            else:
                eligible = np.nonzero(self.stamp <= t0)[0]
                # smallest (stamp, slot): argmin returns the first minimum = lowest slot
                s = int(eligible[np.argmin(self.stamp[eligible])])
                evicted = int(self.owner[s])
                self.table[evicted // self.E, evicted % self.E] = -1
                self.evictions += 1
            self.table[layer, e] = s
            self.owner[s] = layer * self.E + e
            self.tick += 1
            self.stamp[s] = self.tick
            fills.append((s, layer, e, evicted))
        self.hits += len(hit_e)
        self.misses += len(miss_e)
        self.fills_total += len(miss_e)
        return OK, hit_e, fills

    # -- elastic resize at a safe point -------------------------------------------
    def resize(self, n_new: int):
        """Rebuild the cache with ``n_new`` slots; survivors keep their stamps.

        Returns the list of (old slot, new slot) moves."""
        occ = np.nonzero(self.owner >= 0)[0]
        order = occ[np.argsort(-self.stamp[occ], kind="stable")]
        keep = order[:min(n_new, occ.size)]
        owner = np.full(n_new, -1, dtype=np.int64)
        stamp = np.zeros(n_new, dtype=np.int64)
        self.table[:, :] = -1
        moves = []
        for new, old in enumerate(keep):
            owner[new] = self.owner[old]
            stamp[new] = self.stamp[old]
            key = int(owner[new])
            self.table[key // self.E, key % self.E] = new
            moves.append((int(old), new))
        self.owner, self.stamp, self.n_slots = owner, stamp, n_new
        self.resizes += 1
        return moves

    def resident_keys(self):
        """Resident keys ordered least recently used first."""
        occ = np.nonzero(self.owner >= 0)[0]
        return [int(self.owner[s]) for s in occ[np.argsort(self.stamp[occ], kind="stable")]]


class BruteForceLRU:
    """An ordered list with move-to-back, written independently of ``SlotCacheSim``.

    Keys are (layer, expert) tuples; the front of the list is the least recently used.
    Within one call the accesses happen in the order: hits ascending, then misses
    ascending, matching the reading above.  It knows nothing of slots or stamps.
    """

    def __init__(self, capacity: int, warm=()):
        self.capacity = capacity
        self.order = list(warm)[:capacity]

    def call(self, layer, experts):
        keys = sorted({(layer, int(e)) for e in experts})
        if len(keys) > self.capacity:
            return None
        hits = [k for k in keys if k in self.order]
        misses = [k for k in keys if k not in self.order]
        for k in hits:
            self.order.remove(k)
            self.order.append(k)
        evicted = []
        for k in misses:
            if len(self.order) == self.capacity:
                evicted.append(self.order.pop(0))
            self.order.append(k)
        return hits, misses, evicted

    def shrink(self, capacity):
        self.capacity = capacity
        if len(self.order) > capacity:
            self.order = self.order[len(self.order) - capacity:]
