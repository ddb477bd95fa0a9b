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

Admission (optional, ``admission=True``; an extension, not the pages' policy).  The pages let
a miss that is not worth caching be served without entering the GPU cache (FreeToken
benchmark, "how FreeToken serves large MoE models": part of the misses is executed from host
memory instead of being copied in).  The GPU reading here decides by expected reuse, with
frequency counts that age (the TinyLFU admission rule):

* every (layer, expert) key has a count f (0 at start, prewarm included).  A call touching S
  (after the capacity check) adds 1 to f of every key in S and |S| to an access total A; if
  then A >= H = 10 * n_slots, every count is halved (integer division) and H is taken off A;
* hits as above; misses in ascending expert id take the lowest free slot while one exists;
  otherwise the miss is compared with the next victim, the eligible slot with the smallest
  (stamp, slot) not yet evicted in this call: f(miss) >= f(victim's key) admits it (evict,
  take the slot, fresh stamp), else it is bypassed: its weights are staged for this call in
  staging entry n_slots + b (b = bypasses before it in this call) and the cache, the stamps
  and tick are unchanged;
* every miss, admitted or bypassed, has a fill record (destination, layer, expert).
"""
from __future__ import annotations

import numpy as np

OK = 0
ERR_CAPACITY = 5
BYPASS = -2     # fill record of a miss that was not admitted


class SlotCacheSim:
    """Slot-level simulator: the state the GPU keeps, field for field."""

    def __init__(self, L: int, E: int, n_slots: int, entry_bytes: int = 0,
                 prewarm: bool = True, admission: bool = False):
        self.L, self.E, self.n_slots, self.entry_bytes = L, E, n_slots, entry_bytes
        self.table = np.full((L, E), -1, dtype=np.int64)      # (layer, expert) -> slot
        self.owner = np.full(n_slots, -1, dtype=np.int64)     # slot -> layer*E + expert
        self.stamp = np.zeros(n_slots, dtype=np.int64)        # 0 = free
        self.tick = 0
        self.hits = self.misses = self.evictions = self.resizes = 0
        self.fills_total = 0
        self.admission = admission
        self.freq = np.zeros(L * E, dtype=np.int64)           # admission counts per key
        self.acc = 0                                          # accesses since the last halving
        self.bypasses = 0
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

        Returns (status, hit_experts, fills) with fills = [(destination, layer, expert,
        evicted_key, or -1 for a free slot, or BYPASS)] in processing order.
        """
        S = sorted(set(int(e) for e in experts))
        if len(S) > self.n_slots:
            return ERR_CAPACITY, [], []
        if self.admission:
            for e in S:
                self.freq[layer * self.E + e] += 1
            self.acc += len(S)
            H = 10 * self.n_slots
            if self.acc >= H:
                self.freq //= 2
                self.acc -= H
        t0 = self.tick
        hit_e = [e for e in S if self.table[layer, e] >= 0]
        miss_e = [e for e in S if self.table[layer, e] < 0]
        for e in hit_e:
            self.tick += 1
            self.stamp[self.table[layer, e]] = self.tick
        fills = []
        n_bypass = 0
        for e in miss_e:
            free = np.nonzero(self.owner < 0)[0]
            evicted = -1
            if free.size:
                s = int(free[0])
            else:
                eligible = np.nonzero(self.stamp <= t0)[0]
                # smallest (stamp, slot): argmin returns the first minimum = lowest slot
                s = int(eligible[np.argmin(self.stamp[eligible])])
                victim_key = int(self.owner[s])
                if self.admission and self.freq[layer * self.E + e] < self.freq[victim_key]:
                    fills.append((self.n_slots + n_bypass, layer, e, BYPASS))
                    n_bypass += 1
                    continue
                evicted = victim_key
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
        self.bypasses += n_bypass
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
    ascending, matching the reading above.  It knows nothing of slots or stamps.  With
    ``admission`` a dictionary of counts follows the admission rule above: a miss that
    finds the list full replaces the front only if its count is at least the front's;
    otherwise it is bypassed and the list does not change.
    """

    def __init__(self, capacity: int, warm=(), admission: bool = False):
        self.capacity = capacity
        self.order = list(warm)[:capacity]
        self.admission = admission
        self.count = {}
        self.since_halving = 0

    def call(self, layer, experts):
        keys = sorted({(layer, int(e)) for e in experts})
        if len(keys) > self.capacity:
            return None
        if self.admission:
            for k in keys:
                self.count[k] = self.count.get(k, 0) + 1
            self.since_halving += len(keys)
            if self.since_halving >= 10 * self.capacity:
                self.since_halving -= 10 * self.capacity
                self.count = {k: c // 2 for k, c in self.count.items()}
        hits = [k for k in keys if k in self.order]
        misses = [k for k in keys if k not in self.order]
        for k in hits:
            self.order.remove(k)
            self.order.append(k)
        evicted, bypassed = [], []
        for k in misses:
            if len(self.order) == self.capacity:
                front = self.order[0]
                if self.admission and self.count.get(k, 0) < self.count.get(front, 0):
                    bypassed.append(k)
                    continue
                evicted.append(self.order.pop(0))
            self.order.append(k)
        if self.admission:
            return hits, misses, evicted, bypassed
        return hits, misses, evicted

    def shrink(self, capacity):
        self.capacity = capacity
        if len(self.order) > capacity:
            self.order = self.order[len(self.order) - capacity:]
