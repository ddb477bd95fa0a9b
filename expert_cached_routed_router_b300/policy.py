"""Placement policies replayed on a routing trace, for comparison with the device LRU.

FreeToken RTX 4090, "benchmarks, comparison & trade-offs" (engine/strategy table) contrasts
FreeToken's shared routing-aware LRU with a fixed layer-centric placement (llama.cpp hybrid
mode) and a hot placement refreshed by prefill (KTransformers); FreeToken benchmark, "benchmark
results", reports lower decode miss rates for the LRU than for static or prefill-based placement
at the same cache capacity.  These host-side simulators replay the same sequence of touched
(layer, expert) sets that the CUDA path routed, at the same capacity, so the three policies can be
compared on one trace:

* ``StaticLayerSplit``: the first ``capacity`` entries in (layer, expert) order are resident for
  good (whole layers on the GPU, the rest elsewhere).
* ``RefreshedHotSet``: every ``refresh`` steps the ``capacity`` entries touched most often in the
  previous window become the resident set (ties: lower (layer, expert) first); the first window
  uses the static split.

The LRU's own counts come from the library (``ft_cache_stats``), which the parity tests check
against the oracle simulator.  Every access outside the resident set counts as a miss.
"""
from __future__ import annotations

import numpy as np


class StaticLayerSplit:
    def __init__(self, L: int, E: int, capacity: int):
        self.resident = np.zeros((L, E), dtype=bool)
        self.resident.reshape(-1)[:min(capacity, L * E)] = True
        self.hits = self.misses = 0

    def step_begin(self, step: int):
        pass

    def access(self, layer: int, experts):
        s = np.unique(np.asarray(experts, dtype=np.int64))
        h = int(self.resident[layer, s].sum())
        self.hits += h
        self.misses += len(s) - h


class RefreshedHotSet:
    def __init__(self, L: int, E: int, capacity: int, refresh: int):
        self.L, self.E, self.capacity, self.refresh = L, E, capacity, refresh
        self.resident = np.zeros((L, E), dtype=bool)
        self.resident.reshape(-1)[:min(capacity, L * E)] = True
        self.counts = np.zeros((L, E), dtype=np.int64)
        self.hits = self.misses = 0

    def step_begin(self, step: int):
        if step > 0 and step % self.refresh == 0:
            flat = self.counts.reshape(-1)
            # most touched first; stable sort keeps lower (layer, expert) first among ties
            order = np.argsort(-flat, kind="stable")[:min(self.capacity, flat.size)]
            self.resident[:] = False
            self.resident.reshape(-1)[order] = True
            self.counts[:] = 0

    def access(self, layer: int, experts):
        s = np.unique(np.asarray(experts, dtype=np.int64))
        self.counts[layer, s] += 1
        h = int(self.resident[layer, s].sum())
        self.hits += h
        self.misses += len(s) - h


def miss_rate(p) -> float:
    return p.misses / max(1, p.hits + p.misses)
