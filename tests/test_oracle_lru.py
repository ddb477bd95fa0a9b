"""Pins of the slot-level LRU simulator against an independent brute-force LRU and closed forms."""
import itertools

import numpy as np
import pytest

from oracle.lru import ERR_CAPACITY, OK, BruteForceLRU, SlotCacheSim


def _check_same(sim, bf, E):
    assert [(k // E, k % E) for k in sim.resident_keys()] == bf.order
    # slot table, owner and stamps are consistent
    for s in range(sim.n_slots):
        key = sim.owner[s]
        if key >= 0:
            assert sim.table[key // E, key % E] == s and sim.stamp[s] > 0
        else:
            assert sim.stamp[s] == 0
    assert np.count_nonzero(sim.table >= 0) == np.count_nonzero(sim.owner >= 0)
    live = sim.stamp[sim.owner >= 0]
    assert len(set(live.tolist())) == live.size and (live.size == 0 or live.max() <= sim.tick)


def _run_pair(trace, L, E, cap, prewarm):
    sim = SlotCacheSim(L, E, cap, prewarm=prewarm)
    warm = [(k // E, k % E) for k in range(min(cap, L * E))] if prewarm else []
    bf = BruteForceLRU(cap, warm)
    _check_same(sim, bf, E)
    for layer, experts in trace:
        st, hits, fills = sim.access(layer, experts)
        res = bf.call(layer, experts)
        if res is None:
            assert st == ERR_CAPACITY and hits == [] and fills == []
            continue
        assert st == OK
        bhits, bmiss, bevict = res
        assert [(layer, e) for e in hits] == bhits
        assert [(layer, f[2]) for f in fills] == bmiss
        assert [(f[3] // E, f[3] % E) for f in fills if f[3] >= 0] == bevict
        _check_same(sim, bf, E)
    return sim


@pytest.mark.parametrize("cap", [1, 2, 3])
def test_exhaustive_single_key_traces(cap):
    """Every trace of length <= 7 over <= 4 keys (one key per call), capacities 1..3."""
    keys = [(0, 0), (0, 1), (1, 0), (1, 1)]
    n = 0
    for length in range(1, 8):
        for tr in itertools.product(range(4), repeat=length):
            trace = [(keys[i][0], [keys[i][1]]) for i in tr]
            _run_pair(trace, 2, 2, cap, prewarm=False)
            n += 1
    assert n == sum(4 ** m for m in range(1, 8))


def test_random_multi_expert_traces():
    """10,000 random traces of calls touching several experts (hits-then-misses order matters),
    with and without prewarm, against the brute-force LRU model."""
    rng = np.random.default_rng(0)
    for _ in range(10_000):
        L, E = int(rng.integers(1, 4)), int(rng.integers(2, 6))
        cap = int(rng.integers(1, L * E + 2))
        trace = []
        for _ in range(int(rng.integers(1, 12))):
            m = int(rng.integers(1, E + 1))
            trace.append((int(rng.integers(0, L)), list(rng.choice(E, size=m, replace=True))))
        _run_pair(trace, L, E, cap, prewarm=bool(rng.integers(0, 2)))


def test_closed_form_capacity_covers_all_keys():
    rng = np.random.default_rng(1)
    L, E = 3, 5
    sim = SlotCacheSim(L, E, L * E, prewarm=False)
    seen = set()
    for _ in range(200):
        l = int(rng.integers(0, L))
        es = list(rng.choice(E, size=2, replace=False))
        sim.access(l, es)
        seen |= {(l, int(e)) for e in es}
    assert sim.misses == len(seen) and sim.evictions == 0


@pytest.mark.parametrize("C", [1, 2, 5, 9])
def test_closed_form_cyclic_trace_always_misses(C):
    sim = SlotCacheSim(1, C + 1, C, prewarm=False)
    for i in range(10 * (C + 1)):
        sim.access(0, [i % (C + 1)])
    assert sim.hits == 0 and sim.misses == 10 * (C + 1)


def test_free_slot_and_victim_rules():
    sim = SlotCacheSim(1, 8, 3, prewarm=False)
    assert sim.access(0, [5])[2] == [(0, 0, 5, -1)]          # lowest free slot
    assert sim.access(0, [2, 7])[2] == [(1, 0, 2, -1), (2, 0, 7, -1)]
    sim.access(0, [5])                                        # refresh slot 0
    st, hits, fills = sim.access(0, [1])                      # evict LRU = expert 2 in slot 1
    assert fills == [(1, 0, 1, 2)]
    # a call touching a resident expert and a new one never evicts the touched one
    st, hits, fills = sim.access(0, [7, 3])
    assert hits == [7] and fills == [(0, 0, 3, 5)]


def test_capacity_error_changes_nothing():
    sim = SlotCacheSim(2, 4, 2, prewarm=True)
    before = (sim.table.copy(), sim.owner.copy(), sim.stamp.copy(), sim.tick)
    assert sim.access(1, [0, 1, 2])[0] == ERR_CAPACITY
    assert all(np.array_equal(a, b) for a, b in zip(before[:3], (sim.table, sim.owner, sim.stamp)))
    assert sim.tick == before[3] and sim.hits == sim.misses == 0


def test_prewarm_layout():
    sim = SlotCacheSim(3, 4, 6, prewarm=True)
    assert list(sim.owner) == [0, 1, 2, 3, 4, 5] and list(sim.stamp) == [1, 2, 3, 4, 5, 6]
    assert sim.tick == 6 and sim.table[1, 1] == 5 and sim.table[2, 0] == -1
    full = SlotCacheSim(1, 16, 16, prewarm=True)
    full.access(0, range(16))
    assert full.misses == 0 and full.hits == 16


@pytest.mark.parametrize("n_new", [1, 2, 4, 6, 9])
def test_resize_keeps_most_recent_and_continues_like_brute_force(n_new):
    rng = np.random.default_rng(n_new)
    L, E, cap = 2, 6, 5
    sim = SlotCacheSim(L, E, cap, prewarm=True)
    bf = BruteForceLRU(cap, [(k // E, k % E) for k in range(cap)])
    for _ in range(30):
        l = int(rng.integers(0, L))
        es = list(rng.choice(E, size=2, replace=False))
        sim.access(l, es)
        bf.call(l, es)
    stamps_before = {int(sim.owner[s]): int(sim.stamp[s]) for s in range(cap) if sim.owner[s] >= 0}
    tick = sim.tick
    sim.resize(n_new)
    bf.shrink(n_new)
    _check_same(sim, bf, E)
    assert sim.tick == tick and sim.n_slots == n_new
    m = min(n_new, len(stamps_before))
    assert list(sim.stamp[:m]) == sorted(stamps_before.values(), reverse=True)[:m]
    assert np.all(sim.owner[m:] == -1)
    for s in range(m):
        assert stamps_before[int(sim.owner[s])] == sim.stamp[s]
    for _ in range(30):
        l = int(rng.integers(0, L))
        es = list(rng.choice(E, size=min(2, n_new), replace=False))
        sim.access(l, es)
        bf.call(l, es)
        _check_same(sim, bf, E)
