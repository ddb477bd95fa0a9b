"""Pins of the admission rule of the slot-cache simulator (frequency counts halved every
10 * n_slots accesses; a miss that finds no free slot replaces the next victim only if its
count is at least the victim's, else it is bypassed into staging entry n_slots + b)."""
import numpy as np
import pytest

from oracle.lru import BYPASS, ERR_CAPACITY, OK, BruteForceLRU, SlotCacheSim


def _compare(sim, bf, E, layer, experts):
    st, hits, fills = sim.access(layer, experts)
    res = bf.call(layer, experts)
    if res is None:
        assert st == ERR_CAPACITY and hits == [] and fills == []
        return
    assert st == OK
    bhits, bmiss, bevict, bbyp = res
    assert [(layer, e) for e in hits] == bhits
    assert [(layer, f[2]) for f in fills] == bmiss
    assert [(f[3] // E, f[3] % E) for f in fills if f[3] >= 0] == bevict
    assert [(layer, f[2]) for f in fills if f[3] == BYPASS] == bbyp
    # bypass destinations are the staging entries n_slots, n_slots + 1, ... in miss order
    byp = [f[0] for f in fills if f[3] == BYPASS]
    assert byp == list(range(sim.n_slots, sim.n_slots + len(byp)))
    assert all(0 <= f[0] < sim.n_slots for f in fills if f[3] != BYPASS)
    assert [(k // E, k % E) for k in sim.resident_keys()] == bf.order


def test_random_traces_match_brute_force():
    """Long enough for the counts to be halved several times (H = 10 * capacity)."""
    rng = np.random.default_rng(5)
    n_halvings = 0
    for _ in range(400):
        L, E = int(rng.integers(1, 4)), int(rng.integers(2, 7))
        cap = int(rng.integers(1, L * E + 1))
        prewarm = bool(rng.integers(0, 2))
        sim = SlotCacheSim(L, E, cap, prewarm=prewarm, admission=True)
        warm = [(k // E, k % E) for k in range(min(cap, L * E))] if prewarm else []
        bf = BruteForceLRU(cap, warm, admission=True)
        # skewed popularity so that counts differ
        p = 1.0 / np.arange(1, E + 1) ** 1.2
        p /= p.sum()
        acc = 0
        for _ in range(int(rng.integers(5, 120))):
            m = int(rng.integers(1, min(E, cap) + 1))
            es = list(rng.choice(E, size=m, replace=True, p=p))
            layer = int(rng.integers(0, L))
            _compare(sim, bf, E, layer, es)
            acc += len(set(es))
        n_halvings += acc // (10 * cap)
    assert n_halvings > 100


def test_halving_closed_form():
    """Capacity 1 (H = 10): ten calls of key 0 leave f(0) = 10, halved to 5 at the tenth
    access.  A new key 1 is then bypassed on its 1st..4th calls (f = 1..4 < 5) and admitted
    on the 5th (5 >= 5).  Without the halving it would need 10 calls."""
    sim = SlotCacheSim(1, 2, 1, prewarm=False, admission=True)
    for _ in range(10):
        sim.access(0, [0])
    assert sim.freq[0] == 5 and sim.acc == 0
    for j in range(1, 5):
        st, hits, fills = sim.access(0, [1])
        assert fills == [(1, 0, 1, BYPASS)] and sim.owner[0] == 0
    st, hits, fills = sim.access(0, [1])
    assert fills == [(0, 0, 1, 0)] and sim.owner[0] == 1 and sim.bypasses == 4


def test_worked_example_two_slots():
    """Two slots, one layer, no prewarm; each step below is derived by hand from the rule:
    {0}: f0=1, free slot 0.  {1}: f1=1, free slot 1.  {0}, {1}: hits (stamps 3, 4).
    {2}: f2=1 < f0=2 (victim slot 0, stamp 3) -> bypass into staging entry 2.
    {2}: f2=2 >= f0=2 -> admitted into slot 0, evicting 0.
    {0}: f0=3 >= f1=2 (victim slot 1, stamp 4) -> slot 1, evicting 1.
    {1, 3}: victims in order slot 0 (key 2, f=2), slot 1 (key 0, f=3); miss 1 (f=3 >= 2) takes
    slot 0; miss 3 (f=1 < 3) is bypassed into staging entry 2."""
    sim = SlotCacheSim(1, 4, 2, prewarm=False, admission=True)
    steps = [
        ([0], [(0, 0, 0, -1)]),
        ([1], [(1, 0, 1, -1)]),
        ([0], []),
        ([1], []),
        ([2], [(2, 0, 2, BYPASS)]),
        ([2], [(0, 0, 2, 0)]),
        ([0], [(1, 0, 0, 1)]),
        ([1, 3], [(0, 0, 1, 2), (2, 0, 3, BYPASS)]),
    ]
    for experts, want in steps:
        st, hits, fills = sim.access(0, experts)
        assert st == OK and fills == want, (experts, fills)
    assert list(sim.owner) == [1, 0] and list(sim.stamp) == [7, 6] and sim.tick == 7
    assert sim.bypasses == 2 and sim.evictions == 3 and sim.misses == 7


def test_no_bypass_while_everything_fits():
    """Capacity >= distinct keys: admission never triggers; identical to the plain LRU."""
    rng = np.random.default_rng(2)
    L, E = 2, 5
    a = SlotCacheSim(L, E, L * E, prewarm=False, admission=True)
    b = SlotCacheSim(L, E, L * E, prewarm=False)
    for _ in range(300):
        l = int(rng.integers(0, L))
        es = list(rng.choice(E, size=3, replace=False))
        assert a.access(l, es) == b.access(l, es)
    assert a.bypasses == 0
    assert np.array_equal(a.owner, b.owner) and np.array_equal(a.stamp, b.stamp)


@pytest.mark.parametrize("n_new", [1, 3, 6])
def test_resize_keeps_counts_and_continues_like_brute_force(n_new):
    rng = np.random.default_rng(10 + n_new)
    L, E, cap = 2, 6, 4
    sim = SlotCacheSim(L, E, cap, prewarm=True, admission=True)
    bf = BruteForceLRU(cap, [(k // E, k % E) for k in range(cap)], admission=True)
    p = 1.0 / np.arange(1, E + 1) ** 1.5
    p /= p.sum()
    for _ in range(40):
        l = int(rng.integers(0, L))
        _compare(sim, bf, E, l, list(rng.choice(E, size=2, replace=True, p=p)))
    freq = sim.freq.copy()
    sim.resize(n_new)
    bf.shrink(n_new)
    assert np.array_equal(sim.freq, freq)
    for _ in range(60):
        l = int(rng.integers(0, L))
        _compare(sim, bf, E, l, list(rng.choice(E, size=min(2, n_new), replace=True, p=p)))
