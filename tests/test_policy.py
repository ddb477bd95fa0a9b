"""Host-side placement policies used for the LRU comparison (hand-checked tiny traces)."""
from expert_cached_routed_router_b300.policy import RefreshedHotSet, StaticLayerSplit, miss_rate


def test_static_layer_split_counts():
    p = StaticLayerSplit(L=3, E=4, capacity=6)        # layer 0 whole, layer 1 experts 0-1
    p.access(0, [3, 3, 1])                            # 2 distinct, both resident
    p.access(1, [1, 2])                               # 1 hit, 1 miss
    p.access(2, [0])                                  # miss
    assert (p.hits, p.misses) == (3, 2)
    assert miss_rate(p) == 2 / 5


def test_refreshed_hot_set_follows_the_previous_window():
    p = RefreshedHotSet(L=2, E=4, capacity=2, refresh=2)   # starts as (0,0), (0,1)
    for step in range(4):
        p.step_begin(step)
        p.access(1, [3])
        p.access(1, [2] if step % 2 else [3, 2])
    # window 0 (steps 0, 1): 5 accesses, all misses; then (1,3) and (1,2) are the two
    # hottest entries and steps 2, 3 hit all 5 accesses
    assert p.misses == 5 and p.hits == 5
    assert p.resident[1, 3] and p.resident[1, 2] and not p.resident[0].any()
