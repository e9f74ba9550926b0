"""Pins for the LRU slot simulator (no GPU): closed-form hit/miss sequences."""
import pytest

from oracle.cache import LRUSim, NoSlot


def test_fill_then_hits():
    c = LRUSim(layers=2, E=16, slots_per_layer=4)
    assert c.request(0, [3, 5, 7]) == [(0, True), (1, True), (2, True)]
    assert c.request(0, [5, 3]) == [(1, False), (0, False)]
    assert c.request(1, [3]) == [(0, True)]  # layer pools are separate


def test_cyclic_over_capacity_always_misses():
    c = LRUSim(layers=1, E=8, slots_per_layer=3)
    seq = [0, 1, 2, 3] * 5
    res = [c.request(0, [e])[0][1] for e in seq]
    assert all(res)


def test_evicts_least_recently_used():
    c = LRUSim(layers=1, E=8, slots_per_layer=3)
    c.request(0, [0, 1, 2])
    c.request(0, [0])          # 1 is now the oldest
    assert c.request(0, [5]) == [(1, True)]
    assert c.request(0, [1]) == [(2, True)]  # 2 was the oldest now


def test_request_never_evicts_its_own_ids():
    c = LRUSim(layers=1, E=8, slots_per_layer=2)
    c.request(0, [0, 1])
    assert c.request(0, [2, 3]) == [(0, True), (1, True)]
    with pytest.raises(NoSlot):
        c.request(0, [4, 5, 6])


def test_global_pool_is_shared_across_layers():
    c = LRUSim(layers=2, E=4, slots_per_layer=1, policy="global")
    assert c.request(0, [1]) == [(0, True)]
    assert c.request(1, [1]) == [(1, True)]
    assert c.request(1, [2]) == [(0, True)]  # evicts layer 0's expert 1 (oldest)
    assert c.request(0, [1]) == [(1, True)]


def _textbook_lru_misses(trace, capacity, shared):
    """Hit/miss sequence of a textbook LRU (an ordered dict: a hit moves to the most recent
    end, a miss evicts the least recent entry when full) over the same touches."""
    from collections import OrderedDict
    caches = {}
    out = []
    for layer, ids in trace:
        c = caches.setdefault(None if shared else layer, OrderedDict())
        for e in ids:
            key = (layer, int(e))
            if key in c:
                c.move_to_end(key)
                out.append(False)
            else:
                if len(c) >= capacity:
                    c.popitem(last=False)
                c[key] = True
                out.append(True)
    return out


@pytest.mark.parametrize("policy", ["layer", "global"])
def test_misses_equal_a_textbook_lru(policy):
    """Slot numbering aside, the simulator is an LRU: its hit / miss sequence equals an
    independent ordered-dict LRU's on random traces with repeats (requests never larger
    than a pool, so the same-request rule never binds differently)."""
    import numpy as np
    rng = np.random.default_rng(4)
    layers, E, slots, k = 3, 12, 4, 3
    sim = LRUSim(layers, E, slots, policy)
    trace = []
    for _ in range(400):
        layer = int(rng.integers(layers))
        ids = rng.choice(E, size=k, replace=False, p=np.arange(E, 0, -1) / np.arange(E, 0, -1).sum())
        trace.append((layer, ids))
    got = [copied for layer, ids in trace for _, copied in sim.request(layer, ids)]
    cap = slots if policy == "layer" else slots * layers
    assert got == _textbook_lru_misses(trace, cap, policy == "global")


def test_acquired_slots_are_pinned_until_release():
    """A layer's acquired slots cannot be taken by a later request until the layer is
    released: a prefetch that would need them fails with NoSlot and changes nothing."""
    c = LRUSim(layers=2, E=8, slots_per_layer=3, policy="global")  # 6 slots
    assert c.acquire(0, [0, 1, 2, 3]) == [(0, True), (1, True), (2, True), (3, True)]
    before = (list(c.owner[0]), list(c.stamp[0]), dict(c.where), c.clock)
    with pytest.raises(NoSlot):
        c.prefetch(1, [4, 5, 6])          # 3 misses, only slots 4 and 5 unpinned
    assert (list(c.owner[0]), list(c.stamp[0]), dict(c.where), c.clock) == before
    assert c.prefetch(1, [4, 5]) == [(4, True), (5, True)]
    with pytest.raises(NoSlot):
        c.prefetch(1, [4, 5, 6])          # 4, 5 touched by this request, 0..3 pinned
    c.release(0)
    assert c.prefetch(1, [6]) == [(0, True)]  # slot 0 is now the least recently used
    assert c.acquire(0, [1]) == [(1, False)]


def test_pins_count_every_acquire_until_release():
    c = LRUSim(layers=1, E=8, slots_per_layer=2)
    c.acquire(0, [0])
    c.acquire(0, [0, 1])                  # slot 0 pinned twice, slot 1 once
    with pytest.raises(NoSlot):
        c.prefetch(0, [2])
    c.release(0)                          # releases both acquires
    assert c.prefetch(0, [2]) == [(0, True)]


def test_prefetch_pins_nothing():
    c = LRUSim(layers=1, E=8, slots_per_layer=2)
    c.prefetch(0, [0, 1])
    assert c.prefetch(0, [2, 3]) == [(0, True), (1, True)]
