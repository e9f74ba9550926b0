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
