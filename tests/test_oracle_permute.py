"""Pins for the oracle permutation (no GPU): invariants, identity case, library stable sort."""
import numpy as np
import pytest

from oracle import permute


def _check(ids, E, k):
    offsets, sp, inv = permute(ids, E)
    P = ids.size
    flat = ids.reshape(-1)
    assert offsets[0] == 0 and offsets[E] == P
    assert np.all(np.diff(offsets) >= 0)
    assert sorted(sp.tolist()) == list(range(P))
    assert np.all(inv[sp] == np.arange(P))
    for e in range(E):
        grp = sp[offsets[e]:offsets[e + 1]]
        assert np.all(flat[grp] == e)
        assert np.all(np.diff(grp) > 0)
    # every token appears exactly k times
    assert np.all(np.bincount(sp // k, minlength=ids.shape[0]) == k)
    # stable counting sort == the library's stable argsort on the expert ids
    assert np.array_equal(sp, np.argsort(flat, kind="stable"))
    return offsets, sp, inv


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (64, 8, 2), (300, 16, 8), (257, 128, 8), (5, 3, 3)])
def test_invariants_random(T, E, k):
    rng = np.random.default_rng(T + E + k)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    _check(ids, E, k)


def test_single_expert_is_identity():
    ids = np.zeros((37, 1), dtype=np.int32)
    offsets, sp, inv = _check(ids, 1, 1)
    assert sp.tolist() == list(range(37)) and inv.tolist() == list(range(37))
    assert offsets.tolist() == [0, 37]


def test_empty():
    offsets, sp, inv = permute(np.zeros((0, 2), np.int32), 4)
    assert offsets.tolist() == [0, 0, 0, 0, 0] and sp.size == 0 and inv.size == 0


def test_hand_example():
    # tokens: t0 -> (2, 0), t1 -> (0, 1), t2 -> (2, 1)
    ids = np.array([[2, 0], [0, 1], [2, 1]], np.int32)
    offsets, sp, inv = permute(ids, 3)
    assert offsets.tolist() == [0, 2, 4, 6]
    assert sp.tolist() == [1, 2, 3, 5, 0, 4]
    assert inv.tolist() == [4, 0, 1, 2, 5, 3]
