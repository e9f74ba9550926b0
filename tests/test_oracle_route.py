"""Pins for the oracle router (no GPU): brute force over k-subsets, closed forms, invariants."""
import itertools
import math

import numpy as np
import pytest

from oracle import route


@pytest.mark.parametrize("E,k", [(2, 1), (4, 2), (6, 3), (8, 2), (8, 5), (8, 8)])
def test_topk_equals_best_subset_brute_force(E, k):
    rng = np.random.default_rng(100 + E * 10 + k)
    lg = rng.standard_normal((50, E)).astype(np.float32)
    ids, w = route(lg, k)
    for t in range(50):
        best = max(itertools.combinations(range(E), k), key=lambda s: sum(float(lg[t, e]) for e in s))
        assert set(ids[t].tolist()) == set(best)
        # slots in descending logit order
        vals = [float(lg[t, e]) for e in ids[t]]
        assert vals == sorted(vals, reverse=True)


def test_weights_are_softmax_restricted_to_selection():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((40, 16)).astype(np.float32)
    ids, w = route(lg, 4)
    for t in range(40):
        ex = [math.exp(float(lg[t, e])) for e in ids[t]]
        s = math.fsum(ex)
        assert np.allclose(w[t], [v / s for v in ex], rtol=1e-14, atol=0)


def test_invariants_sum_to_one_and_descending():
    rng = np.random.default_rng(4)
    lg = (rng.standard_normal((200, 128)) * 3).astype(np.float32)
    ids, w = route(lg, 8)
    assert np.all(np.abs(w.sum(axis=1) - 1.0) < 1e-14)
    assert np.all(np.diff(w, axis=1) <= 0)
    assert all(len(set(r)) == 8 for r in ids.tolist())


def test_closed_forms():
    # k = 1 -> weight 1
    _, w = route(np.array([[0.3, -1.0, 2.0]], np.float32), 1)
    assert w.tolist() == [[1.0]]
    # equal logits inside the selection -> 1/k
    ids, w = route(np.array([[5.0, 5.0, 5.0, 1.0]], np.float32), 3)
    assert ids.tolist() == [[0, 1, 2]]
    assert np.allclose(w, 1.0 / 3.0, rtol=1e-15)
    # two logits differing by ln 3 -> weights 3/4, 1/4
    ids, w = route(np.array([[0.0, math.log(3.0)]], np.float32), 2)
    assert ids.tolist() == [[1, 0]]
    assert np.allclose(w, [[0.75, 0.25]], rtol=1e-6)


def test_ties_break_toward_lower_id():
    ids, _ = route(np.array([[1.0, 2.0, 2.0, 0.0, 2.0]], np.float32), 2)
    assert ids.tolist() == [[1, 2]]
    ids, _ = route(np.array([[1.0, 2.0, 2.0, 0.0, 2.0]], np.float32), 4)
    assert ids.tolist() == [[1, 2, 4, 0]]


def test_rejects_bad_k_and_nonfinite():
    with pytest.raises(ValueError):
        route(np.zeros((1, 4), np.float32), 5)
    with pytest.raises(ValueError):
        route(np.array([[0.0, np.inf]], np.float32), 1)


def test_large_e_matches_library_sort_and_softmax():
    """E = 1024, k = 32 with many exact ties: the selection equals the library's
    lexicographic sort on (descending logit, ascending id), and the weights equal the
    library softmax of the selected logits (a softmax renormalised over a subset is
    the softmax of that subset)."""
    from scipy.special import softmax
    rng = np.random.default_rng(8)
    lg = np.round(rng.standard_normal((16, 1024)) * 4).astype(np.float32) / 4  # quarter steps: ties
    ids, w = route(lg, 32)
    for t in range(16):
        order = np.lexsort((np.arange(1024), -lg[t].astype(np.float64)))[:32]
        assert np.array_equal(ids[t], order)
        assert np.allclose(w[t], softmax(lg[t, order].astype(np.float64)), rtol=1e-12, atol=0)
