"""Pins for the oracle's top-k selection, gates and router margin.

Selection follows "Mixture-of-Experts Routing at Inference Time" ("How sparse
routing works"; the TopKRouter of its worked example) with the fixed
tie-break "lowest expert index wins on equal scores".  The pins: brute force
over every k-subset, constructed exact ties, NaN and signed-zero cases, the
k=2 closed form of the renormalised softmax, the k=N reduction to the plain
softmax, and hand-computed fixtures.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _beats(la, a, lb, b):
    """Independent statement of the ranking: a number beats NaN; larger beats
    smaller; on equal scores the lower index wins."""
    if math.isnan(la) and math.isnan(lb):
        return a < b
    if math.isnan(lb):
        return True
    if math.isnan(la):
        return False
    return la > lb or (la == lb and a < b)


def _brute_force(l, k):
    N = len(l)
    winners = []
    for S in itertools.combinations(range(N), k):
        rest = [e for e in range(N) if e not in S]
        if all(_beats(l[a], a, l[b], b) for a in S for b in rest):
            winners.append(S)
    assert len(winners) == 1, "the total order must single out exactly one subset"
    return list(winners[0])


@pytest.mark.parametrize("N,k", [(8, 2), (8, 4), (12, 3), (6, 6), (5, 1)])
def test_brute_force_over_all_subsets(N, k):
    rng = np.random.default_rng(N * 10 + k)
    rows = []
    for _ in range(40):
        rows.append(rng.standard_normal(N).astype(np.float32))
    # exact ties at and around the cut, quantised scores, signed zeros
    for _ in range(40):
        rows.append((rng.integers(0, 3, N) * 0.5).astype(np.float32))
    z = np.zeros(N, np.float32)
    z[::2] = -0.0
    rows.append(z)
    l = np.stack(rows)
    idx, _ = oracle.select_topk(l, k)
    for t in range(l.shape[0]):
        assert list(idx[t]) == _brute_force([float(v) for v in l[t]], k)


def test_all_equal_scores_pick_lowest_indices():
    l = np.full((3, 16), 0.75, np.float32)
    idx, g = oracle.select_topk(l, 5)
    assert (idx == np.arange(5)).all()
    np.testing.assert_allclose(g, 0.2, rtol=0, atol=1e-15)


def test_nan_ranks_below_every_number():
    l = np.array([[np.nan, -1e30, np.nan, -np.inf, 3.0]], np.float32)
    idx, _ = oracle.select_topk(l, 3)
    assert list(idx[0]) == [1, 3, 4]
    idx, _ = oracle.select_topk(l, 4)
    assert list(idx[0]) == [0, 1, 3, 4]   # the lower-index NaN is taken first


def test_signed_zeros_tie():
    l = np.array([[-0.0, 0.0, -0.0, -1.0]], np.float32)
    idx, _ = oracle.select_topk(l, 2)
    assert list(idx[0]) == [0, 1]


def test_slots_are_sorted_by_expert_index():
    l = np.array([[0.1, 5.0, -2.0, 4.0, 7.0, 0.0]], np.float32)
    idx, _ = oracle.select_topk(l, 3)
    assert list(idx[0]) == [1, 3, 4]


def test_gates_k2_closed_form():
    # g_first = 1 / (1 + exp(l_second - l_first)) for the renormalised softmax
    rng = np.random.default_rng(3)
    l = rng.standard_normal((200, 8)).astype(np.float32) * 3
    idx, g = oracle.select_topk(l, 2)
    for t in range(200):
        a, b = idx[t]
        la, lb = float(l[t, a]), float(l[t, b])
        np.testing.assert_allclose(g[t, 0], 1 / (1 + math.exp(lb - la)), rtol=1e-14)
        np.testing.assert_allclose(g[t, 1], 1 / (1 + math.exp(la - lb)), rtol=1e-14)
    np.testing.assert_allclose(g.sum(1), 1.0, rtol=0, atol=4e-16)


def test_gates_k_equals_n_is_the_softmax():
    rng = np.random.default_rng(4)
    l = rng.standard_normal((50, 7)).astype(np.float32)
    idx, g = oracle.select_topk(l, 7)
    assert (idx == np.arange(7)).all()
    np.testing.assert_allclose(g, softmax(l.astype(np.float64), axis=1), rtol=1e-13)


def test_gates_hand_fixture():
    with open(os.path.join(GOLDEN, "gates_hand.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        l = np.array([c["logits"]], np.float32)
        idx, g = oracle.select_topk(l, c["k"])
        assert list(idx[0]) == c["experts"]
        np.testing.assert_allclose(g[0], c["gates"], rtol=1e-12)


def test_router_margin_hand_case():
    l = np.array([[1.0, 4.0, 2.5, 2.5, -1.0]], np.float32)
    # ranking: 4.0 (e1), 2.5 (e2), 2.5 (e3), 1.0 (e0), -1.0 (e4)
    assert oracle.router_margin(l, 1)[0] == 1.5    # 4.0 - 2.5
    assert oracle.router_margin(l, 2)[0] == 0.0    # an exact tie at the cut
    assert oracle.router_margin(l, 3)[0] == 1.5    # 2.5 - 1.0
    assert oracle.router_margin(l, 5)[0] == math.inf
