"""Pins for the oracle's routing diagnostics: routing_stats and the margin.

routing_stats follows the instrumentation probe of "Mixture-of-Experts
Routing at Inference Time" (section "The hard part: token dropping is a
silent correctness bug"): per-expert load as a bincount of the routed expert
ids, a probe capacity of floor(mean load x capacity factor), the dropped count
as the sum of overflows (its dropped_tokens formula), the imbalance ratio
max / mean and the drop fraction dropped / total.  The router margin is the
gap between a token's k-th and (k+1)-th scores ("Mixture-of-experts routing
and LLM repeatability").
"""
import math

import numpy as np
import pytest

import oracle


def test_stats_hand_case():
    idx = np.array([[0, 1], [0, 2], [0, 1], [3, 0]], np.int32)
    load, st = oracle.routing_stats(idx, 4, 1.25)
    # load [4, 2, 1, 1], mean 2, capacity floor(2.5) = 2, overflow 4 - 2
    assert load.tolist() == [4, 2, 1, 1]
    assert st == dict(max_expert_load=4, min_expert_load=1, capacity=2, dropped_tokens=2,
                      total_routes=8, imbalance_ratio=2.0, drop_fraction=0.25)
    # a fifth, idle expert: mean 1.6, capacity floor(2.0) = 2, min 0
    load, st = oracle.routing_stats(idx, 5, 1.25)
    assert load.tolist() == [4, 2, 1, 1, 0]
    assert st["min_expert_load"] == 0 and st["capacity"] == 2 and st["dropped_tokens"] == 2
    assert st["imbalance_ratio"] == 2.5


def test_stats_balanced_load_drops_nothing():
    # every expert gets exactly T*k/N routes: ratio 1, no overflow for cf >= 1
    T, N, k = 64, 8, 2
    idx = np.array([[(2 * t) % N, (2 * t + 1) % N] for t in range(T)], np.int32)
    load, st = oracle.routing_stats(idx, N, 1.0)
    assert (load == T * k // N).all()
    assert st["imbalance_ratio"] == 1.0 and st["dropped_tokens"] == 0 and st["drop_fraction"] == 0.0


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_stats_probe_matches_the_dispatch_when_capacities_agree(seed):
    # with T*k/N an integer and cf = 1 the probe's floor(mean * cf) equals the
    # layer's ceil(cf*T*k/N), so its dropped count is the dispatch's
    rng = np.random.default_rng(seed)
    T, N, k = 96, 8, 2
    p = np.exp(-1.0 * np.log(np.arange(N) + 1.0))
    p /= p.sum()
    idx = np.array([np.sort(rng.choice(N, size=k, replace=False, p=p)) for _ in range(T)], np.int32)
    load, st = oracle.routing_stats(idx, N, 1.0)
    cap = oracle.capacity(T, N, k, 1.0)
    assert st["capacity"] == cap
    d = oracle.dispatch(idx, N, 8, cap)
    assert st["dropped_tokens"] == d["num_dropped"] > 0
    assert (load == np.bincount(idx.reshape(-1), minlength=N)).all()
    assert st["drop_fraction"] == d["num_dropped"] / (T * k)


def test_stats_ignore_ids_out_of_range_and_empty_input():
    idx = np.array([[0, 9], [-1, 1]], np.int32)
    load, st = oracle.routing_stats(idx, 4, 1.25)
    assert load.tolist() == [1, 1, 0, 0] and st["total_routes"] == 2
    load, st = oracle.routing_stats(np.zeros((0, 2), np.int32), 4, 1.25)
    assert load.tolist() == [0, 0, 0, 0]
    assert all(v == 0 for v in st.values())


def test_margin_is_the_gap_at_the_cut():
    rng = np.random.default_rng(7)
    l = rng.standard_normal((30, 10)).astype(np.float32)
    for k in (1, 2, 5, 9):
        m = oracle.router_margin(l, k)
        s = -np.sort(-l.astype(np.float64), axis=1)
        assert (m == s[:, k - 1] - s[:, k]).all()
        assert (m >= 0).all()
    assert (oracle.router_margin(l, 10) == math.inf).all()
