"""Pins for the oracle's capacity rule, drops and stable padded-block alignment.

Capacity and drops: "Mixture-of-experts routing and LLM repeatability"
(Switch capacity = tokens / experts x capacity factor, filled in batch order)
and "Mixture-of-Experts Routing at Inference Time" ("The hard part", Figure 2,
and its dropped_tokens formula: sum over experts of max(0, load - capacity)).
Alignment: "Route-Block Membership Selects Packed-AWQ Arithmetic" (routes
grouped by expert and padded into fixed-size blocks; stable construction
orders valid routes by (expert id, flattened route id)).

The pins are invariants that any correct dispatch must satisfy, the closed
form for the drop count, and hand-built cases.
"""
import numpy as np
import pytest

import oracle


def _random_routes(rng, T, N, k, skew=0.0):
    idx = np.empty((T, k), np.int32)
    p = np.exp(-skew * np.log(np.arange(N) + 1.0))
    p /= p.sum()
    for t in range(T):
        idx[t] = np.sort(rng.choice(N, size=k, replace=False, p=p))
    return idx


def _check_invariants(idx, N, B, cap, d):
    T, k = idx.shape
    R = T * k
    e_of = idx.reshape(-1)
    kept, pos, srt, blocks = d["route_kept"], d["route_pos"], d["sorted_route_ids"], d["block_expert"]
    P = d["num_padded"]
    # closed-form drop count (the dropped_tokens formula) and kept counts
    load = np.bincount(e_of, minlength=N)
    c = load if cap < 0 else np.minimum(load, cap)
    assert (d["expert_counts"] == c).all()
    assert d["num_dropped"] == int(np.maximum(load - (load if cap < 0 else cap), 0).sum())
    assert int(kept.sum()) == int(c.sum())
    # capacity filled in batch order: kept routes of e are its first c_e by route id
    for e in range(N):
        routes_e = np.flatnonzero(e_of == e)
        assert (kept[routes_e[:c[e]]] == 1).all() and (kept[routes_e[c[e]:]] == 0).all()
    # padding: every segment a multiple of B, total as the closed form
    padded = (c + B - 1) // B * B
    assert P == int(padded.sum()) and len(srt) == P and len(blocks) == P // B
    # each kept route appears exactly once, at route_pos; dropped routes nowhere
    valid = srt[srt != R]
    assert len(valid) == len(set(valid.tolist())) == int(kept.sum())
    for r in range(R):
        if kept[r]:
            assert srt[pos[r]] == r
        else:
            assert pos[r] == -1 and r not in set(valid.tolist())
    # blocks hold one expert; segments in ascending expert id; routes ascending
    # inside a segment; sentinels only at segment tails
    off = 0
    for e in range(N):
        seg = srt[off:off + padded[e]]
        assert (blocks[off // B:(off + padded[e]) // B] == e).all()
        real = seg[:c[e]]
        assert (np.diff(real) > 0).all() and all(e_of[r] == e for r in real)
        assert (seg[c[e]:] == R).all()
        off += padded[e]


@pytest.mark.parametrize("T,N,k,B,cf,skew", [
    (64, 8, 2, 8, 0.0, 0.0), (100, 8, 2, 64, 0.0, 1.2), (97, 16, 4, 16, 1.0, 1.2),
    (200, 8, 2, 8, 1.0, 2.0), (33, 128, 8, 16, 0.0, 0.0), (50, 5, 5, 8, 1.25, 0.0),
    (1, 256, 8, 16, 0.0, 0.0), (301, 8, 2, 64, 0.5, 1.2)])
def test_dispatch_invariants(T, N, k, B, cf, skew):
    rng = np.random.default_rng(T * 7 + N)
    idx = _random_routes(rng, T, N, k, skew)
    cap = oracle.capacity(T, N, k, cf)
    d = oracle.dispatch(idx, N, B, cap)
    _check_invariants(idx, N, B, cap, d)


def test_capacity_formula():
    assert oracle.capacity(8192, 8, 2, 1.0) == 2048
    assert oracle.capacity(10, 8, 2, 1.0) == 3        # ceil(2.5)
    assert oracle.capacity(4096, 8, 2, 1.25) == 1280
    assert oracle.capacity(7, 3, 1, 1.0) == 3          # ceil(7/3)
    assert oracle.capacity(64, 8, 2, 0.0) == -1
    assert oracle.capacity(64, 8, 2, -1.0) == -1


def test_hot_expert_keeps_the_first_tokens():
    # every token routes to experts {0, 1}; capacity C keeps tokens 0..C-1 and
    # drops the rest (capacity filled in batch order)
    T, N, k, B = 40, 4, 2, 8
    idx = np.tile(np.array([0, 1], np.int32), (T, 1))
    C = 13
    d = oracle.dispatch(idx, N, B, C)
    kept = d["route_kept"].reshape(T, k)
    assert (kept[:C] == 1).all() and (kept[C:] == 0).all()
    assert d["num_dropped"] == 2 * (T - C)
    assert list(d["expert_counts"]) == [C, C, 0, 0]
    # segment 0 = routes 0,2,4,... then pad to 16; segment 1 = routes 1,3,5,...
    srt = d["sorted_route_ids"]
    assert list(srt[:C]) == list(range(0, 2 * C, 2)) and (srt[C:16] == T * k).all()
    assert list(srt[16:16 + C]) == list(range(1, 2 * C, 2))
    assert list(d["block_expert"]) == [0, 0, 1, 1]


def test_out_of_range_expert_ids_are_not_routed():
    idx = np.array([[0, 9], [-1, 2], [2, 3]], np.int32)
    d = oracle.dispatch(idx, 4, 8, -1)
    assert list(d["route_kept"]) == [1, 0, 0, 1, 1, 1]
    assert list(d["route_pos"][[1, 2]]) == [-1, -1]
    assert d["num_dropped"] == 0


def test_empty_experts_get_no_blocks():
    idx = np.array([[3, 5]] * 3, np.int32)
    d = oracle.dispatch(idx, 8, 8, -1)
    assert d["num_padded"] == 16 and list(d["block_expert"]) == [3, 5]
    assert list(d["sorted_route_ids"]) == [0, 2, 4] + [6] * 5 + [1, 3, 5] + [6] * 5
