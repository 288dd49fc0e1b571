"""Pins for the oracle's overflow reroute policy.

"Mixture-of-Experts Routing at Inference Time", Figure 2 (the overflow
policy's reroute branch) and the mitigations after routing_stats: instead of
skipping the expert tier, an overflowing token is sent to its next-choice
expert.  Reading used here: the drop policy's capacity rule runs first
(each expert keeps its first C routes by route id); the routes it would drop
are then taken in ascending route id, and each goes to the best-ranked expert
(the router's total order on that token's logits) that still has room and
that the token does not already use; with no such expert the route stays
dropped.

The pins do not re-run that loop.  They check hand-derived cases and a
declarative characterisation: an assignment is the result of that sequential
rule if and only if (1) phase one matches the drop policy, (2) no expert holds
more than C routes, (3) every target is an expert the token did not use, and
(4) every expert the route ranks above its outcome that it could use is full
at the end, filled only by routes of higher priority (phase one, or a smaller
route id).  Conditions (3)-(4) say that at its turn the route took the best
expert with room, so any assignment that passes them is the sequential one.
"""
import numpy as np
import pytest

import oracle


def _rank_order(lrow):
    """Experts best first: larger logit, then lower index; NaN last."""
    N = len(lrow)
    nan = np.isnan(lrow)
    key = np.where(nan, 0.0, lrow.astype(np.float64))
    return np.lexsort((np.arange(N), -key, nan.astype(np.int8)))


def _check_stable(logits, idx, cap, route_expert):
    T, k = idx.shape
    N = logits.shape[1]
    R = T * k
    d = oracle.dispatch(idx, N, 8, cap)
    kept = d["route_kept"].astype(bool)
    e_of = idx.reshape(-1)
    # (1) phase one is the drop policy
    assert (route_expert[kept] == e_of[kept]).all()
    over = np.flatnonzero(~kept)
    # (2) capacity
    counts = np.bincount(route_expert[route_expert >= 0], minlength=N)
    assert (counts <= cap).all()
    # owner of each overflow assignment (route id), per expert
    for r in over:
        t = r // k
        tgt = route_expert[r]
        mine = set(idx[t].tolist())
        earlier = {int(route_expert[q]) for q in range(t * k, r) if route_expert[q] >= 0}
        # (3) a target the token does not use yet
        if tgt >= 0:
            assert tgt not in mine and tgt not in earlier
            others = {int(route_expert[q]) for q in range(t * k, (t + 1) * k) if q != r}
            assert tgt not in others
        # (4) every better usable expert was full by higher-priority routes
        order = _rank_order(logits[t])
        for e in order:
            if e == tgt:
                break
            if e in mine or e in earlier:
                continue
            assert counts[e] == cap, (r, e)
            holders = np.flatnonzero(route_expert == e)
            assert all(kept[q] or q < r for q in holders), (r, e)


def test_hand_case_top1():
    # Six tokens, four experts, top-1, C = ceil(1.0 * 6 * 1 / 4) = 2.
    logits = np.array([[4, 3, 2, 1],
                       [4, 1, 3, 2],
                       [4, 3, 1, 2],
                       [4, 3, 2, 1],
                       [4, 1, 2, 3],
                       [1, 4, 3, 2]], np.float32)
    idx, _ = oracle.select_topk(logits, 1)
    assert oracle.capacity(6, 4, 1, 1.0) == 2
    re, nr, nd = oracle.reroute(logits, idx, 2)
    # expert 0 keeps tokens 0 and 1; token 5's first choice (expert 1) is
    # kept in phase one although token 2 comes earlier; tokens 2, 3, 4 move
    # to 1, then 2 (1 is full), then 3
    assert re.tolist() == [0, 0, 1, 2, 3, 1]
    assert (nr, nd) == (3, 0)
    # C = 1: tokens 3 and 4 find every expert full
    re, nr, nd = oracle.reroute(logits, idx, 1)
    assert re.tolist() == [0, 2, 3, -1, -1, 1]
    assert (nr, nd) == (2, 2)


def test_hand_case_top2_excludes_the_tokens_own_experts():
    # Six tokens, six experts, top-2, C = ceil(1.0 * 6 * 2 / 6) = 2.
    down = [6, 5, 4, 3, 2, 1]
    up = [1, 2, 3, 4, 5, 6]
    logits = np.array([down, down, down, up, up, up], np.float32)
    idx, _ = oracle.select_topk(logits, 2)
    assert idx.tolist() == [[0, 1]] * 3 + [[4, 5]] * 3
    assert oracle.capacity(6, 6, 2, 1.0) == 2
    re, nr, nd = oracle.reroute(logits, idx, 2)
    # token 2: slot 0 -> 2; slot 1 would take 2 (one place left) but the token
    # already uses it -> 3.  Token 5: slot 0 -> 3 (its best with room), slot 1
    # -> 2 because 3 is now its own.
    assert re.tolist() == [0, 1, 0, 1, 2, 3, 4, 5, 4, 5, 3, 2]
    assert (nr, nd) == (4, 0)
    # C = 1: phase one keeps token 0 on {0, 1} and token 3 on {4, 5}; token 1
    # moves to {2, 3}; every later overflow finds its usable experts full
    assert oracle.capacity(6, 6, 2, 0.5) == 1
    re, nr, nd = oracle.reroute(logits, idx, 1)
    assert re.tolist() == [0, 1, 2, 3, -1, -1, 4, 5, -1, -1, -1, -1]
    assert (nr, nd) == (2, 6)


def test_no_capacity_means_no_reroute():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((50, 8)).astype(np.float32)
    idx, _ = oracle.select_topk(logits, 2)
    re, nr, nd = oracle.reroute(logits, idx, -1)
    assert (re == idx.reshape(-1)).all() and nr == 0 and nd == 0


def test_top1_with_cf_at_least_one_drops_nothing():
    # k = 1 and N*C >= T: when a route overflows, fewer than N*C routes are
    # placed, its own expert is full, so another expert still has room.
    rng = np.random.default_rng(4)
    for N, T, cf in [(4, 37, 1.0), (8, 200, 1.0), (16, 333, 1.25)]:
        bias = -1.5 * np.log(np.arange(N) + 1.0)        # skewed: many overflow
        logits = (rng.standard_normal((T, N)) + bias).astype(np.float32)
        idx, _ = oracle.select_topk(logits, 1)
        cap = oracle.capacity(T, N, 1, cf)
        re, nr, nd = oracle.reroute(logits, idx, cap)
        assert nd == 0 and nr > 0
        assert (re >= 0).all()
        _check_stable(logits, idx, cap, re)


@pytest.mark.parametrize("T,N,k,cf,seed", [(64, 8, 2, 1.0, 0), (300, 8, 2, 0.6, 1),
                                           (120, 16, 4, 0.8, 2), (90, 32, 8, 1.0, 3),
                                           (40, 6, 3, 0.7, 4)])
def test_stable_characterisation(T, N, k, cf, seed):
    rng = np.random.default_rng(seed)
    bias = -1.2 * np.log(np.arange(N) + 1.0)
    logits = (rng.standard_normal((T, N)) * 0.7 + bias).astype(np.float32)
    # exact ties, which the lower-index rule settles, and a NaN
    logits[::7] = np.round(logits[::7])
    logits[5, N - 1] = np.nan
    idx, _ = oracle.select_topk(logits, k)
    cap = oracle.capacity(T, N, k, cf)
    re, nr, nd = oracle.reroute(logits, idx, cap)
    d = oracle.dispatch(idx, N, 8, cap)
    # conservation: kept in phase one + rerouted + still dropped = all routes
    assert int(d["route_kept"].sum()) + nr + nd == T * k
    assert nr > 0
    assert int((re >= 0).sum()) == int(d["route_kept"].sum()) + nr
    _check_stable(logits, idx, cap, re)


def test_stability_check_catches_a_wrong_assignment():
    # the characterisation is strict: moving one rerouted route to a worse
    # expert with room, or swapping the priority of two routes, fails it
    rng = np.random.default_rng(9)
    T, N, k = 80, 8, 2
    bias = -1.2 * np.log(np.arange(N) + 1.0)
    logits = (rng.standard_normal((T, N)) + bias).astype(np.float32)
    idx, _ = oracle.select_topk(logits, k)
    cap = oracle.capacity(T, N, k, 0.8)
    re, nr, nd = oracle.reroute(logits, idx, cap)
    _check_stable(logits, idx, cap, re)
    d = oracle.dispatch(idx, N, 8, cap)
    moved = np.flatnonzero((re >= 0) & (d["route_kept"] == 0))
    assert len(moved) > 0
    caught = 0
    for r in moved[:10]:
        bad = re.copy()
        bad[r] = -1                      # dropped although an expert had room
        with pytest.raises(AssertionError):
            _check_stable(logits, idx, cap, bad)
        caught += 1
    assert caught > 0


def test_forward_with_reroute_equals_drop_when_nothing_overflows():
    import synth
    from synth import workloads as W
    wl = W.WORKLOADS["tiny"]
    h = W.make_h(wl, 24, seed=2)
    wg, bias = W.make_router(wl)
    w13, w2 = W.make_experts(wl)
    cfg = dict(wl.cfg, capacity_factor=8.0)
    a = oracle.moe_forward(dict(cfg, overflow_policy=0), h, wg, bias, w13, w2)
    b = oracle.moe_forward(dict(cfg, overflow_policy=1), h, wg, bias, w13, w2)
    assert a.tobytes() == b.tobytes()
    del synth


def test_forward_rerouted_token_uses_its_new_expert_with_the_old_gate():
    # a token whose route moved gets h + g_j * E_target(h) for that slot
    from synth import workloads as W
    wl = W.WORKLOADS["tiny"]
    T = 48
    h = W.make_h(wl, T, seed=5)
    wg, _ = W.make_router(wl)
    N, k = wl.num_experts, wl.top_k
    bias = (-1.5 * np.log(np.arange(N) + 1.0)).astype(np.float32)
    w13, w2 = W.make_experts(wl)
    cfg = dict(wl.cfg, capacity_factor=0.75, overflow_policy=1)
    out = oracle.moe_forward(cfg, h, wg, bias, w13, w2)
    logits = oracle.router_logits(h, wg, bias)
    idx, gates = oracle.select_topk(logits, k)
    cap = oracle.capacity(T, N, k, 0.75)
    re, nr, nd = oracle.reroute(logits, idx, cap)
    assert nr > 0
    moved_tok = sorted({r // k for r in np.flatnonzero((re >= 0) & (re != idx.reshape(-1)))})
    toks = np.array(moved_tok[:6], np.int32)
    ys = np.zeros((len(toks), k, wl.hidden))
    kept = (re >= 0).astype(np.uint8)
    for i, t in enumerate(toks):
        for j in range(k):
            e = re[t * k + j]
            if e >= 0:
                ys[i, j] = oracle.expert_rows(np.array([t], np.int32), np.array([e], np.int32),
                                              h, w13, w2)[0]
    ref = oracle.combine_rows(toks, h, gates, kept, ys)
    assert ref.tobytes() == out[toks].tobytes()
