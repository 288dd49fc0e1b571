"""Pins for the oracle's expert-choice routing.

"Mixture-of-experts routing and LLM repeatability" (expert-choice routing:
each expert takes its highest-scoring tokens of the batch) and "Mixture-of-
Experts Routing at Inference Time" (section "Integration: where routing lives
in a serving stack", the comparison of routing variants: each expert picks
the tokens it will take, up to its capacity; a token can be taken by no
expert).  Scores are the router's softmax probabilities; capacity is
ceil(cf*T*k/N) (cf = 1 when unset), clipped to T; equal scores go to the
lower token index.

Pins: brute force over token subsets on tiny inputs (the selected set is the
one whose every member outranks every non-member, under probabilities from
numpy's own exp), an exact closed form for two experts (the probability of
expert 0 is monotone in l0 - l1, an exact fp64 difference), exact ties,
conservation laws and the dense reduction (capacity >= T turns expert choice
into the full-softmax mixture, which the token-choice path computes with
k = N).
"""
import itertools

import numpy as np
import pytest

import oracle


def _np_probs(l):
    x = l.astype(np.float64)
    x = x - x.max(axis=1, keepdims=True)
    e = np.exp(x)
    return e / e.sum(axis=1, keepdims=True)


@pytest.mark.parametrize("T,N,C,seed", [(7, 3, 3, 0), (8, 4, 2, 1), (9, 2, 4, 2), (6, 5, 6, 3)])
def test_brute_force_dominant_subset(T, N, C, seed):
    rng = np.random.default_rng(seed)
    l = rng.standard_normal((T, N)).astype(np.float32)
    sel, probs = oracle.expert_choice(l, C)
    p = _np_probs(l)
    np.testing.assert_allclose(probs, p, rtol=1e-12, atol=0)
    for e in range(N):
        winners = []
        for S in itertools.combinations(range(T), min(C, T)):
            rest = [t for t in range(T) if t not in S]
            if all(p[a, e] > p[b, e] or (p[a, e] == p[b, e] and a < b) for a in S for b in rest):
                winners.append(set(S))
        assert len(winners) == 1
        assert set(np.flatnonzero(sel[:, e]).tolist()) == winners[0]


def test_two_experts_closed_form():
    # p0 = 1 / (1 + exp(l1 - l0)) is decreasing in d = l1 - l0 (exact in
    # fp64): expert 0 takes the C smallest d, expert 1 the C largest
    rng = np.random.default_rng(11)
    T, C = 101, 37
    l = (rng.standard_normal((T, 2)) * 3).astype(np.float32)
    sel, _ = oracle.expert_choice(l, C)
    d = l[:, 1].astype(np.float64) - l[:, 0].astype(np.float64)
    order0 = np.lexsort((np.arange(T), d))          # smallest d first, then index
    order1 = np.lexsort((np.arange(T), -d))
    assert set(np.flatnonzero(sel[:, 0])) == set(order0[:C].tolist())
    assert set(np.flatnonzero(sel[:, 1])) == set(order1[:C].tolist())


def test_identical_tokens_go_to_the_lowest_indices():
    row = np.array([0.3, -1.0, 2.0, 0.0], np.float32)
    l = np.tile(row, (10, 1))
    sel, probs = oracle.expert_choice(l, 4)
    for e in range(4):
        assert np.flatnonzero(sel[:, e]).tolist() == [0, 1, 2, 3]
    assert (probs == probs[0]).all()


def test_counts_capacity_and_conservation():
    rng = np.random.default_rng(5)
    T, N, k = 50, 8, 2
    l = rng.standard_normal((T, N)).astype(np.float32)
    C = oracle.ec_capacity(T, N, k, 0.0)
    assert C == int(np.ceil(T * k / N))
    sel, probs = oracle.expert_choice(l, C)
    assert (sel.sum(axis=0) == C).all()                # every expert is full
    np.testing.assert_allclose(probs.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert oracle.ec_capacity(T, N, k, 1.5) == int(np.ceil(1.5 * T * k / N))
    assert oracle.ec_capacity(T, 2, 4, 1.0) == T      # clipped to the batch
    # a token may be taken by no expert (the dual failure of expert choice):
    # tokens 0-3 score 1/N everywhere, every later token is nearly sure of
    # one expert, and each expert has at least four such tokens
    skew = np.zeros((T, N), np.float32)
    skew[:4] = 5.0
    for t in range(4, T):
        skew[t, t % N] = 10.0
    sel, _ = oracle.expert_choice(skew, 4)
    assert not sel[:4].any()
    for e in range(N):
        assert np.flatnonzero(sel[:, e]).tolist() == [t for t in range(4, T) if t % N == e][:4]


def test_shifting_a_token_keeps_its_probabilities_and_the_selection():
    # softmax ignores a per-token constant; the key is computed from l - m,
    # so an exact shift changes no bit (values on a 2^-16 grid, so adding 8
    # or 4*i rounds nothing)
    rng = np.random.default_rng(6)
    l = (np.round(rng.uniform(2.0, 4.0, (40, 6)) * 65536.0) / 65536.0).astype(np.float32)
    sel, probs = oracle.expert_choice(l, 9)
    shifts = np.float32(8.0) * (np.arange(40) % 2).astype(np.float32)[:, None]
    sel2, probs2 = oracle.expert_choice(l + shifts, 9)
    assert (sel == sel2).all()
    assert probs2.tobytes() == probs.tobytes()
    # identical rows at different offsets tie exactly: lower index wins
    tie = np.tile(l[:1], (6, 1)) + (np.float32(4.0) * np.arange(6, dtype=np.float32))[:, None]
    sel3, _ = oracle.expert_choice(tie, 2)
    assert (sel3[:2] == 1).all() and not sel3[2:].any()


def test_nan_scores_rank_last():
    l = np.array([[1.0, 0.0], [np.nan, 0.0], [0.5, 0.0], [2.0, 0.0]], np.float32)
    sel, probs = oracle.expert_choice(l, 3)
    # token 1's expert-0 score is NaN: it goes last for expert 0
    assert np.flatnonzero(sel[:, 0]).tolist() == [0, 2, 3]
    assert np.isnan(probs[1, 0])


def test_capacity_at_least_T_is_the_dense_softmax_mixture():
    # every expert takes every token: out = h + sum_e softmax(l)_e E_e(h),
    # which is the token-choice layer with k = N (renormalising over all N
    # experts is the full softmax)
    from synth import workloads as W
    wl = W.WORKLOADS["tiny"]
    T = 12
    h = W.make_h(wl, T, seed=3)
    wg, bias = W.make_router(wl)
    w13, w2 = W.make_experts(wl)
    N = wl.num_experts
    ec = dict(wl.cfg, routing=1, capacity_factor=float(N) / wl.top_k)
    assert oracle.ec_capacity(T, N, wl.top_k, ec["capacity_factor"]) == T
    dense = dict(wl.cfg, top_k=N, capacity_factor=0.0)
    a = oracle.moe_forward(ec, h, wg, bias, w13, w2)
    b = oracle.moe_forward(dense, h, wg, bias, w13, w2)
    # same experts and terms; the gates come from two exp/renormalise orders,
    # so allow an fp64-rounding difference to flip a bf16 rounding
    diff = np.abs(a.astype(np.int32) - b.astype(np.int32))
    assert (diff <= 1).all() and (diff == 0).mean() > 0.99
