"""Pins for the oracle's SwiGLU experts, combine and whole-layer forward.

Layer output = h + sum of gate * expert(h) over the kept routes ("Mixture-of-
Experts Routing at Inference Time", "How sparse routing works"; the per-token
pseudo-code of "Mixture-of-experts routing and LLM repeatability").  A dropped
route adds nothing and the gates are not renormalised ("The hard part" and
Figure 2 of the first page: the residual plus the routes still kept).  The expert
is SwiGLU: W13 = [gate | up], a = silu(gate) * up, y = a . W2.

Pins: reductions to a dense SwiGLU computed independently in numpy fp64,
exact special cases (zero experts, fully dropped tokens), the closed-form
gates of a constructed router, the no-renormalisation rule, bf16 rounding
against hand values, and permutation equivariance.
"""
import math

import numpy as np
import pytest

import oracle
from synth import bf16_to_f32, f32_to_bf16


def np_bf16(x):
    """bf16 rounding written independently (via fp32; may double-round on
    exact fp32 ties, so comparisons below allow one bf16 ulp)."""
    return f32_to_bf16(np.asarray(x, dtype=np.float64).astype(np.float32))


def np_swiglu(x_bits, w13_bits, w2_bits):
    x = bf16_to_f32(x_bits).astype(np.float64)
    w13 = bf16_to_f32(w13_bits).astype(np.float64)
    w2 = bf16_to_f32(w2_bits).astype(np.float64)
    I = w2.shape[0]
    g = x @ w13[..., :I] if x.ndim == 1 else x @ w13[:, :I]
    u = x @ w13[..., I:] if x.ndim == 1 else x @ w13[:, I:]
    a = bf16_to_f32(np_bf16(g / (1 + np.exp(-g)) * u)).astype(np.float64)
    return a @ w2, a


def assert_bf16_close(got_bits, ref, ulps=1.0):
    got = bf16_to_f32(got_bits).astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -120))) - 7)
    assert np.all(np.abs(got - ref) <= ulps * ulp + 1e-30), np.max(np.abs(got - ref) / ulp)


def _rb(rng, shape, std):
    return f32_to_bf16((rng.standard_normal(shape) * std).astype(np.float32))


def test_bf16_round_hand_values():
    assert oracle.bf16_round(1.0) == 0x3F80
    assert oracle.bf16_round(1.0 + 2 ** -8) == 0x3F80         # tie -> even (1.0)
    assert oracle.bf16_round(1.0 + 3 * 2 ** -8) == 0x3F82     # tie -> even (1 + 2^-6)
    assert oracle.bf16_round(1.0 + 2 ** -8 + 2 ** -30) == 0x3F81
    assert oracle.bf16_round(-2.0) == 0xC000
    assert oracle.bf16_round(0.0) == 0x0000
    assert oracle.bf16_round(-0.0) == 0x8000
    assert oracle.bf16_round(3.140625) == 0x4049              # exactly representable
    assert oracle.bf16_round(2.0 ** -133) == 0x0001           # smallest subnormal
    assert oracle.bf16_round(1e39) == 0x7F80                  # overflow to +inf


def test_bf16_round_matches_single_fp32_rounding():
    # for doubles that are exact fp32 values, rounding to bf16 is one rounding
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(5000) * 10).astype(np.float32)
    ref = f32_to_bf16(x)
    got = np.array([oracle.bf16_round(float(v)) for v in x], np.uint16)
    assert (got == ref).all()


def test_expert_row_is_dense_swiglu():
    rng = np.random.default_rng(1)
    H, I = 256, 512
    x = _rb(rng, H, 1.0)
    w13 = _rb(rng, (H, 2 * I), 0.05)
    w2 = _rb(rng, (I, H), 0.05)
    y, a = oracle.expert_row(x, w13, w2)
    y_ref, a_ref = np_swiglu(x, w13, w2)
    # the activation agrees to one bf16 ulp (double rounding aside)
    assert_bf16_close(a, a_ref, ulps=1.0)
    assert np.mean(a == np_bf16(a_ref)) > 0.99
    # y is a . W2 in fp64 for the oracle's own a
    np.testing.assert_allclose(y, bf16_to_f32(a).astype(np.float64) @ bf16_to_f32(w2).astype(np.float64),
                               rtol=1e-12, atol=1e-12)


def _cfg(H, N, k, I, B, cf=0.0, Is=0):
    return dict(hidden=H, num_experts=N, top_k=k, intermediate=I, block_size=B,
                capacity_factor=cf, shared_intermediate=Is)


def test_single_expert_layer_is_residual_plus_swiglu():
    rng = np.random.default_rng(2)
    T, H, I = 12, 128, 256
    h = _rb(rng, (T, H), 1.0)
    wg = _rb(rng, (H, 1), 0.1)
    w13 = _rb(rng, (1, H, 2 * I), 0.05)
    w2 = _rb(rng, (1, I, H), 0.05)
    out = oracle.moe_forward(_cfg(H, 1, 1, I, 8), h, wg, None, w13, w2)
    y, _ = np_swiglu(h, w13[0], w2[0])
    assert_bf16_close(out, bf16_to_f32(h) + y, ulps=1.0)


def test_shared_expert_is_added_with_gate_one():
    rng = np.random.default_rng(3)
    T, H, I, Is = 8, 128, 256, 384
    h = _rb(rng, (T, H), 1.0)
    wg = _rb(rng, (H, 1), 0.1)
    w13 = _rb(rng, (1, H, 2 * I), 0.05)
    w2 = _rb(rng, (1, I, H), 0.05)
    w13s = _rb(rng, (H, 2 * Is), 0.05)
    w2s = _rb(rng, (Is, H), 0.05)
    out = oracle.moe_forward(_cfg(H, 1, 1, I, 8, Is=Is), h, wg, None, w13, w2, w13s, w2s)
    y, _ = np_swiglu(h, w13[0], w2[0])
    ys, _ = np_swiglu(h, w13s, w2s)
    assert_bf16_close(out, bf16_to_f32(h) + y + ys, ulps=1.0)


def test_zero_experts_return_the_residual_exactly():
    rng = np.random.default_rng(4)
    T, H, N, k, I = 20, 128, 8, 2, 256
    h = _rb(rng, (T, H), 1.0)
    wg = _rb(rng, (H, N), 0.1)
    z13 = np.zeros((N, H, 2 * I), np.uint16)
    z2 = np.zeros((N, I, H), np.uint16)
    out = oracle.moe_forward(_cfg(H, N, k, I, 8), h, wg, None, z13, z2)
    assert (out == h).all()


def test_gates_weight_the_right_experts():
    # W_g = 0 and bias = (0, 1): every token selects both experts with gates
    # 1/(1+e) (expert 0) and e/(1+e) (expert 1).  Expert 1 is all zeros, so
    # out = h + E0(h) / (1 + e); swapping the gates would give e/(1+e).
    rng = np.random.default_rng(5)
    T, H, I = 10, 128, 256
    h = _rb(rng, (T, H), 1.0)
    wg = np.zeros((H, 2), np.uint16)
    bias = np.array([0.0, 1.0], np.float32)
    w13 = np.stack([_rb(rng, (H, 2 * I), 0.05), np.zeros((H, 2 * I), np.uint16)])
    w2 = np.stack([_rb(rng, (I, H), 0.05), np.zeros((I, H), np.uint16)])
    out = oracle.moe_forward(_cfg(H, 2, 2, I, 8), h, wg, bias, w13, w2)
    y0, _ = np_swiglu(h, w13[0], w2[0])
    assert_bf16_close(out, bf16_to_f32(h) + y0 / (1 + math.e), ulps=1.0)


def test_drop_keeps_residual_and_surviving_expert_without_renormalising():
    # token t selects {0, 1} when h[t,0] = +1 and {0, 2} when h[t,0] = -1
    # (logits (10, 5s, -5s)); capacity ceil(0.5*T*2/3) fills expert 0 first
    # for the earliest tokens; later tokens keep only their second expert
    # with its original (not renormalised) gate.
    rng = np.random.default_rng(6)
    T, H, N, k, I, B = 24, 128, 3, 2, 256, 8
    h = _rb(rng, (T, H), 1.0)
    sign = np.where(np.arange(T) % 2 == 0, 1.0, -1.0)
    h[:, 0] = f32_to_bf16(sign.astype(np.float32))
    wg = np.zeros((H, N), np.uint16)
    wg[0] = f32_to_bf16(np.array([0.0, 5.0, -5.0], np.float32))
    bias = np.array([10.0, 0.0, 0.0], np.float32)
    w13 = _rb(rng, (N, H, 2 * I), 0.05)
    w2 = _rb(rng, (N, I, H), 0.05)
    cf = 0.5
    C = oracle.capacity(T, N, k, cf)
    assert C == 8
    out = oracle.moe_forward(_cfg(H, N, k, I, B, cf), h, wg, bias, w13, w2)
    hf = bf16_to_f32(h).astype(np.float64)
    ref = np.empty((T, H))
    load1 = load2 = 0
    for t in range(T):
        other = 1 if sign[t] > 0 else 2
        l_other = 5.0   # 5*s for expert 1 when s = +1, -5*s for expert 2 when s = -1
        g0 = 1 / (1 + math.exp(l_other - 10.0))
        g1 = 1 - g0
        y0, _ = np_swiglu(h[t], w13[0], w2[0])
        yo, _ = np_swiglu(h[t], w13[other], w2[other])
        keep0 = t < C
        if other == 1:
            keep_o = load1 < C
            load1 += 1
        else:
            keep_o = load2 < C
            load2 += 1
        ref[t] = hf[t] + (g0 * y0 if keep0 else 0) + (g1 * yo if keep_o else 0)
    assert_bf16_close(out, ref, ulps=1.0)
    assert not (out[C:] == h[C:]).all()   # the surviving expert still contributes


def test_fully_dropped_tokens_return_the_residual_exactly():
    rng = np.random.default_rng(7)
    T, H, N, k, I = 16, 128, 2, 2, 256
    h = _rb(rng, (T, H), 1.0)
    wg = np.zeros((H, N), np.uint16)
    w13 = _rb(rng, (N, H, 2 * I), 0.05)
    w2 = _rb(rng, (N, I, H), 0.05)
    cf = 1.0 / T           # C = ceil(1/T * T * 2 / 2) = 1
    out = oracle.moe_forward(_cfg(H, N, k, I, 8, cf), h, wg, None, w13, w2)
    assert (out[1:] == h[1:]).all()
    assert not (out[0] == h[0]).all()


def test_identical_experts_sum_to_one_expert():
    rng = np.random.default_rng(8)
    T, H, I = 6, 128, 256
    h = _rb(rng, (T, H), 1.0)
    wg = _rb(rng, (H, 2), 0.3)
    w13 = _rb(rng, (1, H, 2 * I), 0.05)
    w2 = _rb(rng, (1, I, H), 0.05)
    out2 = oracle.moe_forward(_cfg(H, 2, 2, I, 8), h, wg, None, np.concatenate([w13, w13]),
                              np.concatenate([w2, w2]))
    y, _ = np_swiglu(h, w13[0], w2[0])
    assert_bf16_close(out2, bf16_to_f32(h) + y, ulps=1.0)


def test_permuting_tokens_permutes_outputs():
    rng = np.random.default_rng(9)
    T, H, N, k, I = 40, 128, 8, 2, 256
    h = _rb(rng, (T, H), 1.0)
    wg = _rb(rng, (H, N), 1 / np.sqrt(H))
    w13 = _rb(rng, (N, H, 2 * I), 0.02)
    w2 = _rb(rng, (N, I, H), 0.02)
    cfg = _cfg(H, N, k, I, 8)
    out = oracle.moe_forward(cfg, h, wg, None, w13, w2)
    perm = rng.permutation(T)
    out_p = oracle.moe_forward(cfg, h[perm], wg, None, w13, w2)
    assert (out_p == out[perm]).all()


def test_stagewise_equals_whole_layer():
    rng = np.random.default_rng(10)
    T, H, N, k, I, B = 30, 128, 8, 2, 256, 8
    h = _rb(rng, (T, H), 1.0)
    wg = _rb(rng, (H, N), 1 / np.sqrt(H))
    w13 = _rb(rng, (N, H, 2 * I), 0.02)
    w2 = _rb(rng, (N, I, H), 0.02)
    out = oracle.moe_forward(_cfg(H, N, k, I, B), h, wg, None, w13, w2)
    l = oracle.router_logits(h, wg)
    idx, g = oracle.select_topk(l, k)
    d = oracle.dispatch(idx, N, B, -1)
    toks = np.repeat(np.arange(T), k).astype(np.int32)
    y = oracle.expert_rows(toks, idx.reshape(-1), h, w13, w2).reshape(T, k, H)
    out2 = oracle.combine_rows(np.arange(T), h, g, d["route_kept"], y)
    assert (out == out2).all()
