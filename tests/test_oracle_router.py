"""Pins for the oracle's router projection (fp32 logits in the fixed order).

The logits are the router projection h . W_g of "Mixture-of-Experts Routing at
Inference Time" (section "How sparse routing works").  Their fp32 summation
order is the reading of "Why temperature=0 Still Gives Different Answers:
Batch Invariance" (Tier 2): fixed 256-element chunks, each summed in order,
combined in a fixed (ascending) order.  The pins below do not re-run that
formula: they use exact special cases, an error bound against exact
arithmetic, and a hand-built input whose fp32 result is known in closed form
and differs under every other chunking.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from synth import bf16_to_f32, f32_to_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_bf16(rng, shape, std=1.0):
    return f32_to_bf16((rng.standard_normal(shape) * std).astype(np.float32))


def test_one_hot_rows_select_router_columns():
    # h = e_i gives l[e] = W_g[i, e] exactly: catches a transposed W_g or a
    # wrong index in the contraction.
    rng = np.random.default_rng(1)
    H, N = 600, 12
    wg = _rand_bf16(rng, (H, N))
    rows = [0, 1, 255, 256, 257, 511, 599]
    h = np.zeros((len(rows), H), dtype=np.uint16)
    for t, i in enumerate(rows):
        h[t, i] = 0x3F80  # 1.0
    l = oracle.router_logits(h, wg)
    np.testing.assert_array_equal(l, bf16_to_f32(wg[rows]))


def test_zero_tokens_give_the_bias_exactly():
    rng = np.random.default_rng(2)
    H, N = 384, 16
    wg = _rand_bf16(rng, (H, N))
    bias = rng.standard_normal(N).astype(np.float32)
    l = oracle.router_logits(np.zeros((3, H), np.uint16), wg, bias)
    np.testing.assert_array_equal(l, np.broadcast_to(bias, (3, N)))


def test_chunked_order_closed_form():
    # Hand-built products (see tests/golden/router_chunk_order.json): the
    # 256-chunked order gives exactly 1 + 2^-16; a plain sequential sum, a
    # pairwise tree or 128-element chunks all give other values.
    with open(os.path.join(GOLDEN, "router_chunk_order.json")) as f:
        g = json.load(f)
    H = g["H"]
    tiny = np.float32(2.0 ** -24)
    h = np.full((1, H), 0x3F80, dtype=np.uint16)               # all ones
    w = np.full(H, f32_to_bf16(np.array([tiny]))[0], dtype=np.uint16)
    w[0] = 0x3F80
    l = oracle.router_logits(h, w.reshape(H, 1))
    assert l[0, 0] == np.float32(g["expected"])
    assert float(np.float32(g["expected"])) == 1.0 + 2.0 ** -16
    # the alternatives the fixture lists really are different numbers
    for alt in g["other_orders"].values():
        assert np.float32(alt) != l[0, 0]


@pytest.mark.parametrize("H,N", [(128, 8), (300, 5), (2048, 128), (4096, 8), (7168, 16)])
def test_error_bound_against_exact_dot(H, N):
    # |l_fp32 - l_exact| <= gamma * sum|h_i w_ie|, gamma = (256 + chunks + 1) u
    # (each product is exact; at most 255 in-chunk additions, chunks-1
    # combining additions and the bias addition round).
    rng = np.random.default_rng(H + N)
    T = 6
    h = _rand_bf16(rng, (T, H))
    wg = _rand_bf16(rng, (H, N), std=1 / np.sqrt(H))
    bias = rng.standard_normal(N).astype(np.float32)
    l = oracle.router_logits(h, wg, bias).astype(np.float64)
    hf, wf = bf16_to_f32(h).astype(np.float64), bf16_to_f32(wg).astype(np.float64)
    exact = hf @ wf + bias.astype(np.float64)
    mag = np.abs(hf) @ np.abs(wf) + np.abs(bias.astype(np.float64))
    chunks = (H + 255) // 256
    gamma = (256 + chunks + 1) * 2.0 ** -24 * 1.01
    assert np.all(np.abs(l - exact) <= gamma * mag)
    # and not trivially: the result is a genuine fp32 computation, not exact
    assert np.any(l != exact) or H <= 256


def test_summation_order_is_visible_in_fp32():
    # Float addition is not associative (the point of the batch-invariance
    # page): the same fp32 values accumulated left to right and in 3 or 5
    # slices give different bits, so the bit-exact tests can see a change of
    # order in the kernels.
    def left_to_right(v):
        return np.cumsum(v, dtype=np.float32)[-1]

    def sliced(v, n):
        parts = [left_to_right(p) for p in np.array_split(v, n)]
        return left_to_right(np.array(parts, dtype=np.float32))

    differ = 0
    for tid in range(10):
        # full 24-bit mantissas: bf16 draws times an fp32 constant
        vals = bf16_to_f32(synth.normal_bf16((5000,), 9, 100 + tid, 0.05)) * np.float32(1.1)
        results = {float(left_to_right(vals)), float(sliced(vals, 3)), float(sliced(vals, 5))}
        differ += len(results) >= 2
    assert differ >= 5


def test_thread_count_does_not_change_bits():
    rng = np.random.default_rng(5)
    h = _rand_bf16(rng, (37, 1000))
    wg = _rand_bf16(rng, (1000, 24), std=0.03)
    a = oracle.router_logits(h, wg, nthreads=1)
    b = oracle.router_logits(h, wg, nthreads=7)
    assert a.tobytes() == b.tobytes()
