"""Host input generator: determinism, slicing by offset and distribution."""
import numpy as np

import synth
from synth import workloads as W


def test_offsets_slice_the_same_stream():
    full = synth.normal_bf16((1000,), 3, 9, 0.5)
    part = synth.normal_bf16((300,), 3, 9, 0.5, offset=400)
    assert (full[400:700] == part).all()


def test_thread_count_does_not_change_values():
    a = synth.normal_bf16((200000,), 1, 2, 1.0, nthreads=1)
    b = synth.normal_bf16((200000,), 1, 2, 1.0, nthreads=8)
    assert (a == b).all()


def test_distribution_moments():
    x = synth.bf16_to_f32(synth.normal_bf16((400000,), 0, 1, 0.02)).astype(np.float64)
    assert abs(x.mean()) < 1e-4
    assert abs(x.std() / 0.02 - 1) < 0.01
    assert np.abs(x).max() < 6.1 * 0.02


def test_streams_differ_by_seed_and_tensor():
    a = synth.normal_bf16((64,), 0, 1, 1.0)
    assert not (a == synth.normal_bf16((64,), 1, 1, 1.0)).all()
    assert not (a == synth.normal_bf16((64,), 0, 2, 1.0)).all()


def test_expert_slices_match_full_tensor():
    wl = W.Workload("t", 128, 4, 2, 256, 8, wg_std=0.1)
    w13, w2 = W.make_experts(wl)
    for e in range(4):
        assert (W.expert_w13(wl, e) == w13[e]).all()
        assert (W.expert_w2(wl, e) == w2[e]).all()


def test_qw_recipe_has_exact_ties_and_zero_tokens():
    wl = W.WORKLOADS["qw"]
    h = W.make_h(wl, 2000)
    zero_rows = np.flatnonzero((h == 0).all(axis=1))
    assert 5 <= len(zero_rows) <= 40
    _, bias = W.make_router(wl)
    assert set(np.unique(bias).tolist()) <= {0.0, 0.25, 0.5, 0.75}
    assert (bias == bias.max()).sum() > wl.top_k   # the top level is shared by many experts
