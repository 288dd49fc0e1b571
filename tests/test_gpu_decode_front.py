"""The two-launch decode front gives the bits of the separate kernels.

For at most two tokens the forward runs the router's chunk sums, then one
CTA that adds them in chunk order, then the bias, selects the top-k with the
same code, runs the same dispatch body (layout and both tile lists) and
copies the routed rows ("Why temperature=0 Still Gives Different Answers:
Batch Invariance": one reduction order for every batch).  Layer outputs must
be bit-identical with the front switched off (MOE_DEBUG_NO_DECODE_FRONT), for N = 8,
128 and 256 experts, a 40-expert layer with a 128-element last chunk,
capacity drops, the shared expert, and a three-token batch that takes the
separate kernels either way.
"""
import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

_layers = {}

_ODD = W.Workload("odd", 640, 40, 4, 256, 8, tokens=(1,))


def layer(wl):
    from tests.layer_case import LayerCase
    if wl.name not in _layers:
        _layers.clear()
        _layers[wl.name] = LayerCase(wl)
    return _layers[wl.name]


def _forward(c, cfg, h_bits, front):
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16, host_bf16
    T = h_bits.shape[0]
    out = torch.empty((T, c.wl.hidden), dtype=torch.bfloat16, device="cuda")
    cfg = dict(cfg, debug_flags=0 if front else moe.MOE_DEBUG_NO_DECODE_FRONT)
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    moe.moe_forward(cfg, dev_bf16(h_bits), c.wg_d, c.bias_d, c.w13_d, c.w2_d, c.w13s_d, c.w2s_d, out, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    return host_bf16(out)


@pytest.mark.parametrize("name,T,extra", [
    ("tiny", 1, {}), ("tiny", 2, {}), ("tiny", 2, {"capacity_factor": 0.25}),
    ("qw", 1, {}), ("qw", 2, {}),
    ("mix", 1, {}), ("mix", 2, {"capacity_factor": 0.5}),
    ("odd", 1, {}), ("odd", 2, {}), ("odd", 3, {}),
    ("ds", 1, {}), ("ds", 2, {}),
])
def test_decode_front_matches_separate_kernels(name, T, extra):
    wl = _ODD if name == "odd" else W.WORKLOADS[name]
    c = layer(wl)
    cfg = dict(c.cfg, **extra)
    for seed in (3, 4):
        h = W.make_h(wl, T, seed=seed * 100 + T)
        a = _forward(c, cfg, h, front=True)
        b = _forward(c, cfg, h, front=False)
        assert a.shape == (T, wl.hidden)
        assert np.array_equal(a, b), f"seed {seed}"
