"""The two ways of writing the gathered token rows x_perm give the same bits.

The fused forward writes x_perm either in padded-row order (each row read
from h by its route id) or token by token from the inverse map route_pos
(each token row read once, copied to its kept slots, padding rows zeroed);
the second serves batches whose h exceeds half of L2.  The layer output must
be bit-identical either way, with dropped routes, rerouted routes and expert
choice, on ragged batches.
"""
import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

_layers = {}


def layer(name):
    from tests.layer_case import LayerCase
    if name not in _layers:
        _layers.clear()
        _layers[name] = LayerCase(W.WORKLOADS[name])
    return _layers[name]


def _forward(c, cfg, h_bits, mode):
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16, host_bf16
    T = h_bits.shape[0]
    h_d = dev_bf16(h_bits)
    out = torch.empty((T, c.wl.hidden), dtype=torch.bfloat16, device="cuda")
    flag = moe.MOE_DEBUG_ROW_GATHER if mode == "gather" else moe.MOE_DEBUG_ROW_SCATTER
    cfg = dict(cfg, debug_flags=flag)
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    moe.moe_forward(cfg, h_d, c.wg_d, c.bias_d, c.w13_d, c.w2_d, c.w13s_d, c.w2s_d, out, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    return host_bf16(out)


@pytest.mark.parametrize("name,T,extra", [
    ("tiny", 1, {}),
    ("tiny", 203, {}),
    ("tiny", 203, {"capacity_factor": 0.7}),
    ("cap", 2001, {}),
    ("qw", 777, {"capacity_factor": 0.6}),
    ("qw", 777, {"capacity_factor": 0.6, "overflow_policy": 1}),
    ("qw", 300, {"routing": 1}),
])
def test_row_copy_paths_agree(name, T, extra):
    c = layer(name)
    cfg = dict(c.cfg, **extra)
    h = W.make_h(c.wl, T, seed=40 + T)
    a = _forward(c, cfg, h, "gather")
    b = _forward(c, cfg, h, "scatter")
    assert a.shape == (T, c.wl.hidden)
    assert np.array_equal(a, b)
