"""Kernel paths that a configuration's debug flags can force give the bits of
the default path.

The W13 GEMM runs on CTA pairs wherever the intermediate size is a multiple
of 128 (a property of the layer's shape); forced onto single CTAs, the tiny,
Qwen-like and Mixtral-like layers must give the same output bits, because a
pair's M = 256 MMA computes each output element with the same K steps in the
same order as a single CTA's M = 128 MMAs ("Why temperature=0 Still Gives
Different Answers: Batch Invariance": the arithmetic of a row must not depend
on how the work is tiled).  The shared expert of the DeepSeek-like layer runs
on a second stream; run on the caller's stream after the routed GEMMs it
must give the same bits too.
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


def _forward(c, cfg, h_bits):
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16, host_bf16
    T = h_bits.shape[0]
    out = torch.empty((T, c.wl.hidden), dtype=torch.bfloat16, device="cuda")
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    moe.moe_forward(cfg, dev_bf16(h_bits), c.wg_d, c.bias_d, c.w13_d, c.w2_d, c.w13s_d, c.w2s_d, out, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    return host_bf16(out)


@pytest.mark.parametrize("name,T,flag", [
    ("tiny", 64, 0x2000), ("tiny", 1, 0x2000), ("qw", 1, 0x2000), ("qw", 300, 0x2000), ("qw", 4096, 0x2000),
    ("mix", 200, 0x2000), ("ds", 3, 0x400), ("ds", 700, 0x400), ("qw", 4096, 0x1000), ("ds", 700, 0x1000)])
def test_forced_path_gives_default_bits(name, T, flag):
    c = layer(name)
    h = W.make_h(c.wl, T, seed=60 + T)
    a = _forward(c, c.cfg, h)
    b = _forward(c, dict(c.cfg, debug_flags=flag), h)
    assert np.array_equal(a, b)
