"""Negative controls for the parity checker.

Following the evidence design of "Route-Block Membership Selects Packed-AWQ
Arithmetic" (section "The evidence package": a checker must refuse planted
changes to routes, hashes and tensors), each test plants one
mistake in a copy of the oracle's own results, on the CPU, and requires the
checker to reject it.
"""
import numpy as np
import pytest

import oracle
from synth import workloads as W
from tests.checks import ParityError, check_dispatch, check_equal, check_gates, check_outputs, digest


@pytest.fixture(scope="module")
def tiny():
    wl = W.WORKLOADS["tiny"]
    h = W.make_h(wl, 64)
    wg, bias = W.make_router(wl)
    w13, w2 = W.make_experts(wl)
    l = oracle.router_logits(h, wg, bias)
    idx, g = oracle.select_topk(l, wl.top_k)
    d = oracle.dispatch(idx, wl.num_experts, wl.block_size, -1)
    out = oracle.moe_forward(wl.cfg, h, wg, bias, w13, w2)
    return dict(idx=idx, gates=g, d=d, out=out)


def test_checker_accepts_the_truth(tiny):
    check_equal("topk_idx", tiny["idx"], tiny["idx"].copy())
    check_dispatch(tiny["d"], {k: (v.copy() if hasattr(v, "copy") else v) for k, v in tiny["d"].items()})
    check_gates(tiny["gates"].astype(np.float32), tiny["gates"])
    check_outputs(tiny["out"], tiny["out"])


def test_wrong_route_is_rejected(tiny):
    bad = tiny["idx"].copy()
    bad[17, 1] = (bad[17, 1] + 1) % 8
    with pytest.raises(ParityError):
        check_equal("topk_idx", bad, tiny["idx"])


def test_wrong_drop_mask_is_rejected(tiny):
    d = {k: (v.copy() if hasattr(v, "copy") else v) for k, v in tiny["d"].items()}
    d["route_kept"][5] ^= 1
    with pytest.raises(ParityError):
        check_dispatch(d, tiny["d"])


def test_swapped_routes_inside_a_block_are_rejected(tiny):
    d = {k: (v.copy() if hasattr(v, "copy") else v) for k, v in tiny["d"].items()}
    s = d["sorted_route_ids"]
    s[0], s[1] = s[1], s[0]
    with pytest.raises(ParityError):
        check_dispatch(d, tiny["d"])


def test_wrong_block_expert_is_rejected(tiny):
    d = {k: (v.copy() if hasattr(v, "copy") else v) for k, v in tiny["d"].items()}
    d["block_expert"][-1] = 0
    with pytest.raises(ParityError):
        check_dispatch(d, tiny["d"])


def test_perturbed_output_is_rejected(tiny):
    bad = tiny["out"].copy()
    bad[3, 7] ^= 0x0100          # flips an exponent bit: far outside tolerance
    with pytest.raises(ParityError):
        check_outputs(bad, tiny["out"])


def test_perturbed_gate_is_rejected(tiny):
    g = tiny["gates"].astype(np.float32)
    g[9, 0] *= 1.001
    with pytest.raises(ParityError):
        check_gates(g, tiny["gates"])


def test_hash_changes_with_one_bit(tiny):
    a = tiny["out"].copy()
    b = a.copy()
    b[0, 0] ^= 1
    assert digest(a) != digest(b)
