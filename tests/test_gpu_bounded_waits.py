"""Bounded device waits that run out: the status word reports it, nothing hangs.

Every spin of the library's kernels has a time limit ("Mixture-of-Experts
Routing at Inference Time", "The hard part: token dropping is a silent
correctness bug": a failure must be reported, not silent).  A configuration's
debug_wait_ns shortens the limits so that a test can make them run out on
purpose, with no fault and no hang:

* the grouped GEMMs' pipeline waits (mbarriers between the TMA producer, the
  MMA issuer and the epilogue): a wait that gives up sets MOE_DEV_ERR_TIMEOUT,
  lets the copies and MMAs already issued finish, frees the tensor memory and
  returns; the next call with the default limits runs normally (a leaked
  allocation would stall its tcgen05.alloc) and gives the reference bits;
* the device-wide barrier of the reroute's grid-wide acceptance rounds: a
  barrier that gives up releases every CTA, the sequential kernel computes
  the assignment instead (MOE_DEV_NOTE_REROUTE_FALLBACK, informational) and
  the result still equals the oracle's, bit for bit.
"""
import numpy as np
import pytest

import oracle
from synth import workloads as W
from tests.checks import check_dispatch, check_equal

pytestmark = pytest.mark.gpu

_cases = {}


def case(name):
    from tests.layer_case import LayerCase
    if name not in _cases:
        _cases.clear()
        _cases[name] = LayerCase(W.WORKLOADS[name])
    return _cases[name]


def _ffn(moe, c, cfg, h_d, srt, blk, npad, T):
    import torch
    rows = moe.moe_max_padded_rows(cfg, T)
    y = torch.zeros((rows, c.wl.hidden), dtype=torch.bfloat16, device="cuda")
    ysh = (torch.zeros((T, c.wl.hidden), dtype=torch.bfloat16, device="cuda")
           if c.wl.shared_intermediate else None)
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    moe.moe_expert_ffn(cfg, h_d, c.w13_d, c.w2_d, c.w13s_d, c.w2s_d, srt, blk, npad, y, ysh, ws)
    torch.cuda.synchronize()
    return y, ysh, moe.moe_get_device_status(ws)


# tiny: CTA-pair W13, one-CTA W2; qw: CTA-pair W13 and W2; mix: CTA-pair W13
# (gate/up exchange between epilogue warps) and wide CTA-pair W2; with
# MOE_DEBUG_W13_SINGLE (0x2000) W13 runs on the one-CTA kernel, whose work
# items come from a tile counter through a shared-memory ring
@pytest.mark.parametrize("name,T,flags", [("tiny", 64, 0), ("qw", 512, 0), ("mix", 256, 0),
                                          ("tiny", 64, 0x2000), ("qw", 512, 0x2000)])
def test_gemm_pipeline_wait_runs_out_and_reports(name, T, flags):
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16
    c = case(name)
    h = W.make_h(c.wl, T, seed=5)
    h_d = dev_bf16(h)
    st = c.stages(h)   # the routing and layout (checked against the oracle elsewhere)
    assert st["status"] == 0
    N, B = c.wl.num_experts, c.wl.block_size
    rows, nblk = moe.moe_max_padded_rows(c.cfg, T), moe.moe_max_blocks(c.cfg, T)
    srt = torch.full((rows,), T * c.wl.top_k, dtype=torch.int32, device="cuda")
    blk = torch.zeros(nblk, dtype=torch.int32, device="cuda")
    P = st["num_padded"]
    srt[:P] = torch.from_numpy(st["sorted_route_ids"]).cuda()
    blk[:P // B] = torch.from_numpy(st["block_expert"]).cuda()
    npad = torch.tensor([P], dtype=torch.int32, device="cuda")
    cfg = dict(c.cfg, debug_flags=flags)
    y_ref, ysh_ref, s0 = _ffn(moe, c, cfg, h_d, srt, blk, npad, T)
    assert s0 == 0
    # a 1 ns limit: the first pipeline wait that is not already satisfied gives up
    short = dict(cfg, debug_wait_ns=1)
    for _ in range(2):
        _, _, s1 = _ffn(moe, c, short, h_d, srt, blk, npad, T)
        assert s1 & moe.MOE_DEV_ERR_TIMEOUT, f"status {s1:#x}"
    # the default limits again: same bits as before (the GPU and its tensor
    # memory are free again)
    y2, ysh2, s2 = _ffn(moe, c, cfg, h_d, srt, blk, npad, T)
    assert s2 == 0
    assert torch.equal(y2[:P].view(torch.int16), y_ref[:P].view(torch.int16))
    if ysh_ref is not None:
        assert torch.equal(ysh2.view(torch.int16), ysh_ref.view(torch.int16))
    # and the whole layer as usual
    out = c.forward(h)
    assert (out == st["out"]).all()
    del N


def test_forward_with_short_waits_reports_timeout_not_silence():
    # the fused forward on the same short limit: the status word tells the
    # caller the outputs are invalid
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16
    c = case("qw")
    T = 300
    h = W.make_h(c.wl, T, seed=6)
    cfg = dict(c.cfg, debug_wait_ns=1)
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    out = torch.empty((T, c.wl.hidden), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(cfg, dev_bf16(h), c.wg_d, c.bias_d, c.w13_d, c.w2_d, None, None, out, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) & moe.MOE_DEV_ERR_TIMEOUT
    assert (c.forward(h) == c.stages(h)["out"]).all()


def test_reroute_grid_barrier_runs_out_and_sequential_kernel_takes_over():
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16, host
    from tests.test_gpu_routing_modes import _ref_reroute, _reroute_on_gpu
    c = case("qw")
    T, cf = 8192, 1.0
    # the grid-wide rounds (88 of them on this batch) with a 1 ns barrier limit
    cfg = dict(c.cfg, capacity_factor=cf, overflow_policy=1, debug_flags=moe.MOE_DEBUG_REROUTE_GRID,
               debug_wait_ns=1)
    N, k, B = cfg["num_experts"], cfg["top_k"], cfg["block_size"]
    h = W.make_h(c.wl, T, seed=21)
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    g = torch.empty((T, k), dtype=torch.float32, device="cuda")
    lg = torch.empty((T, N), dtype=torch.float32, device="cuda")
    # routing with the default limits (its tensor-core logits are a GEMM too)
    moe.moe_route(dict(cfg, debug_flags=0, debug_wait_ns=0), dev_bf16(h), c.wg_d, c.bias_d, idx, g, lg, ws)
    got = _reroute_on_gpu(moe, cfg, idx, lg, ws)
    status = moe.moe_get_device_status(ws)
    assert status == moe.MOE_DEV_NOTE_REROUTE_FALLBACK, f"status {status:#x}"
    l_ref = oracle.router_logits(h, c.wg, c.bias)
    idx_ref, _ = oracle.select_topk(l_ref, k)
    check_equal("topk_idx", host(idx), idx_ref)
    re, nr, d = _ref_reroute(l_ref, idx_ref, N, B, oracle.capacity(T, N, k, cf))
    check_equal("route_expert", got["route_expert"], re)
    assert got["num_rerouted"] == nr and nr > 0
    check_dispatch(got, d)
