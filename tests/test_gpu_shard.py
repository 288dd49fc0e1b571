"""A capacity-limited batch split into token shards gives the unsharded bits.

Each shard routes its tokens, counts its routes per expert
(moe_routing_stats), and dispatches with moe_dispatch_align_shard given the
routes every expert received in the earlier shards (the sum that the
all-gather of shard.shard_exchange forms across ranks; here the shards run
one after another on one GPU and the sum is taken on the host).  The keep
decisions must equal the oracle's on the whole batch (capacity filled in
batch order: "Mixture-of-Experts Routing at Inference Time"), bit for bit,
and each shard's layer output must equal the unsharded forward's rows.
"""
import numpy as np
import pytest

import oracle
from synth import workloads as W

pytestmark = pytest.mark.gpu

_layers = {}


def layer(name):
    from tests.layer_case import LayerCase
    if name not in _layers:
        _layers.clear()
        _layers[name] = LayerCase(W.WORKLOADS[name])
    return _layers[name]


@pytest.mark.parametrize("name,cf,cuts", [
    ("tiny", 0.7, [0, 90, 91, 203]),
    ("tiny", 1.0, [0, 1, 64]),
    ("cap", 0.8, [0, 1000, 2001]),
    ("qw", 0.6, [0, 300, 777]),
])
def test_shards_reproduce_the_unsharded_batch(name, cf, cuts):
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16, host, host_bf16
    c = layer(name)
    wl = c.wl
    cfg = dict(c.cfg, capacity_factor=cf)
    N, k, B, H = wl.num_experts, wl.top_k, wl.block_size, wl.hidden
    T = cuts[-1]
    h = W.make_h(wl, T, seed=T + 11)
    # the unsharded forward and the oracle's decisions on the whole batch
    out_full = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    moe.moe_forward(cfg, dev_bf16(h), c.wg_d, c.bias_d, c.w13_d, c.w2_d, c.w13s_d, c.w2s_d, out_full, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    l = oracle.router_logits(h, c.wg, c.bias)
    idx_ref, _ = oracle.select_topk(l, k)
    C = oracle.capacity(T, N, k, cf)
    kept_ref = oracle.dispatch(idx_ref, N, B, C)["route_kept"]
    assert 0 < int((kept_ref == 0).sum())            # the capacity binds
    offset = np.zeros(N, np.int64)
    dropped_total = 0
    for lo, hi in zip(cuts[:-1], cuts[1:]):
        Ts, d = hi - lo, "cuda"
        hs = dev_bf16(np.ascontiguousarray(h[lo:hi]))
        wss = moe.workspace(cfg, Ts)
        moe.moe_clear_device_status(wss)
        idx = torch.empty((Ts, k), dtype=torch.int32, device=d)
        gates = torch.empty((Ts, k), dtype=torch.float32, device=d)
        moe.moe_route(cfg, hs, c.wg_d, c.bias_d, idx, gates, None, wss)
        load = torch.empty(N, dtype=torch.int32, device=d)
        stats = torch.empty(64, dtype=torch.uint8, device=d)
        moe.moe_routing_stats(cfg, idx, 1.25, load, stats)
        off_d = torch.from_numpy(offset.astype(np.int32)).to(d)
        R = Ts * k
        rows, nblk = moe.moe_max_padded_rows(cfg, Ts), moe.moe_max_blocks(cfg, Ts)
        kept = torch.empty(R, dtype=torch.uint8, device=d)
        pos = torch.empty(R, dtype=torch.int32, device=d)
        srt = torch.empty(rows, dtype=torch.int32, device=d)
        blk = torch.empty(nblk, dtype=torch.int32, device=d)
        npad = torch.empty(1, dtype=torch.int32, device=d)
        counts = torch.empty(N, dtype=torch.int32, device=d)
        dropped = torch.empty(1, dtype=torch.int32, device=d)
        moe.moe_dispatch_align_shard(cfg, T, idx, off_d, kept, pos, srt, blk, npad, counts, dropped, wss)
        y = torch.empty((rows, H), dtype=torch.bfloat16, device=d)
        ysh = torch.empty((Ts, H), dtype=torch.bfloat16, device=d) if wl.shared_intermediate else None
        moe.moe_expert_ffn(cfg, hs, c.w13_d, c.w2_d, c.w13s_d, c.w2s_d, srt, blk, npad, y, ysh, wss)
        out = torch.empty((Ts, H), dtype=torch.bfloat16, device=d)
        moe.moe_combine(cfg, hs, gates, kept, pos, y, ysh, out)
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(wss) == 0
        assert np.array_equal(host(idx), idx_ref[lo:hi])
        assert np.array_equal(host(kept), kept_ref[lo * k:hi * k]), (lo, hi)
        assert np.array_equal(host_bf16(out), host_bf16(out_full)[lo:hi]), (lo, hi)
        offset += host(load).astype(np.int64)
        dropped_total += int(host(dropped)[0])
    assert dropped_total == int((kept_ref == 0).sum())


def test_forward_shard_through_nccl_on_one_rank():
    # shard.forward_shard end to end (route, counts, NCCL all-gather, shard
    # dispatch, FFN, combine) on a one-rank group: no earlier shards, so the
    # output is moe_forward's, bit for bit
    import os
    import socket
    import torch
    import torch.distributed as dist
    import invariant_expert_routing_gb300 as moe
    from invariant_expert_routing_gb300 import shard
    from tests.gpu_util import dev_bf16, host_bf16
    sk = socket.socket()
    sk.bind(("127.0.0.1", 0))
    port = sk.getsockname()[1]
    sk.close()
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        c = layer("cap")
        cfg = dict(c.cfg, capacity_factor=0.8)
        T, H = 1500, c.wl.hidden
        h_d = dev_bf16(W.make_h(c.wl, T, seed=77))
        ws = moe.workspace(cfg, T)
        moe.moe_clear_device_status(ws)
        a = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        b = torch.empty_like(a)
        moe.moe_forward(cfg, h_d, c.wg_d, c.bias_d, c.w13_d, c.w2_d, c.w13s_d, c.w2s_d, a, ws)
        g, dropped = shard.forward_shard(cfg, h_d, c.wg_d, c.bias_d, c.w13_d, c.w2_d, c.w13s_d, c.w2s_d, b, ws)
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(ws) == 0
        assert g == T and int(dropped.cpu()[0]) > 0
        assert np.array_equal(host_bf16(a), host_bf16(b))
    finally:
        dist.destroy_process_group()
