"""Capacity across token shards: one exchange of N + 1 integers per shard.

A capacity-limited batch split across ranks in token order (rank 0 holds the
first tokens, rank 1 the next, ...) keeps the keep/drop decisions of the
unsharded batch — capacity filled in batch order ("Mixture-of-Experts Routing
at Inference Time", the capacity rule) — when every rank knows how many
routes each expert received on the ranks before it.  shard_exchange
all-gathers every rank's per-expert route counts (moe_routing_stats'
expert_load) together with its token count and sums them over the lower
ranks; integer sums, so every rank derives the same numbers.  The dispatch
itself runs in moe_dispatch_align_shard; this module is plumbing around
torch.distributed (gloo for CPU tensors, NCCL for device tensors).
"""
from __future__ import annotations


def shard_exchange(expert_load, tokens: int, group=None):
    """expert_load: int32 tensor [N] of this rank's routes per expert.
    Returns (expert_offset [N] int32 on expert_load's device: the routes each
    expert received on lower ranks, global_tokens: tokens of all ranks)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    n = expert_load.numel()
    mine = torch.empty(n + 1, dtype=torch.int64, device=expert_load.device)
    mine[:n] = expert_load.to(torch.int64)
    mine[n] = int(tokens)
    gathered = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(gathered, mine, group=group)
    offset = torch.zeros(n, dtype=torch.int64, device=expert_load.device)
    for q in range(rank):
        offset += gathered[q][:n]
    global_tokens = int(sum(int(g[n]) for g in gathered))
    return offset.to(torch.int32), global_tokens


def forward_shard(cfg, h, w_gate, router_bias, w13, w2, w13_shared, w2_shared, out, ws, group=None,
                  stream=None):
    """The layer forward on this rank's token shard of a capacity-limited
    batch: moe_route, moe_routing_stats (per-expert counts), shard_exchange,
    moe_dispatch_align_shard, moe_expert_ffn, moe_combine.  Returns
    (global_tokens, number of routes this shard dropped)."""
    import torch
    from . import (moe_route, moe_routing_stats, moe_dispatch_align_shard, moe_expert_ffn, moe_combine,
                   moe_max_padded_rows, moe_max_blocks)
    T, H = h.shape
    N, k = cfg["num_experts"], cfg["top_k"]
    d = h.device
    idx = torch.empty((T, k), dtype=torch.int32, device=d)
    gates = torch.empty((T, k), dtype=torch.float32, device=d)
    moe_route(cfg, h, w_gate, router_bias, idx, gates, None, ws, stream)
    load = torch.empty(N, dtype=torch.int32, device=d)
    stats = torch.empty(64, dtype=torch.uint8, device=d)
    moe_routing_stats(cfg, idx, 1.25, load, stats, stream)
    offset, global_tokens = shard_exchange(load, T, group)
    R = T * k
    rows, nblk = moe_max_padded_rows(cfg, T), moe_max_blocks(cfg, T)
    kept = torch.empty(R, dtype=torch.uint8, device=d)
    pos = torch.empty(R, dtype=torch.int32, device=d)
    srt = torch.empty(rows, dtype=torch.int32, device=d)
    blk = torch.empty(nblk, dtype=torch.int32, device=d)
    npad = torch.empty(1, dtype=torch.int32, device=d)
    counts = torch.empty(N, dtype=torch.int32, device=d)
    dropped = torch.empty(1, dtype=torch.int32, device=d)
    moe_dispatch_align_shard(cfg, global_tokens, idx, offset, kept, pos, srt, blk, npad, counts, dropped, ws,
                             stream)
    y = torch.empty((rows, H), dtype=torch.bfloat16, device=d)
    ysh = torch.empty((T, H), dtype=torch.bfloat16, device=d) if cfg.get("shared_intermediate", 0) else None
    moe_expert_ffn(cfg, h, w13, w2, w13_shared, w2_shared, srt, blk, npad, y, ysh, ws, stream)
    moe_combine(cfg, h, gates, kept, pos, y, ysh, out, stream)
    return global_tokens, dropped
