"""One synthetic layer instance on the host and the device, and the oracle's
answer for any subset of its tokens.  Shared by the GPU tests, smoke and the
benchmark's full-size parity check (plumbing and bookkeeping only)."""
from __future__ import annotations

import numpy as np

import oracle
from synth import bf16_to_f32
from synth import workloads as W

from .gpu_util import dev, dev_bf16, host, host_bf16


class LayerCase:
    """Weights of workload `wl` (seed 0) resident on the device; routed expert
    weights are also kept on the host when small enough, else regenerated per
    expert for the oracle."""

    HOST_LIMIT = 3 << 30

    def __init__(self, wl: W.Workload, device="cuda", seed: int = 0):
        import torch
        self.wl, self.cfg, self.device, self.seed = wl, wl.cfg, device, seed
        self.wg, self.bias = W.make_router(wl, seed)
        self.wg_d = dev_bf16(self.wg, device)
        self.bias_d = None if self.bias is None else dev(self.bias, device)
        if wl.weight_bytes() <= self.HOST_LIMIT:
            self.w13, self.w2 = W.make_experts(wl, seed)
            self.w13_d, self.w2_d = dev_bf16(self.w13, device), dev_bf16(self.w2, device)
            self.w13s, self.w2s = W.make_shared(wl, seed)
            self.w13s_d = None if self.w13s is None else dev_bf16(self.w13s, device)
            self.w2s_d = None if self.w2s is None else dev_bf16(self.w2s, device)
        else:
            self.w13 = self.w2 = None
            self.w13_d, self.w2_d, self.w13s_d, self.w2s_d = W.make_experts_device(wl, seed, device)
            self.w13s, self.w2s = W.make_shared(wl, seed)
        torch.cuda.synchronize()

    # ---- device runs
    def forward(self, h_bits: np.ndarray, ws=None):
        import torch
        import invariant_expert_routing_gb300 as moe
        T = h_bits.shape[0]
        h_d = dev_bf16(h_bits, self.device)
        out = torch.empty((T, self.wl.hidden), dtype=torch.bfloat16, device=self.device)
        if ws is None:
            ws = moe.workspace(self.cfg, T, self.device)
        moe.moe_clear_device_status(ws)
        moe.moe_forward(self.cfg, h_d, self.wg_d, self.bias_d, self.w13_d, self.w2_d,
                        self.w13s_d, self.w2s_d, out, ws)
        torch.cuda.synchronize()
        status = moe.moe_get_device_status(ws)
        assert status == 0, f"device status {status:#x}"
        return host_bf16(out)

    def stages(self, h_bits: np.ndarray, topk_override=None):
        """Runs the four stage entry points; returns every intermediate."""
        import torch
        import invariant_expert_routing_gb300 as moe
        wl, d = self.wl, self.device
        T, N, k = h_bits.shape[0], wl.num_experts, wl.top_k
        R = T * k
        h_d = dev_bf16(h_bits, d)
        ws = moe.workspace(self.cfg, T, d)
        moe.moe_clear_device_status(ws)
        idx = torch.empty((T, k), dtype=torch.int32, device=d)
        gates = torch.empty((T, k), dtype=torch.float32, device=d)
        logits = torch.empty((T, N), dtype=torch.float32, device=d)
        moe.moe_route(self.cfg, h_d, self.wg_d, self.bias_d, idx, gates, logits, ws)
        if topk_override is not None:
            idx = dev(np.ascontiguousarray(topk_override, dtype=np.int32), d)
        rows = moe.moe_max_padded_rows(self.cfg, T)
        nblk = moe.moe_max_blocks(self.cfg, T)
        kept = torch.empty(R, dtype=torch.uint8, device=d)
        pos = torch.empty(R, dtype=torch.int32, device=d)
        srt = torch.full((rows,), -9, dtype=torch.int32, device=d)
        blk = torch.full((nblk,), -9, dtype=torch.int32, device=d)
        npad = torch.zeros(1, dtype=torch.int32, device=d)
        counts = torch.empty(N, dtype=torch.int32, device=d)
        dropped = torch.zeros(1, dtype=torch.int32, device=d)
        moe.moe_dispatch_align(self.cfg, idx, kept, pos, srt, blk, npad, counts, dropped, ws)
        y = torch.zeros((rows, wl.hidden), dtype=torch.bfloat16, device=d)
        ysh = (torch.zeros((T, wl.hidden), dtype=torch.bfloat16, device=d)
               if wl.shared_intermediate else None)
        moe.moe_expert_ffn(self.cfg, h_d, self.w13_d, self.w2_d, self.w13s_d, self.w2s_d, srt, blk,
                           npad, y, ysh, ws)
        out = torch.empty((T, wl.hidden), dtype=torch.bfloat16, device=d)
        moe.moe_combine(self.cfg, h_d, gates, kept, pos, y, ysh, out)
        torch.cuda.synchronize()
        status = moe.moe_get_device_status(ws)
        P = int(host(npad)[0])
        B = wl.block_size
        return dict(logits=host(logits), topk_idx=host(idx), gates=host(gates),
                    route_kept=host(kept), route_pos=host(pos), sorted_route_ids=host(srt)[:P],
                    block_expert=host(blk)[:P // B], num_padded=P, expert_counts=host(counts),
                    num_dropped=int(host(dropped)[0]), y_perm=bf16_to_f32(host_bf16(y))[:P],
                    y_shared=None if ysh is None else bf16_to_f32(host_bf16(ysh)), out=host_bf16(out),
                    status=status)

    # ---- oracle
    def ref_routing(self, h_bits: np.ndarray):
        l = oracle.router_logits(h_bits, self.wg, self.bias)
        idx, gates = oracle.select_topk(l, self.wl.top_k)
        T = h_bits.shape[0]
        cap = oracle.capacity(T, self.wl.num_experts, self.wl.top_k, self.wl.capacity_factor)
        d = oracle.dispatch(idx, self.wl.num_experts, self.wl.block_size, cap)
        return l, idx, gates, d

    def ref_expert_rows(self, h_bits, tokens, experts) -> np.ndarray:
        """fp64 expert outputs of (token, expert) pairs."""
        tokens = np.asarray(tokens, np.int32)
        experts = np.asarray(experts, np.int32)
        H = self.wl.hidden
        y = np.zeros((len(tokens), H))
        if len(tokens) == 0:
            return y
        if self.w13 is not None:
            return oracle.expert_rows(tokens, experts, h_bits, self.w13, self.w2)
        for e in np.unique(experts):
            sel = np.flatnonzero(experts == e)
            w13 = W.expert_w13(self.wl, int(e), self.seed)[None]
            w2 = W.expert_w2(self.wl, int(e), self.seed)[None]
            y[sel] = oracle.expert_rows(tokens[sel], np.zeros(len(sel), np.int32), h_bits, w13, w2)
        return y

    def ref_outputs(self, h_bits, tokens, idx, gates, route_kept) -> np.ndarray:
        """Oracle layer output (bf16 bits) for the listed tokens of a batch
        whose routing is (idx, gates, route_kept)."""
        tokens = np.asarray(tokens, np.int32)
        k, H = self.wl.top_k, self.wl.hidden
        pairs_t = np.repeat(tokens, k)
        pairs_e = idx[tokens].reshape(-1)
        keep = route_kept.reshape(-1, k)[tokens].reshape(-1).astype(bool)
        y = np.zeros((len(pairs_t), H))
        y[keep] = self.ref_expert_rows(h_bits, pairs_t[keep], pairs_e[keep])
        ysh = None
        if self.wl.shared_intermediate:
            ysh = oracle.expert_rows(tokens, np.zeros(len(tokens), np.int32), h_bits,
                                     self.w13s[None], self.w2s[None])
        return oracle.combine_rows(tokens, h_bits, gates, route_kept, y.reshape(len(tokens), k, H),
                                   ysh)


def edge_tokens(d: dict, T: int, k: int, B: int, tile_rows=(128, 256), small_rows: int = 32,
                limit: int | None = None, seed: int = 0) -> np.ndarray:
    """Tokens whose routes sit where the grouped GEMMs' schedules change: the
    first and last routed row of every tile of each expert segment (tiles of
    each size in tile_rows, cut from the segment's start), the last route of
    every segment, and every route of a tile with at most small_rows routed
    rows (those run the narrow MMA).  From the oracle's dispatch d (block size
    B).  With limit, a seeded subset of at most that many tokens that always
    keeps every segment's last route."""
    counts = np.asarray(d["expert_counts"], np.int64)
    srt = np.asarray(d["sorted_route_ids"], np.int64)
    pads = (counts + B - 1) // B * B
    starts = np.concatenate([[0], np.cumsum(pads)[:-1]])
    must, rows = set(), set()
    for e in np.flatnonzero(counts > 0):
        s0, cnt = int(starts[e]), int(counts[e])
        must.add(s0 + cnt - 1)
        for tr in tile_rows:
            for m in range(0, cnt, tr):
                valid = min(cnt - m, tr)
                rows.update((s0 + m, s0 + m + valid - 1))
                if valid <= small_rows:
                    rows.update(range(s0 + m, s0 + m + valid))
    sentinel = T * k
    keep = {int(srt[r]) // k for r in must if srt[r] != sentinel}
    rest = sorted({int(srt[r]) // k for r in rows if srt[r] != sentinel} - keep)
    if limit is not None and len(keep) + len(rest) > limit:
        n = max(0, limit - len(keep))
        rng = np.random.default_rng(seed)
        rest = [int(x) for x in rng.choice(rest, min(n, len(rest)), replace=False)] if n else []
    return np.array(sorted(keep.union(rest)), np.int64)
