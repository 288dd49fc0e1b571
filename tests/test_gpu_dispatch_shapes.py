"""Dispatch and alignment at expert counts and batch sizes the five workloads
do not reach.

The scan that turns per-tile expert counts into bases gives each of its
1024 threads one (part, expert) pair: expert counts that do not divide 1024,
a single expert, many route tiles per part (large batches), a few tiles and
a batch small enough for the one-CTA dispatch must all give the oracle's
integers bit for bit (keep mask, padded row of every route, sorted route ids,
block experts, per-expert counts, drops), with and without a capacity
("Mixture-of-Experts Routing at Inference Time", "The hard part: token
dropping is a silent correctness bug"; "Route-Block Membership Selects
Packed-AWQ Arithmetic", "The bookkeeping before the matrix multiplication").
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

CASES = [
    # N, k, B, T, capacity factor (0: no capacity)
    (1, 1, 8, 3000, 0.0),
    (5, 2, 16, 40000, 1.0),
    (37, 4, 32, 20000, 0.9),
    (96, 8, 16, 9000, 0.0),
    (200, 6, 64, 12000, 1.1),
    (256, 8, 16, 33000, 0.0),
    (200, 6, 64, 7, 1.0),
    (130, 3, 8, 1500, 0.8),
]


def _skewed_topk(rng, T, N, k):
    """k distinct experts per token, Zipf-skewed popularity (Gumbel top-k)."""
    p = 1.0 / np.arange(1, N + 1) ** 1.1
    rng.shuffle(p)
    keys = np.log(p)[None, :] + rng.gumbel(size=(T, N))
    return np.argsort(-keys, axis=1)[:, :k].astype(np.int32)


@pytest.mark.parametrize("N,k,B,T,cf", CASES)
def test_dispatch_matches_oracle(N, k, B, T, cf):
    import torch
    import invariant_expert_routing_gb300 as moe
    import oracle
    from tests.gpu_util import host
    cfg = dict(hidden=128, num_experts=N, top_k=k, intermediate=128, block_size=B, capacity_factor=cf)
    rng = np.random.default_rng(N * 1000 + T)
    idx = _skewed_topk(rng, T, N, k)
    R = T * k
    d = "cuda"
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    kept = torch.empty(R, dtype=torch.uint8, device=d)
    pos = torch.empty(R, dtype=torch.int32, device=d)
    srt = torch.full((moe.moe_max_padded_rows(cfg, T),), -9, dtype=torch.int32, device=d)
    blk = torch.full((moe.moe_max_blocks(cfg, T),), -9, dtype=torch.int32, device=d)
    npad = torch.zeros(1, dtype=torch.int32, device=d)
    counts = torch.empty(N, dtype=torch.int32, device=d)
    dropped = torch.zeros(1, dtype=torch.int32, device=d)
    moe.moe_dispatch_align(cfg, torch.from_numpy(idx).to(d), kept, pos, srt, blk, npad, counts, dropped, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    ref = oracle.dispatch(idx, N, B, oracle.capacity(T, N, k, cf))
    P = int(host(npad)[0])
    assert P == ref["num_padded"]
    assert np.array_equal(host(kept), ref["route_kept"])
    assert np.array_equal(host(pos), ref["route_pos"])
    assert np.array_equal(host(srt)[:P], ref["sorted_route_ids"])
    assert np.array_equal(host(blk)[:P // B], ref["block_expert"])
    assert np.array_equal(host(counts), ref["expert_counts"])
    assert int(host(dropped)[0]) == ref["num_dropped"]
    if cf > 0:
        assert ref["num_dropped"] > 0 or N == 1   # the capacity cases do drop routes
