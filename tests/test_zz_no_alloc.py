"""moe_dispatch_align_noalloc: the dispatch for callers that cannot allocate.

Callers that cannot allocate device memory (a serving loop whose memory is
fixed at start-up, code running while another framework owns the allocator)
cannot pass a workspace; this entry point keeps its scratch in a fixed array
inside the library.  Its outputs must equal those of moe_dispatch_align, the
workspace version, bit for bit, on two calls in a row (the second call must
not see the first call's leftovers).  This file is collected last on purpose.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _routes(rng, T, N, k, skew):
    p = np.exp(-skew * np.log(np.arange(N) + 1.0))
    p /= p.sum()
    idx = np.empty((T, k), np.int32)
    for t in range(T):
        idx[t] = np.sort(rng.choice(N, size=k, replace=False, p=p))
    return idx


def _outputs(cfg, T, device):
    import torch
    import invariant_expert_routing_gb300 as moe
    R, N = T * cfg["top_k"], cfg["num_experts"]
    rows, nblk = moe.moe_max_padded_rows(cfg, T), moe.moe_max_blocks(cfg, T)
    return dict(route_kept=torch.full((R,), 7, dtype=torch.uint8, device=device),
                route_pos=torch.full((R,), -5, dtype=torch.int32, device=device),
                sorted_route_ids=torch.full((rows,), -5, dtype=torch.int32, device=device),
                block_expert=torch.full((nblk,), -5, dtype=torch.int32, device=device),
                num_padded=torch.full((1,), -5, dtype=torch.int32, device=device),
                expert_counts=torch.full((N,), -5, dtype=torch.int32, device=device),
                num_dropped=torch.full((1,), -5, dtype=torch.int32, device=device))


def _host(o):
    P = int(o["num_padded"].item())
    out = {k: v.cpu().numpy() for k, v in o.items()}
    out["sorted_route_ids"] = out["sorted_route_ids"][:P]
    return out


def test_noalloc_dispatch_matches_workspace_dispatch_twice_in_a_row():
    import torch
    import invariant_expert_routing_gb300 as moe
    dev = torch.device("cuda", torch.cuda.current_device())
    rng = np.random.default_rng(2024)
    calls = [  # (cfg, T, skew): a Qwen-like batch, then a capacity-limited skewed one
        (dict(hidden=2048, num_experts=128, top_k=8, intermediate=768, block_size=16), 4096, 0.0),
        (dict(hidden=4096, num_experts=8, top_k=2, intermediate=14336, block_size=64,
              capacity_factor=1.0), 3000, 1.2),
    ]
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    for cfg, T, skew in calls:
        idx = torch.from_numpy(_routes(rng, T, cfg["num_experts"], cfg["top_k"], skew)).to(dev)
        ws = moe.workspace(cfg, T, dev)
        ref = _outputs(cfg, T, dev)
        moe.moe_dispatch_align(cfg, idx, ref["route_kept"], ref["route_pos"], ref["sorted_route_ids"],
                               ref["block_expert"], ref["num_padded"], ref["expert_counts"],
                               ref["num_dropped"], ws)
        got = _outputs(cfg, T, dev)
        moe.moe_dispatch_align_noalloc(cfg, idx, got["route_kept"], got["route_pos"],
                                       got["sorted_route_ids"], got["block_expert"],
                                       got["num_padded"], got["expert_counts"], got["num_dropped"],
                                       status)
        torch.cuda.synchronize()
        a, b = _host(ref), _host(got)
        for key in a:
            assert np.array_equal(a[key], b[key]), key
        assert int(status.item()) == 0
    assert int(b["num_dropped"][0]) > 0   # the second call really overflowed capacity


def test_noalloc_reports_bad_expert_ids_and_rejects_oversize_batches():
    import torch
    import invariant_expert_routing_gb300 as moe
    dev = torch.device("cuda", torch.cuda.current_device())
    cfg = dict(hidden=128, num_experts=8, top_k=2, intermediate=256, block_size=8)
    idx = torch.tensor([[0, 3], [1, 9]], dtype=torch.int32, device=dev)
    o = _outputs(cfg, 2, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    moe.moe_dispatch_align_noalloc(cfg, idx, *o.values(), status)
    torch.cuda.synchronize()
    assert int(status.item()) & moe.MOE_DEV_ERR_EXPERT_RANGE
    assert o["route_kept"].cpu().tolist() == [1, 1, 1, 0]
    big = dict(cfg, num_experts=128, top_k=8)
    T = 65536 // 8 + 1
    idx = torch.zeros((T, 8), dtype=torch.int32, device=dev)
    o = _outputs(big, T, dev)
    with pytest.raises(moe.MoEError) as e:
        moe.moe_dispatch_align_noalloc(big, idx, *o.values(), status)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
