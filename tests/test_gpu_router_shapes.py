"""The chunked CUDA-core router on shapes the workloads do not cover.

The router's logits follow one order for every batch ("Why temperature=0
Still Gives Different Answers: Batch Invariance", a reduction cut into
constant 256-element pieces added in one order).  Its chunk-sum kernel maps
8, 16 or 32 experts to the lanes of a warp by N, copies W_g with 16-byte
pieces only when N is a multiple of 8, runs one token per thread for at most
64 tokens and four otherwise, and the last chunk of H may be shorter than 256.
Every one of those cases must give the oracle's logits bit for bit, and the
oracle's top-k indices exactly (lowest index on ties), through moe_route.
"""
import numpy as np
import pytest

import oracle
from synth import f32_to_bf16
from tests.checks import check_equal, check_gates

pytestmark = pytest.mark.gpu

# (N, H, k, T): N % 8 != 0 (scalar copies) and == 0, expert blocks of 8 / 16
# / 32 lanes with a partial last block, a partial last chunk of H, T on both
# sides of 64 with ragged token blocks, and k = 1.
CASES = [
    (5, 128, 2, 1), (5, 384, 2, 300), (12, 256, 3, 65), (12, 384, 3, 7),
    (40, 640, 4, 64), (40, 640, 4, 129), (200, 384, 8, 3), (200, 384, 8, 257),
    (8, 128, 1, 1000), (96, 1152, 6, 33),
    # every lane holding eight experts, and up to 16 selected (the top-k's
    # slot ballots over all eight groups of 32 experts)
    (256, 256, 16, 40), (256, 512, 12, 3), (17, 128, 16, 9),
]


def _inputs(N, H, T, seed, with_bias=True, zero_rows=()):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((T, H)).astype(np.float32)
    for t in zero_rows:
        if t < T:
            h[t] = 0.0   # every logit equals the bias: exact ties
    wg = (rng.standard_normal((H, N)) / np.sqrt(H)).astype(np.float32)
    bias = (0.1 * rng.standard_normal(N)).astype(np.float32) if with_bias else None
    return f32_to_bf16(h), f32_to_bf16(wg), bias


def _route(N, H, k, T, h, wg, bias):
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev, dev_bf16, host
    cfg = dict(hidden=H, num_experts=N, top_k=k, intermediate=128, block_size=8)
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    g = torch.empty((T, k), dtype=torch.float32, device="cuda")
    lg = torch.empty((T, N), dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, dev_bf16(h), dev_bf16(wg), None if bias is None else dev(bias), idx, g, lg, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    return host(idx), host(g), host(lg)


@pytest.mark.parametrize("N,H,k,T", CASES)
def test_chunked_router_matches_oracle(N, H, k, T):
    h, wg, bias = _inputs(N, H, T, seed=N * 1000 + T)
    idx, g, lg = _route(N, H, k, T, h, wg, bias)
    l_ref = oracle.router_logits(h, wg, bias)
    check_equal("logits", lg.view(np.uint32), l_ref.view(np.uint32))
    i_ref, g_ref = oracle.select_topk(l_ref, k)
    check_equal("topk_idx", idx, i_ref)
    check_gates(g, g_ref)


@pytest.mark.parametrize("N,T", [(5, 3), (40, 100), (200, 70)])
def test_chunked_router_ties_go_to_the_lowest_index(N, T):
    # tokens with h = 0 and no bias: all N logits are +0, the top-k is 0..k-1
    k = min(4, N)
    h, wg, _ = _inputs(N, 256, T, seed=7 + N, with_bias=False, zero_rows=range(0, T, 3))
    idx, g, lg = _route(N, 256, k, T, h, wg, None)
    l_ref = oracle.router_logits(h, wg, None)
    check_equal("logits", lg.view(np.uint32), l_ref.view(np.uint32))
    i_ref, _ = oracle.select_topk(l_ref, k)
    check_equal("topk_idx", idx, i_ref)
    for t in range(0, T, 3):
        assert list(idx[t]) == list(range(k))
        assert np.all(g[t] == np.float32(1.0 / k))
