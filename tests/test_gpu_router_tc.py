"""The tensor-core router with the certified candidate filter.

For N a multiple of 128 the fused forward (and moe_route without logits)
filters experts with tensor-core logits and recomputes canonical logits only
for the candidates.  Its top-k indices and gates must be bit-identical to the
CUDA-core router's, including exact ties (tokens with h = 0), near-tied
routers and adversarial experts whose columns differ in one element; and the
tensor-core logits must stay well inside the error bound the filter assumes.
"""
import numpy as np
import pytest

from synth import bf16_to_f32, f32_to_bf16
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _route_both(moe, cfg, h_d, wg_d, bias_d, ws, tc_flags=0):
    # with logits: the chunked CUDA-core router (every logit in the canonical
    # order); without: the tensor-core path, forced for any batch size
    # (tc_flags may add a forced token-tile height of its logits)
    import torch
    T, N, k = h_d.shape[0], cfg["num_experts"], cfg["top_k"]
    dev = h_d.device
    out = []
    for with_logits in (True, False):
        idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        g = torch.empty((T, k), dtype=torch.float32, device=dev)
        lg = torch.empty((T, N), dtype=torch.float32, device=dev) if with_logits else None
        flags = moe.MOE_DEBUG_ROUTER_CHUNKED if with_logits else moe.MOE_DEBUG_ROUTER_TC | tc_flags
        moe.moe_route(dict(cfg, debug_flags=flags), h_d, wg_d, bias_d, idx, g, lg, ws)
        out.append((idx, g, lg))
    torch.cuda.synchronize()
    return out


# (layer, T, forced tile height of the tensor-core logits: 0 = the default choice)
_TC_CASES = [("qw", 1, 0), ("qw", 65, 0), ("qw", 700, 0), ("qw", 8192, 0), ("ds", 5, 0), ("ds", 3000, 0),
             ("qw", 700, 128), ("qw", 8192, 128), ("ds", 3000, 128), ("ds", 10000, 0), ("qw", 20000, 0),
             ("qw", 8192, 64), ("ds", 10000, 64)]


@pytest.mark.parametrize("name,T,rows", _TC_CASES)
def test_tensor_core_router_matches_canonical_router(name, T, rows):
    # both router paths against each other bit for bit, and the tensor-core
    # path's top-k directly against the oracle's (indices bit for bit, gates
    # within the gate tolerance); T = 10000 (DeepSeek-like) and 20000
    # (Qwen-like) give every SM a 128-row tile, so the default takes the
    # 128-row logits there; smaller batches take 64-row tiles unless forced
    import torch
    import invariant_expert_routing_gb300 as moe
    import oracle
    from tests.checks import check_equal, check_gates
    from tests.gpu_util import dev, dev_bf16, host
    wl = W.WORKLOADS[name]
    cfg = wl.cfg
    h = W.make_h(wl, T, seed=31)
    wg, bias = W.make_router(wl)
    h_d, wg_d = dev_bf16(h), dev_bf16(wg)
    bias_d = None if bias is None else dev(bias)
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    tile = {0: 0, 128: moe.MOE_DEBUG_ROUTER_TILE128, 64: moe.MOE_DEBUG_ROUTER_TILE64}[rows]
    (i_c, g_c, l_c), (i_t, g_t, _) = _route_both(moe, cfg, h_d, wg_d, bias_d, ws, tile)
    assert torch.equal(i_c, i_t)
    assert torch.equal(g_c.view(torch.int32), g_t.view(torch.int32))
    # the oracle's routing of the same tokens
    l_ref = oracle.router_logits(h, wg, bias)
    idx_ref, g_ref = oracle.select_topk(l_ref, wl.top_k)
    check_equal("topk_idx (tensor-core path vs oracle)", host(i_t), idx_ref)
    check_gates(host(g_t), g_ref)
    # the tensor-core logits stay far inside the assumed bound
    ltc = torch.empty((T, wl.num_experts), dtype=torch.float32, device=h_d.device)
    moe.moe_router_tc_logits(dict(cfg, debug_flags=tile), h_d, wg_d, ltc, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    lc = l_c.double().cpu().numpy() - (0 if bias is None else bias.astype(np.float64))
    lt = ltc.double().cpu().numpy()
    hn = np.linalg.norm(bf16_to_f32(h).astype(np.float64), axis=1)
    wn = np.linalg.norm(bf16_to_f32(wg).astype(np.float64), axis=0).max()
    bound = moe.moe_router_cert_beta(wl.hidden) * hn * wn + 1e-30
    ratio = (np.abs(lt - lc).max(axis=1) / bound).max()
    assert ratio < 1.0 / 16, f"tensor-core error uses {ratio:.3g} of the certified bound"


def test_adversarial_near_identical_experts():
    # 256 experts whose router columns differ from expert 0 in a single
    # element: every logit is within a few ulps of the others, so almost all
    # experts are candidates and the canonical order decides the top-k.
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16
    H, N, k, T = 1024, 256, 8, 96
    cfg = dict(hidden=H, num_experts=N, top_k=k, intermediate=128, block_size=16)
    rng = np.random.default_rng(5)
    base = (rng.standard_normal(H) / np.sqrt(H)).astype(np.float32)
    wg = np.repeat(base[:, None], N, axis=1)
    for e in range(N):
        wg[rng.integers(H), e] *= np.float32(1.0 + 2.0 ** -7)
    wg_b = f32_to_bf16(wg)
    h = f32_to_bf16(rng.standard_normal((T, H)).astype(np.float32))
    h[:4] = 0
    ws = moe.workspace(cfg, T)
    (i_c, g_c, _), (i_t, g_t, _) = _route_both(moe, cfg, dev_bf16(h), dev_bf16(wg_b), None, ws)
    assert torch.equal(i_c, i_t)
    assert torch.equal(g_c.view(torch.int32), g_t.view(torch.int32))
    assert (i_t[:4].cpu().numpy() == np.arange(k)).all()   # exact ties: lowest indices


def test_candidate_tiles_mix_recompute_paths():
    # Tiles of 32 tokens where some tokens have a handful of candidates, some
    # between 17 and 32 (24 near-identical experts aligned with the token),
    # and some every expert (h = 0: exact ties, finished by the filter warp),
    # H with a 128-element last chunk, a ragged last tile, and random tokens
    # whose candidate union fills more than one staging pass.
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16
    H, N, k, T = 1152, 256, 8, 200
    cfg = dict(hidden=H, num_experts=N, top_k=k, intermediate=128, block_size=16)
    rng = np.random.default_rng(11)
    base = (rng.standard_normal(H) / np.sqrt(H)).astype(np.float32)
    wg = (0.3 * rng.standard_normal((H, N)) / np.sqrt(H)).astype(np.float32)
    near = rng.choice(N, 24, replace=False)
    for e in near:
        wg[:, e] = base
        wg[rng.integers(H), e] *= np.float32(1.0 + 2.0 ** -7)
    h = rng.standard_normal((T, H)).astype(np.float32)
    h[0::4] = 8.0 * base + 0.01 * rng.standard_normal((len(range(0, T, 4)), H)).astype(np.float32)
    h[6::16] = 0.0
    h_b, wg_b = f32_to_bf16(h), f32_to_bf16(wg)
    h_d, wg_d = dev_bf16(h_b), dev_bf16(wg_b)
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    (i_c, g_c, _), (i_t, g_t, _) = _route_both(moe, cfg, h_d, wg_d, None, ws)
    assert torch.equal(i_c, i_t)
    assert torch.equal(g_c.view(torch.int32), g_t.view(torch.int32))
    idx = torch.empty((T, k), dtype=torch.int32, device=h_d.device)
    g = torch.empty((T, k), dtype=torch.float32, device=h_d.device)
    nc = torch.empty(T, dtype=torch.int32, device=h_d.device)
    moe.moe_route_filtered(cfg, h_d, wg_d, None, idx, g, nc, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    assert torch.equal(idx, i_c)
    n = nc.cpu().numpy()
    assert (n[6::16] == N).all()                   # every expert: the filter warp finishes
    assert ((n > 16) & (n <= 32)).any()            # the tiled recompute with many candidates
    assert (n <= 12).sum() >= T // 4 and n.min() >= k   # and the usual few candidates
