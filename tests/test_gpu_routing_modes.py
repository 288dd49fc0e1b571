"""GPU parity of the overflow reroute policy, the routing diagnostics and
expert-choice routing, through the C ABI, against the CPU oracle.

Integer results (reroute assignments, layouts, expert-choice selections,
routing_stats counts) must match bit for bit; the fp64 diagnostics (imbalance
ratio, drop fraction, router margin) too, since both sides make the same IEEE
operations on the same inputs; gates and layer outputs within the tolerances
of tests/checks.py.
"""
import numpy as np
import pytest

import oracle
from synth import workloads as W
from tests.checks import check_dispatch, check_equal, check_gates, check_outputs

pytestmark = pytest.mark.gpu

_cases = {}


def case(name):
    from tests.layer_case import LayerCase
    if name not in _cases:
        _cases.clear()
        _cases[name] = LayerCase(W.WORKLOADS[name])
    return _cases[name]


def _logits_and_topk(moe, cfg, c, h_d, ws):
    import torch
    T, N, k = h_d.shape[0], cfg["num_experts"], cfg["top_k"]
    idx = torch.empty((T, k), dtype=torch.int32, device=h_d.device)
    g = torch.empty((T, k), dtype=torch.float32, device=h_d.device)
    lg = torch.empty((T, N), dtype=torch.float32, device=h_d.device)
    moe.moe_route(cfg, h_d, c.wg_d, c.bias_d, idx, g, lg, ws)
    lg2 = torch.empty_like(lg)
    moe.moe_router_logits(cfg, h_d, c.wg_d, c.bias_d, lg2, ws)
    torch.cuda.synchronize()
    assert torch.equal(lg.view(torch.int32), lg2.view(torch.int32))
    return idx, g, lg


def _reroute_on_gpu(moe, cfg, idx, lg, ws):
    import torch
    from tests.gpu_util import host
    T, k = idx.shape
    N = cfg["num_experts"]
    d = idx.device
    R = T * k
    rows, nblk = moe.moe_max_padded_rows(cfg, T), moe.moe_max_blocks(cfg, T)
    kept = torch.empty(R, dtype=torch.uint8, device=d)
    rexp = torch.full((R,), -9, dtype=torch.int32, device=d)
    pos = torch.empty(R, dtype=torch.int32, device=d)
    srt = torch.full((rows,), -9, dtype=torch.int32, device=d)
    blk = torch.full((nblk,), -9, dtype=torch.int32, device=d)
    npad = torch.zeros(1, dtype=torch.int32, device=d)
    counts = torch.empty(N, dtype=torch.int32, device=d)
    nd = torch.full((1,), -1, dtype=torch.int32, device=d)
    nr = torch.full((1,), -1, dtype=torch.int32, device=d)
    moe.moe_dispatch_align_reroute(cfg, idx, lg, kept, rexp, pos, srt, blk, npad, counts, nd, nr, ws)
    torch.cuda.synchronize()
    P = int(host(npad)[0])
    B = cfg["block_size"]
    return dict(route_kept=host(kept), route_expert=host(rexp), route_pos=host(pos),
                sorted_route_ids=host(srt)[:P], block_expert=host(blk)[:P // B], num_padded=P,
                expert_counts=host(counts), num_dropped=int(host(nd)[0]),
                num_rerouted=int(host(nr)[0]))


def _ref_reroute(l, idx, N, B, cap):
    re, nr, nd = oracle.reroute(l, idx, cap)
    d = oracle.dispatch_routes(re, N, B, idx.shape[1])
    d["num_dropped"] = nd
    return re, nr, d


REROUTE_CASES = [("tiny", 64, 0.5), ("tiny", 61, 0.75), ("tiny", 1, 0.5), ("cap", 8192, 1.0),
                 ("cap", 2000, 0.8), ("qw", 512, 1.0), ("qw", 8192, 1.0), ("qw", 777, 0.6),
                 ("ds", 200, 1.0), ("mix", 128, 4.0)]


@pytest.mark.parametrize("name,T,cf", REROUTE_CASES)
def test_reroute_dispatch_is_bit_exact(name, T, cf, extra=None):
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16, host
    c = case(name)
    cfg = dict(c.cfg, capacity_factor=cf, overflow_policy=1, **(extra or {}))
    N, k, B = cfg["num_experts"], cfg["top_k"], cfg["block_size"]
    h = W.make_h(c.wl, T, seed=21)
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    idx, _, lg = _logits_and_topk(moe, cfg, c, dev_bf16(h), ws)
    l_ref = oracle.router_logits(h, c.wg, c.bias)
    check_equal("logits", host(lg).view(np.uint32), l_ref.view(np.uint32))
    idx_ref, _ = oracle.select_topk(l_ref, k)
    check_equal("topk_idx", host(idx), idx_ref)
    got = _reroute_on_gpu(moe, cfg, idx, lg, ws)
    assert moe.moe_get_device_status(ws) == 0
    cap = oracle.capacity(T, N, k, cf)
    re, nr, d = _ref_reroute(l_ref, idx_ref, N, B, cap)
    check_equal("route_expert", got["route_expert"], re)
    assert got["num_rerouted"] == nr
    check_dispatch(got, d)
    if name in ("cap", "qw") and cf <= 1.0:
        assert nr > 0                 # the case exercises the reroute phase


def test_reroute_without_capacity_keeps_every_route():
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16, host
    c = case("tiny")
    cfg = dict(c.cfg, capacity_factor=0.0, overflow_policy=1)
    h = W.make_h(c.wl, 50, seed=2)
    ws = moe.workspace(cfg, 50)
    idx, _, lg = _logits_and_topk(moe, cfg, c, dev_bf16(h), ws)
    got = _reroute_on_gpu(moe, cfg, idx, lg, ws)
    assert (got["route_expert"] == host(idx).reshape(-1)).all()
    assert got["num_rerouted"] == 0 and got["num_dropped"] == 0
    assert got["route_kept"].all()
    del torch


@pytest.mark.parametrize("name,T,cf", [("tiny", 64, 0.9), ("cap", 2048, 1.0), ("qw", 512, 0.8)])
def test_reroute_forward_matches_oracle(name, T, cf):
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16, host_bf16
    c = case(name)
    cfg = dict(c.cfg, capacity_factor=cf, overflow_policy=1)
    N, k, B = cfg["num_experts"], cfg["top_k"], cfg["block_size"]
    h = W.make_h(c.wl, T, seed=4)
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    out = torch.empty((T, c.wl.hidden), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(cfg, dev_bf16(h), c.wg_d, c.bias_d, c.w13_d, c.w2_d, c.w13s_d, c.w2s_d, out, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    got = host_bf16(out)
    l = oracle.router_logits(h, c.wg, c.bias)
    idx, gates = oracle.select_topk(l, k)
    re, nr, nd = oracle.reroute(l, idx, oracle.capacity(T, N, k, cf))
    assert nr > 0
    moved = np.flatnonzero((re >= 0) & (re != idx.reshape(-1)))
    rng = np.random.default_rng(T)
    toks = np.unique(np.concatenate([moved[:24] // k, rng.choice(T, 16, replace=False)]))
    # the oracle's layer output for those tokens: expert per route from the
    # reroute, the slot's gate, kept iff the route has an expert
    kept = (re >= 0).astype(np.uint8)
    pairs_t = np.repeat(toks, k)
    pairs_r = (toks[:, None] * k + np.arange(k)[None, :]).reshape(-1)
    use = kept[pairs_r].astype(bool)
    y = np.zeros((len(pairs_t), c.wl.hidden))
    y[use] = c.ref_expert_rows(h, pairs_t[use], re[pairs_r][use])
    ref = oracle.combine_rows(toks, h, gates, kept, y.reshape(len(toks), k, c.wl.hidden))
    check_outputs(got[toks], ref)
    if name == "tiny":
        full = oracle.moe_forward(cfg, h, c.wg, c.bias, c.w13, c.w2)
        check_outputs(got, full)


@pytest.mark.parametrize("name,T,cf", [("mix", 4096, 1.25), ("qw", 8192, 1.25), ("cap", 8192, 1.0),
                                       ("ds", 333, 1.0), ("tiny", 1, 1.25)])
def test_routing_stats_bit_exact(name, T, cf):
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev, host
    c = case(name)
    N, k = c.wl.num_experts, c.wl.top_k
    h = W.make_h(c.wl, T, seed=6)
    idx, _ = oracle.select_topk(oracle.router_logits(h, c.wg, c.bias), k)
    load = torch.full((N,), -1, dtype=torch.int32, device="cuda")
    raw = torch.zeros(64, dtype=torch.uint8, device="cuda")
    moe.moe_routing_stats(c.cfg, dev(idx), cf, load, raw)
    torch.cuda.synchronize()
    got = moe.route_stats_from_bytes(host(raw).tobytes())
    ref_load, ref = oracle.routing_stats(idx, N, cf)
    check_equal("expert_load", host(load), ref_load)
    for key in ("max_expert_load", "min_expert_load", "capacity", "dropped_tokens", "total_routes"):
        assert got[key] == ref[key], key
    for key in ("imbalance_ratio", "drop_fraction"):
        assert np.float64(got[key]).tobytes() == np.float64(ref[key]).tobytes(), key


@pytest.mark.parametrize("name,T", [("qw", 8192), ("mix", 4096), ("tiny", 64), ("ds", 100)])
def test_router_margin_bit_exact(name, T):
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev, host
    c = case(name)
    k = c.wl.top_k
    h = W.make_h(c.wl, T, seed=7)
    l = oracle.router_logits(h, c.wg, c.bias)
    ref = oracle.router_margin(l, k)
    m = torch.empty(T, dtype=torch.float64, device="cuda")
    moe.moe_router_margin(c.cfg, dev(l), m)
    torch.cuda.synchronize()
    check_equal("margin", host(m).view(np.uint64), ref.view(np.uint64))
    if name == "qw":
        assert (ref == 0).sum() > 0       # the zero tokens tie exactly at the cut


def test_router_margin_special_values():
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev, host
    rng = np.random.default_rng(1)
    N = 40
    l = rng.standard_normal((12, N)).astype(np.float32)
    l[0, 5] = np.nan
    l[1, :] = 1.0                     # all tied
    l[2, :3] = np.inf
    l[3, :] = np.nan
    l[4, 7] = -0.0
    l[4, 8] = 0.0
    for n, k in ((N, 1), (N, 3), (N, 16), (16, 16)):       # k = N: margin +inf
        cfg = dict(hidden=128, num_experts=n, top_k=k, intermediate=128, block_size=8)
        ln = np.ascontiguousarray(l[:, :n])
        m = torch.empty(12, dtype=torch.float64, device="cuda")
        moe.moe_router_margin(cfg, dev(ln), m)
        torch.cuda.synchronize()
        ref = oracle.router_margin(ln, k)
        got = host(m)
        # a NaN result (inf - inf, NaN logits) is a NaN on both sides; its sign
        # and payload are the hardware's choice
        nan = np.isnan(ref)
        assert (np.isnan(got) == nan).all()
        check_equal(f"margin k={k}", got[~nan].view(np.uint64), ref[~nan].view(np.uint64))


def _ec_on_gpu(moe, cfg, lg, ws):
    import torch
    from tests.gpu_util import host
    T, N = lg.shape
    d = lg.device
    R = T * N
    rows, nblk = moe.moe_max_padded_rows(cfg, T), moe.moe_max_blocks(cfg, T)
    gates = torch.empty(R, dtype=torch.float32, device=d)
    kept = torch.empty(R, dtype=torch.uint8, device=d)
    pos = torch.empty(R, dtype=torch.int32, device=d)
    srt = torch.full((rows,), -9, dtype=torch.int32, device=d)
    blk = torch.full((nblk,), -9, dtype=torch.int32, device=d)
    npad = torch.zeros(1, dtype=torch.int32, device=d)
    counts = torch.empty(N, dtype=torch.int32, device=d)
    moe.moe_route_expert_choice(cfg, lg, gates, kept, pos, srt, blk, npad, counts, ws)
    torch.cuda.synchronize()
    P = int(host(npad)[0])
    B = cfg["block_size"]
    return dict(gates=host(gates), route_kept=host(kept), route_pos=host(pos),
                sorted_route_ids=host(srt)[:P], block_expert=host(blk)[:P // B], num_padded=P,
                expert_counts=host(counts), num_dropped=0)


EC_CASES = [("tiny", 64, 0.0), ("tiny", 3, 0.0), ("tiny", 61, 1.5), ("mix", 128, 1.0),
            ("mix", 4096, 1.0), ("qw", 512, 1.0), ("qw", 8192, 1.25), ("ds", 300, 1.0),
            ("cap", 1000, 1.0)]


@pytest.mark.parametrize("name,T,cf", EC_CASES)
def test_expert_choice_selection_is_bit_exact(name, T, cf):
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16
    c = case(name)
    cfg = dict(c.cfg, capacity_factor=cf, routing=1)
    N, k, B = cfg["num_experts"], cfg["top_k"], cfg["block_size"]
    h = W.make_h(c.wl, T, seed=13)
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    import torch
    lg = torch.empty((T, N), dtype=torch.float32, device="cuda")
    moe.moe_router_logits(cfg, dev_bf16(h), c.wg_d, c.bias_d, lg, ws)
    got = _ec_on_gpu(moe, cfg, lg, ws)
    assert moe.moe_get_device_status(ws) == 0
    l = oracle.router_logits(h, c.wg, c.bias)
    C = oracle.ec_capacity(T, N, k, cf)
    sel, probs = oracle.expert_choice(l, C)
    re = np.where(sel.reshape(-1) == 1, np.tile(np.arange(N), T), -1).astype(np.int32)
    d = oracle.dispatch_routes(re, N, B, N)
    check_dispatch(got, d)
    assert (got["expert_counts"] == C).all()
    check_gates(got["gates"], probs.reshape(-1))


@pytest.mark.parametrize("name,T", [("tiny", 64), ("mix", 256), ("qw", 512), ("ds", 40)])
def test_expert_choice_forward_matches_oracle(name, T):
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16, host_bf16
    c = case(name)
    cfg = dict(c.cfg, capacity_factor=0.0, routing=1)
    N, k = cfg["num_experts"], cfg["top_k"]
    h = W.make_h(c.wl, T, seed=17)
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    out = torch.empty((T, c.wl.hidden), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(cfg, dev_bf16(h), c.wg_d, c.bias_d, c.w13_d, c.w2_d, c.w13s_d, c.w2s_d, out, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    got = host_bf16(out)
    l = oracle.router_logits(h, c.wg, c.bias)
    sel, probs = oracle.expert_choice(l, oracle.ec_capacity(T, N, k, 0.0))
    rng = np.random.default_rng(T)
    n_sample = 6 if c.w13 is None else 24       # host-regenerated experts are slow
    toks = np.arange(T) if T <= n_sample else np.sort(rng.choice(T, n_sample, replace=False))
    # include tokens no expert took (they get h plus the shared expert only)
    none = np.flatnonzero(sel.sum(axis=1) == 0)
    toks = np.unique(np.concatenate([toks, none[:4]])).astype(np.int32)
    pairs_t = np.repeat(toks, N)
    pairs_e = np.tile(np.arange(N, dtype=np.int32), len(toks))
    use = sel[toks].reshape(-1).astype(bool)
    y = np.zeros((len(pairs_t), c.wl.hidden))
    y[use] = c.ref_expert_rows(h, pairs_t[use], pairs_e[use])
    ysh = None
    if c.wl.shared_intermediate:
        ysh = oracle.expert_rows(toks, np.zeros(len(toks), np.int32), h, c.w13s[None], c.w2s[None])
    ref = oracle.combine_rows(toks, h, probs, sel.reshape(-1), y.reshape(len(toks), N, c.wl.hidden),
                              ysh)
    check_outputs(got[toks], ref)
    if name == "tiny":
        check_outputs(got, oracle.moe_forward(cfg, h, c.wg, c.bias, c.w13, c.w2))


def test_expert_choice_ties_go_to_the_lowest_token():
    # identical token rows: every expert takes the first C of them
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16, host
    c = case("qw")
    cfg = dict(c.cfg, capacity_factor=1.0, routing=1)
    T, N = 300, c.wl.num_experts
    h = np.tile(W.make_h(c.wl, 1, seed=3), (T, 1))
    ws = moe.workspace(cfg, T)
    lg = torch.empty((T, N), dtype=torch.float32, device="cuda")
    moe.moe_router_logits(cfg, dev_bf16(h), c.wg_d, c.bias_d, lg, ws)
    got = _ec_on_gpu(moe, cfg, lg, ws)
    C = oracle.ec_capacity(T, N, c.wl.top_k, 1.0)
    kept = got["route_kept"].reshape(T, N)
    assert (kept[:C] == 1).all() and not kept[C:].any()
    del host


_FORCED_PATHS = {
    # the sequential kernel (the fallback of the deferred-acceptance rounds) alone
    "sequential": (dict(debug_flags=0x20),        # MOE_DEBUG_REROUTE_SEQUENTIAL
                   [("tiny", 61, 0.75), ("cap", 2000, 0.8), ("qw", 777, 0.6)], []),
    # the grid-wide rounds on small batches (one list tile, ragged tails)
    "grid": (dict(debug_flags=0x40),                    # MOE_DEBUG_REROUTE_GRID
             [("tiny", 61, 0.75), ("tiny", 1, 0.5), ("cap", 2000, 0.8), ("qw", 777, 0.6), ("ds", 200, 1.0)],
             [(200, 8, 2, 0.7), (300, 32, 4, 0.8), (129, 256, 8, 1.0)]),
    # the grid-wide rounds with several 1024-route chunks per CTA
    "grid_chunks": (dict(debug_flags=0x40, debug_grid_ctas=12),
                    [("qw", 777, 0.6), ("cap", 8192, 1.0), ("qw", 8192, 1.0)], []),
    # the one-CTA rounds on batches that default to the grid
    "cta": (dict(debug_flags=0x80), [                   # MOE_DEBUG_REROUTE_ONE_CTA
        ("cap", 8192, 1.0), ("qw", 8192, 1.0)], []),
}


@pytest.mark.parametrize("path", sorted(_FORCED_PATHS))
def test_reroute_forced_path_is_bit_exact(path):
    # each way of computing the reroute on its own, selected by the
    # configuration's path flags (MOE_DEBUG_REROUTE_*)
    extra, cases, nan_cases = _FORCED_PATHS[path]
    for name, T, cf in cases:
        test_reroute_dispatch_is_bit_exact(name, T, cf, extra)
    for args in nan_cases:
        test_reroute_with_nan_and_tied_logits(*args, extra=extra)


def _nan_logits(rng, T, N, ties=True):
    l = (rng.standard_normal((T, N)) - 1.2 * np.log(np.arange(N) + 1.0)).astype(np.float32)
    if ties:
        l[::5] = np.round(l[::5])          # exact ties inside a token
        l[7] = l[3]                        # two identical tokens
    l[2, 1] = np.nan
    l[9, :] = np.nan                       # a token of NaN logits
    l[11, 0] = -np.inf
    return l


@pytest.mark.parametrize("T,N,k,cf", [(200, 8, 2, 0.7), (300, 32, 4, 0.8), (129, 256, 8, 1.0)])
def test_reroute_with_nan_and_tied_logits(T, N, k, cf, extra=None):
    # crafted logits (NaN, -inf, exact ties) fed straight to the reroute
    # dispatch: NaN ranks last, ties go to the lower index, on both sides
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev
    rng = np.random.default_rng(T + N)
    l = _nan_logits(rng, T, N)
    idx, _ = oracle.select_topk(l, k)
    cfg = dict(hidden=128, num_experts=N, top_k=k, intermediate=128, block_size=8,
               capacity_factor=cf, overflow_policy=1, **(extra or {}))
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)
    got = _reroute_on_gpu(moe, cfg, dev(idx), dev(l), ws)
    assert moe.moe_get_device_status(ws) == 0
    re, nr, d = _ref_reroute(l, idx, N, 8, oracle.capacity(T, N, k, cf))
    check_equal("route_expert", got["route_expert"], re)
    assert got["num_rerouted"] == nr and nr > 0
    check_dispatch(got, d)
    del torch


@pytest.mark.parametrize("T,N,cf", [(100, 8, 1.0), (257, 64, 0.5), (40, 256, 2.0)])
def test_expert_choice_with_nan_and_tied_logits(T, N, cf):
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev
    rng = np.random.default_rng(T * N)
    l = _nan_logits(rng, T, N)
    cfg = dict(hidden=128, num_experts=N, top_k=2, intermediate=128, block_size=8,
               capacity_factor=cf, routing=1)
    ws = moe.workspace(cfg, T)
    got = _ec_on_gpu(moe, cfg, dev(l), ws)
    C = oracle.ec_capacity(T, N, 2, cf)
    sel, probs = oracle.expert_choice(l, C)
    re = np.where(sel.reshape(-1) == 1, np.tile(np.arange(N), T), -1).astype(np.int32)
    check_dispatch(got, oracle.dispatch_routes(re, N, 8, N))
    ok = ~np.isnan(probs.reshape(-1))
    check_gates(got["gates"][ok], probs.reshape(-1)[ok])
    assert np.isnan(got["gates"][~ok]).all()
    del torch


@pytest.mark.parametrize("T", [1, 2, 640])
def test_timed_and_host_buffer_forwards_give_the_same_bits(T):
    # moe_forward_timed and moe_forward_hostio run the same launches as
    # moe_forward: identical outputs, bit for bit (T <= 2: the decode front)
    import torch
    import invariant_expert_routing_gb300 as moe
    from tests.gpu_util import dev_bf16, host_bf16
    c = case("mix")
    h = W.make_h(c.wl, T, seed=27)
    h_d = dev_bf16(h)
    ws = moe.workspace(c.cfg, T)
    out = torch.empty((T, c.wl.hidden), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(c.cfg, h_d, c.wg_d, c.bias_d, c.w13_d, c.w2_d, None, None, out, ws)
    ref = host_bf16(out)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
    for e in ev:
        e.record()
    out2 = torch.empty_like(out)
    moe.moe_forward_timed(c.cfg, h_d, c.wg_d, c.bias_d, c.w13_d, c.w2_d, None, None, out2, ws, ev)
    h_host = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).pin_memory()
    out_host = torch.empty((T, c.wl.hidden), dtype=torch.bfloat16).pin_memory()
    moe.moe_forward_hostio(c.cfg, h_host, c.wg_d, c.bias_d, c.w13_d, c.w2_d, None, None, out_host, ws)
    torch.cuda.synchronize()
    assert (host_bf16(out2) == ref).all()
    assert (host_bf16(out_host) == ref).all()
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(7)]
    assert all(t >= 0 for t in times) and times[3] > 0      # the W13 stage took time
