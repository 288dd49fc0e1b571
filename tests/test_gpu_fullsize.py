"""Full-size configurations, in the launch configuration bench.py times.

Routing and dispatch are compared bit for bit over every token (the oracle
does those cheaply); layer outputs are compared on chosen tokens, whose
oracle rows are computed one by one: every token with a route on the first
or last routed row of a 128- or 256-row GEMM tile, on the last row of an
expert segment, or in a tile of at most 32 routed rows (where the grouped
GEMMs' schedules change), plus a seeded random sample.  The DeepSeek-V3-like
layer runs the batch-invariance sweep: 64 probe tokens embedded among
0..16384 filler tokens at shuffled positions give bitwise the probes-alone
outputs, and fillers of the largest batch on tile edges match the oracle.
"""
import numpy as np
import pytest

from synth import workloads as W
from tests.checks import check_dispatch, check_equal, check_gates, check_outputs

pytestmark = pytest.mark.gpu

_cases = {}


def case(name):
    from tests.layer_case import LayerCase
    if name not in _cases:
        _cases.clear()
        import torch
        torch.cuda.empty_cache()
        _cases[name] = LayerCase(W.WORKLOADS[name])
    return _cases[name]


def _full_check(name, T, seed, n_sample=32, must_drop=False, edge_limit=None):
    from tests.layer_case import edge_tokens
    c = case(name)
    h = W.make_h(c.wl, T, seed)
    out = c.forward(h)
    got = c.stages(h)
    assert (got["out"] == out).all()          # stage-wise == fused forward, bitwise
    l, idx, gates, d = c.ref_routing(h)
    check_equal("logits", got["logits"].view(np.uint32), l.view(np.uint32))
    check_equal("topk_idx", got["topk_idx"], idx)
    check_gates(got["gates"], gates)
    check_dispatch(got, d)
    rng = np.random.default_rng(T + seed)
    edges = edge_tokens(d, T, c.wl.top_k, c.wl.block_size, limit=edge_limit, seed=seed)
    toks = np.union1d(np.sort(rng.choice(T, n_sample, replace=False)), edges)
    if must_drop:
        assert d["num_dropped"] > 0
        dropped = np.flatnonzero((d["route_kept"].reshape(T, -1) == 0).any(axis=1))
        toks = np.unique(np.concatenate([toks, dropped[:8], [0, T - 1]]))
    ref = c.ref_outputs(h, toks, idx, gates, d["route_kept"])
    return check_outputs(out[toks], ref), d


def test_mixtral_like_T4096_bench_batch():
    # the exact batch bench.py times (seed 0)
    _full_check("mix", 4096, 0)


def test_qwen_like_T8192():
    # ~600 tiles: a seeded 600 of their edge tokens, every segment's last route
    _full_check("qw", 8192, 0, edge_limit=600)


def test_capacity_T8192_drops_about_15_percent():
    _, d = _full_check("cap", 8192, 0, must_drop=True)
    frac = d["num_dropped"] / (8192 * 2)
    assert 0.12 < frac < 0.18


PROBE_FILLERS = [0, 1, 2, 3, 7, 15, 16, 17, 63, 64, 65, 127, 255, 256, 511, 1000, 1023, 1024, 2047,
                 4095, 4096, 8191, 8192, 16383, 16384]


def test_deepseek_like_probe_sweep():
    c = case("ds")
    wl = c.wl
    probes = W.make_h(wl, 64, seed=1)
    together = c.forward(probes)
    alone = np.stack([c.forward(probes[i:i + 1])[0] for i in range(64)])
    assert (together == alone).all()
    # parity of the probes against the oracle (routed + shared expert)
    l, idx, gates, d = c.ref_routing(probes)
    ref = c.ref_outputs(probes, np.arange(64), idx, gates, d["route_kept"])
    check_outputs(together, ref)
    for F in PROBE_FILLERS:
        fillers = W.make_h(wl, F, seed=1000 + F) if F else np.zeros((0, wl.hidden), np.uint16)
        for shuffle in (0, 1):
            T = 64 + F
            rng = np.random.default_rng(F * 2 + shuffle)
            pos = np.sort(rng.choice(T, 64, replace=False))
            perm = rng.permutation(64)
            batch = np.empty((T, wl.hidden), np.uint16)
            mask = np.zeros(T, bool)
            mask[pos] = True
            batch[pos] = probes[perm]
            batch[~mask] = fillers
            out = c.forward(batch)
            assert (out[pos] == alone[perm]).all(), f"F={F} shuffle={shuffle}"
    # fillers of the largest batch (the last one run) against the oracle:
    # routed on tile edges, segment tails and narrow tiles, plus a few at random
    from tests.layer_case import edge_tokens
    l, idx, gates, d = c.ref_routing(batch)
    fill = np.flatnonzero(~mask)
    edges = np.intersect1d(edge_tokens(d, T, wl.top_k, wl.block_size), fill)
    rng = np.random.default_rng(77)
    sel = np.union1d(rng.choice(edges, min(40, len(edges)), replace=False),
                     rng.choice(fill, 8, replace=False))
    assert len(sel) >= 32
    ref = c.ref_outputs(batch, sel, idx, gates, d["route_kept"])
    check_outputs(out[sel], ref)
