"""The C-ABI library: loads, exports every declared symbol, validates on the host.

No compute call is made here (no GPU in this environment): only entry points
and argument checks that return before any launch.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_api.h")


@pytest.fixture(scope="module")
def moe():
    lib = os.path.join(ROOT, "invariant_expert_routing_gb300", "libmoe_gb300.so")
    if not os.path.exists(lib):
        import __graft_entry__
        __graft_entry__._build_module().build()
    import invariant_expert_routing_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)) - {"moe_config", "moe_status"})


def test_every_declared_symbol_is_exported(moe):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(moe._lib, n), n
        assert n in moe.EXPORTED, n


def test_status_strings(moe):
    for code in range(6):
        assert moe._lib.moe_status_string(code)


TINY = dict(hidden=128, num_experts=8, top_k=2, intermediate=256, block_size=8)


@pytest.mark.parametrize("bad,code", [
    (dict(hidden=100), 2), (dict(hidden=0), 1), (dict(intermediate=200), 2),
    (dict(num_experts=300), 2), (dict(top_k=9), 2), (dict(top_k=17, num_experts=32), 2),
    (dict(block_size=12), 2), (dict(block_size=256), 2), (dict(block_size=24), 2),
    (dict(shared_intermediate=100), 2), (dict(shared_intermediate=-128), 1),
    (dict(capacity_factor=float("nan")), 1)])
def test_config_validation(moe, bad, code):
    cfg = dict(TINY, **bad)
    assert moe.moe_check_config(cfg) == code


@pytest.mark.parametrize("bad", [
    dict(debug_flags=0x4000),                # unknown bit
    dict(debug_flags=0x1 | 0x2),             # tensor-core and chunked router at once
    dict(debug_flags=0x4 | 0x8),             # gather and scatter row copy at once
    dict(debug_flags=0x40 | 0x80),           # grid and one-CTA reroute rounds at once
    dict(debug_flags=0x100 | 0x200),         # two router tile heights
    dict(debug_grid_ctas=-1), dict(debug_wait_ns=-5)])
def test_debug_fields_validation(moe, bad):
    assert moe.moe_check_config(dict(TINY, **bad)) == 1


def test_debug_fields_layout(moe):
    # the C struct: five int32, an fp64 capacity factor, three int32, the
    # debug flags and grid cap, an int64 wait limit (64 bytes)
    assert ctypes.sizeof(moe.moe_config) == 64
    assert moe.moe_config.debug_wait_ns.offset == 56
    for f in (0x1, 0x2, 0x4, 0x8, 0x10, 0x20, 0x40, 0x80, 0x100, 0x200, 0x400, 0x800, 0x1000, 0x2000):
        assert moe.moe_check_config(dict(TINY, debug_flags=f)) == 0
    assert moe.moe_check_config(dict(TINY, debug_grid_ctas=12, debug_wait_ns=1)) == 0


def test_good_configs(moe):
    from synth import workloads as W
    for wl in W.WORKLOADS.values():
        assert moe.moe_check_config(wl.cfg) == 0


def test_capacity_matches_the_oracle(moe):
    import oracle
    # 0.8 is not an fp32 value: carried in fp32 it would make ceil(0.8*2000*2/8) 401
    for T, N, k, cf in [(8192, 8, 2, 1.0), (10, 8, 2, 1.0), (4096, 8, 2, 1.25), (7, 3, 1, 1.0),
                        (64, 8, 2, 0.0), (333, 128, 8, 0.7), (2000, 8, 2, 0.8), (777, 128, 8, 0.6)]:
        cfg = dict(hidden=128, num_experts=N, top_k=k, intermediate=128, block_size=8,
                   capacity_factor=cf)
        assert moe.moe_capacity(cfg, T) == oracle.capacity(T, N, k, cf)


def test_bounds_and_workspace(moe):
    cfg = dict(TINY)
    assert moe.moe_max_padded_rows(cfg, 64) == 64 * 2 + 8 * 7
    assert moe.moe_max_blocks(cfg, 64) == 64 * 2 // 8 + 8
    sizes = [moe.moe_workspace_bytes(cfg, T) for T in (0, 1, 64, 1000)]
    assert all(s > 0 for s in sizes) and sizes == sorted(sizes)
    assert moe.moe_workspace_bytes(dict(cfg, hidden=100), 64) == 0
    assert moe.moe_workspace_bytes(cfg, -1) == 0


def _call_route(moe, cfg, T, ptrs, ws_bytes):
    c = moe.make_config(**cfg)
    return moe._lib.moe_route(ctypes.byref(c), T, *ptrs, ws_bytes, None)


def test_route_argument_errors_return_before_launch(moe):
    cfg = dict(TINY)
    good = [0x10000, 0x20000, None, 0x30000, 0x40000, None, 0x50000]
    ws_need = moe.moe_workspace_bytes(cfg, 64)
    assert _call_route(moe, cfg, 0, good, ws_need) == 0                # T = 0: no-op
    assert _call_route(moe, cfg, -1, good, ws_need) == 1               # negative T
    assert _call_route(moe, cfg, 64, [None] + good[1:], ws_need) == 1  # null h
    assert _call_route(moe, cfg, 64, [0x10008] + good[1:], ws_need) == 1  # misaligned h
    assert _call_route(moe, cfg, 64, good, ws_need - 1) == 3           # workspace too small
    assert _call_route(moe, dict(cfg, hidden=96), 64, good, ws_need) == 2


def test_forward_argument_errors_return_before_launch(moe):
    cfg = dict(TINY, shared_intermediate=128)
    c = moe.make_config(**cfg)
    ws_need = moe.moe_workspace_bytes(cfg, 64)
    p = [0x10000, 0x20000, None, 0x30000, 0x40000, None, None, 0x50000, 0x60000]
    # the shared expert is configured but its weights are missing
    assert moe._lib.moe_forward(ctypes.byref(c), 64, *p, ws_need, None) == 1
    assert moe._lib.moe_forward(ctypes.byref(c), 0, *p, ws_need, None) == 0


def test_binding_refuses_to_import_without_the_library(tmp_path):
    # the package has no CPU fallback: without libmoe_gb300.so the import fails
    import shutil
    import subprocess
    import sys
    pkg = os.path.join(ROOT, "invariant_expert_routing_gb300")
    dst = tmp_path / "invariant_expert_routing_gb300"
    shutil.copytree(pkg, dst, ignore=shutil.ignore_patterns("*.so", "_build", "__pycache__"))
    r = subprocess.run([sys.executable, "-c", "import invariant_expert_routing_gb300"],
                       cwd=tmp_path, capture_output=True, text=True)
    assert r.returncode != 0 and "no CPU fallback" in r.stderr


@pytest.mark.parametrize("bad", [dict(overflow_policy=2), dict(overflow_policy=-1), dict(routing=2)])
def test_policy_and_routing_validation(moe, bad):
    assert moe.moe_check_config(dict(TINY, **bad)) == 1
    assert moe.moe_check_config(dict(TINY, overflow_policy=1, routing=1)) == 0


def test_expert_choice_capacity_and_bounds_match_the_oracle(moe):
    import oracle
    for T, N, k, cf, B in [(64, 8, 2, 0.0, 8), (100, 8, 2, 1.25, 16), (5, 2, 2, 1.5, 8),
                           (8192, 128, 8, 1.0, 16), (1, 256, 8, 0.0, 16)]:
        cfg = dict(hidden=128, num_experts=N, top_k=k, intermediate=128, block_size=B,
                   capacity_factor=cf, routing=1)
        C = oracle.ec_capacity(T, N, k, cf)
        assert moe.moe_capacity(cfg, T) == C
        P = (C + B - 1) // B * B
        assert moe.moe_max_padded_rows(cfg, T) == N * P
        assert moe.moe_max_blocks(cfg, T) == N * P // B
        assert moe.moe_workspace_bytes(cfg, T) > 0


def test_launch_counts(moe):
    mix = dict(hidden=4096, num_experts=8, top_k=2, intermediate=14336, block_size=64)
    qw = dict(hidden=2048, num_experts=128, top_k=8, intermediate=768, block_size=16)
    ds = dict(hidden=7168, num_experts=256, top_k=8, intermediate=2048, block_size=16)
    T = 4096
    # after routing and dispatch: both tile lists with the row copy (one launch), W13, W2, combine = 4
    assert moe.moe_forward_launch_count(mix, T) == 2 + 3 + 4
    assert moe.moe_forward_launch_count(qw, T) == 5 + 3 + 4   # T * H * N above 3 * 2^28: tensor cores
    assert moe.moe_forward_launch_count(qw, 3072) == 2 + 3 + 4   # chunked router up to 3 * 2^28
    assert moe.moe_forward_launch_count(qw, 3073) == 5 + 3 + 4
    assert moe.moe_forward_launch_count(ds, 438) == 2 + 3 + 4
    assert moe.moe_forward_launch_count(ds, 439) == 5 + 3 + 4
    assert moe.moe_forward_launch_count(dict(mix, capacity_factor=1.0, overflow_policy=1), T) == 11 + 4
    assert moe.moe_forward_launch_count(dict(qw, routing=1), T) == 4 + 4
    assert moe.moe_forward_launch_count(dict(ds, routing=1), T) == 4 + 4
    assert moe.moe_forward_launch_count(ds, T) == 5 + 3 + 4
    assert moe.moe_forward_launch_count(dict(mix, shared_intermediate=128), T) == 2 + 3 + 4 + 2
    # up to 64 tokens (or any batch of small router work) are routed in two
    # launches (chunk sums, reduce + top-k), and up to 1024 routes are
    # dispatched with both tile lists in one launch
    assert moe.moe_forward_launch_count(mix, 1) == 2 + 3   # two-launch decode front (T <= 2)
    assert moe.moe_forward_launch_count(mix, 2) == 2 + 3
    assert moe.moe_forward_launch_count(mix, 3) == 2 + 1 + 4
    assert moe.moe_forward_launch_count(dict(ds, shared_intermediate=2048), 1) == 2 + 3 + 2
    assert moe.moe_forward_launch_count(mix, 64) == 2 + 1 + 4
    assert moe.moe_forward_launch_count(mix, 65) == 2 + 1 + 4
    assert moe.moe_forward_launch_count(mix, 512) == 2 + 1 + 4
    assert moe.moe_forward_launch_count(mix, 513) == 2 + 3 + 4
    assert moe.moe_forward_launch_count(qw, 1) == 2 + 3
    assert moe.moe_forward_launch_count(qw, 64) == 2 + 1 + 4
    assert moe.moe_forward_launch_count(qw, 65) == 2 + 1 + 4
    assert moe.moe_forward_launch_count(qw, 128) == 2 + 1 + 4
    assert moe.moe_forward_launch_count(dict(qw, routing=1), 64) == 4 + 4
    assert moe.moe_forward_launch_count(ds, 64) == 2 + 1 + 4
    assert moe.moe_forward_launch_count(ds, 65) == 2 + 1 + 4
    assert moe.moe_forward_launch_count(mix, 0) == 0


def test_drop_only_dispatch_refuses_reroute_and_expert_choice(moe):
    # moe_dispatch_align would drop routes the configuration asks to keep:
    # it refuses before launching anything
    fake = [0x10000 + 0x1000 * i for i in range(8)]
    for extra, code in [(dict(capacity_factor=1.0, overflow_policy=1), 1), (dict(routing=1), 1)]:
        cfg = dict(TINY, **extra)
        c = moe.make_config(**cfg)
        ws = moe.moe_workspace_bytes(cfg, 64)
        assert moe._lib.moe_dispatch_align(ctypes.byref(c), 64, *fake, 0x90000, ws, None) == code
        st = moe._lib.moe_dispatch_align_noalloc(ctypes.byref(c), 64, *fake, None, None)
        assert st == code
    # the expert-choice entry refuses a token-choice configuration, and the
    # reroute entry an expert-choice one
    c = moe.make_config(**TINY)
    assert moe._lib.moe_route_expert_choice(ctypes.byref(c), 64, *fake, 0x90000,
                                            moe.moe_workspace_bytes(TINY, 64), None) == 1
    ce = moe.make_config(**dict(TINY, routing=1))
    assert moe._lib.moe_dispatch_align_reroute(ctypes.byref(ce), 64, *(fake + fake[:3]), 0x90000,
                                               1 << 30, None) == 1


def test_diagnostic_argument_errors(moe):
    c = moe.make_config(**TINY)
    assert moe._lib.moe_routing_stats(ctypes.byref(c), 64, 0x10000, -1.0, 0x20000, 0x30000, None) == 1
    assert moe._lib.moe_routing_stats(ctypes.byref(c), 0, 0x10000, 1.25, 0x20000, 0x30000, None) == 0
    assert moe._lib.moe_routing_stats(ctypes.byref(c), 64, None, 1.25, 0x20000, 0x30000, None) == 1
    assert moe._lib.moe_router_margin(ctypes.byref(c), 64, 0x10004, 0x20000, None) == 1
    assert moe._lib.moe_router_margin(ctypes.byref(c), 0, None, None, None) == 0
    assert ctypes.sizeof(moe.moe_route_stats) == 40
