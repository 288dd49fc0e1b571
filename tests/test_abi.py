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


def test_good_configs(moe):
    from synth import workloads as W
    for wl in W.WORKLOADS.values():
        assert moe.moe_check_config(wl.cfg) == 0


def test_capacity_matches_the_oracle(moe):
    import oracle
    for T, N, k, cf in [(8192, 8, 2, 1.0), (10, 8, 2, 1.0), (4096, 8, 2, 1.25), (7, 3, 1, 1.0),
                        (64, 8, 2, 0.0), (333, 128, 8, 0.7)]:
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
