"""CPU oracle of the batch-invariant MoE layer forward (numpy front end).

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
benchmark's CPU-baseline leg may import this package.  It wraps the plain C++
restatement in moe_oracle.cpp (built with gcc, no CUDA) and shares no code
with the CUDA path.

Each function cites the passage it follows in its C++ implementation.  Pins
(tests/test_oracle_*.py) tie every function to something other than itself:
brute force over expert subsets, closed forms, error bounds against exact
arithmetic, hand-built cases and textbook reductions.  The gate values are
pinned by closed forms and a hand fixture; the GPU's gates are compared with
them within a tolerance, not bit for bit (fp32 expf on the GPU, fp64 here).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

i32p = ctypes.POINTER(ctypes.c_int32)


def build() -> None:
    src = os.path.join(_HERE, "moe_oracle.cpp")
    subprocess.check_call(["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                           "-pthread", "-o", _SO, src])


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_SO):
            build()
        L = ctypes.CDLL(_SO)
        c = ctypes
        vp = c.c_void_p
        L.oracle_router_logits.argtypes = [c.c_int32] * 3 + [vp] * 4 + [c.c_int32]
        L.oracle_select_topk.argtypes = [c.c_int32] * 3 + [vp] * 3
        L.oracle_router_margin.argtypes = [c.c_int32] * 3 + [vp] * 2
        L.oracle_capacity.argtypes = [c.c_int32] * 3 + [c.c_double]
        L.oracle_capacity.restype = c.c_int32
        L.oracle_dispatch.argtypes = [c.c_int32] * 5 + [vp] * 8
        L.oracle_expert_row.argtypes = [c.c_int32] * 2 + [vp] * 5
        L.oracle_expert_rows.argtypes = [c.c_int32, vp, vp, c.c_int32, c.c_int32] + [vp] * 4 + [c.c_int32]
        L.oracle_combine_rows.argtypes = [c.c_int32, vp, c.c_int32, c.c_int32] + [vp] * 6
        L.oracle_moe_forward.argtypes = ([c.c_int32] * 6 + [c.c_double] + [c.c_int32] * 3
                                         + [vp] * 8 + [c.c_int32])
        L.oracle_reroute.argtypes = [c.c_int32] * 4 + [vp] * 5
        L.oracle_routing_stats.argtypes = [c.c_int32] * 3 + [vp, c.c_double] + [vp] * 3
        L.oracle_expert_choice.argtypes = [c.c_int32] * 3 + [vp] * 3
        L.oracle_ec_capacity.argtypes = [c.c_int32] * 3 + [c.c_double]
        L.oracle_ec_capacity.restype = c.c_int32
        L.oracle_bf16_round.argtypes = [c.c_double]
        L.oracle_bf16_round.restype = c.c_uint16
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dt):
    return None if a is None else np.ascontiguousarray(a, dtype=dt)


def router_logits(h, w_gate, bias=None, nthreads: int = 0) -> np.ndarray:
    h = _c(h, np.uint16)
    w_gate = _c(w_gate, np.uint16)
    bias = _c(bias, np.float32)
    T, H = h.shape
    N = w_gate.shape[1]
    out = np.empty((T, N), dtype=np.float32)
    lib().oracle_router_logits(T, H, N, _p(h), _p(w_gate), _p(bias), _p(out), nthreads)
    return out


def select_topk(logits, k: int):
    logits = _c(logits, np.float32)
    T, N = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    gates = np.empty((T, k), dtype=np.float64)
    lib().oracle_select_topk(T, N, k, _p(logits), _p(idx), _p(gates))
    return idx, gates


def router_margin(logits, k: int) -> np.ndarray:
    logits = _c(logits, np.float32)
    T, N = logits.shape
    out = np.empty(T, dtype=np.float64)
    lib().oracle_router_margin(T, N, k, _p(logits), _p(out))
    return out


def capacity(T: int, N: int, k: int, capacity_factor: float) -> int:
    return int(lib().oracle_capacity(T, N, k, float(capacity_factor)))


def dispatch(topk_idx, N: int, B: int, capacity_: int):
    topk_idx = _c(topk_idx, np.int32)
    T, k = topk_idx.shape
    R = T * k
    kept = np.empty(R, dtype=np.uint8)
    pos = np.empty(R, dtype=np.int32)
    sorted_ids = np.full(R + N * B, -7, dtype=np.int32)
    blocks = np.full(R // B + N + 1, -7, dtype=np.int32)
    num_padded = np.zeros(1, dtype=np.int32)
    counts = np.empty(N, dtype=np.int32)
    dropped = np.zeros(1, dtype=np.int32)
    lib().oracle_dispatch(T, N, k, B, capacity_, _p(topk_idx), _p(kept), _p(pos), _p(sorted_ids),
                          _p(blocks), _p(num_padded), _p(counts), _p(dropped))
    P = int(num_padded[0])
    return dict(route_kept=kept, route_pos=pos, sorted_route_ids=sorted_ids[:P],
                block_expert=blocks[:P // B], num_padded=P, expert_counts=counts,
                num_dropped=int(dropped[0]))


def reroute(logits, topk_idx, capacity_: int):
    """Overflow reroute: returns (route_expert [R] int32, -1 = dropped;
    num_rerouted; num_dropped)."""
    logits = _c(logits, np.float32)
    topk_idx = _c(topk_idx, np.int32)
    T, k = topk_idx.shape
    N = logits.shape[1]
    out = np.empty(T * k, dtype=np.int32)
    nr = np.zeros(1, dtype=np.int32)
    nd = np.zeros(1, dtype=np.int32)
    lib().oracle_reroute(T, N, k, capacity_, _p(logits), _p(topk_idx), _p(out), _p(nr), _p(nd))
    return out, int(nr[0]), int(nd[0])


def dispatch_routes(route_expert, N: int, B: int, slots: int):
    """Stable alignment of routes that already have their expert (-1 = not
    routed), `slots` routes per token: the layout after reroute or expert
    choice."""
    route_expert = _c(route_expert, np.int32).reshape(-1, slots)
    return dispatch(route_expert, N, B, -1)


def routing_stats(topk_idx, N: int, capacity_factor: float = 1.25):
    """The routing_stats probe: (load [N], dict)."""
    topk_idx = _c(topk_idx, np.int32)
    T, k = topk_idx.shape
    load = np.empty(N, dtype=np.int32)
    ints = np.empty(5, dtype=np.int32)
    reals = np.empty(2, dtype=np.float64)
    lib().oracle_routing_stats(T, N, k, _p(topk_idx), float(capacity_factor), _p(load), _p(ints),
                               _p(reals))
    return load, dict(max_expert_load=int(ints[0]), min_expert_load=int(ints[1]),
                      capacity=int(ints[2]), dropped_tokens=int(ints[3]), total_routes=int(ints[4]),
                      imbalance_ratio=float(reals[0]), drop_fraction=float(reals[1]))


def ec_capacity(T: int, N: int, k: int, capacity_factor: float) -> int:
    return int(lib().oracle_ec_capacity(T, N, k, float(capacity_factor)))


def expert_choice(logits, capacity_: int):
    """Expert-choice selection: (selected [T, N] uint8, probs [T, N] fp64)."""
    logits = _c(logits, np.float32)
    T, N = logits.shape
    sel = np.empty((T, N), dtype=np.uint8)
    probs = np.empty((T, N), dtype=np.float64)
    lib().oracle_expert_choice(T, N, capacity_, _p(logits), _p(sel), _p(probs))
    return sel, probs


def expert_row(x, w13_e, w2_e):
    """One SwiGLU expert on one row: returns (y fp64 [H], a bf16 bits [I])."""
    x = _c(x, np.uint16)
    w13_e = _c(w13_e, np.uint16)
    w2_e = _c(w2_e, np.uint16)
    H = x.shape[0]
    I = w2_e.shape[0]
    y = np.empty(H, dtype=np.float64)
    a = np.empty(I, dtype=np.uint16)
    lib().oracle_expert_row(H, I, _p(x), _p(w13_e), _p(w2_e), _p(y), _p(a))
    return y, a


def expert_rows(tokens, experts, h, w13, w2, nthreads: int = 0) -> np.ndarray:
    tokens = _c(tokens, np.int32)
    experts = _c(experts, np.int32)
    h = _c(h, np.uint16)
    w13 = _c(w13, np.uint16)
    w2 = _c(w2, np.uint16)
    n = tokens.shape[0]
    H = h.shape[1]
    I = w2.shape[-2]
    y = np.empty((n, H), dtype=np.float64)
    lib().oracle_expert_rows(n, _p(tokens), _p(experts), H, I, _p(h), _p(w13), _p(w2), _p(y),
                             nthreads)
    return y


def combine_rows(tokens, h, gates, route_kept, y_route, y_shared=None) -> np.ndarray:
    tokens = _c(tokens, np.int32)
    h = _c(h, np.uint16)
    gates = _c(gates, np.float64)
    route_kept = _c(route_kept, np.uint8)
    y_route = _c(y_route, np.float64)
    y_shared = _c(y_shared, np.float64)
    n = tokens.shape[0]
    H = h.shape[1]
    k = gates.shape[1]
    out = np.empty((n, H), dtype=np.uint16)
    lib().oracle_combine_rows(n, _p(tokens), H, k, _p(h), _p(gates), _p(route_kept), _p(y_route),
                              _p(y_shared), _p(out))
    return out


def moe_forward(cfg: dict, h, w_gate, bias, w13, w2, w13s=None, w2s=None,
                nthreads: int = 0) -> np.ndarray:
    h = _c(h, np.uint16)
    w_gate = _c(w_gate, np.uint16)
    bias = _c(bias, np.float32)
    w13 = _c(w13, np.uint16)
    w2 = _c(w2, np.uint16)
    w13s = _c(w13s, np.uint16)
    w2s = _c(w2s, np.uint16)
    T, H = h.shape
    N, k, I, B = cfg["num_experts"], cfg["top_k"], cfg["intermediate"], cfg["block_size"]
    Is = cfg.get("shared_intermediate", 0) or 0
    out = np.empty((T, H), dtype=np.uint16)
    lib().oracle_moe_forward(T, H, N, k, I, B, float(cfg.get("capacity_factor", 0.0)),
                             int(cfg.get("overflow_policy", 0)), int(cfg.get("routing", 0)), Is,
                             _p(h), _p(w_gate), _p(bias), _p(w13), _p(w2), _p(w13s), _p(w2s),
                             _p(out), nthreads)
    return out


def bf16_round(x: float) -> int:
    return int(lib().oracle_bf16_round(float(x)))
