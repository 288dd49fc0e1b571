"""Python binding of the batch-invariant MoE layer C ABI (libmoe_gb300.so).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  Functions carry the C names (moe_route, moe_dispatch_align,
moe_expert_ffn, moe_combine, moe_forward, ...) and take torch tensors, whose
device pointers are passed through; PyTorch only provides device memory and
streams.  There is no fallback: if the library is missing, importing this
package raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe_gb300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                      "(nvcc, sm_103a); there is no CPU fallback")

_lib = ctypes.CDLL(LIB_PATH)

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE = 5
MOE_DEV_ERR_EXPERT_RANGE = 0x1
MOE_DEV_ERR_TIMEOUT = 0x2
MOE_DEV_ERR_BAD_BLOCKS = 0x4
MOE_DEV_NOTE_REROUTE_FALLBACK = 0x100
MOE_DEV_ERR_MASK = 0xFF
# debug_flags bits (testing only; each forces one of several equivalent paths)
MOE_DEBUG_ROUTER_TC = 0x1
MOE_DEBUG_ROUTER_CHUNKED = 0x2
MOE_DEBUG_ROW_GATHER = 0x4
MOE_DEBUG_ROW_SCATTER = 0x8
MOE_DEBUG_NO_DECODE_FRONT = 0x10
MOE_DEBUG_REROUTE_SEQUENTIAL = 0x20
MOE_DEBUG_REROUTE_GRID = 0x40
MOE_DEBUG_REROUTE_ONE_CTA = 0x80
MOE_DEBUG_ROUTER_TILE128 = 0x100
MOE_DEBUG_ROUTER_TILE64 = 0x200
MOE_DEBUG_SHARED_SERIAL = 0x400
MOE_DEBUG_W13_PAIR = 0x800
MOE_DEBUG_W2_WIDE = 0x1000
MOE_DEBUG_W13_SINGLE = 0x2000
MOE_OVERFLOW_DROP = 0
MOE_OVERFLOW_REROUTE = 1
MOE_ROUTING_TOKEN_CHOICE = 0
MOE_ROUTING_EXPERT_CHOICE = 1


class moe_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("capacity_factor", ctypes.c_double),
                ("shared_intermediate", ctypes.c_int32), ("overflow_policy", ctypes.c_int32),
                ("routing", ctypes.c_int32), ("debug_flags", ctypes.c_uint32),
                ("debug_grid_ctas", ctypes.c_int32), ("debug_wait_ns", ctypes.c_int64)]


class moe_route_stats(ctypes.Structure):
    _fields_ = [("max_expert_load", ctypes.c_int32), ("min_expert_load", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("dropped_tokens", ctypes.c_int32),
                ("total_routes", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("imbalance_ratio", ctypes.c_double), ("drop_fraction", ctypes.c_double)]


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = _lib.moe_status_string(status).decode()
        super().__init__(f"{fn} failed: {msg} ({status})")


_vp, _i32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
_cfgp = ctypes.POINTER(moe_config)
_SIGS = {
    "moe_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "moe_check_config": ([_cfgp], ctypes.c_int),
    "moe_capacity": ([_cfgp, _i32], _i32),
    "moe_max_padded_rows": ([_cfgp, _i32], ctypes.c_int64),
    "moe_max_blocks": ([_cfgp, _i32], ctypes.c_int64),
    "moe_workspace_bytes": ([_cfgp, _i32], _sz),
    "moe_route": ([_cfgp, _i32] + [_vp] * 6 + [_vp, _sz, _vp], ctypes.c_int),
    "moe_dispatch_align": ([_cfgp, _i32] + [_vp] * 8 + [_vp, _sz, _vp], ctypes.c_int),
    "moe_expert_ffn": ([_cfgp, _i32] + [_vp] * 10 + [_vp, _sz, _vp], ctypes.c_int),
    "moe_combine": ([_cfgp, _i32] + [_vp] * 7 + [_vp], ctypes.c_int),
    "moe_forward": ([_cfgp, _i32] + [_vp] * 8 + [_vp, _sz, _vp], ctypes.c_int),
    "moe_forward_hostio": ([_cfgp, _i32] + [_vp] * 8 + [_vp, _sz, _vp], ctypes.c_int),
    "moe_forward_timed": ([_cfgp, _i32] + [_vp] * 8 + [_vp, _sz, _vp, _i32, _vp], ctypes.c_int),
    "moe_forward_launch_count": ([_cfgp, _i32], _i32),
    "moe_router_cert_beta": ([_i32], ctypes.c_float),
    "moe_route_filtered": ([_cfgp, _i32] + [_vp] * 6 + [_vp, _sz, _vp], ctypes.c_int),
    "moe_router_tc_logits": ([_cfgp, _i32] + [_vp] * 3 + [_vp, _sz, _vp], ctypes.c_int),
    "moe_dispatch_align_noalloc": ([_cfgp, _i32] + [_vp] * 9 + [_vp], ctypes.c_int),
    "moe_dispatch_align_shard": ([_cfgp, _i32, _i32] + [_vp] * 9 + [_vp, _sz, _vp], ctypes.c_int),
    "moe_router_logits": ([_cfgp, _i32] + [_vp] * 4 + [_vp, _sz, _vp], ctypes.c_int),
    "moe_dispatch_align_reroute": ([_cfgp, _i32] + [_vp] * 11 + [_vp, _sz, _vp], ctypes.c_int),
    "moe_route_expert_choice": ([_cfgp, _i32] + [_vp] * 8 + [_vp, _sz, _vp], ctypes.c_int),
    "moe_routing_stats": ([_cfgp, _i32, _vp, ctypes.c_double, _vp, _vp, _vp], ctypes.c_int),
    "moe_router_margin": ([_cfgp, _i32, _vp, _vp, _vp], ctypes.c_int),
    "moe_get_device_status": ([_vp, ctypes.POINTER(_i32), _vp], ctypes.c_int),
    "moe_clear_device_status": ([_vp, _vp], ctypes.c_int),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_SIGS)


def make_config(hidden, num_experts, top_k, intermediate, block_size, capacity_factor=0.0,
                shared_intermediate=0, overflow_policy=MOE_OVERFLOW_DROP,
                routing=MOE_ROUTING_TOKEN_CHOICE, debug_flags=0, debug_grid_ctas=0,
                debug_wait_ns=0) -> moe_config:
    return moe_config(hidden, num_experts, top_k, intermediate, block_size, capacity_factor,
                      shared_intermediate, overflow_policy, routing, debug_flags, debug_grid_ctas,
                      debug_wait_ns)


def _cfg(cfg) -> moe_config:
    if isinstance(cfg, moe_config):
        return cfg
    return make_config(**cfg)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(fn, st):
    if st != MOE_OK:
        raise MoEError(fn, st)


def moe_capacity(cfg, T: int) -> int:
    return int(_lib.moe_capacity(ctypes.byref(_cfg(cfg)), T))


def moe_max_padded_rows(cfg, T: int) -> int:
    return int(_lib.moe_max_padded_rows(ctypes.byref(_cfg(cfg)), T))


def moe_max_blocks(cfg, T: int) -> int:
    return int(_lib.moe_max_blocks(ctypes.byref(_cfg(cfg)), T))


def moe_workspace_bytes(cfg, max_tokens: int) -> int:
    return int(_lib.moe_workspace_bytes(ctypes.byref(_cfg(cfg)), max_tokens))


def moe_check_config(cfg) -> int:
    return int(_lib.moe_check_config(ctypes.byref(_cfg(cfg))))


def workspace(cfg, max_tokens: int, device="cuda"):
    """A torch uint8 tensor sized for moe_* calls with up to max_tokens tokens."""
    import torch
    n = moe_workspace_bytes(cfg, max_tokens)
    if n == 0:
        raise MoEError("moe_workspace_bytes", MOE_ERR_UNSUPPORTED)
    return torch.empty(n, dtype=torch.uint8, device=device)


def moe_route(cfg, h, w_gate, router_bias, topk_idx, topk_gate, logits_out, ws, stream=None):
    T = h.shape[0]
    _check("moe_route", _lib.moe_route(ctypes.byref(_cfg(cfg)), T, _ptr(h), _ptr(w_gate),
                                       _ptr(router_bias), _ptr(topk_idx), _ptr(topk_gate),
                                       _ptr(logits_out), _ptr(ws), ws.numel(), _stream(stream)))


def moe_dispatch_align(cfg, topk_idx, route_kept, route_pos, sorted_route_ids, block_expert,
                       num_padded, expert_counts, num_dropped, ws, stream=None):
    T = topk_idx.shape[0]
    _check("moe_dispatch_align", _lib.moe_dispatch_align(
        ctypes.byref(_cfg(cfg)), T, _ptr(topk_idx), _ptr(route_kept), _ptr(route_pos),
        _ptr(sorted_route_ids), _ptr(block_expert), _ptr(num_padded), _ptr(expert_counts),
        _ptr(num_dropped), _ptr(ws), ws.numel(), _stream(stream)))


def moe_dispatch_align_shard(cfg, global_tokens, topk_idx, expert_offset, route_kept, route_pos,
                             sorted_route_ids, block_expert, num_padded, expert_counts, num_dropped, ws,
                             stream=None):
    """One shard (in token order) of a capacity-limited batch of global_tokens
    tokens; expert_offset: routes each expert received in earlier shards
    (None for the first)."""
    T = topk_idx.shape[0]
    _check("moe_dispatch_align_shard", _lib.moe_dispatch_align_shard(
        ctypes.byref(_cfg(cfg)), T, int(global_tokens), _ptr(topk_idx), _ptr(expert_offset),
        _ptr(route_kept), _ptr(route_pos), _ptr(sorted_route_ids), _ptr(block_expert), _ptr(num_padded),
        _ptr(expert_counts), _ptr(num_dropped), _ptr(ws), ws.numel(), _stream(stream)))


def moe_dispatch_align_noalloc(cfg, topk_idx, route_kept, route_pos, sorted_route_ids,
                               block_expert, num_padded, expert_counts, num_dropped,
                               status_out=None, stream=None):
    """moe_dispatch_align without a workspace (fixed in-library scratch, T*k <= 65536)."""
    T = topk_idx.shape[0]
    _check("moe_dispatch_align_noalloc", _lib.moe_dispatch_align_noalloc(
        ctypes.byref(_cfg(cfg)), T, _ptr(topk_idx), _ptr(route_kept), _ptr(route_pos),
        _ptr(sorted_route_ids), _ptr(block_expert), _ptr(num_padded), _ptr(expert_counts),
        _ptr(num_dropped), _ptr(status_out), _stream(stream)))


def moe_router_logits(cfg, h, w_gate, router_bias, logits_out, ws, stream=None):
    T = h.shape[0]
    _check("moe_router_logits", _lib.moe_router_logits(
        ctypes.byref(_cfg(cfg)), T, _ptr(h), _ptr(w_gate), _ptr(router_bias), _ptr(logits_out),
        _ptr(ws), ws.numel(), _stream(stream)))


def moe_dispatch_align_reroute(cfg, topk_idx, logits, route_kept, route_expert, route_pos,
                               sorted_route_ids, block_expert, num_padded, expert_counts,
                               num_dropped, num_rerouted, ws, stream=None):
    T = topk_idx.shape[0]
    _check("moe_dispatch_align_reroute", _lib.moe_dispatch_align_reroute(
        ctypes.byref(_cfg(cfg)), T, _ptr(topk_idx), _ptr(logits), _ptr(route_kept),
        _ptr(route_expert), _ptr(route_pos), _ptr(sorted_route_ids), _ptr(block_expert),
        _ptr(num_padded), _ptr(expert_counts), _ptr(num_dropped), _ptr(num_rerouted), _ptr(ws),
        ws.numel(), _stream(stream)))


def moe_route_expert_choice(cfg, logits, gates, route_kept, route_pos, sorted_route_ids,
                            block_expert, num_padded, expert_counts, ws, stream=None):
    T = logits.shape[0]
    _check("moe_route_expert_choice", _lib.moe_route_expert_choice(
        ctypes.byref(_cfg(cfg)), T, _ptr(logits), _ptr(gates), _ptr(route_kept), _ptr(route_pos),
        _ptr(sorted_route_ids), _ptr(block_expert), _ptr(num_padded), _ptr(expert_counts),
        _ptr(ws), ws.numel(), _stream(stream)))


def moe_routing_stats(cfg, topk_idx, capacity_factor, expert_load, stats, stream=None):
    """stats: a device uint8 tensor of at least 40 bytes (moe_route_stats);
    read it with route_stats_from_bytes."""
    T = topk_idx.shape[0]
    _check("moe_routing_stats", _lib.moe_routing_stats(
        ctypes.byref(_cfg(cfg)), T, _ptr(topk_idx), float(capacity_factor), _ptr(expert_load),
        _ptr(stats), _stream(stream)))


def route_stats_from_bytes(raw: bytes) -> dict:
    st = moe_route_stats.from_buffer_copy(bytes(raw)[:ctypes.sizeof(moe_route_stats)])
    return {name: getattr(st, name) for name, _ in moe_route_stats._fields_ if name != "reserved"}


def moe_router_margin(cfg, logits, margin, stream=None):
    T = logits.shape[0]
    _check("moe_router_margin", _lib.moe_router_margin(
        ctypes.byref(_cfg(cfg)), T, _ptr(logits), _ptr(margin), _stream(stream)))


def moe_expert_ffn(cfg, h, w13, w2, w13_shared, w2_shared, sorted_route_ids, block_expert,
                   num_padded, y_perm, y_shared, ws, stream=None):
    """y_perm [max padded rows, H] and y_shared [T, H] (or None): bfloat16 tensors."""
    T = h.shape[0]
    _check("moe_expert_ffn", _lib.moe_expert_ffn(
        ctypes.byref(_cfg(cfg)), T, _ptr(h), _ptr(w13), _ptr(w2), _ptr(w13_shared),
        _ptr(w2_shared), _ptr(sorted_route_ids), _ptr(block_expert), _ptr(num_padded),
        _ptr(y_perm), _ptr(y_shared), _ptr(ws), ws.numel(), _stream(stream)))


def moe_combine(cfg, h, topk_gate, route_kept, route_pos, y_perm, y_shared, out, stream=None):
    T = h.shape[0]
    _check("moe_combine", _lib.moe_combine(
        ctypes.byref(_cfg(cfg)), T, _ptr(h), _ptr(topk_gate), _ptr(route_kept), _ptr(route_pos),
        _ptr(y_perm), _ptr(y_shared), _ptr(out), _stream(stream)))


def moe_forward(cfg, h, w_gate, router_bias, w13, w2, w13_shared, w2_shared, out, ws,
                stream=None):
    T = h.shape[0]
    _check("moe_forward", _lib.moe_forward(
        ctypes.byref(_cfg(cfg)), T, _ptr(h), _ptr(w_gate), _ptr(router_bias), _ptr(w13),
        _ptr(w2), _ptr(w13_shared), _ptr(w2_shared), _ptr(out), _ptr(ws), ws.numel(),
        _stream(stream)))


def moe_forward_hostio(cfg, h_host, w_gate, router_bias, w13, w2, w13_shared, w2_shared,
                       out_host, ws, stream=None):
    """h_host / out_host: CPU tensors (pinned for asynchronous copies)."""
    T = h_host.shape[0]
    _check("moe_forward_hostio", _lib.moe_forward_hostio(
        ctypes.byref(_cfg(cfg)), T, _ptr(h_host), _ptr(w_gate), _ptr(router_bias), _ptr(w13),
        _ptr(w2), _ptr(w13_shared), _ptr(w2_shared), _ptr(out_host), _ptr(ws), ws.numel(),
        _stream(stream)))


def moe_forward_timed(cfg, h, w_gate, router_bias, w13, w2, w13_shared, w2_shared, out, ws,
                      events, stream=None):
    """moe_forward recording 8 torch.cuda.Event objects at the stage boundaries
    (each event must have been recorded once, so that torch has created it)."""
    T = h.shape[0]
    if any(e.cuda_event == 0 for e in events):
        raise ValueError("record each torch.cuda.Event once before passing it")
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check("moe_forward_timed", _lib.moe_forward_timed(
        ctypes.byref(_cfg(cfg)), T, _ptr(h), _ptr(w_gate), _ptr(router_bias), _ptr(w13),
        _ptr(w2), _ptr(w13_shared), _ptr(w2_shared), _ptr(out), _ptr(ws), ws.numel(), arr,
        len(events), _stream(stream)))


def moe_router_cert_beta(hidden: int) -> float:
    return float(_lib.moe_router_cert_beta(hidden))


def moe_route_filtered(cfg, h, w_gate, router_bias, topk_idx, topk_gate, n_candidates, ws,
                       stream=None):
    """Tensor-core router path with per-token candidate counts (diagnostic)."""
    T = h.shape[0]
    _check("moe_route_filtered", _lib.moe_route_filtered(
        ctypes.byref(_cfg(cfg)), T, _ptr(h), _ptr(w_gate), _ptr(router_bias), _ptr(topk_idx),
        _ptr(topk_gate), _ptr(n_candidates), _ptr(ws), ws.numel(), _stream(stream)))


def moe_router_tc_logits(cfg, h, w_gate, logits_out, ws, stream=None):
    """Tensor-core logits h . W_g (no bias): the input of the certified filter."""
    T = h.shape[0]
    _check("moe_router_tc_logits", _lib.moe_router_tc_logits(
        ctypes.byref(_cfg(cfg)), T, _ptr(h), _ptr(w_gate), _ptr(logits_out), _ptr(ws), ws.numel(),
        _stream(stream)))


def moe_forward_launch_count(cfg, T: int) -> int:
    return int(_lib.moe_forward_launch_count(ctypes.byref(_cfg(cfg)), T))


def moe_get_device_status(ws, stream=None) -> int:
    v = ctypes.c_int32(0)
    st = _lib.moe_get_device_status(_ptr(ws), ctypes.byref(v), _stream(stream))
    if st not in (MOE_OK, MOE_ERR_DEVICE):
        raise MoEError("moe_get_device_status", st)
    return int(v.value)


def moe_clear_device_status(ws, stream=None) -> None:
    _check("moe_clear_device_status", _lib.moe_clear_device_status(_ptr(ws), _stream(stream)))
