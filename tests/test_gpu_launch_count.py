"""The fused forward launches exactly the kernels moe_forward_launch_count
reports (the figure behind bench.py's gpu_launches).

Each forward is captured in a CUDA graph (kept, not only instantiated) and
its kernel nodes are counted through the driver API: both streams of a layer
with a shared expert land in the one graph.  Cases cover the chunked and the
tensor-core router, the one-CTA small-batch dispatch, the two-launch decode
front, the overflow reroute and expert-choice routing.
"""
import ctypes

import pytest

pytestmark = pytest.mark.gpu

_MIX = dict(hidden=4096, num_experts=8, top_k=2, intermediate=128, block_size=64)
_QW = dict(hidden=2048, num_experts=128, top_k=8, intermediate=128, block_size=16)
_DS = dict(hidden=1024, num_experts=256, top_k=8, intermediate=128, shared_intermediate=128, block_size=16)
CASES = [
    ("mix", _MIX, 4096), ("mix small dispatch", _MIX, 3), ("mix decode", _MIX, 1),
    ("qw tensor-core router", _QW, 8192), ("qw decode", _QW, 1), ("shared expert", _DS, 2048),
    ("reroute", dict(_MIX, capacity_factor=1.0, overflow_policy=1), 4096),
    ("expert choice", dict(_QW, routing=1, capacity_factor=1.0), 1024),
]


def _kernel_nodes(graph_handle: int) -> int:
    cu = ctypes.CDLL("libcuda.so.1")
    n = ctypes.c_size_t(0)
    assert cu.cuGraphGetNodes(ctypes.c_void_p(graph_handle), None, ctypes.byref(n)) == 0
    nodes = (ctypes.c_void_p * n.value)()
    assert cu.cuGraphGetNodes(ctypes.c_void_p(graph_handle), nodes, ctypes.byref(n)) == 0
    kernels = 0
    for i in range(n.value):
        t = ctypes.c_int(-1)
        assert cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) == 0
        kernels += t.value == 0   # CU_GRAPH_NODE_TYPE_KERNEL
    return kernels


@pytest.mark.parametrize("name,cfg,T", CASES, ids=[c[0] for c in CASES])
def test_forward_launch_count(name, cfg, T):
    import torch
    import invariant_expert_routing_gb300 as moe
    try:
        graph = torch.cuda.CUDAGraph(keep_graph=True)
    except TypeError:
        pytest.skip("this PyTorch cannot keep the captured cudaGraph_t")
    g = torch.Generator(device="cuda").manual_seed(7)
    H, N, I = cfg["hidden"], cfg["num_experts"], cfg["intermediate"]
    Is = cfg.get("shared_intermediate", 0)

    def randn(*shape, scale=1.0):
        return (torch.randn(*shape, generator=g, device="cuda") * scale).to(torch.bfloat16)

    h = randn(T, H)
    wg = randn(H, N, scale=H ** -0.5)
    w13 = randn(N, H, 2 * I, scale=H ** -0.5)
    w2 = randn(N, I, H, scale=I ** -0.5)
    w13s = randn(H, 2 * Is, scale=H ** -0.5) if Is else None
    w2s = randn(Is, H, scale=Is ** -0.5) if Is else None
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    ws = moe.workspace(cfg, T)
    moe.moe_clear_device_status(ws)

    def fwd():
        moe.moe_forward(cfg, h, wg, None, w13, w2, w13s, w2s, out, ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fwd()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        fwd()
    counted = _kernel_nodes(graph.raw_cuda_graph())
    assert counted == moe.moe_forward_launch_count(cfg, T), name
    assert moe.moe_get_device_status(ws) == 0
