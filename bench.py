#!/usr/bin/env python
"""Benchmark of the batch-invariant MoE layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

One step = one moe_forward (router, top-k, capacity dispatch, stable padded
alignment, grouped SwiGLU expert GEMMs, combine) over one batch of synthetic
tokens of the Mixtral-like layer (H 4096, 8 experts, top-2, I 14336, block
64, T 4096), inputs resident in HBM.  Prints one JSON line: routed tokens/s
for the whole job, the roofline of the dominant kernel, the end-to-end rate
through the host-buffer entry point, the CPU oracle timed on the host cores,
the SM clocks seen during the timed region, and (key "workloads") one
cold-L2 entry for every other configured layer and batch size: the tiny
layer, the Mixtral-like decode sizes, the Qwen-like layer at T = 1, 32, 512
and 8192, the capacity-limited layer and the DeepSeek-like layer at T = 1,
64 and 16448, each with its fraction of the measured peak of its bound.

Under torchrun (N > 1) every rank runs its own shard of tokens (a different
token seed) against replicated weights: no collective on the data path
(weak scaling); only the barrier and the max-over-ranks time use
torch.distributed.

--impl reference times the CPU oracle (the reference arm of this build) on
the host cores, rank 0 only, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "mix"
TOKENS = 4096
METRIC = "routed tokens/sec per MoE layer"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------- distributed helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_seed(rank: int) -> int:
    """Token seed of a rank's shard (rank 0 holds the reference batch, seed 0)."""
    return 0 if rank == 0 else 1000003 * rank


def reduce_max(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# --------------------------------------------------------------------------- host <-> device plumbing
def dev_bf16(a, device):
    """uint16 bf16 bit patterns (numpy) -> torch.bfloat16 device tensor."""
    import numpy as np
    import torch
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)


def dev(a, device):
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host_bf16(t):
    """torch.bfloat16 tensor -> uint16 bit patterns (numpy)."""
    import numpy as np
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


OUT_ATOL, OUT_RTOL = 2e-2, 1e-2   # |gpu - ref| <= atol + rtol*|ref| (bf16 in, fp32 accumulation)


def max_err_within_tolerance(got_bits, ref_bits):
    """Largest |gpu - ref| over the compared elements; raises if any element
    is outside the layer tolerance."""
    import numpy as np
    from synth import bf16_to_f32
    got = bf16_to_f32(np.asarray(got_bits, np.uint16)).astype(np.float64)
    ref = bf16_to_f32(np.asarray(ref_bits, np.uint16)).astype(np.float64)
    err = np.abs(got - ref)
    if not np.all(err <= OUT_ATOL + OUT_RTOL * np.abs(ref)):
        raise RuntimeError("GPU rows outside the tolerance of the oracle's")
    return float(err.max()) if err.size else 0.0


# --------------------------------------------------------------------------- roofline inputs
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for name in ("expert_gemm.cu", "ptx.cuh", "gemm.h"):
        with open(os.path.join(ROOT, "invariant_expert_routing_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload_tag: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    from the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload_tag}.md")
    if not os.path.exists(path):
        return None, "no ncu summary"
    text = open(path).read()
    m_sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_b:
        return None, "summary lacks dram bytes"
    if not m_sha or m_sha.group(1) != kernel_source_sha():
        return None, "kernel changed since the ncu capture"
    return float(m_b.group(1)), os.path.relpath(path, ROOT)


# --------------------------------------------------------------------------- clocks
def visible_gpu_index(local: int):
    """nvidia-smi index of this process's GPU when CUDA_VISIBLE_DEVICES lists
    plain indices, else None (query every visible GPU)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis is None:
        return local
    parts = [p.strip() for p in vis.split(",") if p.strip()]
    if local < len(parts) and parts[local].isdigit():
        return int(parts[local])
    return None


class ClockSampler:
    """nvidia-smi samples every 200 ms; keeps the ones inside [t0, t1]."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            sel = [] if self.gpu is None else [f"--id={self.gpu}"]
            self.proc = subprocess.Popen(
                ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [s for (t, s) in self.samples if t0 <= t <= t1]
        in_region = len(rows)
        if not rows and self.samples:  # region shorter than one sample period
            mid = 0.5 * (t0 + t1)
            rows = [min(self.samples, key=lambda x: abs(x[0] - mid))[1]]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": in_region}


# --------------------------------------------------------------------------- work accounting
def algorithmic_work(wl, T, kept_routes: int, touched_experts: int):
    """flops and bytes the method must do (not padded or intermediate work)."""
    H, I, N, Is = wl.hidden, wl.intermediate, wl.num_experts, wl.shared_intermediate
    flops = 2.0 * T * H * N + 6.0 * H * I * kept_routes + 6.0 * H * Is * T
    bytes_ = 6.0 * H * I * touched_experts + 6.0 * H * Is + 2.0 * H * N + 4.0 * T * H
    return flops, bytes_


# --------------------------------------------------------------------------- reference arm
def run_reference(args):
    import numpy as np
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from synth import workloads as W
    import oracle
    wl = W.WORKLOADS[WORKLOAD]
    T = TOKENS
    h_all = W.make_h(wl, T, seed=0)
    wg, bias = W.make_router(wl)
    cores = os.cpu_count() or 1
    w13, w2 = W.make_experts(wl)
    steps, warm = args.steps, args.warmup
    # size the per-step sample so that the whole run stays within ~2 minutes
    t0 = time.perf_counter()
    _oracle_tokens(wl, h_all, wg, bias, w13, w2, np.arange(1))
    per_tok = max(time.perf_counter() - t0, 1e-3)
    S = int(max(1, min(64, 120.0 / ((steps + warm) * per_tok))))
    rng = np.random.default_rng(7)
    for _ in range(warm):
        _oracle_tokens(wl, h_all, wg, bias, w13, w2, np.sort(rng.choice(T, S, replace=False)))
    t0 = time.perf_counter()
    for _ in range(steps):
        _oracle_tokens(wl, h_all, wg, bias, w13, w2, np.sort(rng.choice(T, S, replace=False)))
    el = time.perf_counter() - t0
    value = S * steps / el
    sample = (f"{S} tokens per step drawn from the T={T} batch; router, top-k, FFN of their "
              f"{S * wl.top_k} routes and combine, fp64 oracle with {cores} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": warm, "ms_per_step": 1e3 * el / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(wl, T, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def _oracle_tokens(wl, h_all, wg, bias, w13, w2, tokens, nthreads=0):
    import numpy as np
    import oracle
    h = h_all[tokens]
    l = oracle.router_logits(h, wg, bias, nthreads=nthreads)
    idx, gates = oracle.select_topk(l, wl.top_k)
    n = len(tokens)
    toks = np.repeat(np.arange(n), wl.top_k).astype(np.int32)
    y = oracle.expert_rows(toks, idx.reshape(-1), h, w13, w2, nthreads)
    kept = np.ones(idx.size, np.uint8)
    return oracle.combine_rows(np.arange(n), h, gates, kept, y.reshape(n, wl.top_k, wl.hidden))


WORKLOAD_NAMES = {"tiny": "tiny MoE layer", "mix": "mixtral-like MoE layer",
                  "qw": "qwen3-moe-like MoE layer (near-tied router)",
                  "cap": "capacity-limited top-2 MoE layer (cf 1.0, Zipf skew)",
                  "ds": "deepseek-v3-like MoE layer (+1 shared expert)"}


def workload_config(wl, T, world, cfg=None):
    cfg = cfg or wl.cfg
    shared = f", shared expert {wl.shared_intermediate}" if wl.shared_intermediate else ""
    cf = cfg.get("capacity_factor", 0.0)
    cap = f", capacity factor {cf}" if cf > 0 else ""
    mode = ""
    if cfg.get("routing", 0) == 1:
        mode = ", expert-choice routing"
    elif cfg.get("overflow_policy", 0) == 1 and cf > 0:
        mode = ", overflow reroute"
    return {"workload": (f"{WORKLOAD_NAMES.get(wl.name, wl.name)} forward: hidden {wl.hidden}, "
                         f"{wl.num_experts} experts, top-{wl.top_k}, SwiGLU intermediate "
                         f"{wl.intermediate}{shared}, block {wl.block_size}{cap}{mode}, "
                         f"T={T} tokens per GPU"),
            "tokens_per_gpu": T, "global_batch": T * world, "seed": 0,
            "l2": (f"inputs larger than L2: {wl.weight_bytes() / 1e9:.1f} GB of expert weights, "
                   "the touched experts' weights are read every step"),
            "parallelism": ("single GPU" if world == 1
                            else f"{world} token shards, one all-gather of per-expert route counts per step "
                                 "(the capacity of the whole batch)"
                            if cf > 0 and cfg.get("overflow_policy", 0) == 0 and cfg.get("routing", 0) == 0
                            else f"{world} token-shard replicas, no collective")}


def batch_counts(moe, cfg, wl, h_d, wg_d, bias_d, ws, device):
    """Kept routes, touched experts and dropped routes of one batch (for the
    algorithmic work), through the stage entry points of the layer's mode.
    Expert choice drops no route; its third number is the tokens no expert
    took."""
    import torch
    T = h_d.shape[0]
    N = wl.num_experts
    ec = cfg.get("routing", 0) == 1
    slots = N if ec else wl.top_k
    R = T * slots
    kept = torch.empty(R, dtype=torch.uint8, device=device)
    pos = torch.empty(R, dtype=torch.int32, device=device)
    srt = torch.empty(moe.moe_max_padded_rows(cfg, T), dtype=torch.int32, device=device)
    blk = torch.empty(moe.moe_max_blocks(cfg, T), dtype=torch.int32, device=device)
    npad = torch.empty(1, dtype=torch.int32, device=device)
    counts = torch.empty(N, dtype=torch.int32, device=device)
    dropped = torch.zeros(1, dtype=torch.int32, device=device)
    logits = torch.empty((T, N), dtype=torch.float32, device=device)
    if ec:
        gates = torch.empty(R, dtype=torch.float32, device=device)
        moe.moe_router_logits(cfg, h_d, wg_d, bias_d, logits, ws)
        moe.moe_route_expert_choice(cfg, logits, gates, kept, pos, srt, blk, npad, counts, ws)
        third = int((kept.view(T, N).sum(dim=1) == 0).sum().item())
    else:
        idx = torch.empty((T, wl.top_k), dtype=torch.int32, device=device)
        gates = torch.empty((T, wl.top_k), dtype=torch.float32, device=device)
        reroute = cfg.get("overflow_policy", 0) == 1 and cfg.get("capacity_factor", 0.0) > 0
        moe.moe_route(cfg, h_d, wg_d, bias_d, idx, gates, logits if reroute else None, ws)
        if reroute:
            rexp = torch.empty(R, dtype=torch.int32, device=device)
            nrer = torch.zeros(1, dtype=torch.int32, device=device)
            moe.moe_dispatch_align_reroute(cfg, idx, logits, kept, rexp, pos, srt, blk, npad, counts,
                                           dropped, nrer, ws)
        else:
            moe.moe_dispatch_align(cfg, idx, kept, pos, srt, blk, npad, counts, dropped, ws)
        third = int(dropped.item())
    c = counts.cpu().numpy()
    return int(c.sum()), int((c > 0).sum()), third


def time_graph_cold(fwd, n, flush):
    """Per-forward device times of `fwd`, captured once in a CUDA graph and
    replayed n times, each replay between its own pair of CUDA events, with
    `flush` (a buffer larger than L2) written before each replay outside the
    events, so that every replay reads its weights from HBM."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fwd()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fwd()
    for _ in range(3):
        graph.replay()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    del graph
    return [a.elapsed_time(b) for a, b in ev]


# The configured layers and batch sizes (the layer shapes of synth.workloads;
# batch sizes per layer as configured there, the DeepSeek-like layer at its
# decode sizes and its largest invariance batch)
CONFIGURED = [("tiny", (64,)), ("mix", (1, 16, 128, 4096)), ("qw", (1, 32, 512, 8192)),
              ("cap", (8192,)), ("ds", (1, 64, 16448))]


def run_workloads(moe, W, device, peaks, skip):
    """One entry per configured (layer, T) except `skip` (the headline):
    cold-L2 graph-replay time, tokens/s, the layer's algorithmic work and its
    fraction of the bound's measured peak, and one forward's stage times."""
    import numpy as np
    import torch
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_gb = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    ridge = peak_tf * 1e12 / (peak_gb * 1e9)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()
    names = ["router", "dispatch_align", "tile_list_and_row_gather", "w13_gemm", "w2_gemm",
             "shared_expert", "combine"]
    out = []
    for name, Ts in CONFIGURED:
        Ts = [t for t in Ts if (name, t) != tuple(skip)]
        if not Ts:
            continue
        wl = W.WORKLOADS[name]
        cfg = dict(wl.cfg)
        wg, bias = W.make_router(wl)
        wg_d = dev_bf16(wg, device)
        bias_d = None if bias is None else dev(bias, device)
        w13_d, w2_d, w13s_d, w2s_d = W.make_experts_device(wl, 0, device)
        ws = moe.workspace(cfg, max(Ts), device)
        for T in Ts:
            h_d = dev_bf16(W.make_h(wl, T, seed=17), device)
            o_d = torch.empty((T, wl.hidden), dtype=torch.bfloat16, device=device)

            def fwd():
                moe.moe_forward(cfg, h_d, wg_d, bias_d, w13_d, w2_d, w13s_d, w2s_d, o_d, ws)

            moe.moe_clear_device_status(ws)
            for _ in range(3):
                fwd()
            n_it = 30 if T <= 512 else 10
            ms_eager = time_forwards(moe, fwd, 5, stream)
            times = time_graph_cold(fwd, n_it, flush)
            ms = float(np.mean(times))
            # stage split of one more (cold) forward
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
            for e in ev:
                e.record(stream)
            flush.fill_(1)
            moe.moe_forward_timed(cfg, h_d, wg_d, bias_d, w13_d, w2_d, w13s_d, w2s_d, o_d, ws, ev)
            torch.cuda.synchronize()
            stage = {nm: ev[i].elapsed_time(ev[i + 1]) for i, nm in enumerate(names)}
            if moe.moe_get_device_status(ws) & moe.MOE_DEV_ERR_MASK:
                raise RuntimeError(f"device status word set on {name} T={T}")
            kr, tch, dropped = batch_counts(moe, cfg, wl, h_d, wg_d, bias_d, ws, device)
            f_s, b_s = algorithmic_work(wl, T, kr, tch)
            bound = "tensor" if f_s / b_s >= ridge else "hbm"
            e = {"workload": name, "T": T, "ms": ms, "ms_median": float(np.median(times)),
                 "ms_min": float(np.min(times)), "ms_eager_warm": ms_eager, "replays": n_it,
                 "tokens_per_s": T / (ms * 1e-3), "kept_routes": kr, "dropped_routes": dropped,
                 "touched_experts": tch, "algorithmic_gflop": f_s / 1e9, "algorithmic_gb": b_s / 1e9,
                 "tflops": f_s / (ms * 1e-3) / 1e12, "gbs": b_s / (ms * 1e-3) / 1e9, "bound": bound,
                 "launches": moe.moe_forward_launch_count(cfg, T),
                 "stage_ms_one_cold_forward": stage}
            e["frac"] = e["tflops"] / peak_tf if bound == "tensor" else e["gbs"] / peak_gb
            e["peak"] = peak_tf if bound == "tensor" else peak_gb
            e["peak_unit"] = "TFLOP/s (measured bf16 burst)" if bound == "tensor" else "GB/s (measured HBM copy)"
            out.append(e)
            del h_d, o_d
        del w13_d, w2_d, w13s_d, w2s_d, ws, wg_d, bias_d
        torch.cuda.empty_cache()
    return out


def time_forwards(moe, fwd, n, stream):
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        fwd()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


# --------------------------------------------------------------------------- GPU arm
def run_gpu(args):
    import numpy as np
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())

    import invariant_expert_routing_gb300 as moe
    from synth import workloads as W

    wl = W.WORKLOADS[args.workload]
    if args.num_experts is not None:
        # a smaller case of the same layer (fewer routed experts, the same
        # kernels), for profilers: the full-set counters want a few GB on the
        # device at most
        import dataclasses
        wl = dataclasses.replace(wl, name=f"{wl.name}{args.num_experts}", num_experts=args.num_experts)
    T = args.tokens
    if T is None:   # the workload's largest configured batch (the Mixtral-like layer: 4096)
        T = max(wl.tokens)
    cfg = dict(wl.cfg)
    if args.capacity_factor is not None:
        cfg["capacity_factor"] = args.capacity_factor
    cfg["overflow_policy"] = 1 if args.policy == "reroute" else 0
    cfg["routing"] = 1 if args.routing == "expert" else 0
    default_mode = (cfg["overflow_policy"] == 0 and cfg["routing"] == 0
                    and cfg["capacity_factor"] == wl.capacity_factor)
    wg, bias = W.make_router(wl)
    wg_d = dev_bf16(wg, device)
    bias_d = None if bias is None else dev(bias, device)
    w13_d, w2_d, w13s_d, w2s_d = W.make_experts_device(wl, 0, device)
    h = W.make_h(wl, T, seed=shard_seed(rank))
    h_d = dev_bf16(h, device)
    out_d = torch.empty((T, wl.hidden), dtype=torch.bfloat16, device=device)
    ws = moe.workspace(cfg, T, device)
    moe.moe_clear_device_status(ws)
    stream = torch.cuda.current_stream()

    def fwd():
        moe.moe_forward(cfg, h_d, wg_d, bias_d, w13_d, w2_d, w13s_d, w2s_d, out_d, ws)

    if args.profile_run:
        # a short fixed run for profilers: warm-up forwards, then `steps` forwards
        for _ in range(args.warmup + args.steps):
            fwd()
        torch.cuda.synchronize()
        st = moe.moe_get_device_status(ws)
        print(json.dumps({"profile_run": True, "forwards": args.warmup + args.steps, "status": st}))
        return 0 if st == 0 else 1

    for _ in range(max(args.warmup, 3)):
        fwd()
    torch.cuda.synchronize()
    if moe.moe_get_device_status(ws) & moe.MOE_DEV_ERR_MASK:
        raise RuntimeError("device status word set during warm-up")

    # ---- timed region: K forwards, stage events recorded inside each one
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for row in ev:        # torch creates the CUDA event on its first record
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    # a capacity-limited batch sharded over ranks keeps the global batch-order
    # capacity: every step routes, exchanges the per-expert route counts (one
    # all-gather of N + 1 integers) and dispatches with the lower ranks' sums
    shard_mode = (world > 1 and cfg["capacity_factor"] > 0 and cfg["overflow_policy"] == 0
                  and cfg["routing"] == 0)
    if shard_mode:
        from invariant_expert_routing_gb300 import shard

        def fwd_shard():
            return shard.forward_shard(cfg, h_d, wg_d, bias_d, w13_d, w2_d, w13s_d, w2s_d, out_d, ws)

        for _ in range(3):
            fwd_shard()
        torch.cuda.synchronize()
    clocks = ClockSampler(visible_gpu_index(local))
    clocks.start()
    time.sleep(0.6)
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start.record(stream)
    for i in range(K):
        if shard_mode:
            fwd_shard()
        else:
            moe.moe_forward_timed(cfg, h_d, wg_d, bias_d, w13_d, w2_d, w13s_d, w2s_d, out_d, ws, ev[i])
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier()
    time.sleep(0.3)
    clocks.stop()
    ms_total = start.elapsed_time(end)
    ms_total = reduce_max(ms_total, device)
    ms_step = ms_total / K
    if shard_mode:
        # stage times for the roofline: the fused forward on this shard with a
        # local capacity (the staged calls of the shard step have no
        # in-kernel stage marks)
        for i in range(K):
            moe.moe_forward_timed(cfg, h_d, wg_d, bias_d, w13_d, w2_d, w13s_d, w2s_d, out_d, ws, ev[i])
        torch.cuda.synchronize()
    stage = np.array([[ev[i][j].elapsed_time(ev[i][j + 1]) for j in range(7)] for i in range(K)])
    stage_ms = stage.mean(axis=0)
    names = ["router", "dispatch_align", "tile_list_and_row_gather", "w13_gemm", "w2_gemm",
             "shared_expert", "combine"]
    if moe.moe_get_device_status(ws) & moe.MOE_DEV_ERR_MASK:
        raise RuntimeError("device status word set during the timed region")

    # ---- algorithmic work of this batch and the roofline of the dominant kernel
    kept_routes, touched, dropped = batch_counts(moe, cfg, wl, h_d, wg_d, bias_d, ws, device)
    flops, bytes_ = algorithmic_work(wl, T, kept_routes, touched)
    peaks, peak_src = load_peaks()
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_gb = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    i_w13 = names.index("w13_gemm")
    w13_s = stage_ms[i_w13] * 1e-3
    w13_flops = 4.0 * wl.hidden * wl.intermediate * kept_routes
    w13_bytes = 4.0 * wl.hidden * wl.intermediate * touched + 4.0 * kept_routes * wl.hidden
    ridge = peak_tf * 1e12 / (peak_gb * 1e9)
    traffic, traffic_src = profiled_traffic("expert_w13_gemm", f"{wl.name}_T{T}")
    if not default_mode:
        traffic, traffic_src = None, "no ncu summary for this routing mode"
    if w13_flops / w13_bytes >= ridge:
        roof = {"bound": "tensor", "achieved": w13_flops / w13_s / 1e12, "peak": peak_tf,
                "unit": "TFLOP/s", "peak_source": f"{peak_src} bf16 burst",
                "algorithmic_flops_per_launch": w13_flops}
    else:
        roof = {"bound": "hbm", "achieved": w13_bytes / w13_s / 1e9, "peak": peak_gb,
                "unit": "GB/s", "peak_source": f"{peak_src} HBM copy",
                "algorithmic_bytes_per_launch": w13_bytes}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if roof["bound"] == "tensor":
        # the kernel runs inside a loop of forwards long enough for the power
        # cap to lower the SM clock: the sustained GEMM peak is the other yardstick
        sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        roof["peak_sustained"] = sus
        roof["frac_of_sustained"] = roof["achieved"] / sus
    roof.update({"kernel": "expert_w13_gemm (tcgen05 grouped GEMM + SiLU*up)", "traffic": traffic,
                 "traffic_source": traffic_src, "avg_launch_ms": float(stage_ms[i_w13]),
                 "dominant_stage": names[int(np.argmax(stage_ms))]})

    value = world * T / (ms_step * 1e-3)
    layer_tf = flops / (ms_step * 1e-3) / 1e12
    layer_gb = bytes_ / (ms_step * 1e-3) / 1e9
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded counter-based generator; no checkpoints)",
            "config": workload_config(wl, T, world, cfg), "roofline": roof,
            "layer_roofline": {"algorithmic_gflop": flops / 1e9, "algorithmic_gb": bytes_ / 1e9,
                               "kept_routes": kept_routes,
                               ("tokens_without_expert" if cfg["routing"] == 1
                                else "dropped_routes"): dropped,
                               "touched_experts": touched, "tflops": layer_tf,
                               "frac_of_bf16_peak": layer_tf / peak_tf, "gbs": layer_gb,
                               "frac_of_hbm": layer_gb / peak_gb},
            "stage_ms": {n: float(v) for n, v in zip(names, stage_ms)},
            "gpu_launches": (moe.moe_forward_launch_count(cfg, T) + (1 if shard_mode else 0)) * K,
            "clocks": clocks.summary(t_wall0, t_wall1)}
    if shard_mode:
        line["config"]["capacity_exchange"] = (
            "capacity of the whole batch (all ranks' tokens in rank order); per step one all-gather "
            "of each rank's per-expert route counts + token count (N + 1 ints) and "
            "moe_dispatch_align_shard; stage_ms, the roofline, the sweep and e2e from local-capacity "
            "fused forwards")

    # ---- routing diagnostics on this batch: the routing_stats probe and the
    # router margin (device time per call, 50 calls each)
    if cfg["routing"] == 0:
        idx_d = torch.empty((T, wl.top_k), dtype=torch.int32, device=device)
        gate_d = torch.empty((T, wl.top_k), dtype=torch.float32, device=device)
        logit_d = torch.empty((T, wl.num_experts), dtype=torch.float32, device=device)
        moe.moe_route(cfg, h_d, wg_d, bias_d, idx_d, gate_d, logit_d, ws)
        load_d = torch.empty(wl.num_experts, dtype=torch.int32, device=device)
        stats_d = torch.empty(64, dtype=torch.uint8, device=device)
        margin_d = torch.empty(T, dtype=torch.float64, device=device)
        ms_stats = time_forwards(moe, lambda: moe.moe_routing_stats(cfg, idx_d, 1.25, load_d, stats_d),
                                 50, stream)
        ms_margin = time_forwards(moe, lambda: moe.moe_router_margin(cfg, logit_d, margin_d), 50, stream)
        st = moe.route_stats_from_bytes(stats_d.cpu().numpy().tobytes())
        m = margin_d.cpu().numpy()
        line["diagnostics"] = {"routing_stats_us": 1e3 * ms_stats, "router_margin_us": 1e3 * ms_margin,
                               "routing_stats_cf_1.25": st,
                               "margin_quantiles": {q: float(v) for q, v in
                                                    zip(("p01", "p10", "p50"),
                                                        np.quantile(m, [0.01, 0.1, 0.5]))},
                               "tokens_with_zero_margin": int((m == 0).sum())}

    # ---- end to end through the host-buffer entry point
    h_host = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).pin_memory()
    out_host = torch.empty((T, wl.hidden), dtype=torch.bfloat16).pin_memory()

    def fwd_host():
        moe.moe_forward_hostio(cfg, h_host, wg_d, bias_d, w13_d, w2_d, w13s_d, w2s_d, out_host, ws)

    for _ in range(2):
        fwd_host()
    torch.cuda.synchronize()
    barrier()
    ms_e2e = reduce_max(time_forwards(moe, fwd_host, max(5, min(K, 50)), stream), device)
    line["e2e"] = {"value": world * T / (ms_e2e * 1e-3), "unit": UNIT,
                   "h2d_bytes_per_step": T * wl.hidden * 2, "d2h_bytes_per_step": T * wl.hidden * 2,
                   "ms_per_step": ms_e2e, "entry_point": "moe_forward_hostio (pinned host buffers)"}
    e2e_out = host_bf16(out_host)
    fwd()
    torch.cuda.synchronize()
    if not (host_bf16(out_d) == e2e_out).all():
        raise RuntimeError("host-buffer path and device path disagree")

    # ---- CPU oracle on the host cores (rank 0, N = 1)
    if (rank == 0 and world == 1 and not args.no_cpu_baseline and cfg["capacity_factor"] <= 0
            and default_mode and wl.weight_bytes() < (8 << 30)):
        line["cpu_baseline"] = cpu_baseline(wl, h, wg, bias, host_bf16(out_d))

    # ---- every configured layer and batch size (secondary entries, one GPU)
    if not args.no_sweep and default_mode and world == 1:
        del w13_d, w2_d, w13s_d, w2s_d, ws
        torch.cuda.empty_cache()
        line["workloads"] = run_workloads(moe, W, device, peaks, skip=(wl.name, T))
        line["workloads_timing"] = (
            "per configured (layer, T) other than the headline: the forward captured in a CUDA graph, "
            "each replay bracketed by its own CUDA events with a 512 MB buffer written between "
            "replays (cold L2: the weights and tokens come from HBM every time); ms = mean over "
            "the replays; frac against the measured bf16 burst peak (tensor-bound) or the measured "
            "HBM copy bandwidth (HBM-bound) from the layer's algorithmic flops and bytes")

    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))
    return 0


def cpu_baseline(wl, h, wg, bias, gpu_out):
    """The oracle (as it stands) on a bounded sample of the batch; also checks
    the sampled GPU rows against it.  Without capacity a token's routing
    depends on its own row, so a sample of tokens is a faithful sub-batch."""
    import numpy as np
    from synth import workloads as W
    cores = os.cpu_count() or 1
    w13, w2 = W.make_experts(wl)
    rng = np.random.default_rng(123)
    T = h.shape[0]
    S = 16
    toks = np.sort(rng.choice(T, min(S, T), replace=False))
    _oracle_tokens(wl, h, wg, bias, w13, w2, toks[:1])           # warm (page-in)
    t0 = time.perf_counter()
    done = 0
    outs = None
    while done < 4096 and time.perf_counter() - t0 < 15.0:
        sel = toks if done == 0 else np.sort(rng.choice(T, len(toks), replace=False))
        o = _oracle_tokens(wl, h, wg, bias, w13, w2, sel)
        if outs is None:
            outs = o
        done += len(sel)
    el = time.perf_counter() - t0
    err = max_err_within_tolerance(gpu_out[toks], outs)
    return {"value": done / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"{done} tokens of the T={T} batch in groups of {len(toks)} (router, top-k, "
                       f"their {done * wl.top_k} expert FFN routes in fp64, combine), {el:.1f} s"),
            "parity_on_sample": {"tokens": len(toks), "max_abs_err": err,
                                 "tolerance": "2e-2 + 1e-2*|ref|"}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the entries of the other configured layers and batch sizes")
    ap.add_argument("--workload", default=WORKLOAD, choices=["tiny", "mix", "qw", "cap", "ds"])
    ap.add_argument("--tokens", type=int, default=None,
                    help="tokens per GPU (default: the workload's largest configured batch)")
    ap.add_argument("--capacity-factor", type=float, default=None,
                    help="override the workload's capacity factor")
    ap.add_argument("--policy", default="drop", choices=["drop", "reroute"],
                    help="overflow policy for routes past an expert's capacity")
    ap.add_argument("--routing", default="token", choices=["token", "expert"],
                    help="token choice (top-k) or expert choice (top-C tokens per expert)")
    ap.add_argument("--num-experts", type=int, default=None,
                    help="with --profile-run: the layer with this many routed experts (a small case)")
    ap.add_argument("--profile-run", action="store_true",
                    help="only warm-up + steps forwards of the main workload (for ncu)")
    args = ap.parse_args()
    if args.num_experts is not None and not args.profile_run:
        ap.error("--num-experts is for --profile-run captures only")
    if args.warmup < 3 and not args.profile_run:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
