"""Layer shapes and the seeded input recipe for each synthetic workload.

No checkpoints or datasets exist for these model families here, so every
tensor is drawn from the counter-based generator in this package with the
shapes and value distributions stated below (standard deviations, not
variances, except where a variance is written as 1/H):

  tiny  H128  N8   k2 I256   B8   T64            h~N(0,1), W_g~N(0,1/H), experts~N(0,0.02^2)
  mix   H4096 N8   k2 I14336 B64  T in 1,16,128,4096   same distributions
  qw    H2048 N128 k8 I768   B16  T in 1,32,512,8192   near-tied router: a base bias shared
        by every token, b_e = 0.25*U{0..3}, plus noise h.W_g with std 1e-3
        (W_g std 1e-3/sqrt(H)); 1 % of tokens have h = 0, so their logits equal
        b exactly and only the lowest-index tie-break decides their experts
  cap   mix shapes, T8192, capacity factor 1.0, Zipf(s=1.2) skew through the
        router bias b_e = -beta*1.2*ln(e+1); beta is calibrated (on the CPU
        checker) so that about 15 % of routes overflow
  ds    H7168 N256 k8 I2048 B16 + one always-on shared expert (I 2048)

The generator holds none of the layer's arithmetic; it only produces inputs.
"""
from __future__ import annotations

import json
import math
import os
from dataclasses import dataclass, field

import numpy as np

from . import normal_bf16, normal_bf16_device, uniform_u64

# tensor ids of the counter-based streams
TID_H = 1
TID_WG = 2
TID_W13 = 3
TID_W2 = 4
TID_W13S = 5
TID_W2S = 6
TID_BIAS = 7
TID_ZERO_TOKENS = 8

_GOLDEN = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                       "tests", "golden", "cap_bias.json")


@dataclass(frozen=True)
class Workload:
    name: str
    hidden: int
    num_experts: int
    top_k: int
    intermediate: int
    block_size: int
    capacity_factor: float = 0.0
    shared_intermediate: int = 0
    tokens: tuple = field(default=(64,))
    h_std: float = 1.0
    wg_std: float = 0.0
    expert_std: float = 0.02
    bias: str = "none"          # "none" | "qw_base" | "zipf"
    zero_token_pct: int = 0

    @property
    def cfg(self) -> dict:
        return dict(hidden=self.hidden, num_experts=self.num_experts, top_k=self.top_k,
                    intermediate=self.intermediate, block_size=self.block_size,
                    capacity_factor=self.capacity_factor,
                    shared_intermediate=self.shared_intermediate)

    def weight_bytes(self) -> int:
        per = 3 * self.hidden * self.intermediate * 2
        sh = 3 * self.hidden * self.shared_intermediate * 2
        return self.num_experts * per + sh + self.hidden * self.num_experts * 2


WORKLOADS = {
    "tiny": Workload("tiny", 128, 8, 2, 256, 8, tokens=(64,), wg_std=1 / math.sqrt(128)),
    "mix": Workload("mix", 4096, 8, 2, 14336, 64, tokens=(1, 16, 128, 4096),
                    wg_std=1 / math.sqrt(4096)),
    "qw": Workload("qw", 2048, 128, 8, 768, 16, tokens=(1, 32, 512, 8192),
                   wg_std=1e-3 / math.sqrt(2048), bias="qw_base", zero_token_pct=1),
    "cap": Workload("cap", 4096, 8, 2, 14336, 64, capacity_factor=1.0, tokens=(8192,),
                    wg_std=1 / math.sqrt(4096), bias="zipf"),
    "ds": Workload("ds", 7168, 256, 8, 2048, 16, shared_intermediate=2048,
                   tokens=(1, 64, 16448), wg_std=1 / math.sqrt(7168)),
}


def cap_beta() -> float:
    """Zipf strength calibrated by oracle/calibrate_cap_bias.py (seed 0)."""
    with open(_GOLDEN) as f:
        return float(json.load(f)["beta"])


def make_h(wl: Workload, T: int, seed: int = 0) -> np.ndarray:
    """Token hidden states [T, H] as bf16 bit patterns."""
    h = normal_bf16((T, wl.hidden), seed, TID_H, wl.h_std)
    if wl.zero_token_pct:
        u = uniform_u64(T, seed, TID_ZERO_TOKENS)
        h[(u % np.uint64(100)) < np.uint64(wl.zero_token_pct)] = 0
    return h


def make_router(wl: Workload, seed: int = 0, beta: float | None = None):
    """Router weight W_g [H, N] (bf16 bits) and bias [N] (float32 or None)."""
    wg = normal_bf16((wl.hidden, wl.num_experts), seed, TID_WG, wl.wg_std)
    if wl.bias == "none":
        return wg, None
    if wl.bias == "qw_base":
        u = uniform_u64(wl.num_experts, seed, TID_BIAS)
        return wg, (0.25 * (u % np.uint64(4)).astype(np.float64)).astype(np.float32)
    if wl.bias == "zipf":
        b = cap_beta() if beta is None else beta
        e = np.arange(wl.num_experts, dtype=np.float64)
        return wg, (-b * 1.2 * np.log(e + 1.0)).astype(np.float32)
    raise ValueError(wl.bias)


def expert_w13(wl: Workload, e: int, seed: int = 0) -> np.ndarray:
    """W13 of expert e, [H, 2I] (gate columns 0..I-1, up columns I..2I-1)."""
    n = wl.hidden * 2 * wl.intermediate
    return normal_bf16((wl.hidden, 2 * wl.intermediate), seed, TID_W13, wl.expert_std, offset=e * n)


def expert_w2(wl: Workload, e: int, seed: int = 0) -> np.ndarray:
    """W2 of expert e, [I, H]."""
    n = wl.intermediate * wl.hidden
    return normal_bf16((wl.intermediate, wl.hidden), seed, TID_W2, wl.expert_std, offset=e * n)


def make_experts(wl: Workload, seed: int = 0):
    """All routed expert weights on the host: W13 [N,H,2I], W2 [N,I,H]."""
    w13 = normal_bf16((wl.num_experts, wl.hidden, 2 * wl.intermediate), seed, TID_W13, wl.expert_std)
    w2 = normal_bf16((wl.num_experts, wl.intermediate, wl.hidden), seed, TID_W2, wl.expert_std)
    return w13, w2


def make_shared(wl: Workload, seed: int = 0):
    """Shared expert weights W13s [H, 2Is], W2s [Is, H], or (None, None)."""
    if not wl.shared_intermediate:
        return None, None
    Is = wl.shared_intermediate
    return (normal_bf16((wl.hidden, 2 * Is), seed, TID_W13S, wl.expert_std),
            normal_bf16((Is, wl.hidden), seed, TID_W2S, wl.expert_std))


def make_experts_device(wl: Workload, seed: int = 0, device="cuda"):
    """Routed (and shared) expert weights generated directly on the device."""
    import torch
    N, H, I, Is = wl.num_experts, wl.hidden, wl.intermediate, wl.shared_intermediate
    w13 = torch.empty((N, H, 2 * I), dtype=torch.bfloat16, device=device)
    w2 = torch.empty((N, I, H), dtype=torch.bfloat16, device=device)
    normal_bf16_device(w13, seed, TID_W13, wl.expert_std)
    normal_bf16_device(w2, seed, TID_W2, wl.expert_std)
    w13s = w2s = None
    if Is:
        w13s = torch.empty((H, 2 * Is), dtype=torch.bfloat16, device=device)
        w2s = torch.empty((Is, H), dtype=torch.bfloat16, device=device)
        normal_bf16_device(w13s, seed, TID_W13S, wl.expert_std)
        normal_bf16_device(w2s, seed, TID_W2S, wl.expert_std)
    return w13, w2, w13s, w2s
