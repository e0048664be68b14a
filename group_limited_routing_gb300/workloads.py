"""Seeded synthetic inputs for the group-limited MoE layer forward.

This module only draws random tensors with the shapes and distributions of the
five workloads below. It holds none of the layer's arithmetic, imports nothing
from the CUDA binding or from the CPU oracle, and is the one module that both
sides share (the tests feed the same tensors to each).

Shapes follow the hyper-parameter table (section 一) of the article
"InternLumina-U2中256个专家的路由秘密：分组受限Top-K、Expert Bias与Fused MoE详解":
256 experts in 8 groups of 32, 4 groups kept, top-8, expert FFN inner size 512,
hidden size 2048 (the [256, 512, 2048] weight stacks of its section 四), one
shared expert and routed_scaling_factor 2.5.

Seeds: base = 1000 * workload_id + 10 * layer, plus a per-tensor offset
(+0 hidden, +1 router weight, +2 expert bias, +3 expert weights, +4 shared
expert weights, +5 hot-expert set).  Each tensor has its own torch.Generator on
the requested device, so values depend on (seed, device, torch version) only.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes plus the recipe of its random inputs."""
    wid: int
    name: str
    T: int
    H: int
    E: int = 256
    n_group: int = 8
    topk_group: int = 4
    k: int = 8
    I: int = 512
    Is: int = 512
    rsf: float = 2.5
    eps: float = 1e-20
    bias: str = "zero"          # "zero" | "uniform0.01" | "normal0.05"
    hot_experts_per_group: int = 0
    hot_scale: float = 1.0
    layers: int = 1
    residual: bool = False

    def with_T(self, T: int) -> "Workload":
        return dataclasses.replace(self, T=T)


WORKLOADS = {
    1: Workload(1, "tiny T=128 H=512 I=Is=128", T=128, H=512, I=128, Is=128),
    2: Workload(2, "decode T=16 full size", T=16, H=2048, bias="uniform0.01"),
    3: Workload(3, "T=4096 full size, near-uniform routing", T=4096, H=2048),
    4: Workload(4, "T=32768 full size, 16 hot experts (router rows x3), bias~N(0,0.05)",
                T=32768, H=2048, bias="normal0.05", hot_experts_per_group=2, hot_scale=3.0),
    5: Workload(5, "19-layer stack T=8192 full size, residual, per-layer counts and aux loss",
                T=8192, H=2048, layers=19, residual=True),
    # workload 4's recipe with the hot rows scaled x5 instead of x3: about half
    # of all assignments then land on the 16 hot experts (x3 gives ~36%)
    6: Workload(6, "T=32768 full size, 16 hot experts (router rows x5, ~50% of assignments), bias~N(0,0.05)",
                T=32768, H=2048, bias="normal0.05", hot_experts_per_group=2, hot_scale=5.0),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def seed_base(wl: Workload, layer: int = 0) -> int:
    return 1000 * wl.wid + 10 * layer


def hidden(wl: Workload, device="cpu", layer: int = 0) -> torch.Tensor:
    """hidden ~ N(0, 1), stored as bf16 [T, H]."""
    g = _gen(seed_base(wl, layer) + 0, device)
    return torch.randn(wl.T, wl.H, generator=g, device=device).to(torch.bfloat16)


def hot_experts(wl: Workload, device="cpu", layer: int = 0) -> torch.Tensor:
    """Indices of the 'hot' experts: a seeded pick of n per group (empty if none)."""
    if wl.hot_experts_per_group == 0:
        return torch.empty(0, dtype=torch.int64)
    g = _gen(seed_base(wl, layer) + 5, "cpu")
    gs = wl.E // wl.n_group
    picks = []
    for j in range(wl.n_group):
        perm = torch.randperm(gs, generator=g)[: wl.hot_experts_per_group]
        picks.append(perm + j * gs)
    return torch.sort(torch.cat(picks)).values


def router_weight(wl: Workload, device="cpu", layer: int = 0) -> torch.Tensor:
    """Router weight ~ N(0, 0.02), fp32 [E, H]; hot experts' rows scaled."""
    g = _gen(seed_base(wl, layer) + 1, device)
    W = torch.randn(wl.E, wl.H, generator=g, device=device) * 0.02
    hot = hot_experts(wl, layer=layer)
    if hot.numel():
        W[hot.to(device)] *= wl.hot_scale
    return W.contiguous()


def expert_bias(wl: Workload, device="cpu", layer: int = 0) -> torch.Tensor:
    """expert_bias, fp32 [E]: zero, U(-0.01, 0.01) or N(0, 0.05)."""
    g = _gen(seed_base(wl, layer) + 2, device)
    if wl.bias == "zero":
        return torch.zeros(wl.E, device=device)
    if wl.bias == "uniform0.01":
        return (torch.rand(wl.E, generator=g, device=device) * 2.0 - 1.0) * 0.01
    if wl.bias == "normal0.05":
        return torch.randn(wl.E, generator=g, device=device) * 0.05
    raise ValueError(wl.bias)


def expert_weights(wl: Workload, device="cpu", layer: int = 0):
    """Routed expert weights ~ N(0, 0.02), bf16.

    Returns (W_gate_up [E, 2I, H] with rows [0, I) = gate and [I, 2I) = up,
             W_down   [E, I, H]).
    """
    g = _gen(seed_base(wl, layer) + 3, device)
    Wgu = torch.empty(wl.E, 2 * wl.I, wl.H, dtype=torch.bfloat16, device=device)
    Wd = torch.empty(wl.E, wl.I, wl.H, dtype=torch.bfloat16, device=device)
    # drawn expert by expert to bound the fp32 temporary
    for e in range(wl.E):
        Wgu[e] = (torch.randn(2 * wl.I, wl.H, generator=g, device=device) * 0.02).to(torch.bfloat16)
        Wd[e] = (torch.randn(wl.I, wl.H, generator=g, device=device) * 0.02).to(torch.bfloat16)
    return Wgu, Wd


def shared_weights(wl: Workload, device="cpu", layer: int = 0):
    """Shared expert weights ~ N(0, 0.02), bf16: (gate_up [2Is, H], down [Is, H])."""
    g = _gen(seed_base(wl, layer) + 4, device)
    sgu = (torch.randn(2 * wl.Is, wl.H, generator=g, device=device) * 0.02).to(torch.bfloat16)
    sd = (torch.randn(wl.Is, wl.H, generator=g, device=device) * 0.02).to(torch.bfloat16)
    return sgu, sd


def layer_inputs(wl: Workload, device="cpu", layer: int = 0, with_experts: bool = True):
    """Every input of one layer as a dict of tensors on `device`."""
    d = dict(
        hidden=hidden(wl, device, layer),
        W_router=router_weight(wl, device, layer),
        expert_bias=expert_bias(wl, device, layer),
    )
    if with_experts:
        d["W_gate_up"], d["W_down"] = expert_weights(wl, device, layer)
        d["shared_gate_up"], d["shared_down"] = shared_weights(wl, device, layer)
    return d


def token_sample(T: int, n: int, seed: int = 7) -> torch.Tensor:
    """A seeded, sorted sample of n distinct token indices in [0, T)."""
    if n >= T:
        return torch.arange(T, dtype=torch.int32)
    g = _gen(seed, "cpu")
    return torch.sort(torch.randperm(T, generator=g)[:n]).values.to(torch.int32)


def random_routing(T: int, E: int, k: int, seed: int, device="cpu",
                   skew: Optional[torch.Tensor] = None):
    """Random distinct expert ids per token (no group structure) and positive
    weights, for exercising the expert stage on routings the router would not
    produce (empty experts, hot experts, ragged buckets)."""
    g = _gen(seed, "cpu")
    if skew is None:
        keys = torch.rand(T, E, generator=g)
    else:
        keys = torch.rand(T, E, generator=g) * skew.view(1, E)
    idx = torch.topk(keys, k, dim=1).indices.to(torch.int32)
    w = torch.rand(T, k, generator=g) * 0.5
    return idx.to(device), w.to(device)
