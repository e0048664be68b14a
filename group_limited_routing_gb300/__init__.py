"""GB300-native (sm_103a) forward of a fine-grained MoE layer with
group-limited routing.

The layer follows the article "InternLumina-U2中256个专家的路由秘密：分组受限
Top-K、Expert Bias与Fused MoE详解".  The compute runs in libglr_moe.so (C ABI
in include/moe.h, hand-written CUDA kernels); this package is its binding.

Submodules load lazily so that ``group_limited_routing_gb300.workloads`` (the
seeded input generators) imports without the CUDA library.
"""
import importlib

__all__ = ["moe", "workloads", "build", "MoeConfig", "MoELayer", "route", "forward", "router_logits",
           "route_from_logits", "Workspace"]

_FROM_MOE = {"MoeConfig", "MoELayer", "route", "forward", "router_logits", "route_from_logits", "Workspace",
             "last_launch_count", "workspace_bytes"}


def __getattr__(name):
    if name in _FROM_MOE:
        return getattr(importlib.import_module(".moe", __name__), name)
    if name in ("moe", "workloads", "build", "_lib"):
        return importlib.import_module("." + name, __name__)
    raise AttributeError(name)
