"""ctypes binding of libglr_moe.so (include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch provides device memory and the stream.  There is no CPU
fallback: if the library is missing or the device is not sm_103, calls fail.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED_SHAPE = -2
MOE_ERR_MISALIGNED = -3
MOE_ERR_WORKSPACE_TOO_SMALL = -4
MOE_ERR_CUDA = -5
MOE_ERR_DEVICE_STATUS = -6
MOE_ERR_TIMEOUT = -7
MOE_ERR_UNSUPPORTED_DEVICE = -8

MOE_STATUS_NONFINITE_LOGIT = 1
MOE_STATUS_BAD_EXPERT_INDEX = 2
MOE_STATUS_TIMEOUT = 4
MOE_STATUS_COUNT_MISMATCH = 8

MOE_WS_ROUTE = 0
MOE_WS_FORWARD = 1
MOE_WS_BACKWARD = 2

# every symbol include/moe.h declares
EXPORTS = ("moe_workspace_bytes", "moe_workspace_init", "moe_route", "moe_router_logits",
           "moe_route_from_logits", "moe_forward", "moe_get_status", "moe_last_launch_count",
           "moe_profile_enable", "moe_profile_read", "moe_kernel_name", "moe_strerror", "moe_route_static",
           "moe_debug_inject_timeout", "moe_rmsnorm", "moe_expert_feedback", "moe_prepare_router",
           "moe_route_prepared", "moe_dense_workspace_bytes", "moe_dense_ffn", "moe_backward",
           "moe_layer_workspace_bytes", "moe_layer", "moe_router_scores", "moe_ep_dispatch_workspace_bytes",
           "moe_ep_dispatch", "moe_expert_rows_workspace_bytes", "moe_expert_rows", "moe_combine")
MOE_ROUTE_STATIC_SCRATCH_BYTES = 40 << 20
MOE_LAYER_FUSED_ROUTER = 1
MOE_LAYER_FUSED_COMBINE = 2
MOE_KERNEL_COUNT = 19
MOE_KERNEL_STAGE_ROUTE_PERMUTE = 18   # moe_profile_read id of the routing + bucketing stage (mode 2)


class MoeCfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "H", "E", "n_group", "topk_group", "k", "I", "Is")] + \
               [("rsf", ctypes.c_float), ("eps", ctypes.c_float)]


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (what, strerror(code), code))


_lock = threading.Lock()
_handle = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libglr_moe.so (building it first only if asked)."""
    global _handle
    with _lock:
        if _handle is not None:
            return _handle
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError("CUDA library %s is not built; run __graft_entry__.build() "
                                   "or python -m group_limited_routing_gb300.build" % path)
            _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        S = ctypes.c_size_t
        C = ctypes.POINTER(MoeCfg)
        lib.moe_workspace_bytes.argtypes = [C, ctypes.c_int]
        lib.moe_workspace_bytes.restype = S
        lib.moe_workspace_init.argtypes = [P, S, P]
        lib.moe_route.argtypes = [C, P, P, P, P, P, P, P, P, P, S, P]
        lib.moe_router_logits.argtypes = [C, P, P, P, P, S, P]
        I32 = ctypes.c_int32
        lib.moe_dense_workspace_bytes.argtypes = [I32, I32, I32]
        lib.moe_dense_workspace_bytes.restype = S
        lib.moe_dense_ffn.argtypes = [I32, I32, I32, P, P, P, P, P, P, S, P]
        lib.moe_dense_ffn.restype = ctypes.c_int
        lib.moe_prepare_router.argtypes = [C, P, P, P]
        lib.moe_prepare_router.restype = ctypes.c_int
        lib.moe_route_prepared.argtypes = [C, P, P, P, P, P, P, P, P, P, P, S, P]
        lib.moe_route_prepared.restype = ctypes.c_int
        lib.moe_route_from_logits.argtypes = [C, P, P, P, P, P, P, P, P, S, P]
        lib.moe_forward.argtypes = [C, P, P, P, P, P, P, P, P, P, P, S, P]
        lib.moe_backward.argtypes = [C] + [P] * 14 + [P, S, P]
        lib.moe_layer_workspace_bytes.argtypes = [C, ctypes.c_int]
        lib.moe_layer_workspace_bytes.restype = S
        lib.moe_layer.argtypes = [C] + [P] * 15 + [ctypes.c_int, P, S, P]
        lib.moe_layer.restype = ctypes.c_int
        lib.moe_backward.restype = ctypes.c_int
        lib.moe_get_status.argtypes = [P, S, P, ctypes.POINTER(ctypes.c_int32), ctypes.c_int]
        lib.moe_last_launch_count.argtypes = []
        lib.moe_profile_enable.argtypes = [ctypes.c_int]
        lib.moe_profile_enable.restype = ctypes.c_int
        lib.moe_profile_read.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                         ctypes.POINTER(ctypes.c_int32), ctypes.c_int]
        lib.moe_profile_read.restype = ctypes.c_int
        lib.moe_kernel_name.argtypes = [ctypes.c_int]
        lib.moe_kernel_name.restype = ctypes.c_char_p
        lib.moe_expert_feedback.argtypes = [C, P, ctypes.c_float, P, P, P]
        lib.moe_expert_feedback.restype = ctypes.c_int
        lib.moe_rmsnorm.argtypes = [ctypes.c_int32, ctypes.c_int32, P, P, ctypes.c_float, P]
        lib.moe_rmsnorm.restype = ctypes.c_int
        lib.moe_debug_inject_timeout.argtypes = [ctypes.c_int]
        lib.moe_debug_inject_timeout.restype = ctypes.c_int
        lib.moe_route_static.argtypes = [C, P, P, P, P, P, P, P, P, P, P]
        lib.moe_route_static.restype = ctypes.c_int
        lib.moe_ep_dispatch_workspace_bytes.argtypes = [C, I32]
        lib.moe_ep_dispatch_workspace_bytes.restype = S
        lib.moe_ep_dispatch.argtypes = [C, I32, P, P, P, P, P, P, P, S, P]
        lib.moe_ep_dispatch.restype = ctypes.c_int
        lib.moe_expert_rows_workspace_bytes.argtypes = [C, I32]
        lib.moe_expert_rows_workspace_bytes.restype = S
        lib.moe_expert_rows.argtypes = [C, I32, P, P, P, P, P, P, S, P]
        lib.moe_expert_rows.restype = ctypes.c_int
        lib.moe_combine.argtypes = [C, P, ctypes.c_int64, ctypes.c_int64, P, P, P, P, P]
        lib.moe_combine.restype = ctypes.c_int
        lib.moe_router_scores.argtypes = [P, P, ctypes.c_int64, P]
        lib.moe_router_scores.restype = ctypes.c_int
        lib.moe_strerror.argtypes = [ctypes.c_int]
        lib.moe_strerror.restype = ctypes.c_char_p
        for name in ("moe_workspace_init", "moe_route", "moe_router_logits", "moe_route_from_logits",
                     "moe_forward", "moe_get_status", "moe_last_launch_count"):
            getattr(lib, name).restype = ctypes.c_int
        _handle = lib
        return lib


def strerror(code: int) -> str:
    try:
        return load().moe_strerror(code).decode()
    except RuntimeError:
        return "code %d" % code


def check(code: int, what: str) -> None:
    if code != MOE_OK:
        raise MoeError(code, what)
