"""CPU oracle of the group-limited MoE layer forward (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its binding) never imports, links or runs
it, and the two share no code; the oracle's arithmetic lives in
``moe_oracle.c`` (plain loops, double accumulation) and is cited there
against the article "InternLumina-U2中256个专家的路由秘密：分组受限Top-K、
Expert Bias与Fused MoE详解" (the routing page) and the load-balancing-loss
section of the InternLumina-U2 training-pitfalls article.

Arrays are numpy: bf16 tensors travel as their uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


class _Cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("T", "H", "E", "n_group", "topk_group", "k", "I", "Is")] + \
               [("rsf", ctypes.c_float), ("eps", ctypes.c_float)]


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into oracle/_build/liboracle.so with gcc."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            lib.orc_router_logits.argtypes = [ctypes.c_int] * 3 + [P, P, P]
            lib.orc_route.argtypes = [ctypes.POINTER(_Cfg), P, P, P, P, P, P, P]
            lib.orc_route.restype = ctypes.c_int
            lib.orc_counts_aux.argtypes = [ctypes.c_int] * 3 + [P, P, P, P]
            lib.orc_counts_aux.restype = ctypes.c_double
            lib.orc_experts.argtypes = [ctypes.POINTER(_Cfg)] + [P] * 8 + [ctypes.c_int, P, P]
            lib.orc_experts_opt.argtypes = [ctypes.POINTER(_Cfg)] + [P] * 8 + [ctypes.c_int, P, P, ctypes.c_int]
            lib.orc_experts_opt.restype = ctypes.c_int
            lib.orc_experts_backward.argtypes = [ctypes.POINTER(_Cfg)] + [P] * 8 + [ctypes.c_int] + [P] * 6
            lib.orc_experts_backward.restype = ctypes.c_int
            lib.orc_experts.restype = ctypes.c_int
            lib.orc_bf16_round_array.argtypes = [P, P, ctypes.c_long]
            lib.orc_rmsnorm.argtypes = [ctypes.c_int, ctypes.c_int, P, ctypes.c_float, P]
            lib.orc_expert_feedback.argtypes = [ctypes.c_int] * 3 + [P, ctypes.c_float, P, P]
            lib.orc_set_threads.argtypes = [ctypes.c_int]
            lib.orc_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _cfg(T=0, H=0, E=256, n_group=8, topk_group=4, k=8, I=0, Is=0, rsf=2.5, eps=1e-20):
    return _Cfg(T, H, E, n_group, topk_group, k, I, Is, rsf, eps)


def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns as float32."""
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_round(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even (oracle's own rounding)."""
    a = _c(a, np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().orc_bf16_round_array(_p(a), _p(out), a.size)
    return out


def router_logits(x_bf16: np.ndarray, W: np.ndarray) -> np.ndarray:
    """fp32 logits [T, E] = x . W^T, exact in double and rounded once."""
    x = _c(x_bf16, np.uint16)
    W = _c(W, np.float32)
    T, H = x.shape
    E = W.shape[0]
    out = np.empty((T, E), dtype=np.float32)
    _load().orc_router_logits(T, H, E, _p(x), _p(W), _p(out))
    return out


def route(logits: np.ndarray, bias=None, n_group=8, topk_group=4, k=8, rsf=2.5, eps=1e-20):
    """Group-limited top-k from fp32 logits.  Returns a dict with idx [T,k]
    int32, w [T,k] fp32, scores [T,E] fp32 (unbiased), margin_group [T] and
    margin_expert [T] (float64)."""
    L = _c(logits, np.float32)
    T, E = L.shape
    b = _c(bias, np.float32)
    c = _cfg(T=T, E=E, n_group=n_group, topk_group=topk_group, k=k, rsf=rsf, eps=eps)
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    s = np.empty((T, E), dtype=np.float32)
    mg = np.empty(T, dtype=np.float64)
    me = np.empty(T, dtype=np.float64)
    rc = _load().orc_route(ctypes.byref(c), _p(L), _p(b), _p(idx), _p(w), _p(s), _p(mg), _p(me))
    if rc == -1:
        raise ValueError("unsupported routing shape")
    if rc == -2:
        raise FloatingPointError("non-finite logit or bias")
    return dict(idx=idx, w=w, scores=s, margin_group=mg, margin_expert=me)


def counts_aux(idx: np.ndarray, scores=None, E=256):
    """(counts [E] int32, P [E] float64 or None, aux loss float or None)."""
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, dtype=np.int32)
    s = _c(scores, np.float32)
    P = np.empty(E, dtype=np.float64) if s is not None else None
    aux = _load().orc_counts_aux(T, E, k, _p(idx), _p(s), _p(counts), _p(P))
    return counts, P, (aux if s is not None else None)


def experts(x_bf16, W_gate_up, W_down, shared_gate_up, shared_down, idx, w,
            residual=None, tokens=None, E=None, round_act=True):
    """Layer output in float64 for the listed tokens (all by default):
    sum_j w[t,j] * SwiGLU_{idx[t,j]}(x[t]) + shared(x[t]) (+ residual[t]).
    round_act=False keeps the SwiGLU intermediate unrounded (a smooth function
    of every input, for finite-difference checks of the backward)."""
    x = _c(x_bf16, np.uint16)
    T, H = x.shape
    Wgu = _c(W_gate_up, np.uint16)
    Wd = _c(W_down, np.uint16)
    E = Wgu.shape[0] if E is None else E
    I = Wd.shape[1]
    sgu = _c(shared_gate_up, np.uint16)
    sd = _c(shared_down, np.uint16)
    Is = 0 if sd is None else sd.shape[0]
    idx = _c(idx, np.int32)
    w = _c(w, np.float32)
    k = idx.shape[1]
    res = _c(residual, np.uint16)
    tok = None if tokens is None else _c(tokens, np.int32)
    n = T if tok is None else tok.size
    c = _cfg(T=T, H=H, E=E, k=k, I=I, Is=Is)
    out = np.empty((n, H), dtype=np.float64)
    rc = _load().orc_experts_opt(ctypes.byref(c), _p(x), _p(Wgu), _p(Wd), _p(sgu), _p(sd), _p(idx), _p(w),
                                 _p(res), n, _p(tok), _p(out), 1 if round_act else 0)
    if rc != 0:
        raise IndexError("expert index out of range")
    return out


def experts_backward(x_bf16, W_gate_up, W_down, shared_gate_up, shared_down, idx, w, d_out, round_act=True):
    """Backward of experts() for fixed routing, in float64: given d_out [T, H],
    returns dict(dx [T, H], dW_gate_up [E, 2I, H], dW_down [E, I, H],
    d_shared_gate_up [2Is, H], d_shared_down [Is, H], dw [T, k]).  The
    intermediate's bf16 rounding (round_act) passes gradients unchanged."""
    x = _c(x_bf16, np.uint16)
    T, H = x.shape
    Wgu = _c(W_gate_up, np.uint16)
    Wd = _c(W_down, np.uint16)
    E, I = Wgu.shape[0], Wd.shape[1]
    sgu = _c(shared_gate_up, np.uint16)
    sd = _c(shared_down, np.uint16)
    Is = 0 if sd is None else sd.shape[0]
    idx = _c(idx, np.int32)
    w = _c(w, np.float32)
    k = idx.shape[1]
    dout = _c(d_out, np.float64)
    c = _cfg(T=T, H=H, E=E, k=k, I=I, Is=Is)
    r = dict(dx=np.empty((T, H)), dW_gate_up=np.empty((E, 2 * I, H)), dW_down=np.empty((E, I, H)),
             d_shared_gate_up=None if sgu is None else np.empty((2 * Is, H)),
             d_shared_down=None if sd is None else np.empty((Is, H)), dw=np.empty((T, k)))
    rc = _load().orc_experts_backward(ctypes.byref(c), _p(x), _p(Wgu), _p(Wd), _p(sgu), _p(sd), _p(idx), _p(w),
                                      _p(dout), 1 if round_act else 0, _p(r["dx"]), _p(r["dW_gate_up"]),
                                      _p(r["dW_down"]), _p(r["d_shared_gate_up"]), _p(r["d_shared_down"]),
                                      _p(r["dw"]))
    if rc != 0:
        raise IndexError("expert index out of range")
    return r


def dense_ffn(x_bf16, W_gate_up, W_down, residual=None, tokens=None):
    """Dense SwiGLU MLP in float64: down(silu(gate x) * up x) (+ residual),
    with the intermediate rounded to bf16 as in the expert path; it is the
    expert stage with no routed pairs and the dense weights as its one
    always-on MLP."""
    x = _c(x_bf16, np.uint16)
    T, H = x.shape
    gu = _c(W_gate_up, np.uint16)
    dn = _c(W_down, np.uint16)
    I = dn.shape[0]
    dummy_gu = np.zeros((1, 2 * I, H), dtype=np.uint16)
    dummy_dn = np.zeros((1, I, H), dtype=np.uint16)
    return experts(x, dummy_gu, dummy_dn, gu, dn, np.zeros((T, 0), dtype=np.int32),
                   np.zeros((T, 0), dtype=np.float32), residual=residual, tokens=tokens)


def rmsnorm(x_bf16: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """Decoder pre-norm: bf16 bits of x / sqrt(mean(x^2) + eps), row by row."""
    x = _c(x_bf16, np.uint16)
    T, H = x.shape
    out = np.empty_like(x)
    _load().orc_rmsnorm(T, H, _p(x), eps, _p(out))
    return out


def expert_feedback(counts, T, k, gamma, bias=None, totals=None):
    """(new bias or None, new totals or None) after one routing step."""
    c = _c(counts, np.int32)
    E = c.size
    b = None if bias is None else np.array(bias, dtype=np.float32, copy=True)
    tot = None if totals is None else np.array(totals, dtype=np.int64, copy=True)
    _load().orc_expert_feedback(E, T, k, _p(c), gamma, _p(b), _p(tot))
    return b, tot


def set_threads(n: int) -> None:
    """Thread count of the oracle's OpenMP loops."""
    _load().orc_set_threads(int(n))


def max_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().orc_max_threads())
