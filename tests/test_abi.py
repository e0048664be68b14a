"""The C-ABI library builds, loads and exports every symbol include/moe.h
declares, and refuses bad arguments on the host before any CUDA call (so
these run without a GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

from group_limited_routing_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(moe_[a-z_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_binding_exports():
    assert header_functions() == sorted(_lib.EXPORTS)


def test_header_constants_match_the_binding():
    # every #define MOE_* with an integer value in the header has the same
    # value under the same name in the binding
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    defs = dict(re.findall(r"^#define\s+(MOE_\w+)\s+\(?(-?\d+)\)?\s*(?:/\*.*\*/)?\s*$", src, flags=re.M))
    assert {"MOE_LAYER_FUSED_COMBINE", "MOE_KERNEL_COUNT", "MOE_STATUS_TIMEOUT", "MOE_ERR_TIMEOUT"} <= set(defs)
    missing = [n for n in defs if not hasattr(_lib, n)]
    assert not missing, missing
    for name, value in defs.items():
        assert getattr(_lib, name) == int(value), name


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(moe_\w+)", out))
    for name in header_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_library_is_built_for_sm103a_only():
    # cuobjdump --list-elf prints only the names of the embedded images
    r = subprocess.run(["cuobjdump", "--list-elf", build.LIB], capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    arches = set(re.findall(r"sm_(\d+a?)", r.stdout))
    assert arches == {"103a"}, arches


def cfg(**kw):
    base = dict(T=64, H=2048, E=256, n_group=8, topk_group=4, k=8, I=512, Is=512, rsf=2.5, eps=1e-20)
    base.update(kw)
    return _lib.MoeCfg(*[base[n] for n in ("T", "H", "E", "n_group", "topk_group", "k", "I", "Is")],
                       base["rsf"], base["eps"])


def test_workspace_bytes(lib):
    c = cfg()
    r = lib.moe_workspace_bytes(ctypes.byref(c), _lib.MOE_WS_ROUTE)
    f = lib.moe_workspace_bytes(ctypes.byref(c), _lib.MOE_WS_FORWARD)
    # route: header + W split (3 E H bf16) + logits; forward: X_perm + intermediate + Y dominate
    assert r >= 256 + 3 * 256 * 2048 * 2 + 64 * 256 * 4
    assert f >= 8 * 64 * 2048 * 2 + 9 * 64 * 512 * 2 + 9 * 64 * 2048 * 2
    assert r % 256 == 0 and f % 256 == 0
    assert lib.moe_workspace_bytes(ctypes.byref(c), 7) == 0
    assert lib.moe_workspace_bytes(None, _lib.MOE_WS_ROUTE) == 0
    # grows with T
    assert lib.moe_workspace_bytes(ctypes.byref(cfg(T=128)), 1) > f


@pytest.mark.parametrize("kw,code", [
    (dict(T=0), _lib.MOE_ERR_INVALID_ARG),
    (dict(E=250), _lib.MOE_ERR_INVALID_ARG),                 # not divisible by n_group
    (dict(topk_group=9), _lib.MOE_ERR_INVALID_ARG),
    (dict(k=129), _lib.MOE_ERR_INVALID_ARG),                 # more than the surviving experts
    (dict(eps=-1.0), _lib.MOE_ERR_INVALID_ARG),
    (dict(rsf=float("inf")), _lib.MOE_ERR_INVALID_ARG),
    (dict(E=512, n_group=16), _lib.MOE_ERR_UNSUPPORTED_SHAPE),
    (dict(E=256, n_group=4), _lib.MOE_ERR_UNSUPPORTED_SHAPE),  # groups of 64
    (dict(k=33, topk_group=8), _lib.MOE_ERR_UNSUPPORTED_SHAPE),
    (dict(H=2000), _lib.MOE_ERR_UNSUPPORTED_SHAPE),
    (dict(T=(1 << 24) + 1), _lib.MOE_ERR_UNSUPPORTED_SHAPE),
])
def test_route_config_errors(lib, kw, code):
    c = cfg(**kw)
    rc = lib.moe_route(ctypes.byref(c), 16, 16, None, 16, 16, 16, None, None, 256, 1 << 40, None)
    assert rc == code
    assert lib.moe_workspace_bytes(ctypes.byref(c), _lib.MOE_WS_ROUTE) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(I=100), _lib.MOE_ERR_UNSUPPORTED_SHAPE),
    (dict(Is=1024), _lib.MOE_ERR_UNSUPPORTED_SHAPE),
    (dict(H=1000), _lib.MOE_ERR_UNSUPPORTED_SHAPE),
    (dict(k=0), _lib.MOE_ERR_INVALID_ARG),
    (dict(I=0), _lib.MOE_ERR_INVALID_ARG),
])
def test_forward_config_errors(lib, kw, code):
    c = cfg(**kw)
    rc = lib.moe_forward(ctypes.byref(c), 16, 16, 16, 16, 16, 16, 16, None, 16, 256, 1 << 40, None)
    assert rc == code


def test_pointer_and_workspace_errors(lib):
    c = cfg()
    need_r = lib.moe_workspace_bytes(ctypes.byref(c), _lib.MOE_WS_ROUTE)
    need_f = lib.moe_workspace_bytes(ctypes.byref(c), _lib.MOE_WS_FORWARD)
    A = 1 << 20  # a fake, well-aligned address: never dereferenced, the checks fail first
    # null required pointers
    assert lib.moe_route(ctypes.byref(c), None, A, None, A, A, A, None, None, A, need_r, None) == \
        _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_forward(ctypes.byref(c), A, A, A, A, A, None, A, None, A, A, need_f, None) == \
        _lib.MOE_ERR_INVALID_ARG
    # workspace too small / misaligned / null
    assert lib.moe_route(ctypes.byref(c), A, A, None, A, A, A, None, None, A, need_r - 1, None) == \
        _lib.MOE_ERR_WORKSPACE_TOO_SMALL
    assert lib.moe_route(ctypes.byref(c), A, A, None, A, A, A, None, None, A + 16, need_r, None) == \
        _lib.MOE_ERR_MISALIGNED
    assert lib.moe_forward(ctypes.byref(c), A, A, A, A, A, A, A, None, A, None, need_f, None) == \
        _lib.MOE_ERR_INVALID_ARG
    # tensor-core operands must be 16-byte aligned
    assert lib.moe_route(ctypes.byref(c), A + 2, A, None, A, A, A, None, None, A, need_r, None) == \
        _lib.MOE_ERR_MISALIGNED
    assert lib.moe_forward(ctypes.byref(c), A, A + 8, A, A, A, A, A, None, A, A, need_f, None) == \
        _lib.MOE_ERR_MISALIGNED
    assert lib.moe_forward(ctypes.byref(c), A, A, A, A, A, A + 2, A, None, A, A, need_f, None) == \
        _lib.MOE_ERR_MISALIGNED
    # status read needs a workspace and a host destination
    assert lib.moe_get_status(None, 256, None, ctypes.byref(ctypes.c_int32()), 0) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_get_status(A, 256, None, None, 0) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_init(A, 16, None) == _lib.MOE_ERR_WORKSPACE_TOO_SMALL


def test_strerror(lib):
    for code in range(-8, 1):
        s = lib.moe_strerror(code).decode()
        assert s and s != "unknown error code"
    assert lib.moe_strerror(-99).decode() == "unknown error code"


def test_profile_modes(lib):
    """0 off, 1 per kernel, 2 per stage; anything else is refused.  The names
    cover every id, the last one being the routing-and-bucketing stage."""
    assert lib.moe_profile_enable(2) == _lib.MOE_OK
    assert lib.moe_profile_enable(1) == _lib.MOE_OK
    assert lib.moe_profile_enable(0) == _lib.MOE_OK
    assert lib.moe_profile_enable(3) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_profile_enable(-1) == _lib.MOE_ERR_INVALID_ARG
    names = [lib.moe_kernel_name(k).decode() for k in range(_lib.MOE_KERNEL_COUNT)]
    assert all(names) and len(set(names)) == len(names)
    assert names[-1] == "router_plus_permute"
    assert lib.moe_kernel_name(_lib.MOE_KERNEL_COUNT).decode() == ""


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(build, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_handle", None)
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load()


def test_dense_workspace_bytes(lib):
    f = lib.moe_dense_workspace_bytes(1000, 2048, 4608)
    # intermediate + output dominate
    assert f >= 1000 * 4608 * 2 + 1000 * 2048 * 2 and f % 256 == 0
    assert lib.moe_dense_workspace_bytes(1000, 2048, 100) == 0      # I % 128
    assert lib.moe_dense_workspace_bytes(1000, 2000, 4608) == 0     # H % 256
    assert lib.moe_dense_workspace_bytes(0, 2048, 4608) == 0
    assert lib.moe_dense_workspace_bytes(2000, 2048, 4608) > f


def test_layer_workspace_bytes(lib):
    """moe_layer's workspace holds both calls' regions; the fused router's
    buckets (E T rows of X_perm instead of k T) only when asked for and where
    the shape allows it; unknown shapes give 0."""
    c = cfg(T=1024)
    r = lib.moe_workspace_bytes(ctypes.byref(c), _lib.MOE_WS_ROUTE)
    f = lib.moe_workspace_bytes(ctypes.byref(c), _lib.MOE_WS_FORWARD)
    plain = lib.moe_layer_workspace_bytes(ctypes.byref(c), 0)
    fused = lib.moe_layer_workspace_bytes(ctypes.byref(c), _lib.MOE_LAYER_FUSED_ROUTER)
    assert plain >= r + f - 256
    assert fused - plain >= (256 - 8) * 1024 * 2048 * 2
    # 4 groups of 32: not the fused router's shape, the flag changes nothing
    c4 = cfg(T=1024, E=128, n_group=4, topk_group=2)
    assert lib.moe_layer_workspace_bytes(ctypes.byref(c4), _lib.MOE_LAYER_FUSED_ROUTER) == \
        lib.moe_layer_workspace_bytes(ctypes.byref(c4), 0) > 0
    assert lib.moe_layer_workspace_bytes(ctypes.byref(cfg(H=100)), 0) == 0
    assert lib.moe_layer_workspace_bytes(None, 0) == 0
