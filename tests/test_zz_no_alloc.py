"""moe_route_static: the router entry point that takes no workspace.

Some callers cannot allocate device memory where they call the router:
plug-in hosts that hand an operator its tensors but no allocator, runtimes
that keep all device memory to themselves, or tight loops where a cudaMalloc
would stall the device.  moe_route_static keeps the router's scratch in an array inside the
library instead.  These checks call it through the C ABI and compare it with
moe_route (which uses a caller workspace) on two calls in a row: the same
kernels run on the same inputs, so indices, counts, weights and the balance
loss must agree bit for bit.

This file is collected last on purpose, so that a failure here comes after
every other test has run.
"""
import ctypes

import pytest
import torch

from group_limited_routing_gb300 import _lib, moe, workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _outputs(cfg):
    return dict(idx=torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=DEV),
                w=torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=DEV),
                counts=torch.empty(cfg.E, dtype=torch.int32, device=DEV),
                P=torch.empty(cfg.E, dtype=torch.float32, device=DEV),
                loss=torch.empty(1, dtype=torch.float32, device=DEV),
                status=torch.full((1,), -1, dtype=torch.int32, device=DEV))


def _static_route(cfg, x, W, bias, o):
    """One call into the library on outputs allocated beforehand; returns the
    device's free bytes and torch's allocated bytes, both read after it."""
    lib = _lib.load()
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.moe_route_static(ctypes.byref(cfg.c()), x.data_ptr(), W.data_ptr(), bias.data_ptr(),
                              o["idx"].data_ptr(), o["w"].data_ptr(), o["counts"].data_ptr(), o["P"].data_ptr(),
                              o["loss"].data_ptr(), o["status"].data_ptr(), stream)
    assert rc == _lib.MOE_OK, _lib.strerror(rc)
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()


@pytest.mark.parametrize("wid,T", [(4, 32768), (1, 128)])
def test_static_route_matches_workspace_route_twice(wid, T):
    w0 = wl.WORKLOADS[wid].with_T(T)
    d = wl.layer_inputs(w0, DEV, with_experts=False)
    cfg = moe.MoeConfig(T=T, H=w0.H, I=w0.I, Is=w0.Is)
    ref = moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"], aux=True)
    torch.cuda.synchronize()
    outs = [_outputs(cfg), _outputs(cfg)]
    torch.cuda.synchronize()
    mem = [(torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated())]
    for o in outs:
        mem.append(_static_route(cfg, d["hidden"], d["W_router"], d["expert_bias"], o))
        assert int(o["status"].item()) == 0
        assert torch.equal(o["idx"], ref[0])
        assert torch.equal(o["counts"], ref[2])
        assert torch.equal(o["w"], ref[1])
        assert torch.equal(o["P"], ref[3])
        assert torch.equal(o["loss"], ref[4])
    # nothing is allocated by the call itself: after the first call (which may
    # load the library's code onto the device), neither the device's free
    # memory nor torch's allocator moves
    assert mem[2] == mem[1], mem


def test_static_route_rejects_configurations_beyond_its_array():
    lib = _lib.load()
    cfg = moe.MoeConfig(T=65536)            # needs about 70 MiB of scratch
    A = 1 << 20                             # never dereferenced: refused on the host
    rc = lib.moe_route_static(ctypes.byref(cfg.c()), A, A, None, A, A, A, None, None, None, None)
    assert rc == _lib.MOE_ERR_UNSUPPORTED_SHAPE
