"""Failure detection on the GPU without faulting it.

A test hook makes the gate/up GEMM's producer withhold every TMA load, so the
MMA lane's first bounded wait (50 ms) runs out.  The kernel must wind down by
itself -- every role leaves its loop, copies in flight are drained, TMEM is
freed -- report MOE_STATUS_TIMEOUT in the workspace's status word, and leave
the CUDA context usable: the next call gives the normal result.
"""
import time

import pytest
import torch

from group_limited_routing_gb300 import _lib, moe, workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_gemm_wait_timeout_is_reported_and_context_survives():
    T = 512
    w0 = wl.Workload(77, "failure test", T=T, H=512, I=128, Is=128)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T, H=512, I=128, Is=128)
    idx, w = wl.random_routing(T, cfg.E, cfg.k, seed=3, device=DEV)
    args = (cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"], idx, w)
    ws = moe.Workspace(cfg, _lib.MOE_WS_FORWARD, DEV)
    good = moe.forward(*args, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0

    lib = _lib.load()
    assert lib.moe_debug_inject_timeout(1) == _lib.MOE_OK
    try:
        t0 = time.time()
        moe.forward(*args, ws=ws)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
    finally:
        lib.moe_debug_inject_timeout(0)
    st = ws.status()
    assert st & _lib.MOE_STATUS_TIMEOUT, st
    assert elapsed < 10.0

    again = moe.forward(*args, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert torch.equal(again, good)
