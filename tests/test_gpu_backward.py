"""Backward of the expert stage on the GPU (moe_backward) against the oracle's
float64 backward (itself pinned by finite differences and torch autograd):
the input gradient, every expert's and the shared expert's weight gradients
(fp32 sums over the bucket's rows of bf16 products) and the routing-weight
gradients, on random and router routings, with empty experts, a bucket that
holds every row, and ragged sizes."""
import numpy as np
import pytest
import torch

import oracle
from group_limited_routing_gb300 import moe, workloads as wl
from parity import bf16_to_f64, output_errors

pytestmark = pytest.mark.gpu
DEV = "cuda"
# gradients pass through more bf16 roundings than the forward: the saved G
# and U, the weighted intermediate and dG/dU (GEMM operands), each a relative
# 2^-9 at most; measured errors stay under 0.5% of the largest value and 0.4%
# on average, so these bounds keep a margin of about three
GRAD_MAX_REL = 1.5e-2
GRAD_MEAN_REL = 1e-2


def u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def close(got, ref, what):
    e = output_errors(np.asarray(got, dtype=np.float64), ref)
    assert e["max_err"] <= GRAD_MAX_REL * e["max_ref"] + 1e-30, "%s max err %g (max ref %g)" % (
        what, e["max_err"], e["max_ref"])
    assert e["mean_rel"] <= GRAD_MEAN_REL, "%s mean rel %g" % (what, e["mean_rel"])
    return e


def run_case(cfg, d, idx, w, seed=0):
    g = torch.Generator(DEV).manual_seed(1234 + seed)
    dout = torch.randn(cfg.T, cfg.H, device=DEV, generator=g).to(torch.bfloat16)
    ws = moe.Workspace(cfg, 2, DEV)
    got = moe.backward(cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"],
                       idx, w, dout, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    ref = oracle.experts_backward(u16(d["hidden"]), u16(d["W_gate_up"]), u16(d["W_down"]),
                                  u16(d["shared_gate_up"]), u16(d["shared_down"]), idx.cpu().numpy(),
                                  w.cpu().numpy(), bf16_to_f64(dout), round_act=True)
    close(bf16_to_f64(got["d_hidden"]), ref["dx"], "d_hidden")
    used = np.unique(idx.cpu().numpy())
    dWgu = got["dW_gate_up"].cpu().numpy().astype(np.float64)
    dWd = got["dW_down"].cpu().numpy().astype(np.float64)
    close(dWgu[used], ref["dW_gate_up"][used], "dW_gate_up")
    close(dWd[used], ref["dW_down"][used], "dW_down")
    unused = np.setdiff1d(np.arange(cfg.E), used)
    assert not dWgu[unused].any() and not dWd[unused].any()          # experts no token chose
    close(got["d_shared_gate_up"].cpu().numpy(), ref["d_shared_gate_up"], "d_shared_gate_up")
    close(got["d_shared_down"].cpu().numpy(), ref["d_shared_down"], "d_shared_down")
    close(got["d_topk_w"].cpu().numpy(), ref["dw"], "d_topk_w")
    return got


@pytest.mark.parametrize("T", [1, 16, 300, 1000])
def test_backward_random_routing(T):
    H, I, E = 512, 256, 256
    w0 = wl.Workload(80 + T % 7, "bwd", T=T, H=H, E=E, I=I, Is=I)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T, H=H, E=E, I=I, Is=I)
    idx, w = wl.random_routing(T, E, cfg.k, seed=T, device=DEV)
    run_case(cfg, d, idx, w, seed=T)


def test_backward_one_expert_holds_every_row():
    T, H, I = 200, 512, 256
    w0 = wl.Workload(85, "bwd", T=T, H=H, I=I, Is=I)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T, H=H, I=I, Is=I)
    idx = torch.full((T, cfg.k), 9, dtype=torch.int32, device=DEV)
    w = torch.rand(T, cfg.k, device=DEV) * 0.3
    run_case(cfg, d, idx, w, seed=5)


def test_backward_full_size_router_routing():
    T = 64
    w0 = wl.WORKLOADS[3].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T)
    idx, w, _, _, _ = moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"])
    run_case(cfg, d, idx, w, seed=9)


def test_backward_is_deterministic():
    T, H, I = 700, 512, 256
    w0 = wl.Workload(86, "bwd", T=T, H=H, I=I, Is=I)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T, H=H, I=I, Is=I)
    idx, w = wl.random_routing(T, cfg.E, cfg.k, seed=3, device=DEV)
    dout = torch.randn(T, H, device=DEV).to(torch.bfloat16)
    args = (cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"], idx, w, dout)
    a = moe.backward(*args)
    b = moe.backward(*args)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_backward_launch_count():
    T, H, I = 128, 512, 256
    w0 = wl.Workload(87, "bwd", T=T, H=H, I=I, Is=I)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T, H=H, I=I, Is=I)
    idx, w = wl.random_routing(T, cfg.E, cfg.k, seed=4, device=DEV)
    moe.backward(cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"], idx, w,
                 torch.zeros(T, H, device=DEV, dtype=torch.bfloat16))
    # hist, scan, scatter, pad zeroing, recompute, dgrad, dX, combine, dw, 2 weight-gradient GEMMs
    assert moe.last_launch_count() == 11


def test_layer_backward_matches_function_and_reuses_outputs():
    T, H, I = 333, 512, 256
    w0 = wl.Workload(88, "bwd", T=T, H=H, I=I, Is=I)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T, H=H, I=I, Is=I)
    layer = moe.MoELayer(cfg, d["W_router"], d["expert_bias"], d["W_gate_up"], d["W_down"], d["shared_gate_up"],
                         d["shared_down"])
    with pytest.raises(RuntimeError):
        layer.backward(torch.zeros(T, H, device=DEV, dtype=torch.bfloat16))
    layer(d["hidden"])
    dout = torch.randn(T, H, device=DEV).to(torch.bfloat16)
    g = layer.backward(dout)
    ref = moe.backward(cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"],
                       layer.routing[0], layer.routing[1], dout)
    for k in ref:
        assert torch.equal(g[k], ref[k]), k
    ptrs = {k: v.data_ptr() for k, v in g.items()}
    for v in g.values():
        v.fill_(7)
    g2 = layer.backward(dout, out=g)
    torch.cuda.synchronize()
    assert layer.status() == 0
    for k in ref:
        assert g2[k].data_ptr() == ptrs[k], k              # filled in place
        assert torch.equal(g2[k], ref[k]), k
    with pytest.raises(ValueError):
        layer.backward(dout, out={"d_hidden": torch.empty(T, H + 8, device=DEV, dtype=torch.bfloat16)})
