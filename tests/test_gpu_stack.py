"""The 19-layer stack (the first_k_dense_replace=1 layout of the routing
article's §一, dense layer excluded): T=8192, independent seeded weights per
layer, decoder-layer stacking x_{l+1} = bf16(x_l + moe_l(rmsnorm(x_l))),
per-layer expert counts and the balance loss.  (Without the pre-norm, the
SwiGLU's quadratic growth blows a residual stack of random-weight layers up
after about ten layers.)  Parity is teacher-forced: for every layer the oracle
takes the GPU's own layer input (and, for the expert stage, the GPU's
routing), so one layer's rounding cannot drift into the next layer's check."""
import numpy as np
import pytest
import torch

import oracle
from group_limited_routing_gb300 import moe, workloads as wl
from parity import assert_output_close, bf16_to_f64, compare_counts, compare_routing, record

pytestmark = pytest.mark.gpu
DEV = "cuda"
FULL_ROUTE_LAYERS = tuple(range(19))   # every layer's routing on every token


def u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def test_nineteen_layer_stack_teacher_forced():
    w0 = wl.WORKLOADS[5]
    assert w0.layers == 19 and w0.residual
    cfg = moe.MoeConfig(T=w0.T, H=w0.H, I=w0.I, Is=w0.Is)
    x = wl.hidden(w0, DEV)
    tokens = np.union1d(wl.token_sample(w0.T, 64, seed=5).numpy(), [0, w0.T - 1]).astype(np.int32)
    losses, near_total = [], 0
    tally = dict(T=0, near_tie_tokens=0, near_tie_differ=0, order_tie_tokens=0, order_tie_differ=0, max_w_err=0.0)
    for layer in range(w0.layers):
        d = wl.layer_inputs(w0, DEV, layer=layer)
        L = moe.MoELayer(cfg, d["W_router"], d["expert_bias"], d["W_gate_up"], d["W_down"], d["shared_gate_up"],
                         d["shared_down"], aux=True)
        xn = moe.rmsnorm(x)
        out = L(xn, residual=x)
        torch.cuda.synchronize()
        assert L.status() == 0
        idx, w, counts, P, loss = (t.cpu().numpy() for t in L.routing)
        assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=cfg.E))
        xr = u16(x)
        xs = u16(xn)
        ref_norm = oracle.bf16_bits_to_f32(oracle.rmsnorm(xr[tokens])).astype(np.float64)
        got_norm = oracle.bf16_bits_to_f32(xs[tokens]).astype(np.float64)
        assert np.all(np.abs(got_norm - ref_norm) <= np.abs(ref_norm) * 2.0 ** -7 + 1e-30)
        W = d["W_router"].cpu().numpy()
        bias = d["expert_bias"].cpu().numpy()

        rows = np.arange(w0.T) if layer in FULL_ROUTE_LAYERS else tokens
        ref = oracle.route(oracle.router_logits(np.ascontiguousarray(xs[rows]), W), bias=bias)
        rep = {}
        n_near, near = compare_routing(idx[rows], w[rows], ref, cfg.E, rep, bias=bias)
        near_total += n_near
        for key in tally:
            tally[key] = max(tally[key], rep[key]) if key == "max_w_err" else tally[key] + rep[key]
        if layer in FULL_ROUTE_LAYERS:
            rc, rP, _ = oracle.counts_aux(ref["idx"], ref["scores"])
            compare_counts(counts, idx, rc, ref["idx"], near, cfg.E)
            # the loss from the GPU's own selection and the oracle's scores
            _, _, raux = oracle.counts_aux(idx, ref["scores"])
            np.testing.assert_allclose(P, rP, rtol=1e-4, atol=1e-8)
            assert abs(float(loss[0]) - raux) <= 1e-5 * abs(raux)

        ref_out = oracle.experts(xs, u16(d["W_gate_up"]), u16(d["W_down"]), u16(d["shared_gate_up"]),
                                 u16(d["shared_down"]), idx, w, residual=xr, tokens=tokens)
        e = assert_output_close(bf16_to_f64(out)[tokens], ref_out, "layer %d" % layer)
        losses.append(float(loss[0]))
        print("layer %2d: near-tie %d, mean rel %.2e, aux loss %.4f, max |x| %.2f" % (
            layer, n_near, e["mean_rel"], losses[-1], float(out.abs().max())))
        x = out
        del L, d
    record("moe_route in the 19-layer stack, T=8192 per layer (all layers' tokens)", tally)
    assert all(np.isfinite(losses)) and all(0.5 < v < 10.0 for v in losses)
    assert torch.isfinite(x.float()).all()
    assert float(x.float().std()) < 10.0


def test_rmsnorm_matches_oracle():
    x = (torch.randn(1000, 2048, device=DEV) * torch.rand(1000, 1, device=DEV) * 20).to(torch.bfloat16)
    got = oracle.bf16_bits_to_f32(u16(moe.rmsnorm(x))).astype(np.float64)
    ref = oracle.bf16_bits_to_f32(oracle.rmsnorm(u16(x))).astype(np.float64)
    # both round once to bf16 (fp32 vs double before it): at most one bf16 step apart
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30)
    assert (got != ref).mean() < 0.01


def test_moe_stack_object_matches_layer_loop():
    """MoEStack (shared workspaces, ping-pong buffers) computes exactly what the
    layer-by-layer loop above computes: same kernels, deterministic, so bit-equal;
    HostPipeline over the stack gives the same bytes again."""
    w0 = wl.WORKLOADS[5].with_T(1000)
    cfg = moe.MoeConfig(T=w0.T, H=w0.H, I=w0.I, Is=w0.Is)
    ws_l = moe.Workspace(cfg, moe.WS_LAYER, DEV)
    layers = []
    for layer in range(3):
        d = wl.layer_inputs(w0, DEV, layer=layer)
        layers.append(moe.MoELayer(cfg, d["W_router"], d["expert_bias"], d["W_gate_up"], d["W_down"],
                                   d["shared_gate_up"], d["shared_down"], ws_layer=ws_l))
    stack = moe.MoEStack(layers)
    x = wl.hidden(w0, DEV)
    y = torch.empty_like(x)
    got = stack(x, out=y)
    assert got.data_ptr() == y.data_ptr()
    assert stack.last_launches == sum(1 + L.last_launches for L in layers)
    ref = x
    for L in layers:
        ref = L(moe.rmsnorm(ref), residual=ref)
    torch.cuda.synchronize()
    assert stack.status() == 0
    assert torch.equal(y, ref)

    xh = x.cpu().pin_memory()
    outs = [torch.empty_like(xh).pin_memory() for _ in range(3)]
    pipe = moe.HostPipeline(stack)
    pipe.run([xh] * 3, outs)
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, ref.cpu())
