"""moe_layer on the GPU: routing and the expert stage in one call.

With MOE_LAYER_FUSED_ROUTER, for the routing page's setting (256 experts in
8 groups, k <= 8), the router kernel also selects the experts, claims the
bucket rows with integer atomics and copies the hidden rows itself.  Checks:
the fused call against the two-call path bit for bit where both compute the
same logits (the 256-expert router tiles, a token tile for every SM), against
the CPU oracle (routing under the near-tie rules, counts exact, outputs within
the layer tolerance with the GPU's routing as the oracle's input) at small and
ragged T, exact ties built into the logits, a missing bias, determinism,
launch counts and a CUDA-graph replay."""
import numpy as np
import pytest
import torch

import oracle
from group_limited_routing_gb300 import _lib, moe, workloads as wl
from parity import assert_output_close, bf16_to_f64, compare_counts, compare_routing, order_margin

pytestmark = pytest.mark.gpu
DEV = "cuda"
FUSED, PLAIN = _lib.MOE_LAYER_FUSED_ROUTER, 0


def u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def run_layer(cfg, d, flags, residual=None, bias="layer"):
    b = d["expert_bias"] if bias == "layer" else bias
    out, (idx, w, counts) = moe.layer(cfg, d["hidden"], d["W_router"], b, d["W_gate_up"], d["W_down"],
                                      d["shared_gate_up"], d["shared_down"], residual, flags=flags)
    torch.cuda.synchronize()
    return out, idx, w, counts


@pytest.mark.parametrize("T", [32768, 19500])
def test_fused_layer_matches_two_call_path_bit_for_bit(T):
    """Same logits (both paths take the 256-expert router tiles at these T:
    a token tile for every SM), so the same experts, weights and counts, and
    the same output bits although the rows inside each bucket come in a
    scheduling-dependent order."""
    w0 = wl.WORKLOADS[4].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T)
    of, i_f, w_f, c_f = run_layer(cfg, d, FUSED)
    ou, i_u, w_u, c_u = run_layer(cfg, d, PLAIN)
    assert torch.equal(i_f, i_u)
    assert torch.equal(w_f, w_u)
    assert torch.equal(c_f, c_u)
    assert torch.equal(of, ou)
    assert int(c_f.sum()) == T * cfg.k


@pytest.mark.parametrize("T,with_residual,k", [(32768, False, 8), (24780, True, 8), (24576, False, 6),
                                               (4096, False, 8)])
def test_fused_combine_matches_the_default_bit_for_bit(T, with_residual, k):
    """MOE_LAYER_FUSED_COMBINE: the shared expert's down GEMM forms the
    combine in its epilogue (from T = 24576 on, where the down GEMM runs on
    CTA pairs; T = 24780 ends in a 76-token shared tile; k = 6 pads the
    eight-term sum with zero rows; at T = 4096 the flag changes nothing).
    Same routing, same output bits as the default."""
    w0 = wl.WORKLOADS[4].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T, k=k)
    res = (torch.randn(T, cfg.H, device=DEV) * 0.5).to(torch.bfloat16) if with_residual else None
    od, i_d, w_d, c_d = run_layer(cfg, d, PLAIN, residual=res)
    of, i_f, w_f, c_f = run_layer(cfg, d, _lib.MOE_LAYER_FUSED_COMBINE, residual=res)
    assert torch.equal(i_f, i_d) and torch.equal(w_f, w_d) and torch.equal(c_f, c_d)
    assert torch.equal(of, od)


@pytest.mark.parametrize("wid,T,nsample", [(1, 128, None), (2, 16, None), (2, 1, None), (3, 4096, 192),
                                           (4, 2000, 160), (5, 129, None), (3, 300, None)])
def test_fused_layer_matches_oracle(wid, T, nsample):
    w0 = wl.WORKLOADS[wid].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T, H=w0.H, I=w0.I, Is=w0.Is)
    ws = moe.Workspace(cfg, moe.WS_LAYER, DEV, FUSED)
    out, (idx, w, counts) = moe.layer(cfg, d["hidden"], d["W_router"], d["expert_bias"], d["W_gate_up"],
                                      d["W_down"], d["shared_gate_up"], d["shared_down"], flags=FUSED, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    gi, gw, gc = idx.cpu().numpy(), w.cpu().numpy(), counts.cpu().numpy()
    x = u16(d["hidden"])
    bias = d["expert_bias"].cpu().numpy()
    ref = oracle.route(oracle.router_logits(x, d["W_router"].cpu().numpy()), bias=bias)
    n_near, near = compare_routing(gi, gw, ref, cfg.E, bias=bias)
    rc, _, _ = oracle.counts_aux(ref["idx"], ref["scores"])
    compare_counts(gc, gi, rc, ref["idx"], near, cfg.E)
    assert n_near <= max(2, T // 100)
    tok = None
    if nsample is not None:
        tok = np.union1d(wl.token_sample(T, nsample, seed=wid).numpy(), [0, T - 1]).astype(np.int32)
    refo = oracle.experts(x, u16(d["W_gate_up"]), u16(d["W_down"]), u16(d["shared_gate_up"]),
                          u16(d["shared_down"]), gi, gw, tokens=tok)
    got = bf16_to_f64(out)
    if tok is not None:
        got = got[tok]
    assert_output_close(got, refo, "fused layer workload %d T=%d" % (wid, T))


@pytest.mark.parametrize("topk_group,k", [(4, 8), (2, 8), (4, 5), (1, 8)])
def test_fused_exact_ties_go_to_the_lower_index(topk_group, k):
    """One-hot hidden rows and router weights on a 0.25 grid make the logits
    exact grid values (every product exact, every other term zero): equal
    experts inside a group and across the two halves a token's logits are
    split into, equal group scores, equal 4th and 5th groups.  Where the
    oracle sees an exact tie the GPU sees the same one and the lower index
    must win; tokens with a non-zero gap below 1e-5 are left out."""
    rng = np.random.default_rng(50 + 10 * topk_group + k)
    T, H, E = 2048, 512, 256
    W = (0.25 * rng.integers(0, 13, size=(E, H))).astype(np.float32)
    hot = rng.integers(0, H, size=T)
    x = torch.zeros(T, H, dtype=torch.bfloat16)
    x[torch.arange(T), torch.from_numpy(hot)] = 1.0
    w0 = wl.Workload(95, "ties", T=T, H=H, I=128, Is=128)
    d = wl.layer_inputs(w0, DEV)
    d["hidden"] = x.to(DEV)
    d["W_router"] = torch.from_numpy(W).to(DEV)
    cfg = moe.MoeConfig(T=T, H=H, I=128, Is=128, topk_group=topk_group, k=k)
    out, gi, gw, gc = run_layer(cfg, d, FUSED, bias=None)
    gi, gw, gc = gi.cpu().numpy(), gw.cpu().numpy(), gc.cpu().numpy()
    L = W[:, hot].T.copy()
    np.testing.assert_array_equal(oracle.router_logits(u16(d["hidden"]), W), L)
    ref = oracle.route(L, topk_group=topk_group, k=k)

    def clear(m):
        return (m == 0.0) | (m >= 1e-5)
    ok = clear(ref["margin_group"]) & clear(ref["margin_expert"]) & clear(order_margin(ref, None))
    tied = (ref["margin_group"] == 0.0) | (ref["margin_expert"] == 0.0)
    assert ok.sum() >= T * 0.9 and (tied & ok).sum() >= T // 4, (ok.sum(), (tied & ok).sum())
    bad = np.nonzero((gi[ok] != ref["idx"][ok]).any(axis=1))[0]
    assert bad.size == 0, "token %d: gpu %s ref %s" % (np.nonzero(ok)[0][bad[0]], gi[ok][bad[0]],
                                                      ref["idx"][ok][bad[0]])
    assert np.abs(gw[ok].astype(np.float64) - ref["w"][ok]).max() <= 1e-6
    assert np.array_equal(gc, np.bincount(gi.ravel(), minlength=E))
    # the two-call path resolves the same ties the same way
    _, ui, uw, uc = run_layer(cfg, d, PLAIN, bias=None)
    assert np.array_equal(ui.cpu().numpy(), gi) and np.array_equal(uw.cpu().numpy(), gw)


def test_fused_layer_without_bias_and_with_residual():
    T = 700
    w0 = wl.WORKLOADS[3].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T)
    res = torch.randn(T, cfg.H, device=DEV).to(torch.bfloat16)
    out, gi, gw, gc = run_layer(cfg, d, FUSED, residual=res, bias=None)
    x = u16(d["hidden"])
    ref = oracle.route(oracle.router_logits(x, d["W_router"].cpu().numpy()))
    n_near, near = compare_routing(gi.cpu().numpy(), gw.cpu().numpy(), ref, cfg.E)
    assert n_near <= 7
    tok = np.union1d(wl.token_sample(T, 96, seed=3).numpy(), [0, T - 1]).astype(np.int32)
    refo = oracle.experts(x, u16(d["W_gate_up"]), u16(d["W_down"]), u16(d["shared_gate_up"]),
                          u16(d["shared_down"]), gi.cpu().numpy(), gw.cpu().numpy(), residual=u16(res), tokens=tok)
    assert_output_close(bf16_to_f64(out)[tok], refo, "fused layer, no bias, residual")


def test_fused_layer_is_deterministic():
    T = 4096
    w0 = wl.WORKLOADS[4].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T)
    a = run_layer(cfg, d, FUSED)
    b = run_layer(cfg, d, FUSED)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


@pytest.mark.parametrize("flags,kernels", [(FUSED, 5), (PLAIN, 8)])
def test_layer_launch_count(flags, kernels):
    # fused: router (+ routing + bucketing), m-tile list, gate/up, down, combine;
    # two-call path: router, selection, hist, scan, scatter, gate/up, down, combine
    T = 600
    w0 = wl.WORKLOADS[3].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T)
    layer = moe.MoELayer(cfg, d["W_router"], d["expert_bias"], d["W_gate_up"], d["W_down"], d["shared_gate_up"],
                         d["shared_down"], single_call=True, flags=flags)
    layer(d["hidden"])
    assert layer.last_launches == kernels
    assert layer.status() == 0


def test_stage_profile_times_routing_and_bucketing_as_one_interval():
    """moe_profile_enable(2): one router_plus_permute interval per moe_layer
    call, the other kernels one interval each, and no per-kernel records of
    the routing stage's kernels; outputs as with profiling off."""
    T, calls = 4096, 3
    w0 = wl.WORKLOADS[4].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T)
    layer = moe.MoELayer(cfg, d["W_router"], d["expert_bias"], d["W_gate_up"], d["W_down"], d["shared_gate_up"],
                         d["shared_down"], single_call=True)
    ref = layer(d["hidden"]).clone()
    moe.profile_read(reset=True)
    moe.profile_enable(True, stages=True)
    try:
        for _ in range(calls):
            out = layer(d["hidden"])
        torch.cuda.synchronize()
    finally:
        moe.profile_enable(False)
    prof = moe.profile_read(reset=True)
    assert torch.equal(out, ref)
    assert prof["router_plus_permute"][1] == calls and prof["router_plus_permute"][0] > 0
    for name in ("gemm_gate_up_swiglu", "gemm_down", "combine"):
        assert prof[name][1] == calls, name
    for name in ("router_gemm", "route_select", "bucket_scan", "bucket_scatter"):
        assert prof[name][1] == 0, name


def test_graphed_fused_layer_matches_eager():
    T = 1000
    w0 = wl.WORKLOADS[3].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T)
    layer = moe.MoELayer(cfg, d["W_router"], d["expert_bias"], d["W_gate_up"], d["W_down"], d["shared_gate_up"],
                         d["shared_down"], single_call=True, flags=FUSED)
    g = moe.GraphedStep(layer, d["hidden"])
    for seed in range(3):
        x = (torch.randn(T, cfg.H, device=DEV, generator=torch.Generator(DEV).manual_seed(seed))).to(torch.bfloat16)
        ref = layer(x).clone()
        got = g(x).clone()
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
    assert g.status() == 0


def test_layer_rejects_unknown_flags():
    T = 64
    w0 = wl.WORKLOADS[3].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T)
    with pytest.raises(_lib.MoeError):
        moe.layer(cfg, d["hidden"], d["W_router"], d["expert_bias"], d["W_gate_up"], d["W_down"],
                  d["shared_gate_up"], d["shared_down"], flags=4, ws=moe.Workspace(cfg, moe.WS_LAYER, DEV, 0))


@pytest.mark.parametrize("T", [33, 600, 4864, 4865, 8192, 19500, 32768])
def test_layer_matches_the_two_calls_bit_for_bit(T):
    """moe_layer (flags 0, with the balance loss) against moe_route +
    moe_forward on the same inputs: the same routing kernels (from T = 4865
    on, the router's scored output, whose selection kernel also writes the
    bucketing histogram that moe_layer's expert stage then reads instead of
    counting again), so every output agrees bit for bit."""
    w0 = wl.WORKLOADS[4].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T)
    out, (idx, w, counts, P, loss) = moe.layer(cfg, d["hidden"], d["W_router"], d["expert_bias"], d["W_gate_up"],
                                               d["W_down"], d["shared_gate_up"], d["shared_down"], aux=True)
    ri, rw, rc, rP, rl = moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"], aux=True)
    ro = moe.forward(cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"], ri, rw)
    torch.cuda.synchronize()
    for a, b in ((idx, ri), (w, rw), (counts, rc), (P, rP), (loss, rl), (out, ro)):
        assert torch.equal(a, b)
    assert int(counts.sum()) == T * cfg.k
