"""Router parity on the GPU: moe_router_logits, moe_route_from_logits and
moe_route against the CPU oracle, on the five workloads' shapes and on edge
cases (ties, ragged T, other group settings)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from group_limited_routing_gb300 import moe, workloads as wl
from parity import compare_counts, compare_routing, record
from test_oracle_pins import _parse_logits

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def run_route(cfg, x, W, bias, aux=True):
    idx, w, counts, P, loss = moe.route(cfg, x, W, bias, aux=aux)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), counts.cpu().numpy(), \
        (P.cpu().numpy() if P is not None else None), (float(loss.item()) if loss is not None else None)


@pytest.mark.parametrize("wid,T", [(1, 128), (2, 16), (3, 4096), (4, 32768), (5, 8192), (6, 32768)])
def test_route_matches_oracle(wid, T):
    w0 = wl.WORKLOADS[wid].with_T(T)
    d = wl.layer_inputs(w0, DEV, with_experts=False)
    cfg = moe.MoeConfig(T=T, H=w0.H, I=w0.I, Is=w0.Is)
    gi, gw, gc, gP, gloss = run_route(cfg, d["hidden"], d["W_router"], d["expert_bias"])
    x = u16(d["hidden"])
    L = oracle.router_logits(x, d["W_router"].cpu().numpy())
    ref = oracle.route(L, bias=d["expert_bias"].cpu().numpy())
    rep = {}
    n_near, near = compare_routing(gi, gw, ref, cfg.E, rep, bias=d["expert_bias"].cpu().numpy())
    rc, rP, rloss = oracle.counts_aux(ref["idx"], ref["scores"])
    compare_counts(gc, gi, rc, ref["idx"], near, cfg.E)
    np.testing.assert_allclose(gP, rP, rtol=1e-4, atol=1e-7)
    assert abs(gloss - rloss) <= 1e-4 * abs(rloss)
    print("workload %d T=%d near-tie tokens %d (%.3f%%), order-only ties %d, max w err %.2e" % (
        wid, T, n_near, 100.0 * n_near / T, rep["order_tie_tokens"], rep["max_w_err"]))
    record("moe_route, workload %d, T=%d" % (wid, T), rep)
    assert n_near <= max(2, T // 100)


@pytest.mark.parametrize("wid,T", [(1, 128), (2, 16), (2, 1), (2, 31), (4, 32), (3, 4096), (4, 2048), (4, 32768),
                                   (4, 19500)])
def test_router_logits_accuracy(wid, T):
    # T <= 32: the CUDA-core router; T=32768 and 19500 take the 256-expert
    # router tiles (a token tile for every SM), 19500 ending in a part-filled tile
    w0 = wl.WORKLOADS[wid].with_T(T)
    d = wl.layer_inputs(w0, DEV, with_experts=False)
    cfg = moe.MoeConfig(T=T, H=w0.H, I=w0.I, Is=w0.Is)
    g = moe.router_logits(cfg, d["hidden"], d["W_router"]).cpu().numpy()
    L = oracle.router_logits(u16(d["hidden"]), d["W_router"].cpu().numpy())
    err = np.abs(g.astype(np.float64) - L)
    # bf16 x (hi + mid + lo) products are exact; only fp32 accumulation differs
    assert err.max() <= 2e-6 + 2e-6 * np.abs(L).max(), err.max()
    print("workload %d: router logits max abs err %.3e (max |logit| %.2f)" % (wid, err.max(), np.abs(L).max()))
    record("router logits vs exact, workload %d, T=%d" % (wid, T),
           dict(T=int(T), max_abs_err=float(err.max()), max_abs_logit=float(np.abs(L).max())))


def test_router_logits_are_batch_invariant():
    """Within the CTA-pair router's range (T >= 19456) a token's logits and
    routing do not depend on the batch around it: the first 19456 tokens of a
    32768-token batch (128 tiles on the pairs, some pairs taking two) come out
    bit for bit as in a 19456-token batch (one tile per pair).  (Below that
    range the router splits K over SMs for small batches, which changes the
    summation order.)"""
    w0 = wl.WORKLOADS[4].with_T(32768)
    d = wl.layer_inputs(w0, DEV, with_experts=False)
    cfg = moe.MoeConfig(T=32768, H=w0.H, I=w0.I, Is=w0.Is)
    n = 19456
    cfg1 = cfg.with_T(n)
    x1 = d["hidden"][:n].contiguous()
    big = moe.router_logits(cfg, d["hidden"], d["W_router"])
    small = moe.router_logits(cfg1, x1, d["W_router"])
    torch.cuda.synchronize()
    assert torch.equal(big[:n], small)
    bi, bw, bc, _, _ = moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"], aux=False)
    si, sw, sc, _, _ = moe.route(cfg1, x1, d["W_router"], d["expert_bias"], aux=False)
    torch.cuda.synchronize()
    assert torch.equal(bi[:n], si) and torch.equal(bw[:n], sw)
    # and the same batch again
    again = moe.router_logits(cfg, d["hidden"], d["W_router"])
    torch.cuda.synchronize()
    assert torch.equal(again, big)


def test_router_sigmoid_ulp_distance():
    """The routing kernels' fp32 sigmoid (the hardware 2^x on a compensated
    argument, then the hardware reciprocal of 1 + exp(-L) with one Newton
    step) against the oracle's sigmoid (double, rounded once to fp32): how
    many fp32 steps apart they are, and the absolute error that matters for
    the 1e-5 near-tie margin."""
    rng = np.random.default_rng(5)
    grid = np.linspace(-30.0, 30.0, 1 << 20, dtype=np.float32)
    L = np.concatenate([grid, rng.standard_normal(1 << 20).astype(np.float32) * 3.0])
    L = L[: (L.size // 256) * 256]
    got = moe.router_scores(torch.from_numpy(L).to(DEV)).cpu().numpy()
    ref = oracle.route(L.reshape(-1, 256))["scores"].ravel()
    # positive floats: the distance in fp32 steps is the difference of the bit patterns
    ulps = np.abs(got.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    hist = {int(u): int(c) for u, c in zip(*np.unique(ulps, return_counts=True))}
    abs_err = float(np.abs(got.astype(np.float64) - ref.astype(np.float64)).max())
    print("router sigmoid: fp32 steps from the exact sigmoid (count by distance): %s; max abs err %.3g" % (
        hist, abs_err))
    record("router sigmoid vs exact (fp32 steps), %d logits in [-30, 30] and N(0, 9)" % L.size,
           dict(T=int(L.size), ulp_hist=hist, max_ulps=int(ulps.max()), max_abs_err=abs_err,
                frac_exact=float((ulps == 0).mean())))
    assert ulps.max() <= 16
    assert abs_err <= 5e-7


@pytest.mark.parametrize("wid,T", [(4, 4865), (5, 8192), (3, 9000), (4, 32768)])
def test_scored_router_output_selects_like_the_logits(wid, T):
    """From T = 4865 on, moe_route takes the router's scored output (sigmoid
    scores and group scores formed in the GEMM's epilogue); routing the same
    batch from moe_router_logits' logits with moe_route_from_logits must give
    the same experts, weights and counts bit for bit (same sigmoid, same fp32
    additions), and the same balance-loss terms up to summation order."""
    w0 = wl.WORKLOADS[wid].with_T(T)
    d = wl.layer_inputs(w0, DEV, with_experts=False)
    cfg = moe.MoeConfig(T=T, H=w0.H, I=w0.I, Is=w0.Is)
    gi, gw, gc, gP, gl = moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"], aux=True)
    logits = moe.router_logits(cfg, d["hidden"], d["W_router"])
    li, lw, lc, lP, ll = moe.route_from_logits(cfg, logits, d["expert_bias"], aux=True)
    torch.cuda.synchronize()
    assert torch.equal(gi, li) and torch.equal(gw, lw) and torch.equal(gc, lc)
    np.testing.assert_allclose(gP.cpu().numpy(), lP.cpu().numpy(), rtol=1e-5, atol=1e-9)
    assert abs(float(gl.item()) - float(ll.item())) <= 1e-5 * abs(float(ll.item()))


@pytest.mark.parametrize("wid,T", [(4, 4865), (5, 8192), (3, 9001), (6, 19500), (4, 32768), (4, 131072)])
def test_thread_per_token_selection_equals_the_warp_kernel(wid, T):
    """Without the balance loss, the scored routing runs one thread per token;
    with it, one warp per token (the kernel the oracle tests above check).
    Both must give the same experts, weights and counts bit for bit."""
    w0 = wl.WORKLOADS[wid].with_T(T)
    d = wl.layer_inputs(w0, DEV, with_experts=False)
    cfg = moe.MoeConfig(T=T, H=w0.H, I=w0.I, Is=w0.Is)
    ti, tw, tc, _, _ = moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"], aux=False)
    gi, gw, gc, _, _ = moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"], aux=True)
    torch.cuda.synchronize()
    assert torch.equal(ti, gi) and torch.equal(tw, gw) and torch.equal(tc, gc)


@pytest.mark.parametrize("T,n_group,topk_group,k,scale", [
    (1, 8, 4, 8, 1.0), (130, 8, 4, 8, 1.0), (1000, 8, 1, 8, 2.0), (777, 8, 8, 8, 1.0),
    (513, 8, 4, 1, 1.0), (300, 8, 4, 32, 1.0), (257, 4, 2, 6, 1.0), (129, 4, 4, 32, 3.0),
])
def test_route_from_logits_edge_shapes(T, n_group, topk_group, k, scale):
    rng = np.random.default_rng(T * 7 + k)
    E = 32 * n_group
    L = (rng.standard_normal((T, E)) * scale).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.05).astype(np.float32)
    cfg = moe.MoeConfig(T=T, H=2048, E=E, n_group=n_group, topk_group=topk_group, k=k)
    gi, gw, gc, gP, gl = [a.cpu().numpy() if a is not None else None for a in
                          moe.route_from_logits(cfg, torch.from_numpy(L).to(DEV), torch.from_numpy(bias).to(DEV),
                                                aux=True)]
    ref = oracle.route(L, bias=bias, n_group=n_group, topk_group=topk_group, k=k)
    n_near, near = compare_routing(gi, gw, ref, E, bias=bias, n_group=n_group, topk_group=topk_group)
    rc, rP, rl = oracle.counts_aux(ref["idx"], ref["scores"], E=E)
    compare_counts(gc, gi, rc, ref["idx"], near, E)
    np.testing.assert_allclose(gP, rP, rtol=1e-4, atol=1e-7)
    assert abs(gl[0] - rl) <= 1e-4 * abs(rl)


def test_route_handworked_golden_tokens():
    with open(os.path.join(GOLDEN, "route_handworked.json")) as f:
        fx = json.load(f)
    for tok in fx["tokens"]:
        L, bias = _parse_logits(tok)
        cfg = moe.MoeConfig(T=1)
        gi, gw, gc, _, _ = moe.route_from_logits(cfg, torch.from_numpy(L[None, :]).to(DEV),
                                                 torch.from_numpy(bias).to(DEV))
        assert gi.cpu().numpy()[0].tolist() == tok["idx"], tok["name"]
        np.testing.assert_allclose(gw.cpu().numpy()[0], tok["w"], atol=1e-6, err_msg=tok["name"])
        assert gc.sum().item() == 8


def test_route_is_deterministic():
    w0 = wl.WORKLOADS[4].with_T(8192)
    d = wl.layer_inputs(w0, DEV, with_experts=False)
    cfg = moe.MoeConfig(T=8192)
    a = run_route(cfg, d["hidden"], d["W_router"], d["expert_bias"])
    b = run_route(cfg, d["hidden"], d["W_router"], d["expert_bias"])
    for x, y in zip(a[:4], b[:4]):
        assert np.array_equal(x, y)
    assert a[4] == b[4]


def test_nonfinite_logits_set_status():
    T = 64
    L = torch.zeros(T, 256, device=DEV)
    L[5, 17] = float("nan")
    cfg = moe.MoeConfig(T=T)
    ws = moe.Workspace(cfg, 0, DEV)
    moe.route_from_logits(cfg, L, None, ws=ws)
    assert ws.status() & 1
    assert ws.status() == 0          # reset by the previous read
    moe.route_from_logits(cfg, torch.zeros(T, 256, device=DEV), None, ws=ws)
    assert ws.status() == 0


@pytest.mark.parametrize("T,kernels", [(16, 2), (256, 3)])
def test_route_launch_count(T, kernels):
    # small T: CUDA-core router + select; otherwise W split + tensor-core router + select
    cfg = moe.MoeConfig(T=T)
    d = wl.layer_inputs(wl.WORKLOADS[3].with_T(T), DEV, with_experts=False)
    moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"])
    assert moe.last_launch_count() == kernels
    moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"], aux=True)
    assert moe.last_launch_count() == kernels + 1   # + the balance-loss reduction


def test_expert_feedback_matches_oracle():
    w0 = wl.WORKLOADS[4].with_T(4096)
    d = wl.layer_inputs(w0, DEV, with_experts=False)
    cfg = moe.MoeConfig(T=4096)
    idx, w, counts, _, _ = moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"])
    bias = d["expert_bias"].clone()
    totals = torch.arange(256, dtype=torch.int64, device=DEV)
    moe.expert_feedback(cfg, counts, 1e-3, bias, totals)
    torch.cuda.synchronize()
    ref_b, ref_t = oracle.expert_feedback(counts.cpu().numpy(), 4096, 8, 1e-3,
                                          bias=d["expert_bias"].cpu().numpy(), totals=np.arange(256))
    assert np.array_equal(bias.cpu().numpy(), ref_b)
    assert np.array_equal(totals.cpu().numpy(), ref_t)
    # the hot experts of this workload get their bias lowered
    hot = wl.hot_experts(w0).numpy()
    assert (bias.cpu().numpy()[hot] < d["expert_bias"].cpu().numpy()[hot]).all()


@pytest.mark.parametrize("T", [16, 33, 1000])
def test_prepared_router_matches_route_bit_for_bit(T):
    """moe_prepare_router writes an exact split (hi + mid + lo == W) and
    moe_route_prepared gives moe_route's outputs bit for bit; the prepared
    tensor-core path launches the router GEMM and the selection only."""
    w0 = wl.WORKLOADS[4].with_T(T)
    d = wl.layer_inputs(w0, DEV, with_experts=False)
    cfg = moe.MoeConfig(T=T)
    W = d["W_router"]
    W3 = moe.prepare_router(cfg, W)
    torch.cuda.synchronize()
    parts = W3.float().double()
    assert torch.equal(parts[0] + parts[1] + parts[2], W.double())
    assert torch.equal(W3[0], W.to(torch.bfloat16))                    # hi = RN(W)
    a = moe.route(cfg, d["hidden"], W, d["expert_bias"], aux=True)
    b = moe.route(cfg, d["hidden"], W, d["expert_bias"], aux=True, W_split=W3)
    assert moe.last_launch_count() == 3      # router (CUDA-core or tensor-core) + select + loss
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_decode_router_with_weight_only_4_byte_aligned():
    """The CUDA-core router for decode sizes reads W_router in 16-byte pieces;
    a W_router that is only 4-byte aligned goes to the tensor-core router
    instead, with the same accuracy against the oracle."""
    T = 16
    w0 = wl.WORKLOADS[2].with_T(T)
    d = wl.layer_inputs(w0, DEV, with_experts=False)
    cfg = moe.MoeConfig(T=T)
    W = d["W_router"]
    buf = torch.empty(W.numel() + 1, dtype=torch.float32, device=DEV)
    Wu = buf[1:].view_as(W)
    Wu.copy_(W)
    assert Wu.data_ptr() % 16 == 4
    L = oracle.router_logits(u16(d["hidden"]), W.cpu().numpy())
    for Wx, kernels in ((W, 1), (Wu, 2)):          # CUDA-core router / split + tensor-core router
        g = moe.router_logits(cfg, d["hidden"], Wx).cpu().numpy()
        assert moe.last_launch_count() == kernels
        err = np.abs(g.astype(np.float64) - L)
        assert err.max() <= 2e-6 + 2e-6 * np.abs(L).max(), err.max()


@pytest.mark.parametrize("n_group,topk_group,k", [(8, 4, 8), (8, 2, 8), (4, 2, 6), (8, 4, 32)])
def test_exact_ties_go_to_the_lower_index(n_group, topk_group, k):
    """Logits on a coarse grid (13 values 0.25 apart, bias 0) make exact ties
    at every level: equal experts, equal group scores, equal 4th and 5th
    groups.  Distinct grid values give distinct scores on both sides, and equal
    logits give equal scores and equal sums on both sides, so wherever the
    oracle sees an exact tie the GPU sees the same tie, and the lower index must
    win on both.  Tokens where some gap is non-zero but below 1e-5 (two
    different pairs whose sums nearly coincide) are left out."""
    rng = np.random.default_rng(1000 * n_group + 10 * topk_group + k)
    T, E = 2048, 32 * n_group
    L = (0.25 * rng.integers(0, 13, size=(T, E))).astype(np.float32)
    cfg = moe.MoeConfig(T=T, H=2048, E=E, n_group=n_group, topk_group=topk_group, k=k)
    gi, gw, gc, _, _ = [a.cpu().numpy() if a is not None else None for a in
                        moe.route_from_logits(cfg, torch.from_numpy(L).to(DEV), None)]
    ref = oracle.route(L, n_group=n_group, topk_group=topk_group, k=k)
    from parity import order_margin

    def clear(m):
        return (m == 0.0) | (m >= 1e-5)
    ok = clear(ref["margin_group"]) & clear(ref["margin_expert"]) & clear(order_margin(ref, None))
    tied = (ref["margin_group"] == 0.0) | (ref["margin_expert"] == 0.0)
    assert ok.sum() >= T * 0.9 and (tied & ok).sum() >= T // 4, (ok.sum(), (tied & ok).sum())
    bad = np.nonzero((gi[ok] != ref["idx"][ok]).any(axis=1))[0]
    assert bad.size == 0, "token %d: gpu %s ref %s" % (np.nonzero(ok)[0][bad[0]], gi[ok][bad[0]], ref["idx"][ok][bad[0]])
    assert np.abs(gw[ok].astype(np.float64) - ref["w"][ok]).max() <= 1e-6
    assert np.array_equal(gc, np.bincount(gi.ravel(), minlength=E))


@pytest.mark.parametrize("case", range(12))
def test_route_from_logits_random_settings(case):
    """Seeded random group settings (the supported 4 or 8 groups of 32, any
    number kept, k up to 32), ragged T, random logit scale and bias: the GPU
    selection against the oracle under the usual near-tie rules, counts exact,
    balance-loss terms close."""
    rng = np.random.default_rng(7000 + case)
    n_group = int(rng.choice([4, 8]))
    topk_group = int(rng.integers(1, n_group + 1))
    k = int(rng.integers(1, min(32, 32 * topk_group) + 1))
    T = int(rng.integers(1, 3000))
    E = 32 * n_group
    L = (rng.standard_normal((T, E)) * rng.uniform(0.2, 4.0)).astype(np.float32)
    bias = None if case % 3 == 0 else (rng.standard_normal(E) * rng.uniform(0.0, 0.2)).astype(np.float32)
    cfg = moe.MoeConfig(T=T, H=2048, E=E, n_group=n_group, topk_group=topk_group, k=k)
    gi, gw, gc, gP, gl = [a.cpu().numpy() if a is not None else None for a in
                          moe.route_from_logits(cfg, torch.from_numpy(L).to(DEV),
                                                None if bias is None else torch.from_numpy(bias).to(DEV), aux=True)]
    ref = oracle.route(L, bias=bias, n_group=n_group, topk_group=topk_group, k=k)
    n_near, near = compare_routing(gi, gw, ref, E, bias=bias, n_group=n_group, topk_group=topk_group)
    rc, rP, rl = oracle.counts_aux(ref["idx"], ref["scores"], E=E)
    compare_counts(gc, gi, rc, ref["idx"], near, E)
    np.testing.assert_allclose(gP, rP, rtol=1e-4, atol=1e-7)
    assert abs(gl[0] - rl) <= 1e-4 * abs(rl)
    assert n_near <= max(2, T // 50), (n_group, topk_group, k, T, n_near)
