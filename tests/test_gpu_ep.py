"""Expert parallelism's CUDA kernels on one GPU: moe_ep_dispatch,
moe_expert_rows and moe_combine, driven by ep_forward_local for R = 2 and 4
ranks (each with its own batch and its slice of the experts; the exchanges are
row copies in one process -- no rank waits on another).  Every rank's output
must equal moe_forward's on the same routing bit for bit, since each pair's
expert row does not depend on where it is computed and the combine adds in
moe_forward's order."""
import numpy as np
import pytest
import torch

from group_limited_routing_gb300 import _lib, ep, moe, workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _shards(cfg, d, world, bias=None):
    per = cfg.E // world
    b = d["expert_bias"] if bias is None else bias
    return [ep.ExpertShard(cfg, r, world, d["W_router"], b, d["W_gate_up"][r * per:(r + 1) * per],
                           d["W_down"][r * per:(r + 1) * per], d["shared_gate_up"], d["shared_down"])
            for r in range(world)]


@pytest.mark.parametrize("world,T,wid", [(2, 600, 3), (4, 4096, 4), (2, 40, 2), (4, 30000, 6), (2, 12000, 4)])
def test_ep_local_equals_moe_forward(world, T, wid):
    """(2, 12000): moe_forward's 12000 tokens take the single-CTA down GEMM,
    the ~48000 rows each rank receives the CTA-pair one: the two give the
    same rows."""
    w0 = wl.WORKLOADS[wid].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T, H=w0.H, I=w0.I, Is=w0.Is)
    shards = _shards(cfg, d, world)
    xs = [wl.hidden(w0, DEV, layer=r) for r in range(world)]
    outs = ep.ep_forward_local(shards, xs)
    snap = [o.clone() for o in outs]
    for r in range(world):
        idx, w, _, _, _ = moe.route(cfg, xs[r], d["W_router"], d["expert_bias"])
        ref = moe.forward(cfg, xs[r], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"], idx, w)
        torch.cuda.synchronize()
        assert torch.equal(outs[r], ref), "rank %d of %d: %s" % (r, world, _mismatch_report(
            cfg, d, shards, xs, outs, r, ref, idx, w, snap))


def _mismatch_report(cfg, d, shards, xs, outs, r, ref, idx, w, snap):
    """What differs when a rank's output is not moe_forward's: the tokens,
    the routing, and whether each side repeats itself."""
    bad = (outs[r] != ref).any(1).nonzero().flatten()
    disp = shards[r].dispatch(xs[r])
    ref2 = moe.forward(cfg, xs[r], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"], idx, w)
    outs2 = ep.ep_forward_local(shards, xs)
    torch.cuda.synchronize()
    t0 = int(bad[0])
    return ("%d tokens differ (first %s, max |diff| %g); EP routing equals moe_route: %s / %s; token %d experts %s; "
            "moe_forward repeats itself: %s; the EP step repeats itself: %s, and then equals moe_forward: %s; "
            "the output changed after the EP step: %s" % (
                bad.numel(), bad[:8].tolist(), (outs[r].float() - ref.float()).abs().max().item(),
                torch.equal(disp.idx, idx), torch.equal(disp.w, w), t0, idx[t0].tolist(), torch.equal(ref2, ref),
                torch.equal(outs2[r], outs[r]), torch.equal(outs2[r], ref), not torch.equal(snap[r], outs[r])))


def test_ep_with_residual_equals_moe_forward():
    """The residual is added in the combine on each rank as moe_forward adds
    it: bit for bit."""
    T, world = 2048, 2
    w0 = wl.WORKLOADS[4].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T)
    shards = _shards(cfg, d, world)
    xs = [wl.hidden(w0, DEV, layer=r) for r in range(world)]
    res = [wl.hidden(w0, DEV, layer=10 + r) for r in range(world)]
    outs = ep.ep_forward_local(shards, xs, res)
    for r in range(world):
        idx, w, _, _, _ = moe.route(cfg, xs[r], d["W_router"], d["expert_bias"])
        ref = moe.forward(cfg, xs[r], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"], idx, w,
                          res[r])
        torch.cuda.synchronize()
        assert torch.equal(outs[r], ref), "rank %d" % r


def test_ep_rank_that_receives_nothing():
    """A bias that keeps every token off rank 1's experts: rank 1 receives no
    rows (moe_expert_rows with 0 rows), and both outputs still equal
    moe_forward's."""
    T, world = 500, 2
    w0 = wl.WORKLOADS[3].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T)
    bias = d["expert_bias"].clone()
    bias[128:] = -100.0
    shards = _shards(cfg, d, world, bias)
    xs = [wl.hidden(w0, DEV, layer=r) for r in range(world)]
    disp = shards[0].dispatch(xs[0])
    assert disp.send_counts == [T * cfg.k, 0]
    outs = ep.ep_forward_local(shards, xs)
    for r in range(world):
        idx, w, _, _, _ = moe.route(cfg, xs[r], d["W_router"], bias)
        ref = moe.forward(cfg, xs[r], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"], idx, w)
        torch.cuda.synchronize()
        assert torch.equal(outs[r], ref)


def test_ep_dispatch_layout():
    """moe_ep_dispatch: counts per rank, rows grouped by rank in ascending
    (token, j) order, local expert ids, and slot_of pointing at each pair's row."""
    T, world = 1000, 4
    w0 = wl.WORKLOADS[4].with_T(T)
    d = wl.layer_inputs(w0, DEV, with_experts=False)
    cfg = moe.MoeConfig(T=T)
    idx, _, _, _, _ = moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"])
    counts, x_send, e_send, slot_of = moe.ep_dispatch(cfg, world, d["hidden"], idx)
    torch.cuda.synchronize()
    idx_h = idx.cpu().numpy()
    per = cfg.E // world
    dest = (idx_h // per).ravel()
    order = np.argsort(dest, kind="stable")
    assert counts.cpu().tolist() == np.bincount(dest, minlength=world).tolist()
    slots = slot_of.cpu().numpy().ravel()
    assert np.array_equal(np.sort(slots), np.arange(T * cfg.k))
    assert np.array_equal(slots[order], np.arange(T * cfg.k))
    assert np.array_equal(e_send.cpu().numpy()[slots], idx_h.ravel() % per)
    xh = d["hidden"].cpu()
    assert torch.equal(x_send.cpu()[torch.from_numpy(slots).long()], xh[torch.arange(T).repeat_interleave(cfg.k)])


def test_ep_calls_reject_bad_arguments():
    T = 64
    cfg = moe.MoeConfig(T=T)
    x = torch.zeros(T, cfg.H, dtype=torch.bfloat16, device=DEV)
    idx = torch.zeros(T, cfg.k, dtype=torch.int32, device=DEV)
    with pytest.raises(_lib.MoeError):
        moe.ep_dispatch(cfg, 3, x, idx)                 # 256 experts do not split over 3 ranks
    Y = torch.zeros(10, cfg.H, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(_lib.MoeError):                  # the shared rows would run past Y
        moe.combine(cfg, Y, 0, idx, torch.zeros(T, cfg.k, device=DEV))
