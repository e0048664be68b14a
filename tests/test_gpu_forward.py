"""Expert-stage parity on the GPU: moe_forward against the CPU oracle.

The oracle takes the routing the GPU uses as its input (teacher forcing), so
near-tie routing decisions cannot pollute the output check.  Cases cover the
five workloads' shapes (sampled tokens at full size), ragged T, empty and
overfull buckets (0, 1, 127, 128, 129 rows and one expert holding every
row), zero weights (shared expert only), the residual, bad indices and
determinism."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from group_limited_routing_gb300 import moe, workloads as wl
from parity import assert_output_close, bf16_to_f64, covering_tokens

pytestmark = pytest.mark.gpu
DEV = "cuda"


def u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class Host:
    """Host copies of a layer's bf16 weights for the oracle (bit patterns)."""

    def __init__(self, d):
        self.x = u16(d["hidden"])
        self.gu = u16(d["W_gate_up"])
        self.dn = u16(d["W_down"])
        self.sgu = u16(d["shared_gate_up"])
        self.sd = u16(d["shared_down"])


def check(cfg, d, idx, w, tokens=None, residual=None, what="", host=None):
    out = moe.forward(cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"],
                      idx, w, residual)
    torch.cuda.synchronize()
    h = host or Host(d)
    tok = None if tokens is None else np.asarray(tokens, dtype=np.int32)
    ref = oracle.experts(h.x, h.gu, h.dn, h.sgu, h.sd, idx.cpu().numpy(), w.cpu().numpy(),
                         residual=None if residual is None else u16(residual), tokens=tok)
    got = bf16_to_f64(out)
    if tok is not None:
        got = got[tok]
    e = assert_output_close(got, ref, what)
    print("%s: max err %.3e (max ref %.3e), mean rel %.3e, rel-L2 %.3e" % (what, e["max_err"], e["max_ref"],
                                                                             e["mean_rel"], e["rel_l2"]))
    return out


def small_layer(T, H=512, I=128, E=256, seed=0):
    w0 = wl.Workload(90 + seed, "test", T=T, H=H, E=E, n_group=E // 32, I=I, Is=I)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T, H=H, E=E, n_group=E // 32, I=I, Is=I)
    return cfg, d


@pytest.mark.parametrize("wid,T,nsample", [(1, 128, None), (2, 16, None), (3, 4096, 256), (4, 32768, "cover"),
                                           (5, 8192, 192), (6, 32768, "cover")])
def test_forward_matches_oracle_on_workloads(wid, T, nsample):
    """nsample "cover": every m-tile of both grouped GEMMs (each bucket's
    128-row tiles, its part-filled last tile, the shared expert's tiles) has
    at least one compared row; workload 6 puts ~half of all rows on 16 hot
    experts (~8k rows each)."""
    w0 = wl.WORKLOADS[wid].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T, H=w0.H, I=w0.I, Is=w0.Is)
    idx, w, counts, _, _ = moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"])
    tokens = None
    if nsample == "cover":
        tokens = covering_tokens(idx.cpu().numpy(), T, cfg.E)
    elif nsample is not None:
        tokens = np.union1d(wl.token_sample(T, nsample, seed=wid).numpy(), [0, T - 1]).astype(np.int32)
    if w0.hot_experts_per_group:
        c = counts.cpu().numpy()
        print("workload %d: hot-expert share %.3f" % (wid, c[wl.hot_experts(w0).numpy()].sum() / c.sum()))
    check(cfg, d, idx, w, tokens, what="workload %d T=%d (%s tokens)" % (wid, T, "all" if tokens is None
                                                                           else len(tokens)))


@pytest.mark.parametrize("T", [1, 7, 16, 17, 32, 33, 128, 300, 1000])
def test_forward_ragged_T_random_routing(T):
    # T <= 16 runs the small-T GEMM kinds (16 A rows per stage), 17 the others
    cfg, d = small_layer(T, seed=T % 7)
    idx, w = wl.random_routing(T, cfg.E, cfg.k, seed=T, device=DEV)
    check(cfg, d, idx, w, what="ragged T=%d" % T)


def test_forward_bucket_sizes_and_empty_experts():
    # bucket sizes 0, 1, 127, 128, 129 and one large bucket, by construction
    T, k, E = 1200, 8, 256
    cfg, d = small_layer(T, E=E, seed=3)
    rng = np.random.default_rng(5)
    sizes = {10: 1, 11: 127, 12: 128, 13: 129, 14: 255}
    pairs = []
    for e, n in sizes.items():
        pairs += [e] * n
    rest = [e for e in range(20, 200)] * 100
    need = T * k - len(pairs)
    pairs += rest[:need]
    pairs = np.array(pairs, dtype=np.int32)
    # token t gets pairs[t::T]; a token may hold an expert twice, which the
    # expert stage treats as two separate (token, expert) pairs
    idx = pairs.reshape(k, T).T.copy()
    counts = np.bincount(idx.ravel(), minlength=E)
    assert [counts[e] for e in sizes] == list(sizes.values()) and counts[0] == 0
    w = rng.random((T, k)).astype(np.float32)
    check(cfg, d, torch.from_numpy(idx).to(DEV), torch.from_numpy(w).to(DEV), what="bucket sizes")


@pytest.mark.parametrize("H,k,T", [(512, 4, 300), (512, 1, 97), (512, 12, 300), (1536, 8, 257), (2048, 5, 130),
                                   (4096, 8, 40)])
def test_forward_other_k_and_hidden_sizes(H, k, T):
    # k < 8 pads the combine's eight-term sum with zero rows, k > 8 takes its
    # batches of eight; H = 512 puts four tokens in a combine block, H = 4096
    # gives a thread two column vectors of a row; H = 1536 and 4096 run the
    # bucketing's row gather without its loads-first path
    cfg, d = small_layer(T, H=H, seed=k)
    cfg = dataclasses.replace(cfg, k=k)
    idx, w = wl.random_routing(T, cfg.E, k, seed=H + k, device=DEV)
    check(cfg, d, idx, w, what="H=%d k=%d T=%d" % (H, k, T))
    r = (torch.randn(T, H, device=DEV) * 0.5).to(torch.bfloat16)
    check(cfg, d, idx, w, residual=r, what="H=%d k=%d T=%d with residual" % (H, k, T))


@pytest.mark.parametrize("T", [500, 32, 16, 5])
def test_forward_one_expert_holds_every_row(T):
    # T <= 32: one-launch bucketing; T <= 16: 16-row m-tiles of the small GEMM
    # kinds (a bucket of k T rows is then split into k T / 16 tiles)
    cfg, d = small_layer(T, seed=4)
    idx = torch.full((T, cfg.k), 77, dtype=torch.int32, device=DEV)   # every slot to expert 77
    w = torch.rand(T, cfg.k, device=DEV) * 0.3
    check(cfg, d, idx, w, what="one expert, %d rows" % (T * cfg.k))


def test_forward_zero_weights_is_shared_expert_only():
    T = 256
    cfg, d = small_layer(T, seed=5)
    idx, _ = wl.random_routing(T, cfg.E, cfg.k, seed=9, device=DEV)
    w = torch.zeros(T, cfg.k, device=DEV)
    out = check(cfg, d, idx, w, what="zero weights")
    # the same as routing every token nowhere useful: equals shared(x) computed with other indices
    idx2, _ = wl.random_routing(T, cfg.E, cfg.k, seed=10, device=DEV)
    out2 = moe.forward(cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"],
                       idx2, w)
    assert torch.equal(out, out2)


def test_forward_with_residual_full_size():
    w0 = wl.WORKLOADS[5].with_T(1024)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=1024)
    idx, w, _, _, _ = moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"])
    res = torch.randn(1024, 2048, device=DEV).to(torch.bfloat16)
    tokens = wl.token_sample(1024, 128, seed=2).numpy()
    check(cfg, d, idx, w, tokens, residual=res, what="residual")


def test_forward_out_may_alias_residual():
    T = 200
    cfg, d = small_layer(T, seed=6)
    idx, w = wl.random_routing(T, cfg.E, cfg.k, seed=11, device=DEV)
    res = torch.randn(T, cfg.H, device=DEV).to(torch.bfloat16)
    expect = moe.forward(cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"],
                         idx, w, res.clone())
    buf = res.clone()
    moe.forward(cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"], idx, w,
                buf, out=buf)
    assert torch.equal(buf, expect)


@pytest.mark.parametrize("T", [64, 16])
def test_forward_bad_index_is_skipped_and_reported(T):
    cfg, d = small_layer(T, seed=7)
    idx, w = wl.random_routing(T, cfg.E, cfg.k, seed=12, device=DEV)
    bad = idx.clone()
    bad[3, 2] = cfg.E          # out of range: the kernels skip it and flag it
    bad[9, 0] = -1
    ws = moe.Workspace(cfg, 1, DEV)
    out = moe.forward(cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"],
                      bad, w, ws=ws)
    st = ws.status()
    assert st & 2 and st & 8
    # the skipped pairs contribute nothing: same as weight 0 for them
    w2 = w.clone()
    w2[3, 2] = 0.0
    w2[9, 0] = 0.0
    ok = moe.forward(cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"],
                     idx, w2)
    assert torch.equal(out, ok)
    assert ws.status() == 0


def test_forward_is_deterministic():
    w0 = wl.WORKLOADS[3].with_T(4096)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=4096)
    idx, w, _, _, _ = moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"])
    a = moe.forward(cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"], idx, w)
    b = moe.forward(cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"], idx, w)
    assert torch.equal(a, b)


@pytest.mark.parametrize("wid,T", [(4, 8192), (6, 30000)])
def test_forward_on_freshly_mapped_memory_repeats_itself(wid, T):
    """The grouped GEMMs on a workspace and outputs the driver has just
    mapped (the allocator's cache emptied first: cold address translation,
    slow TMA stores) must give the warm run's rows bit for bit, through
    moe_forward and through moe_expert_rows on ~2T rows.  A bucket's
    part-filled output piece once reused a staging buffer that the previous
    TMA store of the same warp could still be reading."""
    w0 = wl.WORKLOADS[wid].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T, H=w0.H, I=w0.I, Is=w0.Is)
    idx, w, _, _, _ = moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"])
    ref = moe.forward(cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"], idx, w)
    cfg_r = moe.MoeConfig(T=T, H=w0.H, I=w0.I, Is=w0.Is, E=64, n_group=2)
    n = 2 * T
    xr = d["hidden"].repeat(2, 1).contiguous()
    er = (idx.flatten()[:n] % 64).to(torch.int32).contiguous()
    ref_rows = moe.expert_rows(cfg_r, xr, er, d["W_gate_up"][:64], d["W_down"][:64])
    torch.cuda.synchronize()
    for rep in range(3):
        torch.cuda.empty_cache()
        out = moe.forward(cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"],
                          idx, w)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), "moe_forward, repetition %d" % rep
        torch.cuda.empty_cache()
        rows = moe.expert_rows(cfg_r, xr, er, d["W_gate_up"][:64], d["W_down"][:64])
        torch.cuda.synchronize()
        assert torch.equal(rows, ref_rows), "moe_expert_rows, repetition %d" % rep


@pytest.mark.parametrize("T,kernels", [(128, 6), (32, 4), (16, 4)])
def test_forward_launch_count(T, kernels):
    # hist, scan, scatter (one launch for T <= 32), gate/up GEMM, down GEMM, combine
    cfg, d = small_layer(T, seed=8)
    idx, w = wl.random_routing(T, cfg.E, cfg.k, seed=13, device=DEV)
    moe.forward(cfg, d["hidden"], d["W_gate_up"], d["W_down"], d["shared_gate_up"], d["shared_down"], idx, w)
    assert moe.last_launch_count() == kernels


def test_host_pipeline_matches_the_layer():
    """Batches streamed from pinned host memory give the layer's own outputs."""
    T = 1024
    w0 = wl.WORKLOADS[3].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T)
    layer = moe.MoELayer(cfg, d["W_router"], d["expert_bias"], d["W_gate_up"], d["W_down"], d["shared_gate_up"],
                         d["shared_down"])
    xs = [torch.randn(T, cfg.H).to(torch.bfloat16).pin_memory() for _ in range(5)]
    outs = [torch.empty(T, cfg.H, dtype=torch.bfloat16).pin_memory() for _ in range(5)]
    pipe = moe.HostPipeline(layer)
    pipe.run(xs, outs)
    torch.cuda.synchronize()
    for xh, oh in zip(xs, outs):
        ref = layer(xh.to(DEV)).cpu()
        assert torch.equal(oh, ref)
    assert pipe.launches == 5 * 8      # prepared router: GEMM + select, then 6 forward kernels


@pytest.mark.parametrize("T", [16, 1000])
def test_graphed_step_matches_eager(T):
    """A MoELayer step captured in a CUDA graph gives the eager step's output
    bit for bit, replay after replay, on new inputs copied into it."""
    w0 = wl.WORKLOADS[3].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T)
    layer = moe.MoELayer(cfg, d["W_router"], d["expert_bias"], d["W_gate_up"], d["W_down"], d["shared_gate_up"],
                         d["shared_down"])
    g = moe.GraphedStep(layer, d["hidden"])
    for seed in range(3):
        x = (torch.randn(T, cfg.H, device=DEV, generator=torch.Generator(DEV).manual_seed(seed))).to(torch.bfloat16)
        ref = layer(x).clone()
        got = g(x).clone()
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
    assert g.status() == 0


@pytest.mark.parametrize("T,I,nsample", [(1, 4608, None), (16, 4608, None), (17, 1024, None), (300, 4608, None),
                                         (4096, 4608, 128)])
def test_dense_ffn_matches_oracle(T, I, nsample):
    """The dense first-layer MLP (one weight group through the grouped GEMMs,
    T <= 16 on the small-T kinds) against the oracle, with a residual."""
    H = 2048
    g = torch.Generator(DEV).manual_seed(T + I)
    x = torch.randn(T, H, device=DEV, generator=g).to(torch.bfloat16)
    gu = (torch.randn(2 * I, H, device=DEV, generator=g) * 0.02).to(torch.bfloat16)
    dn = (torch.randn(I, H, device=DEV, generator=g) * 0.02).to(torch.bfloat16)
    res = torch.randn(T, H, device=DEV, generator=g).to(torch.bfloat16)
    ws = moe.DenseWorkspace(T, H, I, DEV)
    out = moe.dense_ffn(x, gu, dn, res, ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert moe.last_launch_count() == 4          # tile list, gate/up GEMM, down GEMM, combine
    tokens = None
    if nsample is not None:
        tokens = np.union1d(wl.token_sample(T, nsample, seed=3).numpy(), [0, T - 1]).astype(np.int32)
    ref = oracle.dense_ffn(u16(x), u16(gu), u16(dn), residual=u16(res), tokens=tokens)
    got = bf16_to_f64(out)
    if tokens is not None:
        got = got[tokens]
    assert_output_close(got, ref, "dense T=%d I=%d" % (T, I))
    # no residual: the MLP alone
    out2 = moe.dense_ffn(x, gu, dn, ws=ws)
    ref2 = oracle.dense_ffn(u16(x), u16(gu), u16(dn), tokens=tokens)
    got2 = bf16_to_f64(out2)
    assert_output_close(got2 if tokens is None else got2[tokens], ref2, "dense T=%d I=%d, no residual" % (T, I))


def test_large_batch_sampled_parity():
    """T = 131072 (4x the bench batch; ~1M bucket rows, 32-bit row indices and
    byte offsets well past 2^31 bytes in X_perm and Y): routing counts are
    exact, and sampled outputs match the oracle."""
    T = 131072
    w0 = wl.WORKLOADS[4].with_T(T)
    d = wl.layer_inputs(w0, DEV)
    cfg = moe.MoeConfig(T=T, H=w0.H, I=w0.I, Is=w0.Is)
    idx, w, counts, _, _ = moe.route(cfg, d["hidden"], d["W_router"], d["expert_bias"])
    torch.cuda.synchronize()
    assert int(counts.sum()) == 8 * T
    assert torch.equal(counts.cpu(), torch.bincount(idx.cpu().view(-1).long(), minlength=256).to(torch.int32))
    tokens = covering_tokens(idx.cpu().numpy(), T, cfg.E)
    check(cfg, d, idx, w, tokens, what="T=%d, a row in every m-tile (%d tokens)" % (T, len(tokens)))


@pytest.mark.parametrize("T", [24576, 24780, 30000])
def test_forward_pair_tiles_edge_buckets(T):
    """The CTA-pair down GEMM (256-row pair tiles, T >= 24576) on bucket
    sizes that end a pair tile in every way: empty, 1, 127, 128, 129, 255,
    256, 257 and 383 rows, one bucket of ~half of all rows, the rest spread;
    every m-tile compared.  The shared expert's last pair tile holds 48 rows
    at T = 30000 and 204 at T = 24780."""
    k, E = 8, 256
    cfg, d = small_layer(T, seed=6)
    rng = np.random.default_rng(T)
    sizes = {3: 1, 4: 127, 5: 128, 6: 129, 7: 255, 8: 256, 9: 257, 10: 383}
    pairs = []
    for e, n in sizes.items():
        pairs += [e] * n
    pairs += [40] * (T * k // 2)                   # one hot bucket, half of all rows
    rest = list(range(50, 250))
    need = T * k - len(pairs)
    pairs += (rest * (need // len(rest) + 1))[:need]
    pairs = np.array(pairs, dtype=np.int32)
    rng.shuffle(pairs)
    idx = pairs.reshape(T, k).copy()
    counts = np.bincount(idx.ravel(), minlength=E)
    assert [counts[e] for e in sizes] == list(sizes.values()) and counts[0] == 0
    w = rng.random((T, k)).astype(np.float32)
    tokens = covering_tokens(idx, T, E)
    check(cfg, d, torch.from_numpy(idx).to(DEV), torch.from_numpy(w).to(DEV), tokens,
          what="pair tiles T=%d (%d tokens)" % (T, len(tokens)))
