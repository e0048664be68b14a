"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against what the routing article ("InternLumina-U2
中256个专家的路由秘密：分组受限Top-K、Expert Bias与Fused MoE详解") and plain
mathematics fix: brute-force enumeration of every group subset and every
k-subset on tiny shapes, special cases that reduce to a plain top-k or to a
library matmul, hand-worked fixtures, invariants and closed forms.  No GPU.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(a, seed=None):
    return oracle.bf16_round(np.asarray(a, dtype=np.float32))


def f32_of(u16):
    return oracle.bf16_bits_to_f32(u16)


# ------------------------------------------------------------------ helpers

def brute_route(b, s, n_group, topk_group, k, rsf=2.5):
    """Selection by exhaustive search, written from the article's definition
    (section 二 step 2) without sorting: a group's score is its best pair sum,
    the kept groups are the topk_group-subset with the largest total, and the
    chosen experts are the k-subset of the kept experts with the largest total
    biased score.  Sums of pairs are fp32 (as the group score is); totals in
    float64.  Returns (set of groups, set of experts, weights by expert)."""
    E = len(b)
    gs = E // n_group
    gscore = []
    for j in range(n_group):
        mem = range(j * gs, (j + 1) * gs)
        gscore.append(max(float(np.float32(b[p]) + np.float32(b[q]))
                          for p, q in itertools.combinations(mem, 2)))
    best_groups = max(itertools.combinations(range(n_group), topk_group),
                      key=lambda S: sum(gscore[j] for j in S))
    surv = [e for j in best_groups for e in range(j * gs, (j + 1) * gs)]
    best = max(itertools.combinations(surv, k), key=lambda S: sum(float(b[e]) for e in S))
    tot = sum(float(s[e]) for e in best)
    wts = {e: float(s[e]) / tot * rsf for e in best}
    return set(best_groups), set(best), wts


def fp32_b(logits, bias):
    s = oracle.route(logits[None, :], bias=bias, n_group=1, topk_group=1, k=1)["scores"][0]
    return s, (s + (bias if bias is not None else np.float32(0))).astype(np.float32)


# --------------------------------------------------------------- bf16, logits

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 20000),
        np.array([0.0, -0.0, 1.0, np.inf, -np.inf, 3.0e38, 1e-40, -1e-41], dtype=np.float32),
        # exact ties between two bf16 values: must go to the even one
        (np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 2.0 + 2 ** -7], dtype=np.float32)),
    ]).astype(np.float32)
    ours = oracle.bf16_round(vals)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    nan = oracle.bf16_round(np.array([np.nan], dtype=np.float32))
    assert np.isnan(f32_of(nan)[0])


def test_router_logits_match_numpy_matmul():
    rng = np.random.default_rng(2)
    x = bf16(rng.standard_normal((37, 256)))
    W = (rng.standard_normal((256, 256)) * 0.02).astype(np.float32)
    ours = oracle.router_logits(x, W)
    ref = (f32_of(x).astype(np.float64) @ W.astype(np.float64).T).astype(np.float32)
    # both are double sums rounded once; they may differ only at a rounding boundary
    np.testing.assert_array_max_ulp(ours, ref, maxulp=1)


def test_router_logits_not_transposed():
    rng = np.random.default_rng(3)
    x = bf16(rng.standard_normal((8, 64)))
    W = (rng.standard_normal((256, 64)) * 0.02).astype(np.float32)
    ours = oracle.router_logits(x, W)
    assert ours.shape == (8, 256)
    # logit of expert e is the dot product with row e of W
    e = 77
    np.testing.assert_allclose(ours[:, e], f32_of(x).astype(np.float64) @ W[e].astype(np.float64), rtol=1e-6)


def test_sigmoid_scores_match_scipy():
    rng = np.random.default_rng(4)
    L = (rng.standard_normal((64, 256)) * 4).astype(np.float32)
    s = oracle.route(L)["scores"]
    ref = expit(L.astype(np.float64)).astype(np.float32)
    np.testing.assert_array_max_ulp(s, ref, maxulp=1)


# ---------------------------------------------------------- brute force pins

@pytest.mark.parametrize("E,n_group,topk_group,k", [
    (16, 4, 2, 3), (24, 6, 3, 4), (12, 3, 1, 2), (16, 4, 4, 5), (20, 5, 2, 7), (8, 2, 1, 4),
])
def test_brute_force_tiny_shapes(E, n_group, topk_group, k):
    rng = np.random.default_rng(E * 100 + k)
    for trial in range(40):
        L = (rng.standard_normal(E) * 1.5).astype(np.float32)
        bias = (rng.standard_normal(E) * 0.1).astype(np.float32) if trial % 2 else None
        r = oracle.route(L[None, :], bias=bias, n_group=n_group, topk_group=topk_group, k=k)
        s, b = fp32_b(L, bias)
        groups, chosen, wts = brute_route(b, s, n_group, topk_group, k)
        idx = r["idx"][0]
        assert set(idx.tolist()) == chosen
        gs = E // n_group
        assert {e // gs for e in idx} <= groups
        # order: biased score descending
        assert all(b[idx[i]] >= b[idx[i + 1]] for i in range(k - 1))
        for j, e in enumerate(idx):
            assert abs(r["w"][0, j] - wts[e]) <= 5e-7 * max(1.0, wts[e])


def test_group_stage_brute_force_full_shape():
    """E=256 in 8 groups of 32, keep 4: all 70 subsets of 4 groups enumerated."""
    rng = np.random.default_rng(5)
    T = 200
    L = rng.standard_normal((T, 256)).astype(np.float32)
    bias = (rng.standard_normal(256) * 0.05).astype(np.float32)
    r = oracle.route(L, bias=bias)
    for t in range(T):
        s, b = fp32_b(L[t], bias)
        gscore = [max(float(np.float32(b[p]) + np.float32(b[q]))
                      for p, q in itertools.combinations(range(32 * j, 32 * j + 32), 2))
                  for j in range(8)]
        best = max(itertools.combinations(range(8), 4), key=lambda S: sum(gscore[j] for j in S))
        used = {e // 32 for e in r["idx"][t]}
        assert used <= set(best)
        # the top-8 of the survivors: no surviving expert outside the choice beats the worst chosen
        surv = [e for j in best for e in range(32 * j, 32 * j + 32)]
        chosen = set(r["idx"][t].tolist())
        worst = min(b[e] for e in chosen)
        assert all(b[e] <= worst for e in surv if e not in chosen)


@pytest.mark.parametrize("n_group,topk_group", [(1, 1), (8, 8), (4, 4)])
def test_plain_topk_special_cases(n_group, topk_group):
    """With one group, or with every group kept, the method is a plain top-k
    over s + bias (ties to the lower index)."""
    rng = np.random.default_rng(6 + n_group)
    T, E, k = 300, 256, 8
    L = rng.standard_normal((T, E)).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.05).astype(np.float32)
    r = oracle.route(L, bias=bias, n_group=n_group, topk_group=topk_group, k=k)
    s = expit(L.astype(np.float64)).astype(np.float32)
    b = (s + bias).astype(np.float32)
    ref = np.argsort(-b, axis=1, kind="stable")[:, :k]
    assert np.array_equal(r["idx"], ref)
    den = s[np.arange(T)[:, None], ref].astype(np.float64).sum(1, keepdims=True)
    np.testing.assert_allclose(r["w"], s[np.arange(T)[:, None], ref] / den * 2.5, atol=1e-6)


# ---------------------------------------------------------------- fixtures

def _parse_logits(tok):
    def val(v):
        if v == "0":
            return np.float32(0.0)
        if v == "ln3":
            return np.float32(np.log(3.0))
        if v == "-ln3":
            return np.float32(-np.log(3.0))
        return np.float32(float(v))
    L = np.full(256, val(tok["logit_default"]), dtype=np.float32)
    for key, v in tok["logit_exceptions"].items():
        L[int(key)] = val(v)
    bias = np.zeros(256, dtype=np.float32)
    for key, v in tok["bias"].items():
        if ".." in key:
            lo, hi = map(int, key.split(".."))
            bias[lo:hi + 1] = v
        else:
            bias[int(key)] = v
    return L, bias


def test_handworked_golden_routes():
    with open(os.path.join(GOLDEN, "route_handworked.json")) as f:
        fx = json.load(f)
    c = fx["config"]
    for tok in fx["tokens"]:
        L, bias = _parse_logits(tok)
        r = oracle.route(L[None, :], bias=bias, n_group=c["n_group"], topk_group=c["topk_group"],
                         k=c["k"], rsf=c["rsf"], eps=c["eps"])
        assert r["idx"][0].tolist() == tok["idx"], tok["name"]
        np.testing.assert_allclose(r["w"][0], tok["w"], atol=1e-7, err_msg=tok["name"])
        assert r["margin_group"][0] == pytest.approx(tok["margin_group"], abs=1e-12)
        assert r["margin_expert"][0] == pytest.approx(tok["margin_expert"], abs=1e-7)


# -------------------------------------------------------------- invariants

def test_routing_invariants():
    rng = np.random.default_rng(8)
    T = 2000
    L = (rng.standard_normal((T, 256))).astype(np.float32)
    bias = (rng.standard_normal(256) * 0.05).astype(np.float32)
    r = oracle.route(L, bias=bias)
    idx, w, s = r["idx"], r["w"], r["scores"]
    b = (s + bias).astype(np.float32)
    for t in range(T):
        groups = {e // 32 for e in idx[t]}
        assert len(groups) <= 4
        assert len(set(idx[t].tolist())) == 8
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 2.5) <= 2e-6)
    # w is proportional to the unbiased score
    ratio = w / s[np.arange(T)[:, None], idx]
    assert np.all(np.abs(ratio / ratio[:, :1] - 1) < 1e-6)
    # ordered by biased score
    bs = b[np.arange(T)[:, None], idx]
    assert np.all(np.diff(bs, axis=1) <= 0)
    counts, _, _ = oracle.counts_aux(idx)
    assert counts.sum() == 8 * T
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=256))


def test_huge_bias_forces_expert_but_not_its_weight():
    rng = np.random.default_rng(9)
    T = 500
    L = rng.standard_normal((T, 256)).astype(np.float32)
    bias = np.zeros(256, dtype=np.float32)
    bias[123] = 10.0
    r = oracle.route(L, bias=bias)
    assert np.all(r["idx"][:, 0] == 123)
    s = r["scores"]
    den = s[np.arange(T)[:, None], r["idx"]].astype(np.float64).sum(1)
    np.testing.assert_allclose(r["w"][:, 0], s[:, 123] / den * 2.5, rtol=2e-6)


def test_bias_shift_leaves_selection():
    """A constant added to every expert's bias shifts every biased score and
    group score alike; the choice is unchanged (away from near-ties)."""
    rng = np.random.default_rng(10)
    T = 1000
    L = rng.standard_normal((T, 256)).astype(np.float32)
    bias = (rng.standard_normal(256) * 0.05).astype(np.float32)
    r0 = oracle.route(L, bias=bias)
    r1 = oracle.route(L, bias=(bias + np.float32(0.125)).astype(np.float32))
    clear = (r0["margin_group"] > 1e-5) & (r0["margin_expert"] > 1e-5)
    assert clear.mean() > 0.9
    assert np.array_equal(r0["idx"][clear], r1["idx"][clear])
    # the weights come from the unbiased scores, so they do not move either
    np.testing.assert_array_equal(r0["w"][clear], r1["w"][clear])


def test_bias_changes_selection_not_weight_formula():
    rng = np.random.default_rng(11)
    T = 400
    L = rng.standard_normal((T, 256)).astype(np.float32)
    bias = (rng.standard_normal(256) * 0.5).astype(np.float32)
    r0 = oracle.route(L)
    r1 = oracle.route(L, bias=bias)
    assert (r0["idx"] != r1["idx"]).any()
    s = r1["scores"]
    sel = s[np.arange(T)[:, None], r1["idx"]].astype(np.float64)
    np.testing.assert_allclose(r1["w"], sel / sel.sum(1, keepdims=True) * 2.5, atol=1e-6)


def test_eps_only_matters_for_zero_scores():
    L = np.full((1, 256), -200.0, dtype=np.float32)       # sigmoid underflows to 0 in fp32
    r = oracle.route(L)
    assert np.all(r["w"] == 0.0) and np.all(np.isfinite(r["w"]))


def test_non_finite_logits_are_refused():
    L = np.zeros((2, 256), dtype=np.float32)
    L[1, 5] = np.nan
    with pytest.raises(FloatingPointError):
        oracle.route(L)


# ------------------------------------------------------------------ aux loss

def test_aux_loss_identities():
    rng = np.random.default_rng(12)
    T = 700
    L = rng.standard_normal((T, 256)).astype(np.float32)
    r = oracle.route(L)
    counts, P, aux = oracle.counts_aux(r["idx"], r["scores"])
    f = counts / (8.0 * T)
    assert f.sum() == pytest.approx(1.0, abs=1e-12)
    assert P.sum() == pytest.approx(1.0, abs=1e-9)
    assert aux == pytest.approx(256 * float((f * P).sum()), rel=1e-12)
    # uniform: every score equal and every expert hit equally often -> loss 1
    idx = np.arange(256, dtype=np.int32).reshape(32, 8)
    s = np.full((32, 256), 0.5, dtype=np.float32)
    c2, P2, aux2 = oracle.counts_aux(idx, s)
    assert np.all(c2 == 1) and np.allclose(P2, 1 / 256)
    assert aux2 == pytest.approx(1.0, abs=1e-12)
    # all selections on one expert that also holds all the score mass -> loss E
    idx3 = np.zeros((4, 8), dtype=np.int32)
    s3 = np.zeros((4, 256), dtype=np.float32)
    s3[:, 0] = 1.0
    _, _, aux3 = oracle.counts_aux(idx3, s3)
    assert aux3 == pytest.approx(256.0)


# --------------------------------------------------------------- expert math

def _textbook_swiglu(x_bf16, Wgu, Wd):
    """SwiGLU FFN from numpy matmuls and torch's bf16 rounding of the
    intermediate: down(silu(gate x) * up x), Wgu = [gate; up] rows, Wd [I, H]."""
    X = f32_of(x_bf16).astype(np.float64)
    I = Wd.shape[0]
    Wg = f32_of(Wgu[:I]).astype(np.float64)
    Wu = f32_of(Wgu[I:]).astype(np.float64)
    G = X @ Wg.T
    U = X @ Wu.T
    act = (G * expit(G) * U).astype(np.float32)
    act = torch.from_numpy(act).to(torch.bfloat16).to(torch.float64).numpy()
    return act @ f32_of(Wd).astype(np.float64)


def _expert_setup(T=24, H=128, I=64, E=6, k=3, seed=13):
    rng = np.random.default_rng(seed)
    x = bf16(rng.standard_normal((T, H)))
    Wgu = bf16(rng.standard_normal((E, 2 * I, H)) * 0.05)
    Wd = bf16(rng.standard_normal((E, I, H)) * 0.05)
    sgu = bf16(rng.standard_normal((2 * I, H)) * 0.05)
    sd = bf16(rng.standard_normal((I, H)) * 0.05)
    return rng, x, Wgu, Wd, sgu, sd


def test_forced_routing_is_textbook_swiglu():
    rng, x, Wgu, Wd, sgu, sd = _expert_setup()
    T, k = x.shape[0], 3
    zero_sgu = np.zeros_like(sgu)
    for e in range(Wgu.shape[0]):
        idx = np.full((T, k), e, dtype=np.int32)
        w = np.full((T, k), 1.0 / k, dtype=np.float32)
        w[:, 0] = 1.0 - np.float32(2.0 / k)
        out = oracle.experts(x, Wgu, Wd, zero_sgu, sd, idx, w)
        ref = _textbook_swiglu(x, Wgu[e], Wd[e]) * w.astype(np.float64).sum(1, keepdims=True)
        np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12)


def test_zero_weights_leave_the_shared_expert():
    rng, x, Wgu, Wd, sgu, sd = _expert_setup(seed=14)
    T = x.shape[0]
    idx = rng.integers(0, Wgu.shape[0], (T, 3)).astype(np.int32)
    w = np.zeros((T, 3), dtype=np.float32)
    out = oracle.experts(x, Wgu, Wd, sgu, sd, idx, w)
    np.testing.assert_allclose(out, _textbook_swiglu(x, sgu, sd), rtol=1e-9, atol=1e-12)


def test_dense_mlp_is_textbook_swiglu_with_its_own_size():
    # the dense first layer: one SwiGLU MLP of intermediate size I != the experts'
    rng = np.random.default_rng(21)
    T, H, I = 9, 128, 96
    x = bf16(rng.standard_normal((T, H)))
    gu = bf16(rng.standard_normal((2 * I, H)) * 0.05)
    dn = bf16(rng.standard_normal((I, H)) * 0.05)
    res = bf16(rng.standard_normal((T, H)))
    np.testing.assert_allclose(oracle.dense_ffn(x, gu, dn), _textbook_swiglu(x, gu, dn), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(oracle.dense_ffn(x, gu, dn, residual=res),
                               _textbook_swiglu(x, gu, dn) + f32_of(res).astype(np.float64), rtol=1e-9,
                               atol=1e-12)
    # gate and up are not interchangeable (silu(gate) * up)
    swapped = np.concatenate([gu[I:], gu[:I]])
    assert np.abs(oracle.dense_ffn(x, swapped, dn) - oracle.dense_ffn(x, gu, dn)).max() > 1e-3


def test_weighted_sum_of_experts_plus_shared_and_residual():
    rng, x, Wgu, Wd, sgu, sd = _expert_setup(seed=15)
    T = x.shape[0]
    idx = np.stack([rng.permutation(Wgu.shape[0])[:3] for _ in range(T)]).astype(np.int32)
    w = rng.random((T, 3)).astype(np.float32)
    res = bf16(rng.standard_normal(x.shape))
    out = oracle.experts(x, Wgu, Wd, sgu, sd, idx, w, residual=res)
    per_e = [_textbook_swiglu(x, Wgu[e], Wd[e]) for e in range(Wgu.shape[0])]
    ref = _textbook_swiglu(x, sgu, sd) + f32_of(res)
    for t in range(T):
        for j in range(3):
            ref[t] += float(w[t, j]) * per_e[idx[t, j]][t]
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12)
    # token subsets give the same rows
    tok = np.array([5, 0, 17], dtype=np.int32)
    sub = oracle.experts(x, Wgu, Wd, sgu, sd, idx, w, residual=res, tokens=tok)
    np.testing.assert_array_equal(sub, out[tok])


def test_down_projection_is_linear_and_untransposed():
    rng, x, Wgu, Wd, sgu, sd = _expert_setup(seed=16)
    T = x.shape[0]
    idx = np.zeros((T, 3), dtype=np.int32)
    idx[:, 1], idx[:, 2] = 1, 2
    w = np.full((T, 3), 0.25, dtype=np.float32)
    z = np.zeros_like(sgu)
    a = oracle.experts(x, Wgu, Wd, z, sd, idx, w)
    Wd2 = bf16(f32_of(Wd) * 2)          # doubling a bf16 value is exact
    b = oracle.experts(x, Wgu, Wd2, z, sd, idx, w)
    np.testing.assert_array_equal(b, 2 * a)


def test_out_of_range_expert_index_is_reported():
    rng, x, Wgu, Wd, sgu, sd = _expert_setup(seed=17)
    idx = np.zeros((x.shape[0], 3), dtype=np.int32)
    idx[3, 1] = Wgu.shape[0]
    with pytest.raises(IndexError):
        oracle.experts(x, Wgu, Wd, sgu, sd, idx, np.ones(idx.shape, np.float32))


# ------------------------------------------------------------- stacking norm

def test_rmsnorm_matches_numpy():
    rng = np.random.default_rng(18)
    x = bf16(rng.standard_normal((50, 512)) * rng.uniform(0.01, 30, (50, 1)))
    ours = f32_of(oracle.rmsnorm(x, 1e-6)).astype(np.float64)
    X = f32_of(x).astype(np.float64)
    ref = X / np.sqrt((X * X).mean(axis=1, keepdims=True) + 1e-6)
    # the oracle rounds once to bf16: within half a bf16 ulp (2^-9 relative)
    assert np.all(np.abs(ours - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)
    np.testing.assert_allclose(np.sqrt((ours ** 2).mean(axis=1)), 1.0, atol=1e-2)


# ------------------------------------------------------ bias feedback (NEXT)

def test_expert_feedback_moves_bias_toward_balance():
    """Routing article §三: cold experts are raised, hot ones lowered; an
    expert at exactly the balanced load k T / E is left alone; totals add up."""
    E, T, k, g = 8, 4, 2, 0.001
    counts = np.array([0, 1, 2, 3, 1, 1, 0, 0], dtype=np.int32)   # sum = 8 = k T, mean = 1
    bias = np.linspace(-0.1, 0.1, E).astype(np.float32)
    nb, tot = oracle.expert_feedback(counts, T, k, g, bias=bias, totals=np.arange(E))
    step = nb.astype(np.float64) - bias.astype(np.float64)
    assert np.all(step[counts < 1] > 0) and np.all(step[counts > 1] < 0) and np.all(step[counts == 1] == 0)
    np.testing.assert_allclose(np.abs(step[counts != 1]), g, rtol=1e-5)
    assert np.array_equal(tot, np.arange(E) + counts)
    # perfectly balanced counts leave the bias unchanged
    nb2, _ = oracle.expert_feedback(np.full(E, 1, np.int32), T, k, g, bias=bias)
    assert np.array_equal(nb2, bias)
    # repeated feedback on a routed batch lowers the most-hit expert's bias
    rng = np.random.default_rng(19)
    L = rng.standard_normal((256, 256)).astype(np.float32)
    L[:, 7] += 3.0
    r = oracle.route(L)
    c, _, _ = oracle.counts_aux(r["idx"])
    nb3, _ = oracle.expert_feedback(c, 256, 8, 0.01, bias=np.zeros(256, np.float32))
    assert nb3[7] == np.float32(-0.01) and c[7] == c.max()
