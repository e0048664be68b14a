"""Shared comparison rules of the GPU-vs-oracle parity tests.

Routing: indices and counts bit-exact, except tokens whose oracle margin at
the group boundary (4th vs 5th group score) or the expert boundary (8th vs
9th surviving biased score) is below 1e-5; those are counted and reported,
and the GPU's answer for them must be one the method allows when the close
scores fall either way.  Where only the order inside the chosen k hangs on a
gap below 1e-5, the chosen set must match, each expert its weight, and the
order must descend up to 1e-5; those tokens are counted and reported too.
Weights within 1e-6 absolute.

Layer output: max |out - ref| <= 2e-2 * max |ref| and
sum |out - ref| / sum |ref| <= 5e-3, ref the oracle's float64 output.
"""
import numpy as np

NEAR_TIE = 1e-5
W_ATOL = 1e-6
MAX_REL = 2e-2
MEAN_REL = 5e-3


def bf16_tensor_bits(t):
    """torch bf16 tensor -> numpy uint16 bit patterns (on the host)."""
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(t):
    import torch
    return t.detach().cpu().to(torch.float64).numpy()


def biased_scores(ref, bias):
    """The oracle's biased scores fp32(s + bias) [T, E] (what selection ranks)."""
    s = ref["scores"].astype(np.float32)
    b = np.float32(0.0) if bias is None else np.asarray(bias, dtype=np.float32)
    return (s + b).astype(np.float32)


def order_margin(ref, bias):
    """Smallest gap between consecutive chosen experts' biased scores (the
    order inside the chosen k), per token, in float64."""
    b = biased_scores(ref, bias)
    bs = np.take_along_axis(b, ref["idx"].astype(np.int64), axis=1).astype(np.float64)
    if bs.shape[1] < 2:
        return np.full(bs.shape[0], np.inf)
    return (bs[:, :-1] - bs[:, 1:]).min(axis=1)


def valid_selection(sel, wts, s, b, n_group, topk_group, rsf=2.5, eps=1e-20, tol=NEAR_TIE):
    """Whether one token's selection `sel` (k expert ids, in output order) with
    weights `wts` is one of the answers the method allows when scores closer
    than `tol` may fall either way.  s, b: the oracle's unbiased and biased
    fp32 scores [E] of that token.  Returns (ok, reason).

    Allowed means: k distinct ids; a kept set of topk_group groups, every one
    of them within tol of the topk_group-th best group score (top-1 + top-2
    of the group's biased scores) and no dropped group above the weakest kept
    one by more than tol, that holds all chosen ids; the chosen ids are a
    top-k of that set's experts up to tol and come out in descending biased
    score up to tol; each weight is s / (sum of the chosen s + eps) * rsf."""
    from itertools import combinations
    sel = np.asarray(sel, dtype=np.int64)
    E = b.shape[0]
    gs = E // n_group
    k = sel.size
    if sel.min() < 0 or sel.max() >= E or np.unique(sel).size != k:
        return False, "ids out of range or repeated"
    bb = b.astype(np.float32).reshape(n_group, gs)
    top2 = np.sort(bb, axis=1)[:, -2:]
    g = (top2[:, 1] + top2[:, 0]).astype(np.float32).astype(np.float64)
    g_cut = np.sort(g)[::-1][topk_group - 1]
    used = set((sel // gs).tolist())
    if len(used) > topk_group:
        return False, "more than %d groups" % topk_group
    cand = [j for j in range(n_group) if g[j] >= g_cut - tol]
    if not used.issubset(cand):
        return False, "a chosen expert lies in a group that is not among the best %d" % topk_group
    bd = b.astype(np.float64)
    chosen = bd[sel]
    if k > 1 and (chosen[:-1] - chosen[1:]).min() < -tol:
        return False, "order inside the chosen k is not descending"
    found = False
    for kept in combinations(cand, topk_group):
        if not used.issubset(kept):
            continue
        gmin = min(g[j] for j in kept)
        if any(g[j] > gmin + tol for j in range(n_group) if j not in kept):
            continue
        surv = np.concatenate([np.arange(j * gs, (j + 1) * gs) for j in kept])
        rest = np.setdiff1d(surv, sel)
        if rest.size == 0 or bd[rest].max() <= chosen.min() + tol:
            found = True
            break
    if not found:
        return False, "not a top-%d of any allowed kept group set" % k
    sc = s.astype(np.float64)[sel]
    wref = sc / (sc.sum() + eps) * rsf
    werr = np.abs(np.asarray(wts, dtype=np.float64) - wref).max()
    if werr > W_ATOL:
        return False, "weight error %g" % werr
    return True, ""


def compare_routing(gpu_idx, gpu_w, ref, E, report=None, bias=None, n_group=8, topk_group=4, rsf=2.5,
                    eps=1e-20):
    """Returns (number of boundary near-tie tokens, their mask); asserts the
    rest match.

    * Tokens clear of every near tie: indices bit-exact, weights within W_ATOL.
    * Boundary near ties (group topk_group / topk_group+1 or expert k / k+1
      margin below NEAR_TIE): the GPU's answer must be one the method allows
      when those scores fall either way (valid_selection).
    * Tokens whose chosen set is clear but whose order inside it hangs on a
      gap below NEAR_TIE: the same set, each expert with its own weight, and
      an order that descends up to NEAR_TIE.
    The report gives each class's size and how many of its tokens differ from
    the oracle's answer."""
    gi = np.asarray(gpu_idx)
    gw = np.asarray(gpu_w)
    near = (ref["margin_group"] < NEAR_TIE) | (ref["margin_expert"] < NEAR_TIE)
    loose = (~near) & (order_margin(ref, bias) < NEAR_TIE)
    strict = ~near & ~loose
    mism = np.nonzero((gi[strict] != ref["idx"][strict]).any(axis=1))[0]
    assert mism.size == 0, "index mismatch on %d non-tie tokens, first %s: gpu %s ref %s" % (
        mism.size, np.nonzero(strict)[0][mism[0]], gi[strict][mism[0]], ref["idx"][strict][mism[0]])
    werr = np.abs(gw[strict].astype(np.float64) - ref["w"][strict].astype(np.float64))
    werr = werr.ravel()
    b = biased_scores(ref, bias)
    # order near-ties: same set, a descending order up to NEAR_TIE, each expert its own weight
    for t in np.nonzero(loose)[0]:
        og, orf = np.argsort(gi[t], kind="stable"), np.argsort(ref["idx"][t], kind="stable")
        assert np.array_equal(gi[t][og], ref["idx"][t][orf]), "set mismatch on token %d" % t
        bo = b[t][gi[t].astype(np.int64)].astype(np.float64)
        assert gi.shape[1] < 2 or (bo[:-1] - bo[1:]).min() >= -NEAR_TIE, "order on token %d not descending" % t
        werr = np.concatenate([werr, np.abs(gw[t][og].astype(np.float64) - ref["w"][t][orf])])
    assert werr.size == 0 or werr.max() <= W_ATOL, "weight error %g" % werr.max()
    # boundary near-ties: the GPU's answer must be an allowed one
    for t in np.nonzero(near)[0]:
        ok, why = valid_selection(gi[t], gw[t], ref["scores"][t], b[t], n_group, topk_group, rsf, eps)
        assert ok, "near-tie token %d: %s (gpu %s, oracle %s)" % (t, why, gi[t], ref["idx"][t])
    if report is not None:
        T = gi.shape[0]
        differs = (gi != ref["idx"]).any(axis=1)
        report.update(T=int(T), near_tie_tokens=int(near.sum()), near_tie_differ=int((near & differs).sum()),
                      order_tie_tokens=int(loose.sum()), order_tie_differ=int((loose & differs).sum()),
                      max_w_err=float(werr.max()) if werr.size else 0.0)
    return int(near.sum()), near


def record(name, rep):
    """Appends one parity report (a JSON line) to the file named by the
    GLR_PARITY_RECORD environment variable, when it is set."""
    import json
    import os
    path = os.environ.get("GLR_PARITY_RECORD")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(dict(case=name, **rep)) + "\n")


def compare_counts(gpu_counts, gpu_idx, ref_counts, ref_idx, near, E):
    gc = np.asarray(gpu_counts).astype(np.int64)
    assert np.array_equal(gc, np.bincount(np.asarray(gpu_idx).ravel(), minlength=E)), "counts != bincount(idx)"
    assert gc.sum() == np.asarray(gpu_idx).size
    g_excl = gc - np.bincount(np.asarray(gpu_idx)[near].ravel(), minlength=E)
    r_excl = np.asarray(ref_counts).astype(np.int64) - np.bincount(np.asarray(ref_idx)[near].ravel(), minlength=E)
    assert np.array_equal(g_excl, r_excl)


def covering_tokens(idx, T, E, mt=128):
    """Tokens that put at least one compared row into every m-tile of the
    grouped GEMMs, from a routing idx [T, k] (host numpy): the bucket of expert
    e holds its (token, j) pairs in ascending (token, j) order, cut into
    mt-row m-tiles; one token per m-tile (its first row), the token of every
    bucket's last row (its part-filled last tile), and for the shared expert
    (all T tokens in order) one token per m-tile plus the last."""
    idx = np.asarray(idx)
    k = idx.shape[1]
    flat = idx.ravel().astype(np.int64)
    order = np.argsort(flat, kind="stable")          # pair ids, by expert then (token, j)
    experts = flat[order]
    starts = np.searchsorted(experts, np.arange(E))
    r = np.arange(flat.size) - starts[experts]
    first_of_tile = (r % mt) == 0
    last_of_bucket = np.r_[experts[1:] != experts[:-1], True]
    tok = order[first_of_tile | last_of_bucket] // k
    shared = np.r_[np.arange(0, T, mt), T - 1]
    return np.unique(np.concatenate([tok, shared])).astype(np.int32)


def output_errors(out, ref):
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(out - ref)
    return dict(max_err=float(err.max()), max_ref=float(np.abs(ref).max()),
                mean_rel=float(err.sum() / max(np.abs(ref).sum(), 1e-300)),
                rel_l2=float(np.linalg.norm(out - ref) / max(np.linalg.norm(ref), 1e-10)))


def assert_output_close(out, ref, what=""):
    e = output_errors(out, ref)
    assert e["max_err"] <= MAX_REL * e["max_ref"], "%s max err %g > %g * %g" % (what, e["max_err"], MAX_REL,
                                                                                e["max_ref"])
    assert e["mean_rel"] <= MEAN_REL, "%s mean relative error %g" % (what, e["mean_rel"])
    return e
