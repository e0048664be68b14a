"""Shared comparison rules of the GPU-vs-oracle parity tests.

Routing: indices and counts bit-exact, except tokens whose oracle margin at
the group boundary (4th vs 5th group score) or the expert boundary (8th vs
9th surviving biased score) is below 1e-5; those are counted and reported.
Where only the order inside the chosen k hangs on a gap below 1e-5, the
chosen set must match and each expert its weight.  Weights within 1e-6
absolute.

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


def order_margin(ref, bias):
    """Smallest gap between consecutive chosen experts' biased scores (the
    order inside the chosen k), per token, in float64."""
    s = ref["scores"]
    b = s + (0.0 if bias is None else np.asarray(bias, dtype=np.float32))
    b = b.astype(np.float32)
    bs = np.take_along_axis(b, ref["idx"].astype(np.int64), axis=1).astype(np.float64)
    if bs.shape[1] < 2:
        return np.full(bs.shape[0], np.inf)
    return (bs[:, :-1] - bs[:, 1:]).min(axis=1)


def compare_routing(gpu_idx, gpu_w, ref, E, report=None, bias=None):
    """Returns (number of boundary near-tie tokens, their mask); asserts the
    rest match.  Tokens whose chosen set is clear but whose order inside the
    set hangs on a gap below NEAR_TIE are compared as sets, each expert with
    its own weight."""
    gi = np.asarray(gpu_idx)
    gw = np.asarray(gpu_w)
    near = (ref["margin_group"] < NEAR_TIE) | (ref["margin_expert"] < NEAR_TIE)
    loose = (~near) & (order_margin(ref, bias) < NEAR_TIE)
    strict = ~near & ~loose
    mism = np.nonzero((gi[strict] != ref["idx"][strict]).any(axis=1))[0]
    assert mism.size == 0, "index mismatch on %d non-tie tokens, first %s: gpu %s ref %s" % (
        mism.size, np.nonzero(strict)[0][mism[0]], gi[strict][mism[0]], ref["idx"][strict][mism[0]])
    werr = np.abs(gw[strict].astype(np.float64) - ref["w"][strict].astype(np.float64))
    # order near-ties: same set, and each expert carries the same weight
    for t in np.nonzero(loose)[0]:
        og, orf = np.argsort(gi[t], kind="stable"), np.argsort(ref["idx"][t], kind="stable")
        assert np.array_equal(gi[t][og], ref["idx"][t][orf]), "set mismatch on token %d" % t
        werr = np.concatenate([werr.ravel(), np.abs(gw[t][og].astype(np.float64) - ref["w"][t][orf])])
    assert werr.size == 0 or werr.max() <= W_ATOL, "weight error %g" % werr.max()
    if report is not None:
        report["near_tie_tokens"] = int(near.sum())
        report["order_tie_tokens"] = int(loose.sum())
        report["max_w_err"] = float(werr.max()) if werr.size else 0.0
    return int(near.sum()), near


def compare_counts(gpu_counts, gpu_idx, ref_counts, ref_idx, near, E):
    gc = np.asarray(gpu_counts).astype(np.int64)
    assert np.array_equal(gc, np.bincount(np.asarray(gpu_idx).ravel(), minlength=E)), "counts != bincount(idx)"
    assert gc.sum() == np.asarray(gpu_idx).size
    g_excl = gc - np.bincount(np.asarray(gpu_idx)[near].ravel(), minlength=E)
    r_excl = np.asarray(ref_counts).astype(np.int64) - np.bincount(np.asarray(ref_idx)[near].ravel(), minlength=E)
    assert np.array_equal(g_excl, r_excl)


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
