"""The parity rules themselves (tests/parity.py), checked on the CPU.

The GPU tests accept, for a token whose oracle margin at the group or expert
boundary is below 1e-5, any answer the method allows when those close scores
fall either way.  These checks make sure that rule is not a blank cheque: the
oracle's own answers pass; an expert from a dropped group, a repeated expert,
a wrong order, a wrong weight or a non-top-k pick fail; and on a token built
with an exact group tie, both sides of the tie pass while a third group does
not.
"""
import numpy as np

import oracle
from parity import NEAR_TIE, biased_scores, compare_routing, valid_selection


def _ref(L, bias=None):
    return oracle.route(L.astype(np.float32), bias=bias)


def _weights(s, sel, rsf=2.5, eps=1e-20):
    sc = s.astype(np.float64)[np.asarray(sel)]
    return sc / (sc.sum() + eps) * rsf


def test_oracle_answers_are_valid():
    rng = np.random.default_rng(11)
    L = rng.standard_normal((300, 256)).astype(np.float32)
    bias = (rng.standard_normal(256) * 0.05).astype(np.float32)
    ref = _ref(L, bias)
    b = biased_scores(ref, bias)
    for t in range(L.shape[0]):
        ok, why = valid_selection(ref["idx"][t], ref["w"][t], ref["scores"][t], b[t], 8, 4)
        assert ok, (t, why)
    rep = {}
    compare_routing(ref["idx"], ref["w"], ref, 256, rep, bias=bias)
    assert rep["near_tie_differ"] == 0 and rep["order_tie_differ"] == 0


def test_invalid_answers_fail():
    rng = np.random.default_rng(12)
    L = (rng.standard_normal((200, 256)) * 2.0).astype(np.float32)
    ref = _ref(L)
    b = biased_scores(ref, None)
    clear = np.nonzero((ref["margin_group"] > 1e-3) & (ref["margin_expert"] > 1e-3))[0]
    assert clear.size > 50
    for t in clear[:50]:
        sel = ref["idx"][t].copy()
        s = ref["scores"][t]
        groups = set((sel // 32).tolist())
        dropped = [j for j in range(8) if j not in groups]
        # an expert of a dropped group (its best one) in place of the last pick
        j = dropped[0]
        alt = sel.copy()
        alt[-1] = 32 * j + int(np.argmax(b[t][32 * j:32 * j + 32]))
        assert not valid_selection(alt, _weights(s, alt), s, b[t], 8, 4)[0]
        # a repeated expert
        rep_ = sel.copy()
        rep_[-1] = rep_[0]
        assert not valid_selection(rep_, _weights(s, rep_), s, b[t], 8, 4)[0]
        # the first two swapped (their gap is far above the tolerance here)
        if b[t][sel[0]] - b[t][sel[1]] > 10 * NEAR_TIE:
            sw = sel.copy()
            sw[[0, 1]] = sw[[1, 0]]
            assert not valid_selection(sw, _weights(s, sw), s, b[t], 8, 4)[0]
        # a weight off by ten times the tolerance
        w = _weights(s, sel)
        w[3] += 1e-5
        assert not valid_selection(sel, w, s, b[t], 8, 4)[0]
        # the 9th-best survivor in place of the 8th (not a top-8)
        kept = sorted(groups)
        surv = np.concatenate([np.arange(32 * g, 32 * g + 32) for g in kept])
        rest = np.setdiff1d(surv, sel)
        ninth = rest[np.argmax(b[t][rest])]
        if b[t][sel[-1]] - b[t][ninth] > 10 * NEAR_TIE:
            alt2 = sel.copy()
            alt2[-1] = ninth
            assert not valid_selection(alt2, _weights(s, alt2), s, b[t], 8, 4)[0]


def test_exact_group_tie_allows_either_side_only():
    # groups 3 and 4 tie exactly for the 4th place; every other expert is far below
    L = np.full((1, 256), -10.0, dtype=np.float32)
    L[0, [0, 1]] = 3.0
    L[0, [32, 33]] = 2.9
    L[0, [64, 65]] = 2.8
    L[0, [96, 97]] = 2.0
    L[0, [128, 129]] = 2.0
    L[0, [160, 161]] = -1.0
    ref = _ref(L)
    assert ref["margin_group"][0] == 0.0
    assert ref["idx"][0].tolist() == [0, 1, 32, 33, 64, 65, 96, 97]     # the lower group wins the tie
    s, b = ref["scores"][0], biased_scores(ref, None)[0]
    other = np.array([0, 1, 32, 33, 64, 65, 128, 129])
    assert valid_selection(ref["idx"][0], ref["w"][0], s, b, 8, 4)[0]
    assert valid_selection(other, _weights(s, other), s, b, 8, 4)[0]
    third = np.array([0, 1, 32, 33, 64, 65, 160, 161])
    assert not valid_selection(third, _weights(s, third), s, b, 8, 4)[0]
    # the same through compare_routing: a GPU answer on the other side of the tie passes
    rep = {}
    compare_routing(other[None, :].astype(np.int32), _weights(s, other)[None, :].astype(np.float32), ref, 256, rep)
    assert rep["near_tie_tokens"] == 1 and rep["near_tie_differ"] == 1


def test_covering_tokens_reach_every_m_tile():
    """covering_tokens picks, from a routing, tokens whose rows fall into every
    128-row m-tile of every bucket (stable (token, j) order inside a bucket),
    into every bucket's last row, and into every m-tile of the shared expert."""
    from parity import covering_tokens
    rng = np.random.default_rng(3)
    T, k, E = 3000, 8, 256
    p = np.ones(E)
    p[:4] = 200.0                                    # a few long buckets
    p[200:] = 0.0                                    # and empty ones
    idx = rng.choice(E, size=(T, k), p=p / p.sum()).astype(np.int32)
    tok = set(covering_tokens(idx, T, E).tolist())
    for e in range(E):
        rows = [t for t in range(T) for j in range(k) if idx[t, j] == e]   # bucket order
        for r0 in range(0, len(rows), 128):
            assert any(t in tok for t in rows[r0:r0 + 128]), (e, r0)
        if rows:
            assert rows[-1] in tok
    for r0 in range(0, T, 128):
        assert any(t in tok for t in range(r0, min(T, r0 + 128)))
    assert T - 1 in tok
