"""Pins of the oracle's backward of the expert stage (CPU, no GPU).

The backward is pinned to the forward it differentiates: central differences of
the oracle's own forward (with the intermediate left unrounded, so the forward
is smooth) over every input element of a tiny layer, stepping bf16 inputs to
their neighbouring bf16 values; and to float64 torch autograd of a textbook
SwiGLU MoE written with torch matmuls on a small layer."""
import numpy as np
import pytest
import torch

import oracle


def bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def val(u):
    return oracle.bf16_bits_to_f32(u).astype(np.float64)


def _tiny(seed=3, T=3, H=16, I=8, E=3, k=2):
    rng = np.random.default_rng(seed)
    x = bf16(rng.standard_normal((T, H)))
    gu = bf16(rng.standard_normal((E, 2 * I, H)) * 0.3)
    dn = bf16(rng.standard_normal((E, I, H)) * 0.3)
    sgu = bf16(rng.standard_normal((2 * I, H)) * 0.3)
    sd = bf16(rng.standard_normal((I, H)) * 0.3)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    R = rng.standard_normal((T, H))
    return x, gu, dn, sgu, sd, idx, w, R


def _loss(x, gu, dn, sgu, sd, idx, w, R):
    return float((oracle.experts(x, gu, dn, sgu, sd, idx, w, round_act=False) * R).sum())


def _fd_bf16(arr, pos, f):
    """Central difference of f over arr[pos], stepping to the neighbouring bf16 values."""
    a = arr.copy()
    u = int(a[pos])
    up = (u + 1) if u & 0x8000 == 0 else (u - 1)      # one ulp away from zero ...
    dn_ = (u - 1) if u & 0x8000 == 0 else (u + 1)     # ... and one toward it
    if u in (0x0000, 0x8000):
        up, dn_ = 0x0001, 0x8001
    a[pos] = up
    fp, vp = f(a), val(np.uint16(up))
    a[pos] = dn_
    fm, vm = f(a), val(np.uint16(dn_))
    return (fp - fm) / (vp - vm)


def test_backward_matches_finite_differences():
    x, gu, dn, sgu, sd, idx, w, R = _tiny()
    g = oracle.experts_backward(x, gu, dn, sgu, sd, idx, w, R, round_act=False)
    T, H = x.shape

    def close(fd, an, what):
        assert abs(fd - an) <= 2e-3 * max(1.0, abs(an)), (what, fd, an)

    for pos in np.ndindex(x.shape):
        close(_fd_bf16(x, pos, lambda a: _loss(a, gu, dn, sgu, sd, idx, w, R)), g["dx"][pos], ("x", pos))
    for pos in np.ndindex(gu.shape):
        close(_fd_bf16(gu, pos, lambda a: _loss(x, a, dn, sgu, sd, idx, w, R)), g["dW_gate_up"][pos], ("gu", pos))
    for pos in np.ndindex(dn.shape):
        close(_fd_bf16(dn, pos, lambda a: _loss(x, gu, a, sgu, sd, idx, w, R)), g["dW_down"][pos], ("dn", pos))
    for pos in np.ndindex(sgu.shape):
        close(_fd_bf16(sgu, pos, lambda a: _loss(x, gu, dn, a, sd, idx, w, R)), g["d_shared_gate_up"][pos],
              ("sgu", pos))
    for pos in np.ndindex(sd.shape):
        close(_fd_bf16(sd, pos, lambda a: _loss(x, gu, dn, sgu, a, idx, w, R)), g["d_shared_down"][pos],
              ("sd", pos))
    # the output is linear in w: any step is exact up to rounding
    for pos in np.ndindex(w.shape):
        wp, wm = w.copy(), w.copy()
        wp[pos] += np.float32(0.125)
        wm[pos] -= np.float32(0.125)
        fd = (_loss(x, gu, dn, sgu, sd, idx, wp, R) - _loss(x, gu, dn, sgu, sd, idx, wm, R)) / \
            (float(wp[pos]) - float(wm[pos]))
        close(fd, g["dw"][pos], ("w", pos))
    # experts no token routed to get zero gradients
    used = set(idx.ravel().tolist())
    for e in range(gu.shape[0]):
        if e not in used:
            assert not g["dW_gate_up"][e].any() and not g["dW_down"][e].any()


def test_backward_matches_torch_autograd_of_a_textbook_moe():
    rng = np.random.default_rng(11)
    T, H, I, E, k = 20, 64, 32, 6, 3
    x = bf16(rng.standard_normal((T, H)))
    gu = bf16(rng.standard_normal((E, 2 * I, H)) * 0.1)
    dn = bf16(rng.standard_normal((E, I, H)) * 0.1)
    sgu = bf16(rng.standard_normal((2 * I, H)) * 0.1)
    sd = bf16(rng.standard_normal((I, H)) * 0.1)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    dout = rng.standard_normal((T, H))
    g = oracle.experts_backward(x, gu, dn, sgu, sd, idx, w, dout, round_act=False)

    tx = torch.tensor(val(x), requires_grad=True)
    tgu = torch.tensor(val(gu), requires_grad=True)
    tdn = torch.tensor(val(dn), requires_grad=True)
    tsgu = torch.tensor(val(sgu), requires_grad=True)
    tsd = torch.tensor(val(sd), requires_grad=True)
    tw = torch.tensor(w.astype(np.float64), requires_grad=True)

    def mlp(xx, wgu, wd):
        gate, up = xx @ wgu[:I].T, xx @ wgu[I:].T
        return (torch.nn.functional.silu(gate) * up) @ wd

    out = mlp(tx, tsgu, tsd)
    for j in range(k):
        rows = []
        for t in range(T):
            rows.append(tw[t, j] * mlp(tx[t:t + 1], tgu[idx[t, j]], tdn[idx[t, j]])[0])
        out = out + torch.stack(rows)
    (out * torch.tensor(dout)).sum().backward()
    for name, t in (("dx", tx), ("dW_gate_up", tgu), ("dW_down", tdn), ("d_shared_gate_up", tsgu),
                    ("d_shared_down", tsd), ("dw", tw)):
        np.testing.assert_allclose(g[name], t.grad.numpy(), rtol=1e-9, atol=1e-11, err_msg=name)


def test_rounded_intermediate_only_changes_what_uses_it():
    # with the bf16 rounding of the intermediate (the GPU's forward), the
    # gradients move by at most the rounding's relative size
    x, gu, dn, sgu, sd, idx, w, R = _tiny(seed=5)
    a = oracle.experts_backward(x, gu, dn, sgu, sd, idx, w, R, round_act=False)
    b = oracle.experts_backward(x, gu, dn, sgu, sd, idx, w, R, round_act=True)
    np.testing.assert_array_equal(a["dx"], b["dx"])                      # da does not use a
    np.testing.assert_array_equal(a["dW_gate_up"], b["dW_gate_up"])
    for name in ("dW_down", "dw"):
        assert np.abs(a[name] - b[name]).max() <= 2 ** -8 * np.abs(a[name]).max() * 4
