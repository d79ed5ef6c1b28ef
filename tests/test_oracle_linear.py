"""Pins of the LoRA linear oracle (forward, backward, SiLU glue).

No GPU.  The forward is checked against the merge identity (a different order
of evaluation that the Day 25 notes state, section 2.6), the backward against
adjoint identities, central finite differences and torch autograd in float64.
"""

import numpy as np
import pytest
import torch

from oracle import linear


def _case(m=12, n=40, k=64, r=8, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((m, k))
    w = rng.standard_normal((n, k)) * 0.02
    a = rng.standard_normal((r, k)) / np.sqrt(k)
    b = rng.standard_normal((n, r)) * 0.01
    dy = rng.standard_normal((m, n))
    return x, w, a, b, dy


def test_forward_merge_identity():
    x, w, a, b, _ = _case()
    alpha, r = 16.0, 8
    y, t = linear.lora_forward(x, w, a, b, alpha, r)
    merged = w + (alpha / r) * (b @ a)
    assert np.allclose(y, x @ merged.T, rtol=1e-12, atol=1e-13)
    assert np.allclose(t, np.einsum("mk,rk->mr", x, a), rtol=1e-12, atol=1e-14)


def test_forward_special_cases():
    x, w, a, b, _ = _case()
    y0, _ = linear.lora_forward(x, w, a, np.zeros_like(b), 16.0, 8)
    assert np.allclose(y0, np.einsum("mk,nk->mn", x, w), rtol=1e-12, atol=1e-14)
    ya, _ = linear.lora_forward(x, w, a, b, 0.0, 8)
    assert np.array_equal(ya, y0)


def test_backward_adjoint_identities():
    x, w, a, b, dy = _case(seed=1)
    alpha, r = 32.0, 8
    s = alpha / r
    y, t = linear.lora_forward(x, w, a, b, alpha, r)
    dx, da, db, _ = linear.lora_backward(dy, x, w, a, b, alpha, r, t)
    # Y is linear in X
    assert np.isclose(np.sum(dy * y), np.sum(dx * x), rtol=1e-11)
    # the LoRA term is linear in B and in A separately
    assert np.isclose(np.sum(dy * (s * t @ b.T)), np.sum(db * b), rtol=1e-11)
    assert np.isclose(np.sum(dy * (s * (x @ a.T) @ b.T)), np.sum(da * a), rtol=1e-11)


def test_backward_matches_autograd_float64():
    x, w, a, b, dy = _case(m=9, n=24, k=128, r=4, seed=2)
    alpha, r = 8.0, 4
    tx, ta, tb = (torch.tensor(v, requires_grad=True) for v in (x, a, b))
    tw = torch.tensor(w)
    y = tx @ tw.T + (alpha / r) * (tx @ ta.T) @ tb.T
    y.backward(torch.tensor(dy))
    dx, da, db, _ = linear.lora_backward(dy, x, w, a, b, alpha, r)
    assert np.allclose(dx, tx.grad.numpy(), rtol=1e-12, atol=1e-13)
    assert np.allclose(da, ta.grad.numpy(), rtol=1e-12, atol=1e-13)
    assert np.allclose(db, tb.grad.numpy(), rtol=1e-12, atol=1e-13)


def test_backward_finite_differences():
    x, w, a, b, dy = _case(m=4, n=8, k=64, r=2, seed=3)
    alpha, r = 4.0, 2

    def loss(xx, aa, bb):
        y, _ = linear.lora_forward(xx, w, aa, bb, alpha, r)
        return float(np.sum(y * dy))

    dx, da, db, _ = linear.lora_backward(dy, x, w, a, b, alpha, r)
    h = 1e-6
    rng = np.random.default_rng(0)
    for arr, grad, which in ((x, dx, 0), (a, da, 1), (b, db, 2)):
        for _ in range(6):
            idx = tuple(rng.integers(0, s) for s in arr.shape)
            p, mi = arr.copy(), arr.copy()
            p[idx] += h
            mi[idx] -= h
            args_p = [x, a, b]
            args_m = [x, a, b]
            args_p[which], args_m[which] = p, mi
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd))


def test_backward_b_zero():
    x, w, a, b, dy = _case(seed=4)
    dx, da, db, _ = linear.lora_backward(dy, x, w, a, np.zeros_like(b), 16.0, 8)
    assert np.all(da == 0)
    assert np.allclose(dx, dy @ w, rtol=1e-12, atol=1e-14)


def test_rows_helpers_agree_with_full():
    x, w, a, b, dy = _case(seed=5)
    y, _ = linear.lora_forward(x, w, a, b, 16.0, 8)
    dx, _, _, _ = linear.lora_backward(dy, x, w, a, b, 16.0, 8)
    rows = [0, 3, 7]
    yr, _ = linear.lora_forward_rows(x[rows], w, a, b, 16.0, 8)
    assert np.allclose(yr, y[rows], rtol=1e-13, atol=1e-15)
    assert np.allclose(linear.lora_backward_dx_rows(dy[rows], w, a, b, 16.0, 8), dx[rows], rtol=1e-13, atol=1e-15)


def test_silu_mul_matches_autograd():
    rng = np.random.default_rng(6)
    g, u, dh = (rng.standard_normal(1000) * 3 for _ in range(3))
    tg, tu = torch.tensor(g, requires_grad=True), torch.tensor(u, requires_grad=True)
    h = torch.nn.functional.silu(tg) * tu
    h.backward(torch.tensor(dh))
    assert np.allclose(linear.silu_mul_forward(g, u), h.detach().numpy(), rtol=1e-13, atol=1e-15)
    dg, du = linear.silu_mul_backward(dh, g, u)
    assert np.allclose(dg, tg.grad.numpy(), rtol=1e-12, atol=1e-14)
    assert np.allclose(du, tu.grad.numpy(), rtol=1e-12, atol=1e-14)
    assert linear.silu_mul_forward(0.0, 5.0) == 0.0
    dg0, _ = linear.silu_mul_backward(1.0, 0.0, 1.0)
    assert dg0 == pytest.approx(0.5)


def test_lora_grads_helper_agrees_with_backward():
    x, w, a, b, dy = _case(seed=7)
    _, da, db, _ = linear.lora_backward(dy, x, w, a, b, 16.0, 8)
    da2, db2 = linear.lora_grads(dy, x, a, b, 16.0, 8)
    assert np.array_equal(da, da2) and np.array_equal(db, db2)
