"""Pins of the LoRA-dropout oracle (no GPU): the Philox4x32-10 generator against its
published known-answer vectors, the statistics and layout of the keep mask, and
the dropout layer's backward against the adjoint identities of a layer that is
linear in X, A and B for a fixed mask, plus finite differences."""

import json
import os

import numpy as np
import pytest

from oracle import dropout, linear

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.json")) as f:
        kat = json.load(f)["vectors"]
    for v in kat:
        ctr = np.array([[int(h, 16) for h in v["ctr"]]], dtype=np.uint64)
        key = np.array([[int(h, 16) for h in v["key"]]], dtype=np.uint64)
        out = dropout.philox4x32_10(ctr, key)[0]
        assert [int(x) for x in out] == [int(h, 16) for h in v["out"]]


def test_keep_fraction_and_independence():
    m, k, p = 64, 1024, 0.05
    keep = dropout.keep_mask(1234, 0, m, k, p)
    n = keep.size
    frac_drop = 1.0 - keep.mean()
    assert abs(frac_drop - p) < 5 * np.sqrt(p * (1 - p) / n)
    other = dropout.keep_mask(1234, 1, m, k, p)
    assert 0.8 * 2 * p * (1 - p) < np.mean(keep != other) < 1.2 * 2 * p * (1 - p)   # independent draws
    assert dropout.keep_mask(7, 3, 4, 64, 0.0).all()


def test_mask_counter_layout():
    """Element e uses word e % 4 of the Philox block with counter e // 4: rebuild one row by hand."""
    seed, offset, k, p = 99, 5, 128, 0.3
    keep = dropout.keep_mask(seed, offset, 2, k, p)
    thr = dropout.keep_threshold(p)
    e0 = k  # row 1
    for e in range(e0, e0 + k):
        ctr = np.array([[e // 4, 0, offset, 0]], dtype=np.uint64)
        key = np.array([[seed, 0]], dtype=np.uint64)
        word = int(dropout.philox4x32_10(ctr, key)[0][e % 4])
        assert keep[1, e - e0] == (word >= thr)
    packed = dropout.pack_mask(keep)
    assert packed.shape == (2, k // 8)
    assert ((packed[1, 0] >> 3) & 1) == keep[1, 3]
    assert np.array_equal(dropout.unpack_mask(packed, k), keep)


def _case(m=12, n=20, k=64, r=4, seed=0, p=0.25):
    rng = np.random.default_rng(seed)
    x, dy = rng.standard_normal((m, k)), rng.standard_normal((m, n))
    w, a, b = rng.standard_normal((n, k)), rng.standard_normal((r, k)), rng.standard_normal((n, r))
    keep = rng.random((m, k)) >= p
    return x, dy, w, a, b, keep, p


def test_no_drop_is_the_plain_layer():
    x, dy, w, a, b, _, _ = _case()
    keep = np.ones_like(x, dtype=bool)
    y, t = dropout.lora_forward(x, w, a, b, 8.0, 4, keep, 0.0)
    y0, t0 = linear.lora_forward(x, w, a, b, 8.0, 4)
    assert np.allclose(y, y0, rtol=1e-14, atol=1e-12) and np.allclose(t, t0, rtol=1e-14, atol=1e-12)
    g = dropout.lora_backward(dy, x, w, a, b, 8.0, 4, keep, 0.0)
    g0 = linear.lora_backward(dy, x, w, a, b, 8.0, 4)[:3]
    for u, v in zip(g, g0):
        assert np.allclose(u, v, rtol=1e-13, atol=1e-12)


def test_adjoint_identities_with_a_fixed_mask():
    x, dy, w, a, b, keep, p = _case(seed=1)
    alpha, r = 6.0, 4
    s = alpha / r
    y, t = dropout.lora_forward(x, w, a, b, alpha, r, keep, p)
    dx, da, db = dropout.lora_backward(dy, x, w, a, b, alpha, r, keep, p)
    # Y is linear in X: <dY, Y(X)> = <dX, X>
    assert abs(np.sum(dy * y) - np.sum(dx * x)) < 1e-11 * np.sum(np.abs(dy * y))
    # the branch is linear in B and in A
    yb = s * (t @ b.T)
    assert abs(np.sum(dy * yb) - np.sum(db * b)) < 1e-11 * np.sum(np.abs(dy * yb))
    assert abs(np.sum(dy * yb) - np.sum(da * a)) < 1e-11 * np.sum(np.abs(dy * yb))


@pytest.mark.parametrize("which", ["x", "a", "b"])
def test_finite_differences(which):
    x, dy, w, a, b, keep, p = _case(m=5, n=6, k=64, r=3, seed=2, p=0.4)
    alpha, r = 3.0, 3
    args = {"x": x, "a": a, "b": b}
    grads = dict(zip(("x", "a", "b"), dropout.lora_backward(dy, x, w, a, b, alpha, r, keep, p)))

    def loss(v):
        kw = dict(args)
        kw[which] = v
        y, _ = dropout.lora_forward(kw["x"], w, kw["a"], kw["b"], alpha, r, keep, p)
        return np.sum(dy * y)

    base = args[which]
    rng = np.random.default_rng(3)
    d = rng.standard_normal(base.shape)
    h = 1e-6
    fd = (loss(base + h * d) - loss(base - h * d)) / (2 * h)
    assert abs(fd - np.sum(grads[which] * d)) < 1e-6 * (1 + abs(fd))
