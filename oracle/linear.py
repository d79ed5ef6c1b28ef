"""LoRA linear forward / backward through the dequantised NF4 weight (float64).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Notation (Day 25 notes "Fine-tuning and LoRA/QLoRA", section 2.1 "Core
idea"): frozen weight ``W0`` of shape [d, k] (here [N, K], PyTorch
out x in), ``B`` in R^{d x r}, ``A`` in R^{r x k}, output ``W0 x + B A x``;
section 6.2 "Choosing alpha": the LoRA branch is scaled by ``s = alpha / r``.
Glossary "QLoRA", "How QLoRA works": the frozen layer dequantises NF4 to
bfloat16 before the matmul and adds the LoRA output; backpropagation goes
through the dequantised weight but only the two low-rank matrices are updated
(no gradient for W).

Rows are tokens: ``X`` is [M, K], ``Y = X Wdeq^T + s (X A^T) B^T`` is [M, N].
The backward is the derivative of that expression:

    U  = dY B                   [M, r]
    dX = dY Wdeq + s U A        [M, K]
    dA = s U^T X                [r, K]
    dB = s dY^T T               [N, r]   with T = X A^T from the forward.

Inputs are the exact values the GPU path sees (bfloat16 activations and LoRA
matrices, the dequantised bfloat16 weight) promoted to float64; every sum is
float64.  The SiLU * up glue between the MLP linears is not on the pages: it is
the plain definition ``h = silu(g) * u`` with ``silu(g) = g * sigmoid(g)``.
"""

from __future__ import annotations

import numpy as np

F64 = np.float64


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=F64)


def lora_scale(alpha: float, r: int) -> float:
    """``s = alpha / r`` (Day 25 notes, section 6.2)."""
    return float(alpha) / float(r)


def lora_forward(x, wdeq, a, b, alpha: float, r: int):
    """Return ``(Y, T)`` with ``T = X A^T`` and ``Y = X Wdeq^T + s T B^T``."""
    x, wdeq, a, b = _f64(x), _f64(wdeq), _f64(a), _f64(b)
    s = lora_scale(alpha, r)
    t = x @ a.T
    y = x @ wdeq.T + s * (t @ b.T)
    return y, t


def lora_backward(dy, x, wdeq, a, b, alpha: float, r: int, t=None):
    """Return ``(dX, dA, dB, U)`` for upstream gradient ``dY`` (no dW)."""
    dy, x, wdeq, a, b = _f64(dy), _f64(x), _f64(wdeq), _f64(a), _f64(b)
    s = lora_scale(alpha, r)
    if t is None:
        t = x @ a.T
    t = _f64(t)
    u = dy @ b
    dx = dy @ wdeq + s * (u @ a)
    da = s * (u.T @ x)
    db = s * (dy.T @ t)
    return dx, da, db, u


def lora_grads(dy, x, a, b, alpha: float, r: int, t=None):
    """``(dA, dB)`` of :func:`lora_backward` without dX (the same two formulas)."""
    dy, x, a, b = _f64(dy), _f64(x), _f64(a), _f64(b)
    s = lora_scale(alpha, r)
    if t is None:
        t = x @ a.T
    u = dy @ b
    return s * (u.T @ x), s * (dy.T @ _f64(t))


def lora_forward_rows(x_rows, wdeq, a, b, alpha: float, r: int):
    """:func:`lora_forward` on a subset of token rows (rows are independent)."""
    return lora_forward(x_rows, wdeq, a, b, alpha, r)


def lora_backward_dx_rows(dy_rows, wdeq, a, b, alpha: float, r: int):
    """dX on a subset of token rows (each row of dX depends only on that row of dY)."""
    dy_rows, wdeq, a, b = _f64(dy_rows), _f64(wdeq), _f64(a), _f64(b)
    s = lora_scale(alpha, r)
    return dy_rows @ wdeq + s * ((dy_rows @ b) @ a)


def sigmoid(g):
    g = _f64(g)
    return 1.0 / (1.0 + np.exp(-g))


def silu_mul_forward(g, u):
    """``h = silu(g) * u`` (float64)."""
    g, u = _f64(g), _f64(u)
    return g * sigmoid(g) * u


def silu_mul_backward(dh, g, u):
    """Return ``(dg, du)`` of ``h = silu(g) * u``.

    ``d silu/dg = sigma(g) (1 + g (1 - sigma(g)))``.
    """
    dh, g, u = _f64(dh), _f64(g), _f64(u)
    sg = sigmoid(g)
    du = dh * g * sg
    dg = dh * u * sg * (1.0 + g * (1.0 - sg))
    return dg, du
