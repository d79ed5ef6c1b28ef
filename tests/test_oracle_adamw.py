"""Pins of the AdamW oracle (no GPU): closed forms of the first step and of pure
weight decay, and agreement with an independent implementation of the same
published algorithm (torch.optim.AdamW, float64) over several steps."""

import numpy as np
import torch

from oracle import adamw

F32 = np.float32


def test_first_step_closed_form():
    """With zero moments, the bias-corrected moments of step 1 are g and g^2, so the update
    is lr g / (|g| + eps) (about lr sign(g) when |g| >> eps), evaluated here in float64; the
    float32 chain stays within a few float32 units of p."""
    rng = np.random.default_rng(0)
    p = rng.standard_normal(1000).astype(F32)
    g = (rng.standard_normal(1000) * 1e-2).astype(F32)
    g[:3] = [1e-7, -3e-8, 0.0]  # |g| near eps: the update is far from lr sign(g)
    z = np.zeros_like(p)
    lr, eps = 1e-3, 1e-8
    p1, m1, v1, _ = adamw.adamw_step(p, g, z, z, lr, 0.9, 0.999, eps, 0.0, 1)
    g64 = g.astype(np.float64)
    ref = p.astype(np.float64) - float(F32(lr)) * g64 / (np.abs(g64) + float(F32(eps)))
    assert np.all(np.abs(p1 - ref) <= 4 * np.spacing(np.abs(p).astype(F32)) + 1e-9)
    assert p1[2] == p[2]
    assert np.array_equal(m1, (F32(1.0 - float(F32(0.9))) * g).astype(F32))  # 1 - b1 from the float32 b1


def test_weight_decay_alone():
    """Zero gradient and zero moments: only the decoupled decay acts, p (1 - lr wd) exactly."""
    p = np.linspace(-2, 2, 101).astype(F32)
    z = np.zeros_like(p)
    p1, m1, v1, _ = adamw.adamw_step(p, z, z, z, 0.01, 0.9, 0.999, 1e-8, 0.1, 3)
    assert np.array_equal(p1, (p * F32(1 - 0.01 * 0.1)).astype(F32))
    assert not m1.any() and not v1.any()


def test_matches_torch_adamw_over_steps():
    """torch.optim.AdamW (decoupled weight decay, float64, CPU, unfused) as an independent
    implementation: after 5 steps the float32 oracle agrees to float32 accuracy."""
    rng = np.random.default_rng(1)
    p0 = rng.standard_normal(4096).astype(F32)
    grads = [(rng.standard_normal(4096) * 0.1).astype(F32) for _ in range(5)]
    lr, b1, b2, eps, wd = 2e-3, 0.9, 0.999, 1e-8, 0.05
    tp = torch.nn.Parameter(torch.tensor(p0.astype(np.float64)))
    opt = torch.optim.AdamW([tp], lr=float(F32(lr)), betas=(float(F32(b1)), float(F32(b2))), eps=float(F32(eps)),
                            weight_decay=float(F32(wd)), foreach=False, fused=False)
    p, m, v = p0, np.zeros_like(p0), np.zeros_like(p0)
    for t, g in enumerate(grads, start=1):
        tp.grad = torch.tensor(g.astype(np.float64))
        opt.step()
        p, m, v, _ = adamw.adamw_step(p, g, m, v, lr, b1, b2, eps, wd, t)
    ref = tp.detach().numpy()
    assert np.max(np.abs(p - ref)) < 1e-5 * np.max(np.abs(ref))
    assert np.max(np.abs(m - opt.state[tp]["exp_avg"].numpy())) < 1e-6
