"""AdamW step on the trained LoRA matrices (float32 state).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The pages train only the LoRA matrices with a paged AdamW (P1 tutorial "QLoRA:
fine-tuning 7B on a 24 GB card", section 3.3; tbr8.org "QLoRA on consumer
GPUs", section 5, ``paged_adamw_32bit``; glossary "QLoRA", "How QLoRA works":
the optimizer state sits in unified memory and is paged to CPU RAM during
memory spikes).  Paging moves the state, it does not change the arithmetic,
which is AdamW with decoupled weight decay as published (Loshchilov and
Hutter, "Decoupled Weight Decay Regularization", 2019):

    p  <- p (1 - lr wd)
    m  <- b1 m + (1 - b1) g
    v  <- b2 v + (1 - b2) g^2
    p  <- p - lr / (1 - b1^t) * m / (sqrt(v) / sqrt(1 - b2^t) + eps)

Reading (the order and precision, which the publication leaves open): state
and weights in float32, each operation above rounded once in float32 in the
order written; the scalar factors 1 - lr wd, 1 - b1, 1 - b2, lr / (1 - b1^t)
and sqrt(1 - b2^t) formed in float64 from the float32 hyper-parameters and
rounded to float32; the bf16 copy the linear reads is bf16_rn(p).
"""

from __future__ import annotations

import math

import numpy as np

from . import nf4

F32 = np.float32


def _f(x) -> float:
    """A hyper-parameter as the float32 value the caller passes, widened to float64."""
    return float(F32(x))


def factors(lr, beta1, beta2, eps, weight_decay, step: int) -> dict:
    """The float32 scalar factors of step ``step`` (the first step is 1)."""
    lr, b1, b2, eps, wd = (_f(v) for v in (lr, beta1, beta2, eps, weight_decay))
    return {"decay": F32(1.0 - lr * wd), "b1": F32(b1), "omb1": F32(1.0 - b1), "b2": F32(b2), "omb2": F32(1.0 - b2),
            "step_size": F32(lr / (1.0 - b1 ** step)), "bc2_sqrt": F32(math.sqrt(1.0 - b2 ** step)), "eps": F32(eps)}


def adamw_step(master, grad, exp_avg, exp_avg_sq, lr, beta1, beta2, eps, weight_decay, step: int):
    """One step; returns new ``(master, exp_avg, exp_avg_sq, param_bf16_bits)`` (float32 / uint16)."""
    f = factors(lr, beta1, beta2, eps, weight_decay, step)
    p = np.asarray(master, dtype=F32)
    g = np.asarray(grad, dtype=F32)
    m = np.asarray(exp_avg, dtype=F32)
    v = np.asarray(exp_avg_sq, dtype=F32)
    p = (p * f["decay"]).astype(F32)
    m = ((f["b1"] * m).astype(F32) + (f["omb1"] * g).astype(F32)).astype(F32)
    gg = (g * g).astype(F32)
    v = ((f["b2"] * v).astype(F32) + (f["omb2"] * gg).astype(F32)).astype(F32)
    denom = ((np.sqrt(v).astype(F32) / f["bc2_sqrt"]).astype(F32) + f["eps"]).astype(F32)
    upd = (f["step_size"] * (m / denom).astype(F32)).astype(F32)
    p = (p - upd).astype(F32)
    return p, m, v, nf4.f32_to_bf16_bits(p)
