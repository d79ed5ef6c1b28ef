"""LoftQ initialisation: a 4-bit base plus a LoRA branch fitted to what
quantisation loses.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

P1 tutorial "QLoRA: fine-tuning 7B on a 24 GB card", section 3.10: SVD of the
weight, the top-r part becomes the LoRA branch with A = sqrt(S_r) V_r and
B = U_r sqrt(S_r), the rest is quantised to 4 bits, and the two steps repeat
so the residual converges.  Reading taken (the page lists the steps without
their exact loop):

    B, A = factors of the rank-r truncation of W
    for each iteration:  Q = NF4(W - s B A);  B, A = factors of the rank-r truncation of W - deq(Q)

with s = alpha / r folded into A (so s B A is the truncation itself) and A, B
rounded to bfloat16, the precision the linear layer reads them in.  The SVD is
numpy's (float64); the dense steps are :mod:`oracle.lowrank` and the
quantisation :mod:`oracle.nf4`.
"""

from __future__ import annotations

import numpy as np

from . import lowrank, nf4


def rank_r_factors(res, r: int, scale: float, round_bf16: bool = True):
    """(A [r, k], B [n, r]) with scale * B A the best rank-r approximation of ``res``
    (float64 SVD); rounded to bfloat16 values unless ``round_bf16`` is False."""
    u, sv, vh = np.linalg.svd(np.asarray(res, dtype=np.float64), full_matrices=False)
    root = np.sqrt(sv[:r])
    b = u[:, :r] * root[None, :]
    a = (root[:, None] * vh[:r, :]) / scale
    if round_bf16:
        b = nf4.bf16_bits_to_f32(nf4.f32_to_bf16_bits(b.astype(np.float32)))
        a = nf4.bf16_bits_to_f32(nf4.f32_to_bf16_bits(a.astype(np.float32)))
    return a, b


def loftq(w, r: int, alpha: float, iters: int):
    """Run the iteration on a float32 [n, k] weight; returns a list with, per
    iteration, the record, the factors fed to the quantiser, the new factors and
    the relative error ||W - deq(Q) - s B A|| / ||W||."""
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    s = float(lowrank.lora_scale_f32(alpha, r))
    a, b = rank_r_factors(w, r, s)
    out = []
    for _ in range(iters):
        target = lowrank.lowrank_update_f32(w, None, a, b, -s, n, k)
        rec = nf4.quantize(target, n, k)
        res = lowrank.lowrank_update_f32(w, rec, None, None, 0.0, n, k)
        a_new, b_new = rank_r_factors(res, r, s)
        err = lowrank.lowrank_update_f32(w, rec, a_new, b_new, -s, n, k)
        out.append({"record": rec, "a_in": a, "b_in": b, "a": a_new, "b": b_new,
                    "rel_err": float(np.linalg.norm(err.astype(np.float64)) / np.linalg.norm(w.astype(np.float64)))})
        a, b = a_new, b_new
    return out
