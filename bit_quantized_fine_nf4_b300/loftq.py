"""LoftQ initialisation of a QLoRA layer: a 4-bit base plus a LoRA branch that
together approximate the full-precision weight.

P1 tutorial "QLoRA: fine-tuning 7B on a 24 GB card", section 3.10: with B = 0
a QLoRA layer starts as the 4-bit base alone, which has already lost
precision; LoftQ instead takes an SVD, keeps the top-r part as the LoRA
branch (A = sqrt(S_r) V_r, B = U_r sqrt(S_r)), quantises what remains to 4
bits, and iterates so the residual converges.  The steps, as taken here:

    B, A  = rank-r factors of W                      (the SVD of W itself)
    repeat `iters` times:
        Q     = NF4(W - s B A)                       qlora_lowrank_update + qlora_nf4_quantize
        R     = W - deq(Q)                           qlora_lowrank_update
        B, A  = rank-r factors of R                  (SVD)

with s = alpha / r and the factors split as the page prints them, 1/s folded
into A so that s B A is the rank-r truncation; A and B are rounded to bf16
(the precision the linear reads them in) before they are used.  The
arithmetic steps run in the library's kernels; the rank-r SVD of the float32
residual is a library primitive (torch.linalg.svd, cuSOLVER on the GPU).
"""

from __future__ import annotations

import torch

from . import _binding as q


def _rank_r_factors(res: torch.Tensor, r: int, scale: float):
    """(A [r, k] bf16, B [n, r] bf16) with scale * B A the best rank-r approximation of `res`."""
    u, sv, vh = torch.linalg.svd(res, full_matrices=False)
    root = sv[:r].sqrt()
    b = (u[:, :r] * root[None, :]).to(torch.bfloat16).contiguous()
    a = ((root[:, None] * vh[:r, :]) / scale).to(torch.bfloat16).contiguous()
    return a, b


def loftq_init(w: torch.Tensor, r: int, alpha: float, iters: int = 1, history: list | None = None,
               trace: list | None = None):
    """LoftQ initialisation of one [n, k] weight (float32 or bfloat16, on the GPU).

    Returns ``(record, A, B)``: the NF4 record of the base and the bf16 LoRA pair,
    with deq(record) + (alpha/r) B A close to W.  If ``history`` is a list, the
    relative error ||W - deq(Q) - s B A|| / ||W|| after each iteration is appended;
    if ``trace`` is a list, each iteration appends the factors it quantised against
    (``a_in``, ``b_in``), its record and the new factors (``a``, ``b``).
    """
    if iters < 1:
        raise ValueError("iters must be >= 1")
    n, k = w.shape
    s = float(alpha) / float(r)
    wf = w.float()
    a, b = _rank_r_factors(wf, r, s)
    rec = q.NF4Weight.empty(n, k, w.device)
    target = torch.empty((n, k), dtype=torch.float32, device=w.device)
    res = torch.empty_like(target)
    ws = torch.empty(q.quantize_workspace_bytes(n, k), dtype=torch.uint8, device=w.device)
    wnorm = float(wf.norm())
    for _ in range(iters):
        if trace is not None:
            rec = q.NF4Weight.empty(n, k, w.device)            # keep each iteration's record
        a_in, b_in = a, b
        q.lowrank_update(w, None, a, b, -s, out=target)       # W - s B A
        q.quantize(target, out=rec, workspace=ws)              # Q = NF4(W - s B A)
        q.lowrank_update(w, rec, None, None, 0.0, out=res)    # R = W - deq(Q)
        a, b = _rank_r_factors(res, r, s)
        if trace is not None:
            trace.append({"a_in": a_in, "b_in": b_in, "record": rec, "a": a, "b": b})
        if history is not None:
            err = q.lowrank_update(w, rec, a, b, -s)           # W - deq(Q) - s B A
            history.append(float(err.norm()) / wnorm)
    return rec, a, b
