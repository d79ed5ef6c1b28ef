"""Merge / export and the dense low-rank update (float32 by definition).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources (page title, section):

* Day 25 notes "Fine-tuning and LoRA/QLoRA", section 2.6 ("merging at
  inference"): after training, ``W_merged = W0 + B A`` and the layer is a
  plain linear again; section 6.2: the branch carries the scale ``s = alpha/r``.
* P1 tutorial "QLoRA: fine-tuning 7B on a 24 GB card", section 3.8: a 4-bit
  base is not merged as is; it is dequantised to bfloat16 and then merged.
* Ultralytics glossary "QLoRA", section "Trade-offs": the merged 16-bit model
  is usually quantised again for serving.
* P1 tutorial, section 3.10 (LoftQ): the base is quantised after removing the
  LoRA branch, and the branch is fitted to what quantisation lost -- the two
  dense combinations ``W - s B A`` and ``W - deq(Q)``.

Readings (the pages give the formula, not the arithmetic):

* the merge adds ``s * (B A)`` to the dequantised bfloat16 base and rounds the
  sum to bfloat16 once;
* ``(B A)[n, k]`` is summed in float32 over ``j = 0 .. r-1`` in that order,
  each step rounding once (the bfloat16 products are exact in float32, so a
  fused multiply-add and a multiply-then-add give the same bits); ``s * (B A)``
  is rounded to float32 before the add;
* ``s = float32(alpha) / float32(r)`` in float32;
* the dense update is ``(W - deq(Q)) + c * (B A)``, every operation rounded
  once in float32.
"""

from __future__ import annotations

import numpy as np

from . import nf4

F32 = np.float32


def lora_product_f32(b, a) -> np.ndarray:
    """``(B A)`` as float32 [n, k]: a running float32 sum over j = 0 .. r-1 of the
    exact products ``B[n, j] * A[j, k]`` (B [n, r], A [r, k] hold bfloat16 values)."""
    b = np.asarray(b, dtype=F32)
    a = np.asarray(a, dtype=F32)
    n, r = b.shape
    acc = np.zeros((n, a.shape[1]), dtype=F32)
    for j in range(r):
        term = (b[:, j:j + 1] * a[j:j + 1, :]).astype(F32)   # exact: two 8-bit significands
        acc = (acc + term).astype(F32)                          # one rounding per step
    return acc


def lora_scale_f32(alpha: float, r: int) -> np.float32:
    """``s = alpha / r`` as one float32 division."""
    return F32(F32(alpha) / F32(r))


def merge_bf16_bits(record: dict, a, b, alpha: float, n: int, k: int) -> np.ndarray:
    """bfloat16 bits [n, k] of ``deq(W) + s (B A)`` (Day 25 notes 2.6; P1 3.8).

    ``record`` is a quantised weight as :func:`oracle.nf4.quantize` returns it.
    """
    r = np.asarray(a).shape[0]
    wd = nf4.bf16_bits_to_f32(nf4.dequantize_bf16_bits(record["codes"], record["q"], record["step"], record["mu"],
                                                       n, k))
    s = lora_scale_f32(alpha, r)
    delta = (s * lora_product_f32(b, a)).astype(F32)
    return nf4.f32_to_bf16_bits((wd + delta).astype(F32))


def lowrank_update_f32(w, sub: dict | None, a, b, coef: float, n: int, k: int) -> np.ndarray:
    """``(W - deq(sub)) + coef (B A)`` in float32 [n, k]; ``sub`` (a quantised record) and
    the LoRA pair (``a is None``) are optional."""
    out = np.asarray(w, dtype=F32).reshape(n, k).copy()
    if sub is not None:
        q = nf4.bf16_bits_to_f32(nf4.dequantize_bf16_bits(sub["codes"], sub["q"], sub["step"], sub["mu"], n, k))
        out = (out - q).astype(F32)
    if a is not None and np.asarray(a).shape[0] > 0:
        delta = (F32(coef) * lora_product_f32(b, a)).astype(F32)
        out = (out + delta).astype(F32)
    return out
