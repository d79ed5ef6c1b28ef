"""Pins of the merge / low-rank-update oracle (no GPU).

Each check ties ``oracle.lowrank`` to something other than its own formula:
the merge identity of the Day 25 notes (section 2.6: the merged layer computes
what the frozen layer plus its LoRA branch computes), the dequantised weight
itself when B = 0, an independent float64 evaluation that must agree to one
bfloat16 unit in the last place, a rank-1 closed form, and the algebra of the
dense update.
"""

import numpy as np
import pytest

from oracle import linear, lowrank, nf4


def _bf16(x):
    return nf4.bf16_bits_to_f32(nf4.f32_to_bf16_bits(np.asarray(x, dtype=np.float32)))


def _problem(n, k, r, seed):
    rng = np.random.default_rng(seed)
    w = _bf16(rng.standard_normal((n, k)) * 0.02)
    a = _bf16(rng.uniform(-1, 1, (r, k)) / np.sqrt(k))
    b = _bf16(rng.standard_normal((n, r)) * 0.05)
    rec = nf4.quantize(w, n, k)
    wd = nf4.dequantize(rec["codes"], rec["q"], rec["step"], rec["mu"], n, k)
    return w, a, b, rec, wd


def test_merge_with_zero_b_is_the_dequantised_weight():
    n, k, r = 64, 192, 8
    _, a, b, rec, _ = _problem(n, k, r, 0)
    got = lowrank.merge_bf16_bits(rec, a, np.zeros_like(b), 16.0, n, k)
    assert np.array_equal(got, nf4.dequantize_bf16_bits(rec["codes"], rec["q"], rec["step"], rec["mu"], n, k))


def test_merge_identity():
    """X merged^T equals the frozen layer plus its LoRA branch (float64 oracle) up to the
    bfloat16 rounding of the merged weight (relative 2^-9 per entry)."""
    n, k, r, m, alpha = 96, 256, 16, 24, 32.0
    _, a, b, rec, wd = _problem(n, k, r, 1)
    x = _bf16(np.random.default_rng(2).standard_normal((m, k)))
    merged = nf4.bf16_bits_to_f32(lowrank.merge_bf16_bits(rec, a, b, alpha, n, k)).astype(np.float64)
    y_merged = x.astype(np.float64) @ merged.T
    y_fused, _ = linear.lora_forward(x, wd, a, b, alpha, r)
    err = np.linalg.norm(y_merged - y_fused) / np.linalg.norm(y_fused)
    assert err < 2e-3


def test_merge_agrees_with_float64_within_one_bf16_ulp():
    """An independent evaluation: deq(W) + s B A in float64 (BLAS product), rounded once to
    bfloat16.  The float32 chain differs from it only when the exact value lies within the
    chain's rounding error of a bfloat16 rounding boundary: at most one unit in the last place,
    and rarely."""
    n, k, r, alpha = 128, 512, 32, 64.0
    _, a, b, rec, wd = _problem(n, k, r, 3)
    s = float(lowrank.lora_scale_f32(alpha, r))
    exact = wd + s * (b.astype(np.float64) @ a.astype(np.float64))
    ref = nf4.f32_to_bf16_bits(exact.astype(np.float32)).astype(np.int32)
    got = lowrank.merge_bf16_bits(rec, a, b, alpha, n, k).astype(np.int32)
    diff = np.abs(got - ref)
    assert diff.max() <= 1
    assert np.count_nonzero(diff) <= 0.002 * diff.size


def test_merge_rank_one_closed_form():
    """r = 1: (B A)[n, k] is the single exact product b_n a_k, so the merge is
    bf16(w' + RN32(s b_n a_k)); evaluated here in float64 then rounded."""
    n, k, alpha = 32, 128, 2.0
    _, a, b, rec, wd = _problem(n, k, 1, 4)
    s = np.float64(lowrank.lora_scale_f32(alpha, 1))
    delta = (s * b.astype(np.float64) * a.astype(np.float64)).astype(np.float32)   # s b a exact in float64
    ref = nf4.f32_to_bf16_bits((wd + delta.astype(np.float64)).astype(np.float32))
    assert np.array_equal(lowrank.merge_bf16_bits(rec, a, b, alpha, n, k), ref)


def test_lora_product_is_a_sequential_float32_sum():
    """Two terms: (b0 a0 + b1 a1) rounded once; checked against an exactly representable case
    and against a case where the order of the two additions matters in float32."""
    b = np.array([[1.0, 2.0 ** -24]], dtype=np.float32)
    a = np.array([[1.0], [1.0]], dtype=np.float32)
    # 1 + 2^-24 rounds to 1 in float32 (ties to even)
    assert lowrank.lora_product_f32(b, a)[0, 0] == np.float32(1.0)
    b = np.array([[2.0 ** -24, 1.0]], dtype=np.float32)
    assert lowrank.lora_product_f32(b, a)[0, 0] == np.float32(1.0)
    b = np.array([[2.0 ** -24, 2.0 ** -24, 1.0]], dtype=np.float32)
    a = np.ones((3, 1), dtype=np.float32)
    # j order: 2^-24 + 2^-24 = 2^-23 exactly, then 1 + 2^-23 is representable
    assert lowrank.lora_product_f32(b, a)[0, 0] == np.float32(1.0 + 2.0 ** -23)


@pytest.mark.parametrize("with_sub", [False, True])
def test_dense_update_algebra(with_sub):
    n, k, r = 48, 128, 4
    w, a, b, rec, wd = _problem(n, k, r, 5)
    c = -0.75
    got = lowrank.lowrank_update_f32(w, rec if with_sub else None, a, b, c, n, k)
    base = w.astype(np.float64) - (wd if with_sub else 0.0)
    exact = base + c * (b.astype(np.float64) @ a.astype(np.float64))
    assert np.max(np.abs(got - exact)) <= 1e-6 * np.max(np.abs(exact)) + 1e-9
    # without the LoRA pair it is the plain difference, exactly
    plain = lowrank.lowrank_update_f32(w, rec if with_sub else None, None, None, 0.0, n, k)
    assert np.array_equal(plain, base.astype(np.float32))
