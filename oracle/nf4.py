"""NF4 quantisation oracle: levels, blockwise absmax, encode, pack, double quant, dequant.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources (page title, section):

* Ultralytics glossary "QLoRA", section "How QLoRA works": 16 NF4 levels at
  quantiles of the standard normal with an exact zero, normalised so the
  largest is 1; one absmax scale per block of 64 weights; the 4-bit code of a
  weight is the index of the level nearest to ``w / absmax``; the restored
  weight is ``level[code] * absmax``; the block scales are themselves
  quantised to 8 bits in blocks of 256 ("double quantisation"), which takes the
  scale overhead from 0.5 to about 0.127 bit per parameter.  The same section
  states that the forward pass dequantises NF4 to bfloat16 before the matmul.
* fedte.cc "QLoRA fine-tuning on 4 GB", section 1 ("4-bit NormalFloat",
  "double quantisation"): 64 parameters share one fp32 scale; 0.5 byte per
  parameter for the codes.

Readings taken where the pages are silent:

* table built in float64 and rounded once to float32 (the page builds it in
  torch float32; both give the page's worked-example MSE to 4 digits);
* ties in the nearest-level search go to the lower index (first occurrence,
  as ``argmin`` on the page does);
* a block is 64 consecutive elements of the row-major weight;
* two codes per byte, the even-indexed element in the high nibble;
* codes use the raw float32 absmax; double quantisation is a second, separate
  step on the absmax array;
* double quantisation (scheme fixed by the benchmark spec): subtract the
  per-tensor mean ``mu`` of all block absmax values, then symmetric int8 in
  groups of 256 consecutive absmax values with one float32 step per group,
  ``step = max|a - mu| / 127``, ``q = clamp(rint((a - mu) / step), -127, 127)``,
  ``q = 0`` where ``step == 0``;
* ``mu`` = float32( (correctly rounded float64 sum of the absmax values) / n )
  with the division done in float64, i.e. independent of summation order;
* an all-zero block has absmax 0 and takes ``x = 0`` (code of the zero level);
* a non-finite weight is an error (the GPU path reports NONFINITE).
"""

from __future__ import annotations

import math

import numpy as np
from scipy.special import ndtri

BLOCK = 64          # weights per absmax block
DQ_GROUP = 256      # absmax values per double-quantisation group
F32 = np.float32


# --------------------------------------------------------------------------
# bfloat16 helpers (round-to-nearest-even from float32), written out here so
# the oracle depends on no bfloat16 implementation of the product path.
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x) -> np.ndarray:
    """float32 -> bfloat16 bit pattern (uint16), round to nearest, ties to even."""
    x = np.ascontiguousarray(np.asarray(x, dtype=F32))
    u = x.view(np.uint32).astype(np.uint64)
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        rounded = np.where(nan, np.uint16(0x7FC0), rounded)
    return rounded.reshape(x.shape)


def bf16_bits_to_f32(b) -> np.ndarray:
    """bfloat16 bit pattern (uint16) -> float32 (exact)."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(F32)


# --------------------------------------------------------------------------
# NF4 level table
# --------------------------------------------------------------------------
# Largest probability at which the levels take a normal quantile (glossary
# "QLoRA", "How QLoRA works"); the two halves of the table use evenly spaced
# probabilities from here down toward one half.
P_TOP = 0.9677083


def _side_quantiles(count: int) -> list:
    """Standard-normal quantiles at ``count`` probabilities, the first P_TOP,
    then equal steps of (1/2 - P_TOP) / count toward 1/2 (1/2 itself is not
    taken, so no quantile here is zero).  Largest quantile first.  ``ndtri``
    (the inverse normal CDF) is the library step."""
    probs = [P_TOP + i * (0.5 - P_TOP) / count for i in range(count)]
    return [float(ndtri(pr)) for pr in probs]


def nf4_levels_f64() -> np.ndarray:
    """The 16 NF4 levels in float64, ascending.

    Glossary "QLoRA", "How QLoRA works": the levels sit at quantiles of the
    standard normal with one exact zero, 7 below it and 8 above it, and the
    table is scaled so its ends are -1 and +1.  The 8 positive levels take the
    quantiles of :func:`_side_quantiles` with 8 steps; the 7 negative levels
    take the negated quantiles with 7 steps (so the two sides are not mirror
    images); every level is divided by the largest quantile, which both sides
    share (the one at P_TOP).
    """
    q_hi = _side_quantiles(8)          # largest first; q_hi[0] is the quantile at P_TOP
    q_lo = _side_quantiles(7)
    scale = q_hi[0]
    below = [-q / scale for q in q_lo]            # -1 first, rising toward 0
    above = [q / scale for q in q_hi[::-1]]       # smallest first, +1 last
    return np.array(below + [0.0] + above, dtype=np.float64)


def nf4_levels_f32() -> np.ndarray:
    """The NF4 levels rounded once to float32 (the table the codes index)."""
    return nf4_levels_f64().astype(F32)


def int4_levels_f32() -> np.ndarray:
    """16 evenly spaced levels on [-1, 1]: the glossary page's INT4 comparison grid."""
    return np.linspace(-1.0, 1.0, 16).astype(F32)


# --------------------------------------------------------------------------
# Quantisation of the weights
# --------------------------------------------------------------------------
def _check_finite(w: np.ndarray) -> None:
    if not np.all(np.isfinite(w)):
        raise ValueError("non-finite weight: NF4 quantisation is undefined")


def blockwise_absmax(w: np.ndarray) -> np.ndarray:
    """float32 absmax of every 64 consecutive elements of the flattened weight.

    Glossary "QLoRA", "How QLoRA works": one absolute-maximum scale per block
    of 64 weights.
    """
    w = np.asarray(w, dtype=F32).reshape(-1)
    if w.size % BLOCK:
        raise ValueError("weight size must be a multiple of 64")
    _check_finite(w)
    return np.abs(w.reshape(-1, BLOCK)).max(axis=1).astype(F32)


def encode_nearest(x: np.ndarray, levels: np.ndarray) -> np.ndarray:
    """Index of the nearest level for each float32 ``x`` (brute force).

    Distances ``|x - L_j|`` are float32 (one rounding of the difference); the
    scan is ascending with a strict ``<`` so ties keep the lower index.
    """
    x = np.asarray(x, dtype=F32).reshape(-1)
    levels = np.asarray(levels, dtype=F32)
    best = np.zeros(x.shape, dtype=np.uint8)
    best_d = np.abs(x - levels[0])
    for j in range(1, levels.size):
        d = np.abs(x - levels[j])
        better = d < best_d
        best = np.where(better, np.uint8(j), best)
        best_d = np.where(better, d, best_d)
    return best


def nf4_encode(w: np.ndarray, absmax: np.ndarray, levels: np.ndarray | None = None) -> np.ndarray:
    """4-bit codes (uint8 in 0..15, one per element) of a flattened weight.

    Glossary "QLoRA", "How QLoRA works": code = argmin_j |w / absmax - L_j|.
    ``w / absmax`` is one float32 IEEE division; a block whose absmax is 0 takes
    ``x = 0``.
    """
    if levels is None:
        levels = nf4_levels_f32()
    w = np.asarray(w, dtype=F32).reshape(-1, BLOCK)
    a = np.asarray(absmax, dtype=F32).reshape(-1, 1)
    out = np.empty(w.shape, dtype=np.uint8)
    rows = max(1, (1 << 20) // BLOCK)
    for s in range(0, w.shape[0], rows):
        wb, ab = w[s:s + rows], a[s:s + rows]
        safe = np.where(ab == 0, F32(1), ab)
        x = np.where(ab == 0, F32(0), (wb / safe).astype(F32))
        out[s:s + rows] = encode_nearest(x, levels).reshape(wb.shape)
    return out.reshape(-1)


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """Two codes per byte: element 2i in the high nibble, element 2i+1 in the low."""
    c = np.asarray(codes, dtype=np.uint8).reshape(-1, 2)
    return ((c[:, 0] << 4) | c[:, 1]).astype(np.uint8)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """Inverse of :func:`pack_codes`."""
    p = np.asarray(packed, dtype=np.uint8).reshape(-1)
    out = np.empty(p.size * 2, dtype=np.uint8)
    out[0::2] = p >> 4
    out[1::2] = p & 0x0F
    return out


def restore_with_levels(codes: np.ndarray, absmax: np.ndarray, levels: np.ndarray) -> np.ndarray:
    """Reconstruction ``levels[code] * absmax`` in float32 with the raw block scale
    (glossary "QLoRA", "How QLoRA works": the restored weight is the level times
    the block's scale).  ``codes`` holds one code per element (not packed)."""
    c = np.asarray(codes, dtype=np.uint8).reshape(-1, BLOCK)
    a = np.asarray(absmax, dtype=F32).reshape(-1, 1)
    return (np.asarray(levels, dtype=F32)[c] * a).astype(F32).reshape(-1)


# --------------------------------------------------------------------------
# Double quantisation of the block absmax values
# --------------------------------------------------------------------------
def absmax_mean(absmax: np.ndarray) -> np.float32:
    """Per-tensor mean of the absmax values.

    float32( fsum(a) / n ): ``math.fsum`` returns the correctly rounded float64
    sum (the library step); the division is one float64 IEEE division; the
    result is rounded once to float32.
    """
    a = np.asarray(absmax, dtype=F32).reshape(-1)
    if a.size == 0:
        raise ValueError("empty absmax array")
    s = math.fsum(a.astype(np.float64).tolist())
    return F32(s / float(a.size))


def double_quant(absmax: np.ndarray):
    """Quantise the absmax array to int8 in groups of 256 after mean subtraction.

    Glossary "QLoRA", "How QLoRA works" (8-bit scales in blocks of 256) with the
    scheme the benchmark spec fixes.  Returns ``(q int8 [n_a], step float32
    [ceil(n_a/256)], mu float32)``.
    """
    a = np.asarray(absmax, dtype=F32).reshape(-1)
    mu = absmax_mean(a)
    d = (a - mu).astype(F32)
    n_a = a.size
    groups = (n_a + DQ_GROUP - 1) // DQ_GROUP
    step = np.zeros(groups, dtype=F32)
    q = np.zeros(n_a, dtype=np.int8)
    for g in range(groups):
        dg = d[g * DQ_GROUP:(g + 1) * DQ_GROUP]
        m = np.abs(dg).max()
        st = F32(m / F32(127))
        step[g] = st
        if st == 0:
            continue
        r = np.rint((dg / st).astype(F32))
        q[g * DQ_GROUP:(g + 1) * DQ_GROUP] = np.clip(r, -127, 127).astype(np.int8)
    return q, step, mu


def dequant_absmax(q: np.ndarray, step: np.ndarray, mu) -> np.ndarray:
    """Restored absmax ``a' = (float(q) * step) + mu``, two float32 roundings."""
    q = np.asarray(q, dtype=np.int8).reshape(-1)
    g = np.arange(q.size) // DQ_GROUP
    prod = (q.astype(F32) * np.asarray(step, dtype=F32)[g]).astype(F32)
    return (prod + F32(mu)).astype(F32)


# --------------------------------------------------------------------------
# Whole-weight helpers
# --------------------------------------------------------------------------
def quantize(w: np.ndarray, n: int, k: int) -> dict:
    """NF4 + double-quant record of a row-major [n, k] weight (float32 or bf16 values).

    Returns ``codes`` (packed uint8 [n*k/2]), ``absmax`` (float32 [n*k/64], the
    raw scales the codes were made with), ``q`` (int8 [n*k/64]), ``step``
    (float32 [ceil(n*k/64/256)]) and ``mu`` (float32).
    """
    if k % BLOCK:
        raise ValueError("k must be a multiple of 64")
    w = np.asarray(w, dtype=F32).reshape(n * k)
    a = blockwise_absmax(w)
    codes = nf4_encode(w, a)
    q, step, mu = double_quant(a)
    return {"codes": pack_codes(codes), "absmax": a, "q": q, "step": step, "mu": mu}


def dequantize_bf16_bits(codes_packed, q, step, mu, n: int, k: int) -> np.ndarray:
    """bfloat16 bits [n, k] of the dequantised weight.

    ``w' = bf16_rn(float32(L[code] * a'))`` with ``a'`` from
    :func:`dequant_absmax`: glossary "QLoRA", "How QLoRA works" (restored weight
    = level * scale; dequantised to bfloat16 before the matmul).
    """
    levels = nf4_levels_f32()
    c = unpack_codes(codes_packed)[: n * k].reshape(-1, BLOCK)
    a2 = dequant_absmax(q, step, mu).reshape(-1, 1)
    prod = (levels[c] * a2).astype(F32)
    return f32_to_bf16_bits(prod).reshape(n, k)


def dequantize(codes_packed, q, step, mu, n: int, k: int) -> np.ndarray:
    """Dequantised weight as float64 [n, k] (the exact bfloat16 values)."""
    return bf16_bits_to_f32(dequantize_bf16_bits(codes_packed, q, step, mu, n, k)).astype(np.float64)


def overhead_bits_per_param(n_params: int) -> float:
    """Storage of the double-quantised scales in bits per parameter.

    int8 per 64 parameters, one float32 step per 256 absmax values and one
    float32 mean, measured from the record sizes this module produces.
    """
    n_a = n_params // BLOCK
    groups = (n_a + DQ_GROUP - 1) // DQ_GROUP
    return (8 * n_a + 32 * groups + 32) / n_params
