"""Pins of the NF4 / double-quantisation oracle against what the pages and mathematics fix.

No GPU.  Each test checks the oracle against something other than itself: the
glossary page's printed worked example, closed forms, exact rational
arithmetic, an independent search method, or an independent library.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import nf4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------- levels
def test_levels_invariants():
    lv = nf4.nf4_levels_f32()
    assert lv.shape == (16,)
    assert lv[0] == -1.0 and lv[15] == 1.0
    assert np.all(np.diff(lv) > 0), "levels must be strictly increasing"
    assert np.count_nonzero(lv == 0) == 1 and lv[7] == 0.0
    assert np.count_nonzero(lv < 0) == 7 and np.count_nonzero(lv > 0) == 8


def test_levels_are_normal_quantiles():
    """Un-normalised levels satisfy Phi(q) = p, checked with math.erfc (not ndtri)."""
    lv = nf4.nf4_levels_f64()
    # positive side: divided by its own max, the largest positive quantile
    p_pos = [0.9677083 + i * (0.5 - 0.9677083) / 8 for i in range(8)]
    q_top = math.sqrt(2.0) * _erfcinv_bisect(2.0 * (1.0 - p_pos[0]))
    for j, p in enumerate(p_pos):
        q = lv[15 - j] * q_top
        assert abs(0.5 * math.erfc(-q / math.sqrt(2.0)) - p) < 1e-12
    p_neg = [0.9677083 + i * (0.5 - 0.9677083) / 7 for i in range(7)]
    for j, p in enumerate(p_neg):
        q = -lv[j] * q_top
        assert abs(0.5 * math.erfc(-q / math.sqrt(2.0)) - p) < 1e-12


def _erfcinv_bisect(y):
    lo, hi = 0.0, 10.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if math.erfc(mid) > y:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def test_levels_regression_fixture():
    with open(os.path.join(GOLDEN, "nf4_levels_f32.txt")) as f:
        hexes = [ln for ln in f if not ln.startswith("#")][0].split()
    assert [int(h, 16) for h in hexes] == [int(v) for v in nf4.nf4_levels_f32().view(np.uint32)]


# ----------------------------------------------------------------- worked example
def test_glossary_worked_example_mse():
    """The glossary page prints NF4 MSE 3.395e-06 and INT4 MSE 4.053e-06 for 4096 blocks
    of 64 N(0, 0.02^2) weights (torch seed 0): the oracle's own encode and
    reconstruction, with either table, must print the same figures."""
    g = _golden("glossary_worked_example.json")
    torch.manual_seed(g["input"]["torch_seed"])
    w = (torch.randn(*g["input"]["shape"]) * g["input"]["std"]).numpy().reshape(-1)
    a = nf4.blockwise_absmax(w)

    def reconstruction_mse(table):
        back = nf4.restore_with_levels(nf4.nf4_encode(w, a, table), a, table)
        return float(np.mean(np.square(back.astype(np.float64) - w.astype(np.float64))))

    nf4_mse = reconstruction_mse(nf4.nf4_levels_f32())
    int4_mse = reconstruction_mse(nf4.int4_levels_f32())
    assert "%.3e" % nf4_mse == g["printed"]["NF4"]
    assert "%.3e" % int4_mse == g["printed"]["INT4"]
    reduction = 100.0 * (1.0 - nf4_mse / int4_mse)
    assert abs(reduction - g["stated_reduction_about_percent"]) < 1.0


# ----------------------------------------------------------------- encode
def test_encode_matches_threshold_search():
    """Nearest level by sorted float64 midpoints + searchsorted (a different method)."""
    lv = nf4.nf4_levels_f32()
    mids = (lv[:-1].astype(np.float64) + lv[1:].astype(np.float64)) / 2.0
    rng = np.random.default_rng(1)
    x = rng.uniform(-1.0, 1.0, 200_000).astype(np.float32)
    far = np.min(np.abs(x.astype(np.float64)[:, None] - mids[None, :]), axis=1) > 1e-6
    ref = np.searchsorted(mids, x.astype(np.float64), side="left")
    got = nf4.encode_nearest(x, lv)
    assert np.array_equal(got[far], ref[far].astype(np.uint8))


def test_encode_exact_levels_and_ties():
    lv = nf4.nf4_levels_f32()
    assert np.array_equal(nf4.encode_nearest(lv, lv), np.arange(16, dtype=np.uint8))
    # halfway between L6 and 0 and between 0 and L8: exactly representable, exact ties
    x = np.array([lv[6] / 2, lv[8] / 2], dtype=np.float32)
    assert np.abs(x[0] - lv[6]) == np.abs(x[0] - lv[7])
    assert np.abs(x[1] - lv[7]) == np.abs(x[1] - lv[8])
    assert list(nf4.encode_nearest(x, lv)) == [6, 7], "ties go to the lower index"


def test_encode_blocks_absmax_element_and_zero_block():
    rng = np.random.default_rng(2)
    w = (rng.standard_normal((32, 64)) * 0.02).astype(np.float32)
    w[3] = 0.0
    a = nf4.blockwise_absmax(w)
    codes = nf4.nf4_encode(w, a).reshape(32, 64)
    for i in range(32):
        if i == 3:
            assert np.all(codes[i] == 7)
            continue
        j = int(np.argmax(np.abs(w[i])))
        assert codes[i, j] == (15 if w[i, j] > 0 else 0)


def test_encode_rejects_nonfinite():
    w = np.zeros(64, dtype=np.float32)
    w[5] = np.nan
    with pytest.raises(ValueError):
        nf4.blockwise_absmax(w)


def test_pack_roundtrip_and_nibble_order():
    codes = np.array([0x1, 0xF, 0x7, 0x8], dtype=np.uint8)
    p = nf4.pack_codes(codes)
    assert list(p) == [0x1F, 0x78]
    rng = np.random.default_rng(3)
    c = rng.integers(0, 16, 4096).astype(np.uint8)
    assert np.array_equal(nf4.unpack_codes(nf4.pack_codes(c)), c)


# ----------------------------------------------------------------- double quantisation
def test_mean_is_correctly_rounded_exact_sum():
    rng = np.random.default_rng(4)
    for n in (1, 7, 256, 1000, 4097):
        a = np.abs(rng.standard_normal(n) * rng.choice([1e-30, 1e-3, 1.0, 1e20], n)).astype(np.float32)
        exact = sum((Fraction(float(v)) for v in a), Fraction(0))
        ref = np.float32(float(exact) / float(n))
        assert nf4.absmax_mean(a) == ref


def test_double_quant_constant_and_bounds():
    a = np.full(600, 0.0375, dtype=np.float32)
    q, step, mu = nf4.double_quant(a)
    assert mu == np.float32(0.0375) and np.all(step == 0) and np.all(q == 0)
    assert np.array_equal(nf4.dequant_absmax(q, step, mu), a)

    rng = np.random.default_rng(5)
    w = (rng.standard_normal((128, 64 * 40)) * 0.02).astype(np.float32)
    a = nf4.blockwise_absmax(w)
    q, step, mu = nf4.double_quant(a)
    assert q.dtype == np.int8 and q.min() >= -127 and q.max() <= 127
    assert step.size == (a.size + 255) // 256
    a2 = nf4.dequant_absmax(q, step, mu)
    g = np.arange(a.size) // 256
    err = np.abs(a2.astype(np.float64) - a.astype(np.float64))
    assert np.all(err <= step[g].astype(np.float64) * 0.5 * (1 + 1e-5) + 4 * np.spacing(np.float32(a.max())))
    for gi in range(step.size):
        if step[gi] > 0:
            assert np.abs(q[gi * 256:(gi + 1) * 256].astype(int)).max() == 127


def test_double_quant_overhead_closed_form():
    g = _golden("pages_sizes.json")["double_quant_overhead"]
    n = 4096 * 4096
    bits = nf4.overhead_bits_per_param(n)
    closed = 8 / 64 + 32 / (64 * 256)
    # the closed form plus the one float32 mean per tensor
    assert abs(bits - (closed + 32 / n)) < 1e-12
    assert round(bits, 3) == g["after_bits_per_param_about"]
    assert 32 / 64 == g["before_bits_per_param"]


def test_resident_sizes_match_pages():
    """Record sizes for the Llama-65B and 7B linear stacks against the pages' sizes."""
    from synthetic import LLAMA65B_LAYER, LLAMA7B_LAYER
    sizes = _golden("pages_sizes.json")

    def record_bytes(shapes, layers):
        tot = 0
        for n, k in shapes:
            p = n * k
            n_a = p // 64
            tot += p // 2 + n_a + 4 * ((n_a + 255) // 256) + 4
        return tot * layers

    gb65 = record_bytes(LLAMA65B_LAYER, 80) / 1e9
    assert abs(gb65 - sizes["resident_65b"]["gb_about"]) / sizes["resident_65b"]["gb_about"] < 0.05
    codes7 = sum(n * k for n, k in LLAMA7B_LAYER) * 32 * sizes["codes_7b"]["bytes_per_param"] / 1e9
    assert abs(codes7 - sizes["codes_7b"]["gb_about"]) / sizes["codes_7b"]["gb_about"] < 0.10


# ----------------------------------------------------------------- dequantisation
def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(6)
    x = np.concatenate([
        rng.standard_normal(100_000).astype(np.float32) * 0.05,
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, 1e-40, -1e-40, np.inf, -np.inf], dtype=np.float32),
        # exact halfway patterns (low 16 bits 0x8000) with even and odd kept bits
        np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x3F80FFFF], dtype=np.uint32).view(np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(nf4.f32_to_bf16_bits(x), ref)


def test_dequant_error_bound():
    rng = np.random.default_rng(7)
    n, k = 64, 512
    w = (rng.standard_normal((n, k)) * 0.02).astype(np.float32)
    rec = nf4.quantize(w, n, k)
    wd = nf4.dequantize(rec["codes"], rec["q"], rec["step"], rec["mu"], n, k)
    a = np.repeat(rec["absmax"], 64).reshape(n, k).astype(np.float64)
    a2 = np.repeat(nf4.dequant_absmax(rec["q"], rec["step"], rec["mu"]), 64).reshape(n, k).astype(np.float64)
    lv = nf4.nf4_levels_f64()
    half_gap = float(np.max(np.diff(lv)) / 2)
    bound = a2 * half_gap * (1 + 1e-6) + np.abs(a - a2) + np.abs(wd) * 2.0 ** -8 + 1e-30
    assert np.all(np.abs(w - wd) <= bound)
    assert abs(half_gap - 0.15190) < 1e-4


def test_dequant_reproduces_levels_times_restored_scale():
    """A block whose codes are 0..15 (x4) restores bf16(L[c] * a') exactly."""
    lv = nf4.nf4_levels_f32()
    w = np.tile(np.concatenate([lv, lv, lv, lv]), 3).astype(np.float32) * np.float32(0.5)
    rec = nf4.quantize(w, 3, 64)
    codes = nf4.unpack_codes(rec["codes"])
    assert np.array_equal(codes, np.tile(np.arange(16, dtype=np.uint8), 12))
    a2 = nf4.dequant_absmax(rec["q"], rec["step"], rec["mu"])
    assert np.all(a2 == np.float32(0.5))
    wd = nf4.dequantize(rec["codes"], rec["q"], rec["step"], rec["mu"], 3, 64)
    expect = torch.from_numpy(w).to(torch.bfloat16).to(torch.float64).numpy().reshape(3, 64)
    assert np.array_equal(wd, expect)
