"""Pins of the LoftQ oracle (no GPU): the SVD identity it rests on (Eckart-Young:
the rank-r truncation leaves exactly the energy of the other singular values),
and the properties the page claims for the method (P1 tutorial, section 3.10):
base + branch approximate the weight better than the 4-bit base alone with
B = 0, and the error does not grow over the iterations."""

import numpy as np
import pytest

import synthetic
from oracle import loftq, lowrank, nf4


def test_rank_r_factors_leave_the_tail_energy():
    rng = np.random.default_rng(0)
    res = rng.standard_normal((96, 160))
    r, s = 8, 0.5
    a, b = loftq.rank_r_factors(res, r, s, round_bf16=False)
    sv = np.linalg.svd(res, compute_uv=False)
    left = np.sum((res - s * (b @ a)) ** 2)
    assert abs(left - np.sum(sv[r:] ** 2)) < 1e-9 * np.sum(sv ** 2)
    # and the bf16-rounded factors stay close to that optimum
    a16, b16 = loftq.rank_r_factors(res, r, s)
    left16 = np.sum((res - s * (b16.astype(np.float64) @ a16.astype(np.float64))) ** 2)
    assert left16 >= left * (1 - 1e-12) and left16 < left * 1.001


@pytest.fixture(scope="module")
def structured():
    return synthetic.structured_weight(256, 512, rank=8, seed=4).numpy()


def test_loftq_beats_the_plain_4bit_base(structured):
    w = structured
    n, k = w.shape
    rec = nf4.quantize(w, n, k)
    base_err = np.linalg.norm(w - nf4.dequantize(rec["codes"], rec["q"], rec["step"], rec["mu"], n, k)) / \
        np.linalg.norm(w)
    hist = loftq.loftq(w, 16, 32.0, 3)
    assert hist[-1]["rel_err"] < 0.8 * base_err


def test_loftq_error_does_not_grow(structured):
    hist = loftq.loftq(structured, 16, 32.0, 4)
    errs = [h["rel_err"] for h in hist]
    for e0, e1 in zip(errs, errs[1:]):
        assert e1 <= e0 * (1 + 1e-3), errs


def test_first_branch_is_the_truncated_svd_of_w(structured):
    """Before any quantisation the branch is the rank-r truncation of W itself, so the first
    quantised weight is W minus its top-r part."""
    w = structured.astype(np.float64)
    hist = loftq.loftq(structured, 8, 16.0, 1)
    s = float(lowrank.lora_scale_f32(16.0, 8))
    a, b = hist[0]["a_in"], hist[0]["b_in"]
    u, sv, vh = np.linalg.svd(w, full_matrices=False)
    top = (u[:, :8] * sv[:8]) @ vh[:8]
    assert np.linalg.norm(s * (b.astype(np.float64) @ a.astype(np.float64)) - top) < 5e-3 * np.linalg.norm(top)
