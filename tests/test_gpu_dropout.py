"""GPU parity: LoRA dropout (mask generation, forward and backward) against the oracle.

The mask from qlora_dropout_mask must equal the oracle's Philox4x32-10 mask bit
for bit; the dropped input x_drop = x * mask is exact; the layer's outputs and
gradients with that mask are compared with the float64 oracle (GEMM tolerance,
whole tensor and every row) on the small-token GEMMs and on the CTA-pair GEMMs,
including gradient accumulation and p = 0.
"""

import numpy as np
import pytest
import torch

import synthetic
from oracle import dropout, nf4
from tests._helpers import GEMM_TOL, assert_close, rel_fro, t_save_tol, to_np32, to_np64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed,offset,m,k,p", [(0, 0, 16, 256, 0.05), (2 ** 40 + 7, 2 ** 33 + 1, 33, 4160, 0.05),
                                               (5, 9, 8, 64, 0.5), (1, 2, 3, 128, 0.0), (123, 0, 300, 1024, 0.1)])
def test_mask_bit_exact(lib, seed, offset, m, k, p):
    got = lib.dropout_mask(seed, offset, m, k, p)
    lib.check_status()
    want = dropout.pack_mask(dropout.keep_mask(seed, offset, m, k, p))
    assert np.array_equal(got.cpu().numpy(), want)


def _deq(w):
    n, k = w.shape
    rec = nf4.quantize(to_np32(w.cpu()), n, k)
    return nf4.dequantize(rec["codes"], rec["q"], rec["step"], rec["mu"], n, k)


@pytest.mark.parametrize("m,n,k,r,p", [(96, 320, 448, 16, 0.05), (600, 512, 768, 16, 0.05), (2048, 1024, 1024, 8, 0.1),
                                       (130, 264, 320, 5, 0.3)])
def test_dropout_layer_against_oracle(lib, m, n, k, r, p):
    alpha = 2.0 * r
    case = synthetic.linear_case(n, k, m, r, alpha, device="cuda", base_seed=m + n + r)
    rec = lib.quantize(case.w)
    mask = lib.dropout_mask(2024, m, m, k, p)
    y, t, x_drop = lib.linear_fwd_dropout(case.x, rec, case.a, case.b, alpha, mask, p)
    dx, da, db = lib.linear_bwd_dropout(case.dy, x_drop, rec, case.a, case.b, alpha, mask, p, t)
    lib.check_status()
    keep = dropout.unpack_mask(mask.cpu().numpy(), k)
    x, a, b, dy = (to_np64(v) for v in (case.x, case.a, case.b, case.dy))
    assert np.array_equal(to_np64(x_drop), x * keep)
    wd = _deq(case.w)
    yr, tr = dropout.lora_forward(x, wd, a, b, alpha, r, keep, p)
    dxr, dar, dbr = dropout.lora_backward(dy, x, wd, a, b, alpha, r, keep, p, tr)
    assert rel_fro(to_np64(t), tr) < t_save_tol(k)
    for name, got, want in (("y", y, yr), ("dx", dx, dxr), ("da", da, dar), ("db", db, dbr)):
        assert_close(to_np64(got), want, GEMM_TOL, name)


def test_dropout_accumulate_and_p_zero(lib):
    """Gradient accumulation through the dropout path, and p = 0 (every element kept) giving
    the same outputs as the layer without dropout."""
    m, n, k, r, alpha = 520, 384, 512, 16, 32.0
    case = synthetic.linear_case(n, k, m, r, alpha, device="cuda", base_seed=8)
    rec = lib.quantize(case.w)
    mask = lib.dropout_mask(1, 1, m, k, 0.05)
    y, t, xd = lib.linear_fwd_dropout(case.x, rec, case.a, case.b, alpha, mask, 0.05)
    dx, da, db = lib.linear_bwd_dropout(case.dy, xd, rec, case.a, case.b, alpha, mask, 0.05, t)
    dx2, da2, db2 = dx.clone(), da.clone(), db.clone()
    lib.linear_bwd_dropout(case.dy, xd, rec, case.a, case.b, alpha, mask, 0.05, t, dx=dx2, da=da2, db=db2,
                           flags=lib.ACCUM_DX | lib.ACCUM_DA | lib.ACCUM_DB)
    lib.check_status()
    assert_close(to_np64(da2), 2 * to_np64(da), 1e-6, "dA accumulated")
    assert_close(to_np64(db2), 2 * to_np64(db), 1e-6, "dB accumulated")
    assert_close(to_np64(dx2), 2 * to_np64(dx), 1e-2, "dX accumulated")
    # p = 0
    ones = lib.dropout_mask(1, 1, m, k, 0.0)
    assert int(ones.min()) == 255
    y0, t0, xd0 = lib.linear_fwd_dropout(case.x, rec, case.a, case.b, alpha, ones, 0.0)
    y1, t1 = lib.linear_fwd(case.x, rec, case.a, case.b, alpha)
    dx0, da0, db0 = lib.linear_bwd_dropout(case.dy, xd0, rec, case.a, case.b, alpha, ones, 0.0, t0)
    dx1, da1, db1 = lib.linear_bwd(case.dy, case.x, rec, case.a, case.b, alpha, t1)
    lib.check_status()
    assert torch.equal(y0, y1) and torch.equal(t0, t1) and torch.equal(xd0, case.x)
    assert torch.equal(da0, da1) and torch.equal(db0, db1)
    assert_close(to_np64(dx0), to_np64(dx1), 1e-2, "dX p=0")
