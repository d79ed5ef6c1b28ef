"""GPU parity: QLoRA linear forward / backward / decode against the float64 oracle.

The CUDA path (through the C ABI) and the oracle see the same seeded bf16
inputs; the oracle quantises W itself.  The bar is GEMM_TOL, the relative
Frobenius error for bf16-in / fp32-accumulate outputs and gradients, applied
to the whole tensor and to every row on its own.  Cases span several tiles
with ragged tails, forwards of 1..16 tokens (the decode kernel), ranks 8 / 16 / 64 /
128, the isolated LoRA path (W = 0) and B = 0, and the full-size workloads:
the 4096^2 attention projection and the 4096 x 11008 MLP down projection at
2048 tokens (every row), the 11008 x 4096 gate shape and the 65B up projection
(sampled rows).
"""

import numpy as np
import pytest
import torch

import synthetic
from oracle import linear, nf4
from tests._helpers import GEMM_TOL, t_save_tol, assert_close, rel_fro, to_np32, to_np64

pytestmark = pytest.mark.gpu


def _deq_oracle(w_cpu):
    n, k = w_cpu.shape
    rec = nf4.quantize(to_np32(w_cpu), n, k)
    return nf4.dequantize(rec["codes"], rec["q"], rec["step"], rec["mu"], n, k)


def _run(lib, case, flags=0):
    w = case.w.cuda()
    rec = lib.quantize(w)
    x, a, b, dy = (t.cuda() for t in (case.x, case.a, case.b, case.dy))
    y, t = lib.linear_fwd(x, rec, a, b, case.alpha)
    dx, da, db = lib.linear_bwd(dy, x, rec, a, b, case.alpha, t, flags=flags)
    lib.check_status()
    return rec, y, t, dx, da, db


def _check_all(lib, case, rows=None, flags=0):
    rec, y, t, dx, da, db = _run(lib, case, flags)
    wd = _deq_oracle(case.w)
    x, a, b, dy = (to_np64(v) for v in (case.x, case.a, case.b, case.dy))
    r = case.r
    t_ref = x @ a.T
    assert rel_fro(to_np64(t), t_ref) < t_save_tol(case.k)
    dar, dbr = linear.lora_grads(dy, x, a, b, case.alpha, r, t_ref)
    assert_close(to_np64(da), dar, GEMM_TOL, "dA")
    assert_close(to_np64(db), dbr, GEMM_TOL, "dB")
    if rows is None:
        dxr, _, _, _ = linear.lora_backward(dy, x, wd, a, b, case.alpha, r, t_ref)
        yr, _ = linear.lora_forward(x, wd, a, b, case.alpha, r)
        assert_close(to_np64(y), yr, GEMM_TOL, "Y")
        assert_close(to_np64(dx), dxr, GEMM_TOL, "dX")
    else:
        yr, _ = linear.lora_forward_rows(x[rows], wd, a, b, case.alpha, r)
        assert_close(to_np64(y)[rows], yr, GEMM_TOL, "Y rows")
        dxr_rows = linear.lora_backward_dx_rows(dy[rows], wd, a, b, case.alpha, r)
        assert_close(to_np64(dx)[rows], dxr_rows, GEMM_TOL, "dX rows")
    return y, dx, da, db


def test_tiny_case(lib):
    _check_all(lib, synthetic.tiny_case())


@pytest.mark.parametrize("m,n,k,r", [(300, 640, 512, 16), (129, 264, 320, 8), (260, 384, 1024, 64),
                                     (130, 256, 256, 128), (17, 512, 512, 16), (64, 136, 448, 24)])
def test_ragged_tiles(lib, m, n, k, r):
    case = synthetic.linear_case(n, k, m, r, 2.0 * r, base_seed=m + n + k + r)
    _check_all(lib, case)


# 17..256 tokens run the small-token GEMMs with k split over up to four CTAs per 128-row tile and
# the partials added by the tile's last CTA: 65..128 tokens (the 128-token variant), a ragged
# row tail (1000 = 7 x 128 + 104), and the 4096^2 weight at 128 tokens.
@pytest.mark.parametrize("m,n,k,r", [(100, 1000, 2048, 16), (128, 4096, 4096, 16), (65, 384, 768, 8)])
def test_small_token_split_k(lib, m, n, k, r):
    _check_all(lib, synthetic.linear_case(n, k, m, r, 2.0 * r, base_seed=m * 7 + n + k))


@pytest.mark.parametrize("m", [1, 4, 16])
def test_decode_tokens(lib, m):
    case = synthetic.linear_case(4096, 4096, m, 16, 32.0, base_seed=100 + m)
    _check_all(lib, case)


def test_decode_down_proj_shape(lib):
    case = synthetic.linear_case(4096, 11008, 4, 16, 32.0, base_seed=7)
    _check_all(lib, case)


def _device_case(n, k, m, r, alpha, seed):
    """A large case drawn on the device (the bench's generators), then moved to the host."""
    case = synthetic.linear_case(n, k, m, r, alpha, device="cuda", base_seed=seed)
    return synthetic.LinearCase(*(t.cpu() for t in (case.w, case.x, case.a, case.b, case.dy)), case.alpha, case.r)


def test_attention_projection_every_row(lib):
    """The 4096^2, 2048-token, r=16 workload the bench times: every row of Y and dX, full dA / dB."""
    _check_all(lib, _device_case(4096, 4096, 2048, 16, 32.0, 0))


def test_mlp_down_projection_every_row(lib):
    """The Llama-7B MLP down projection, W 4096 x 11008, 2048 tokens, r=16: the CTA-pair backward
    with an 11008-wide dX (43 column tiles of 256, 172 CTA pairs), every row checked."""
    _check_all(lib, _device_case(4096, 11008, 2048, 16, 32.0, 41))


def test_lora_path_alone_with_zero_weight(lib):
    """W = 0 dequantises to 0, so Y and dX are the LoRA terms alone (large B)."""
    case = synthetic.linear_case(384, 512, 200, 16, 32.0, base_seed=11)
    case.w.zero_()
    case.b.copy_((torch.randn(case.b.shape, generator=torch.Generator().manual_seed(5))).to(torch.bfloat16))
    y, dx, _, _ = _check_all(lib, case)
    assert float(y.float().abs().max()) > 0 and float(dx.float().abs().max()) > 0


def test_b_zero_is_plain_dequantised_linear(lib):
    """B = 0: Y is the oracle's X deq(W)^T exactly as a plain linear, dA = 0, dB = s dY^T T."""
    case = synthetic.linear_case(256, 512, 96, 16, 32.0, base_seed=12)
    case.b.zero_()
    rec, y, t, dx, da, db = _run(lib, case)
    wd = _deq_oracle(case.w)
    x, dy = to_np64(case.x), to_np64(case.dy)
    assert_close(to_np64(y), x @ wd.T, GEMM_TOL, "Y")
    assert_close(to_np64(dx), dy @ wd, GEMM_TOL, "dX")
    assert float(da.abs().max()) == 0.0
    _, dbr = linear.lora_grads(dy, x, to_np64(case.a), to_np64(case.b), case.alpha, case.r)
    assert_close(to_np64(db), dbr, GEMM_TOL, "dB")


def _accumulate_against_oracle(lib, case):
    """Gradient accumulation: a second backward with all three ACCUM flags adds the same
    gradients again, so the buffers hold twice the oracle's dX, dA and dB."""
    rec, y, t, dx, da, db = _run(lib, case)
    x, a, b, dy = (v.cuda() for v in (case.x, case.a, case.b, case.dy))
    lib.linear_bwd(dy, x, rec, a, b, case.alpha, t, dx=dx, da=da, db=db,
                   flags=lib.ACCUM_DX | lib.ACCUM_DA | lib.ACCUM_DB)
    lib.check_status()
    wd = _deq_oracle(case.w)
    xn, an, bn, dyn = (to_np64(v) for v in (case.x, case.a, case.b, case.dy))
    dxr, dar, dbr, _ = linear.lora_backward(dyn, xn, wd, an, bn, case.alpha, case.r)
    assert_close(to_np64(dx), 2 * dxr, GEMM_TOL, "dX accumulated")
    assert_close(to_np64(da), 2 * dar, GEMM_TOL, "dA accumulated")
    assert_close(to_np64(db), 2 * dbr, GEMM_TOL, "dB accumulated")


def test_accumulate_flags(lib):
    _accumulate_against_oracle(lib, synthetic.linear_case(256, 256, 64, 16, 32.0, base_seed=13))


def test_zero_tokens(lib):
    case = synthetic.linear_case(256, 256, 8, 16, 32.0, base_seed=14)
    rec = lib.quantize(case.w.cuda())
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    a, b = case.a.cuda(), case.b.cuda()
    y, t = lib.linear_fwd(x, rec, a, b, 32.0)
    da = torch.full((16, 256), 3.0, device="cuda")
    db = torch.full((256, 16), 3.0, device="cuda")
    lib.linear_bwd(torch.empty((0, 256), dtype=torch.bfloat16, device="cuda"), x, rec, a, b, 32.0, t,
                   dx=torch.empty((0, 256), dtype=torch.bfloat16, device="cuda"), da=da, db=db)
    lib.check_status()
    assert y.shape == (0, 256) and float(da.abs().max()) == 0.0 and float(db.abs().max()) == 0.0


@pytest.mark.parametrize("r", [0, 129])
def test_rank_outside_the_boundary_rejected(lib, r):
    case = synthetic.linear_case(256, 256, 8, 16, 32.0, base_seed=15)
    rec = lib.quantize(case.w.cuda())
    a = torch.zeros((max(r, 1), 256), dtype=torch.bfloat16, device="cuda")[:r]
    b = torch.zeros((256, max(r, 1)), dtype=torch.bfloat16, device="cuda")[:, :r].contiguous()
    with pytest.raises(lib.QloraError) as e:
        lib.linear_fwd(case.x.cuda(), rec, a, b, 24.0)
    assert e.value.code == lib.QLORA_ERR_UNSUPPORTED


# Every rank the boundary accepts, 1 <= r <= 128: ranks that are not multiples of 8 (odd ones
# too) on the small-token GEMMs (<= 256 tokens) and on the CTA-pair GEMMs (> 256 tokens).
@pytest.mark.parametrize("m", [96, 600])
@pytest.mark.parametrize("r", [1, 4, 12, 100, 127])
def test_any_rank(lib, m, r):
    case = synthetic.linear_case(320, 448, m, r, 2.0 * r, base_seed=5 * m + r)
    _check_all(lib, case)


def test_odd_rank_accumulate(lib):
    """Rank 5 (rows of t_save and dB not 16-byte aligned) with gradient accumulation."""
    _accumulate_against_oracle(lib, synthetic.linear_case(264, 320, 520, 5, 10.0, base_seed=23))


def _sampled_big(lib, n, k, m, r, alpha, seed, nrows=24):
    case = _device_case(n, k, m, r, alpha, seed)
    rows = np.concatenate([np.random.default_rng(seed).choice(m, nrows, replace=False), [0, m - 1]])
    _check_all(lib, case, rows=rows)


def test_mlp_gate_shape_sampled_rows(lib):
    """11008 x 4096 (Llama-7B gate / up projection), 2048 tokens, r=16."""
    _sampled_big(lib, 11008, 4096, 2048, 16, 32.0, seed=31)


def test_65b_upproj_sampled_rows(lib):
    """22016 x 8192 (Llama-65B up-projection), 4096 tokens, r=64, alpha=16."""
    _sampled_big(lib, 22016, 8192, 4096, 64, 16.0, seed=65, nrows=12)


# More than 256 tokens take the CTA-pair GEMMs (512-token tiles, 256-row / 256-column pair tiles).
@pytest.mark.parametrize("m,n,k,r", [(600, 320, 448, 16), (777, 1024, 768, 128), (1030, 136, 64, 8),
                                     (257, 512, 1280, 32), (1536, 768, 512, 64)])
def test_pair_tiles_ragged(lib, m, n, k, r):
    case = synthetic.linear_case(n, k, m, r, 2.0 * r, base_seed=3 * m + n + k + r)
    _check_all(lib, case)


# U = dY B of the backward with k split over a cluster of up to four CTAs per 64-row block: four
# shares with a ragged k (n = 1000 ends inside a 32-wide chunk), two shares (65 row blocks), one
# share (141 row blocks, the whole of B staged per CTA) and, past a wave of row blocks, the
# persistent kernel over 16-row tiles.
# The CTA-pair dX GEMM shapes around it: a ragged n = 1000 with r = 12 (scalar staging of B) and
# 15 column tiles of dX at 1900 tokens.
@pytest.mark.parametrize("m,n,k,r", [(700, 1000, 256, 16), (4100, 512, 256, 8), (9000, 264, 128, 16),
                                     (9500, 256, 128, 12), (2000, 1000, 4096, 12), (1900, 4096, 3840, 16)])
def test_u_split_over_cluster(lib, m, n, k, r):
    _check_all(lib, synthetic.linear_case(n, k, m, r, 2.0 * r, base_seed=m + n + k + r))


def test_pair_accumulate_flags(lib):
    _accumulate_against_oracle(lib, synthetic.linear_case(384, 320, 520, 16, 32.0, base_seed=21))


# More tiles than CTA pairs fit at once (74 on a B300): 1030 tokens make 3 token tiles (the last
# ragged), 32 x 3 = 96 pair tiles in two waves -- in the forward (n = 8192) and in the backward
# (k = 8192); U = dY B of the backward runs on the k-major copy of B beside the dX GEMM.
@pytest.mark.parametrize("m,n,k,r", [(1030, 8192, 2048, 16), (1030, 2048, 8192, 16)])
def test_pair_multi_wave(lib, m, n, k, r):
    _check_all(lib, synthetic.linear_case(n, k, m, r, 2.0 * r, base_seed=m + n // 64 + k // 64))


def test_pair_multi_wave_accumulate(lib):
    """Gradient accumulation into dX (16-byte read-modify-write in the GEMM epilogue), two waves."""
    _accumulate_against_oracle(lib, synthetic.linear_case(2048, 8192, 1030, 16, 32.0, base_seed=77))


def test_pair_lora_path_alone_with_zero_weight(lib):
    case = synthetic.linear_case(512, 256, 600, 16, 32.0, base_seed=22)
    case.w.zero_()
    case.b.copy_((torch.randn(case.b.shape, generator=torch.Generator().manual_seed(6))).to(torch.bfloat16))
    y, dx, _, _ = _check_all(lib, case)
    assert float(y.float().abs().max()) > 0 and float(dx.float().abs().max()) > 0
