"""GPU parity: NF4 quantise / double quant / dequantise, bit-exact against the oracle.

Calls the CUDA path through the C ABI (ctypes binding) on seeded synthetic
weights and compares every output byte with ``oracle.nf4``.
"""

import numpy as np
import pytest
import torch

import synthetic
from oracle import nf4
from tests._helpers import to_np32

pytestmark = pytest.mark.gpu


def _oracle_record(w_cpu: torch.Tensor):
    n, k = w_cpu.shape
    return nf4.quantize(to_np32(w_cpu), n, k)


def _assert_record_equal(lib, rec, ref, n, k):
    assert np.array_equal(rec.codes.cpu().numpy(), ref["codes"]), "4-bit codes differ"
    assert np.array_equal(rec.absmax_q.cpu().numpy(), ref["q"]), "int8 absmax codes differ"
    assert np.array_equal(rec.absmax_step.cpu().numpy().view(np.uint32), ref["step"].view(np.uint32)), "steps differ"
    assert rec.absmax_mean.cpu().numpy().view(np.uint32)[0] == np.float32(ref["mu"]).view(np.uint32), "mean differs"
    wd = lib.dequantize(rec)
    lib.check_status()
    ref_bits = nf4.dequantize_bf16_bits(ref["codes"], ref["q"], ref["step"], ref["mu"], n, k)
    got_bits = wd.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got_bits, ref_bits), "dequantised bf16 differs"


def test_tiny_case_fp32(lib):
    case = synthetic.tiny_case()
    w = case.w.cuda()
    rec = lib.quantize(w)
    lib.check_status()
    _assert_record_equal(lib, rec, _oracle_record(case.w), 256, 256)


@pytest.mark.parametrize("n,k", [(8, 64), (24, 192), (136, 640), (512, 4160)])
def test_ragged_shapes_bf16(lib, n, k):
    w = synthetic.weight(n, k, device="cuda", seed=n * 7 + k)
    rec = lib.quantize(w)
    lib.check_status()
    _assert_record_equal(lib, rec, _oracle_record(w.cpu()), n, k)


def test_attention_projection_4096(lib):
    w = synthetic.weight(4096, 4096, device="cuda", seed=0)
    rec = lib.quantize(w)
    lib.check_status()
    _assert_record_equal(lib, rec, _oracle_record(w.cpu()), 4096, 4096)


def test_encode_boundaries_and_special_blocks(lib):
    """Blocks of absmax 1 (so x = w exactly) filled with every fp32 value near each
    decision boundary, exact levels, exact ties, zeros and an all-zero block."""
    lv = nf4.nf4_levels_f32()
    vals = []
    for j in range(15):
        mid = np.float32((np.float64(lv[j]) + np.float64(lv[j + 1])) / 2)
        v = mid
        for _ in range(6):
            v = np.nextafter(v, np.float32(-2))
        for _ in range(13):
            vals.append(v)
            v = np.nextafter(v, np.float32(2))
    vals += list(lv) + [lv[6] / 2, lv[8] / 2, np.float32(0), np.float32(-0.0)]
    vals = np.array(vals, dtype=np.float32)
    per = 63
    nb = (vals.size + per - 1) // per
    w = np.zeros((nb + 1, 64), dtype=np.float32)
    for b in range(nb):
        chunk = vals[b * per:(b + 1) * per]
        w[b, :chunk.size] = chunk
        w[b, 63] = 1.0
    # last block stays all zero
    n = 8 * ((w.size // 64 + 7) // 8)
    full = np.zeros((n * 64,), dtype=np.float32)
    full[: w.size] = w.reshape(-1)
    full = full.reshape(n, 64)
    rec = lib.quantize(torch.from_numpy(full).cuda())
    lib.check_status()
    _assert_record_equal(lib, rec, nf4.quantize(full, n, 64), n, 64)


def _bf16_threshold_blocks():
    """bf16 blocks of 64: for absmax values a spread over the whole bf16 exponent
    range (subnormal to 2^126), the eight bf16 values on each side of a * m_j for
    every decision boundary m_j (the midpoint of two neighbouring NF4 levels),
    both signs, with a itself in the block's last slot."""
    lv = nf4.nf4_levels_f32().astype(np.float64)
    mids = (lv[:-1] + lv[1:]) / 2
    abits = sorted(set(list(range(0x0001, 0x7f80, 0x00c7)) +
                       [0x0080, 0x00ff, 0x0100, 0x0101, 0x3f80, 0x3f81, 0x3fff, 0x7dff, 0x7e00, 0x7e01, 0x7f7f]))
    blocks = []
    for ab in abits:
        a = nf4.bf16_bits_to_f32(np.array([ab], dtype=np.uint16))[0]
        vals = []
        for m in mids:
            tb = int(nf4.f32_to_bf16_bits(np.array([abs(a * m)], dtype=np.float32))[0])
            for mag in range(max(tb - 8, 0), tb + 9):
                if mag <= ab:
                    vals.append(mag | (0x8000 if m < 0 else 0))
        vals = np.array(vals, dtype=np.uint16)
        for c0 in range(0, vals.size, 63):
            blk = np.zeros(64, dtype=np.uint16)
            chunk = vals[c0:c0 + 63]
            blk[:chunk.size] = chunk
            blk[63] = ab
            blocks.append(blk)
    while len(blocks) % 8:  # rows of the [n, 64] weight: n a multiple of 8
        blocks.append(np.zeros(64, dtype=np.uint16))
    bits = np.stack(blocks)
    return nf4.bf16_bits_to_f32(bits.reshape(-1)).reshape(bits.shape)


def test_bf16_codes_near_every_boundary_all_exponents(lib):
    """The bf16 path takes the quotient from the rounded reciprocal with one
    correction and the code from a bucket table; its codes must equal the
    oracle's (IEEE quotient, nearest level, lower index on ties) for weights
    packed around every decision boundary at every block-scale exponent."""
    w = _bf16_threshold_blocks()
    n = w.shape[0]
    rec = lib.quantize(torch.from_numpy(w).to(torch.bfloat16).cuda())
    lib.check_status()
    a = nf4.blockwise_absmax(w)
    ref = nf4.pack_codes(nf4.nf4_encode(w.reshape(-1), a))
    assert np.array_equal(rec.codes.cpu().numpy(), ref), "4-bit codes differ"


def test_bf16_every_weight_value_for_sampled_scales(lib):
    """For 200 block scales a (bf16) spread over the whole exponent range --
    subnormal, both edges of the range where the bf16 path decides without a
    quotient (2^-90 and 2^120), and ordinary values -- blocks holding every bf16
    weight w with |w| <= a, both signs: all codes equal the oracle's."""
    rng = np.random.default_rng(2024)
    edges = [0x0001, 0x007f, 0x0080, 0x0100, 0x127f, 0x1280, 0x1281, 0x3c00, 0x3f80, 0x3fff,
             0x7b7f, 0x7b80, 0x7b81, 0x7f7f]
    abits = sorted(set(edges + list(rng.integers(1, 0x7f80, size=186))))
    blocks = []
    for ab in abits:
        mags = np.arange(0, ab + 1, dtype=np.uint32)
        vals = np.concatenate([mags, mags[1:] | 0x8000]).astype(np.uint16)
        nb = (vals.size + 62) // 63
        blk = np.zeros((nb, 64), dtype=np.uint16)
        flat = blk[:, :63].reshape(-1)
        flat[:vals.size] = vals
        blk[:, :63] = flat.reshape(nb, 63)
        blk[:, 63] = ab
        blocks.append(blk)
    bits = np.concatenate(blocks)
    pad = (-bits.shape[0]) % 8
    if pad:
        bits = np.concatenate([bits, np.zeros((pad, 64), dtype=np.uint16)])
    w = nf4.bf16_bits_to_f32(bits.reshape(-1)).reshape(bits.shape)
    rec = lib.quantize(torch.from_numpy(w).to(torch.bfloat16).cuda())
    lib.check_status()
    ref = nf4.pack_codes(nf4.nf4_encode(w.reshape(-1), nf4.blockwise_absmax(w)))
    assert np.array_equal(rec.codes.cpu().numpy(), ref), "4-bit codes differ"


def test_nonfinite_is_reported(lib):
    w = synthetic.weight(16, 128, device="cuda", seed=3)
    w[5, 17] = float("nan")
    lib.quantize(w)
    assert lib.get_status() == lib.QLORA_ERR_NONFINITE
    assert lib.get_status() == lib.QLORA_OK  # cleared
    w2 = synthetic.weight(16, 128, device="cuda", seed=4)
    rec = lib.quantize(w2)
    lib.check_status()
    _assert_record_equal(lib, rec, _oracle_record(w2.cpu()), 16, 128)


def test_invalid_arguments_are_rejected(lib):
    w = synthetic.weight(16, 96, device="cuda", seed=5)  # k not a multiple of 64
    with pytest.raises(lib.QloraError) as e:
        lib.quantize(w)
    assert e.value.code in (lib.QLORA_ERR_INVALID_ARGUMENT, lib.QLORA_ERR_UNSUPPORTED)
    w = synthetic.weight(16, 128, device="cuda", seed=5)
    rec = lib.NF4Weight.empty(16, 128)
    bad = torch.empty(16 * 128 + 8, dtype=torch.bfloat16, device="cuda")[1:].view(-1)[: 16 * 128].view(16, 128)
    with pytest.raises(lib.QloraError) as e:
        lib.quantize(bad, rec)
    assert e.value.code == lib.QLORA_ERR_INVALID_ARGUMENT
    lib.check_status()


def test_bounded_wait_timeout_keeps_context(lib):
    lib.selftest_wait_timeout(20_000_000)  # 20 ms on a barrier nothing arrives on
    assert lib.get_status() == lib.QLORA_ERR_TIMEOUT
    w = synthetic.weight(8, 64, device="cuda", seed=6)
    rec = lib.quantize(w)
    lib.check_status()
    _assert_record_equal(lib, rec, _oracle_record(w.cpu()), 8, 64)


def test_65b_upproj_weight_sampled_rows(lib):
    """22016 x 8192 (Llama-65B up-projection): the double quantisation of all
    2.8 M block scales bit-exact, codes and dequantised rows on 64 sampled rows."""
    n, k = 22016, 8192
    w = synthetic.weight(n, k, device="cuda", seed=4242)
    rec = lib.quantize(w)
    lib.check_status()
    wc = to_np32(w.cpu())
    a = nf4.blockwise_absmax(wc)
    q, step, mu = nf4.double_quant(a)
    assert np.array_equal(rec.absmax_q.cpu().numpy(), q)
    assert np.array_equal(rec.absmax_step.cpu().numpy().view(np.uint32), step.view(np.uint32))
    assert rec.absmax_mean.cpu().numpy().view(np.uint32)[0] == np.float32(mu).view(np.uint32)
    rows = np.sort(np.random.default_rng(1).choice(n, 64, replace=False))
    codes_gpu = rec.codes.cpu().numpy().reshape(n, k // 2)
    bpr = k // 64
    for r0 in rows:
        ref = nf4.pack_codes(nf4.nf4_encode(wc[r0], a[r0 * bpr:(r0 + 1) * bpr]))
        assert np.array_equal(codes_gpu[r0], ref)
    wd = lib.dequantize(rec)[torch.from_numpy(rows).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    lv = nf4.nf4_levels_f32()
    a2 = nf4.dequant_absmax(q, step, mu).reshape(n, bpr)
    for i, r0 in enumerate(rows):
        c = nf4.unpack_codes(codes_gpu[r0]).reshape(bpr, 64)
        ref = nf4.f32_to_bf16_bits((lv[c] * a2[r0][:, None]).astype(np.float32)).reshape(-1)
        assert np.array_equal(wd[i], ref)
