"""GPU parity: merge / export and the dense low-rank update, bit-exact against the oracle.

qlora_nf4_merge gives bf16(deq(W) + s B A) with a fixed float32 order, so the
bits must equal ``oracle.lowrank.merge_bf16_bits`` (Day 25 notes section 2.6;
P1 tutorial section 3.8).  The merged weight re-quantised by qlora_nf4_quantize
must equal the oracle's quantisation of the oracle's merge (glossary "QLoRA",
"Trade-offs": merged to 16 bits, quantised again for serving).  The dense
update (the arithmetic of the LoftQ initialisation) is bit-exact too.
"""

import numpy as np
import pytest
import torch

import synthetic
from oracle import lowrank, nf4
from tests._helpers import to_np32

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _f32(t):
    return t.float().cpu().numpy()


@pytest.mark.parametrize("n,k,r,alpha", [(256, 256, 8, 16.0), (264, 320, 5, 10.0), (4096, 4096, 16, 32.0),
                                         (136, 4160, 1, 2.0), (512, 1024, 128, 256.0), (320, 448, 12, 24.0)])
def test_merge_bit_exact(lib, n, k, r, alpha):
    case = synthetic.linear_case(n, k, 1, r, alpha, device="cuda", base_seed=n + k + r)
    rec = lib.quantize(case.w)
    out = lib.merge(rec, case.a, case.b, alpha)
    lib.check_status()
    ref_rec = nf4.quantize(to_np32(case.w.cpu()), n, k)
    ref = lowrank.merge_bf16_bits(ref_rec, _f32(case.a), _f32(case.b), alpha, n, k)
    assert np.array_equal(_bits(out), ref)


def test_merge_then_requantise(lib):
    """Export: merge, then quantise the merged bf16 weight again; codes, scales and the
    dequantised weight equal the oracle's quantisation of its own merge."""
    n, k, r, alpha = 1024, 2048, 16, 32.0
    case = synthetic.linear_case(n, k, 1, r, alpha, device="cuda", base_seed=77)
    # a trained branch is larger than the initial B: scale B up so the merge moves weights
    b = (case.b.float() * 20).to(torch.bfloat16)
    rec = lib.quantize(case.w)
    merged = lib.merge(rec, case.a, b, alpha)
    rec2 = lib.quantize(merged)
    lib.check_status()
    ref_merged = nf4.bf16_bits_to_f32(lowrank.merge_bf16_bits(nf4.quantize(to_np32(case.w.cpu()), n, k),
                                                              _f32(case.a), _f32(b), alpha, n, k))
    ref2 = nf4.quantize(ref_merged, n, k)
    assert np.array_equal(rec2.codes.cpu().numpy(), ref2["codes"])
    assert np.array_equal(rec2.absmax_q.cpu().numpy(), ref2["q"])
    assert np.array_equal(rec2.absmax_step.cpu().numpy().view(np.uint32), ref2["step"].view(np.uint32))
    assert rec2.absmax_mean.cpu().numpy().view(np.uint32)[0] == np.float32(ref2["mu"]).view(np.uint32)
    # the export changed the codes (the branch was not negligible)
    assert not np.array_equal(rec2.codes.cpu().numpy(), rec.codes.cpu().numpy())


@pytest.mark.parametrize("w_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("with_sub,r", [(False, 16), (True, 0), (True, 7)])
def test_lowrank_update_bit_exact(lib, w_dtype, with_sub, r):
    n, k = 520, 1088
    case = synthetic.linear_case(n, k, 1, max(r, 1), 2.0, device="cuda", base_seed=31 + r, w_dtype=w_dtype)
    rec = lib.quantize(case.w) if with_sub else None
    a, b = (case.a, case.b) if r > 0 else (None, None)
    coef = -0.625
    out = lib.lowrank_update(case.w, rec, a, b, coef)
    lib.check_status()
    ref_rec = nf4.quantize(to_np32(case.w.cpu()), n, k) if with_sub else None
    ref = lowrank.lowrank_update_f32(to_np32(case.w.cpu()), ref_rec, _f32(a) if r else None, _f32(b) if r else None,
                                     coef, n, k)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
