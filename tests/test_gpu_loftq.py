"""GPU check of the LoftQ initialisation (P1 tutorial, section 3.10).

The SVD runs in float32 on the GPU and in float64 in the oracle, so the factors
are not bit-comparable (the tail of a quantisation residual's spectrum is
nearly flat, so its top-r subspace is not well determined).  What is unique is
checked against the oracle -- the error of base + branch after each iteration
-- and the rest is checked for validity: every record is exactly the NF4
quantisation of W - s B A for the factors that went in, and every new branch
leaves the residual the energy of its discarded singular values.
"""

import numpy as np
import pytest
import torch

import synthetic
from bit_quantized_fine_nf4_b300 import loftq as gpu_loftq
from oracle import loftq, lowrank, nf4

pytestmark = pytest.mark.gpu


def test_loftq_matches_oracle_errors_and_each_step_is_exact(lib):
    n, k, r, alpha, iters = 512, 1024, 16, 32.0, 3
    w = synthetic.structured_weight(n, k, rank=8, device="cuda", seed=5)
    hist = []
    trace = []
    rec, a, b = gpu_loftq.loftq_init(w, r, alpha, iters=iters, history=hist, trace=trace)
    lib.check_status()
    ref = loftq.loftq(w.cpu().numpy(), r, alpha, iters)
    for h, rr in zip(hist, ref):
        assert abs(h - rr["rel_err"]) < 0.01 * rr["rel_err"], (hist, [x["rel_err"] for x in ref])
    # the plain 4-bit base for comparison: LoftQ must be well below it
    q0 = nf4.quantize(w.cpu().numpy(), n, k)
    base_err = np.linalg.norm(w.cpu().numpy() - nf4.dequantize(q0["codes"], q0["q"], q0["step"], q0["mu"], n, k)) / \
        np.linalg.norm(w.cpu().numpy())
    assert hist[-1] < 0.8 * base_err
    s = float(lowrank.lora_scale_f32(alpha, r))
    f = lambda t: t.float().cpu().numpy()  # noqa: E731
    for step in trace:
        target = lowrank.lowrank_update_f32(w.cpu().numpy(), None, f(step["a_in"]), f(step["b_in"]), -s, n, k)
        want = nf4.quantize(target, n, k)
        assert np.array_equal(step["record"].codes.cpu().numpy(), want["codes"])
        assert np.array_equal(step["record"].absmax_q.cpu().numpy(), want["q"])
        res = lowrank.lowrank_update_f32(w.cpu().numpy(), want, None, None, 0.0, n, k).astype(np.float64)
        sv = np.linalg.svd(res, compute_uv=False)
        left = np.sum((res - s * (f(step["b"]).astype(np.float64) @ f(step["a"]).astype(np.float64))) ** 2)
        tail = np.sum(sv[r:] ** 2)
        assert tail * (1 - 1e-6) <= left < tail * 1.01
    assert torch.equal(trace[-1]["record"].codes, rec.codes) and torch.equal(trace[-1]["a"], a)
