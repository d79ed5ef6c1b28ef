"""GPU test of qlora_nf4_quantize_noalloc, the quantiser that allocates nothing.

Some callers cannot allocate device memory on the call path (a framework that
owns the whole device pool, a memory budget fixed at start-up, code where a
cudaMalloc/cudaFree would stall the device).  This entry point gives them the
same quantisation as qlora_nf4_quantize, with its scratch in a fixed device
array inside the library instead of a caller workspace.  The test calls it
through the C ABI twice in a row, on two different weights, and compares each
record bit for bit with the one the workspace entry point produces (the
tolerance the quantiser tests use: exact).  It also checks that a weight above
the fixed limit is refused before anything runs.

This file is named so that pytest collects it after every other test file.
"""

import numpy as np
import pytest

import synthetic

pytestmark = pytest.mark.gpu


def _same_record(a, b):
    assert np.array_equal(a.codes.cpu().numpy(), b.codes.cpu().numpy())
    assert np.array_equal(a.absmax_q.cpu().numpy(), b.absmax_q.cpu().numpy())
    assert np.array_equal(a.absmax_step.cpu().numpy().view(np.uint32), b.absmax_step.cpu().numpy().view(np.uint32))
    assert np.array_equal(a.absmax_mean.cpu().numpy().view(np.uint32), b.absmax_mean.cpu().numpy().view(np.uint32))


def test_noalloc_quantize_matches_workspace_quantize_twice(lib):
    # two calls in a row with different shapes: the shared scratch must not carry over
    for n, k, seed in ((4096, 4096, 0), (1024, 8256, 1)):
        w = synthetic.weight(n, k, device="cuda", seed=seed)
        ref = lib.quantize(w)
        got = lib.quantize_noalloc(w)
        lib.check_status()
        _same_record(got, ref)


def test_noalloc_largest_accepted_weight(lib):
    """n*k == 2^26 exactly (8192 x 8192, the limit): bit-exact against the workspace quantiser,
    twice in a row; one row more (8200 x 8192) is refused before anything runs."""
    w = synthetic.weight(8192, 8192, device="cuda", seed=3)
    ref = lib.quantize(w)
    for _ in range(2):
        got = lib.quantize_noalloc(w)
        lib.check_status()
        _same_record(got, ref)
    import torch
    big = torch.zeros((8200, 8192), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.QloraError) as e:
        lib.quantize_noalloc(big)
    assert e.value.code == lib.QLORA_ERR_UNSUPPORTED
    lib.check_status()


def test_noalloc_quantize_float32_input(lib):
    case = synthetic.tiny_case()
    w = case.w.cuda()
    ref = lib.quantize(w)
    got = lib.quantize_noalloc(w)
    lib.check_status()
    _same_record(got, ref)


def test_noalloc_rejects_weights_above_the_limit(lib):
    import torch
    n, k = 8192, 8256  # 67,633,152 weights > 2^26
    w = torch.empty((n, k), dtype=torch.bfloat16, device="cuda")
    out = lib.NF4Weight.empty(n, k)
    with pytest.raises(lib.QloraError) as e:
        lib.quantize_noalloc(w, out)
    assert e.value.code == lib.QLORA_ERR_UNSUPPORTED
    assert "fixed scratch" in str(e.value)
    lib.check_status()
