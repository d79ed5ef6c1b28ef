"""GPU parity: the grouped small-token forward (decode over a list of matrices).

A list of independent problems with mixed shapes (Llama-7B projection shapes,
ragged rows), token counts 1..16 and ranks 1..128 runs as one
qlora_linear_fwd_grouped call; every output is compared with the float64
oracle (GEMM tolerance, whole tensor and every row) and with the
single-problem entry point.  A chain of dependent calls (each input the
previous call's output, as a decoder's layers are) checks that the weights
the next call prefetches early never let it read its input early, and a CUDA
graph replay of the chain checks the per-call counters start clean every time.
"""

import numpy as np
import pytest
import torch

import synthetic
from oracle import linear, nf4
from tests._helpers import GEMM_TOL, assert_close, t_save_tol, rel_fro, to_np32, to_np64

pytestmark = pytest.mark.gpu

SHAPES = [  # (n, k, m, r)
    (4096, 4096, 1, 16), (4096, 4096, 4, 16), (11008, 4096, 16, 16), (4096, 11008, 4, 16),
    (136, 640, 3, 8), (264, 320, 16, 64), (512, 512, 7, 24), (128, 64, 1, 8),
    (200, 1088, 9, 1), (72, 256, 12, 5), (384, 512, 16, 128), (1032, 2112, 2, 100),
]


def _problems(device="cuda"):
    out = []
    for i, (n, k, m, r) in enumerate(SHAPES):
        c = synthetic.linear_case(n, k, m, r, 2.0 * r, device=device, base_seed=500 + 10 * i)
        out.append(c)
    return out


def test_grouped_matches_oracle_and_single_calls(lib):
    cases = _problems()
    recs = [lib.quantize(c.w) for c in cases]
    probs = [(c.x, rec, c.a, c.b, c.alpha, None, torch.empty((c.m, c.r), dtype=torch.float32, device="cuda"))
             for c, rec in zip(cases, recs)]
    g = lib.GroupedForward(probs)
    ys = g.run()
    ys2 = g.run()  # a second call on the same prepared list gives the same bits
    lib.check_status()
    for i, (c, rec) in enumerate(zip(cases, recs)):
        assert torch.equal(ys[i], ys2[i])
        n, k = c.w.shape
        ref = nf4.quantize(to_np32(c.w.cpu()), n, k)
        wd = nf4.dequantize(ref["codes"], ref["q"], ref["step"], ref["mu"], n, k)
        yr, tr = linear.lora_forward(to_np64(c.x), wd, to_np64(c.a), to_np64(c.b), c.alpha, c.r)
        assert_close(to_np64(ys[i]), yr, GEMM_TOL, str(SHAPES[i]))
        assert rel_fro(to_np64(probs[i][6]), tr) < t_save_tol(c.k), SHAPES[i]
        # the single-problem path keeps bf16_rn(L a') per weight, the grouped path bf16(L) a':
        # within 2^-8 of each other per weight, far less over a sum
        y1, _ = lib.linear_fwd(c.x, rec, c.a, c.b, c.alpha)
        assert rel_fro(to_np64(ys[i]), to_np64(y1)) < 5e-3, SHAPES[i]


def test_grouped_rejects_large_token_counts(lib):
    c = synthetic.linear_case(256, 256, 17, 16, 32.0, device="cuda", base_seed=9)
    rec = lib.quantize(c.w)
    with pytest.raises(lib.QloraError) as e:
        lib.linear_fwd_grouped([(c.x, rec, c.a, c.b, c.alpha, None, None)])
    assert e.value.code == lib.QLORA_ERR_UNSUPPORTED
    lib.check_status()


def test_grouped_long_rows_and_k_limit(lib):
    """k = 32768: 64 absmax blocks per warp and row (the cp.async ring wraps many times, the
    block steps change group inside a warp's range); k above 131072 is refused."""
    c = synthetic.linear_case(24, 32768, 2, 8, 16.0, device="cuda", base_seed=77)
    rec = lib.quantize(c.w)
    t = torch.empty((c.m, c.r), dtype=torch.float32, device="cuda")
    (y,) = lib.linear_fwd_grouped([(c.x, rec, c.a, c.b, c.alpha, None, t)])
    lib.check_status()
    n, k = c.w.shape
    ref = nf4.quantize(to_np32(c.w.cpu()), n, k)
    wd = nf4.dequantize(ref["codes"], ref["q"], ref["step"], ref["mu"], n, k)
    yr, tr = linear.lora_forward(to_np64(c.x), wd, to_np64(c.a), to_np64(c.b), c.alpha, c.r)
    assert_close(to_np64(y), yr, GEMM_TOL, "k=32768")
    assert rel_fro(to_np64(t), tr) < t_save_tol(k)
    big = synthetic.linear_case(8, 131136, 1, 1, 2.0, device="cuda", base_seed=78)
    brec = lib.quantize(big.w)
    with pytest.raises(lib.QloraError) as e:
        lib.linear_fwd_grouped([(big.x, brec, big.a, big.b, big.alpha, None, None)])
    assert e.value.code == lib.QLORA_ERR_UNSUPPORTED
    lib.check_status()


SMALL_SHAPES = [  # lists capped at 1, 2 or 4 tokens (one token group of the MMA), k of 1 to 172 blocks
    (4096, 4096, 1, 16), (4096, 11008, 4, 16), (11008, 4096, 2, 16), (136, 640, 3, 8),
    (264, 320, 4, 64), (128, 64, 1, 8), (512, 4160, 2, 24), (1032, 2112, 1, 32),
]


@pytest.mark.parametrize("mmax", [1, 2, 4])
def test_grouped_small_token_path(lib, mmax):
    shapes = [(n, k, min(m, mmax), r) for (n, k, m, r) in SMALL_SHAPES]
    cases = [synthetic.linear_case(n, k, m, r, 2.0 * r, device="cuda", base_seed=700 + 10 * i + mmax)
             for i, (n, k, m, r) in enumerate(shapes)]
    recs = [lib.quantize(c.w) for c in cases]
    probs = [(c.x, rec, c.a, c.b, c.alpha, None, None) for c, rec in zip(cases, recs)]
    ys = lib.linear_fwd_grouped(probs)
    lib.check_status()
    for i, (c, rec) in enumerate(zip(cases, recs)):
        n, k = c.w.shape
        ref = nf4.quantize(to_np32(c.w.cpu()), n, k)
        wd = nf4.dequantize(ref["codes"], ref["q"], ref["step"], ref["mu"], n, k)
        yr, _ = linear.lora_forward(to_np64(c.x), wd, to_np64(c.a), to_np64(c.b), c.alpha, c.r)
        assert rel_fro(to_np64(ys[i]), yr) < GEMM_TOL, shapes[i]


SHORT_LISTS = [  # short lists at 1-2 tokens: one 16-row tile per CTA, its k range split over 8 warps
    [(4096, 4096, 1, 16)],                        # 256 tiles, 8 blocks per warp
    [(4096, 11008, 1, 16)],                       # the down projection: 21-22 blocks per warp
    [(296, 1088, 2, 8), (264, 2112, 1, 16)],      # ragged rows; 17 and 33 blocks a row (odd warp ranges)
    [(1032, 4160, 2, 24)],                        # 65 blocks a row, 65 tiles of which the last is half full
]


@pytest.mark.parametrize("which", range(len(SHORT_LISTS)))
def test_grouped_short_lists_match_oracle_and_are_deterministic(lib, which):
    shapes = SHORT_LISTS[which]
    cases = [synthetic.linear_case(n, k, m, r, 2.0 * r, device="cuda", base_seed=900 + 10 * i + which)
             for i, (n, k, m, r) in enumerate(shapes)]
    recs = [lib.quantize(c.w) for c in cases]
    ts = [torch.full((c.m, c.r), float("nan"), dtype=torch.float32, device="cuda") for c in cases]
    probs = [(c.x, rec, c.a, c.b, c.alpha, None, t) for c, rec, t in zip(cases, recs, ts)]
    g = lib.GroupedForward(probs)
    ys = [y.clone() for y in g.run()]
    ys2 = g.run()
    lib.check_status()
    for i, (c, rec) in enumerate(zip(cases, recs)):
        assert torch.equal(ys[i], ys2[i]), shapes[i]
        n, k = c.w.shape
        ref = nf4.quantize(to_np32(c.w.cpu()), n, k)
        wd = nf4.dequantize(ref["codes"], ref["q"], ref["step"], ref["mu"], n, k)
        yr, tr = linear.lora_forward(to_np64(c.x), wd, to_np64(c.a), to_np64(c.b), c.alpha, c.r)
        assert rel_fro(to_np64(ys[i]), yr) < GEMM_TOL, shapes[i]
        assert rel_fro(to_np64(ts[i]), tr) < t_save_tol(c.k), shapes[i]


def test_grouped_long_list_one_and_two_tokens(lib):
    """A list long enough to give every CTA slot a 128-row tile of its own (48
    problems, 312 tiles for a 148-SM B300): the layout streamed for long lists,
    ragged rows, 1 and 2 tokens, against the oracle; a second call gives the same bits."""
    base = [(768, 256, 1, 8), (776, 320, 2, 16), (1024, 1088, 1, 16), (520, 512, 2, 24)]
    shapes = [base[i % 4] for i in range(48)]
    cases = [synthetic.linear_case(n, k, m, r, 2.0 * r, device="cuda", base_seed=1300 + 7 * i)
             for i, (n, k, m, r) in enumerate(shapes)]
    recs = [lib.quantize(c.w) for c in cases]
    probs = [(c.x, rec, c.a, c.b, c.alpha, None, None) for c, rec in zip(cases, recs)]
    g = lib.GroupedForward(probs)
    ys = [y.clone() for y in g.run()]
    ys2 = g.run()
    lib.check_status()
    for i, (c, rec) in enumerate(zip(cases, recs)):
        assert torch.equal(ys[i], ys2[i]), shapes[i]
        n, k = c.w.shape
        ref = nf4.quantize(to_np32(c.w.cpu()), n, k)
        wd = nf4.dequantize(ref["codes"], ref["q"], ref["step"], ref["mu"], n, k)
        yr, _ = linear.lora_forward(to_np64(c.x), wd, to_np64(c.a), to_np64(c.b), c.alpha, c.r)
        assert rel_fro(to_np64(ys[i]), yr) < GEMM_TOL, shapes[i]


def _chain(lib, recs, loras, x0, graph_replays=0):
    """Dependent calls: call i reads call i-1's output (every matrix is square)."""
    outs = [torch.empty_like(x0) for _ in recs]
    steps = []
    prev = x0
    for i, rec in enumerate(recs):
        steps.append(lib.GroupedForward([(prev, rec, loras[i][0], loras[i][1], 32.0, outs[i], None)]))
        prev = outs[i]

    def run():
        for g in steps:
            g.run()

    run()
    torch.cuda.synchronize()
    first = [o.clone() for o in outs]
    if graph_replays:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run()
        for _ in range(graph_replays):
            for o in outs:
                o.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            for a, b in zip(first, outs):
                assert torch.equal(a, b)
    return first


@pytest.mark.parametrize("m", [1, 4, 16])
def test_grouped_chain_of_dependent_calls(lib, m):
    n = 1024
    layers = 6
    recs, loras = [], []
    for i in range(layers):
        w = synthetic.weight(n, n, device="cuda", seed=3000 + i)
        recs.append(lib.quantize(w))
        loras.append(synthetic.lora_pair(n, n, 16, device="cuda", seed=3100 + 2 * i))
    x0 = synthetic.activations(m, n, device="cuda", seed=3200)
    outs = _chain(lib, recs, loras, x0, graph_replays=2)
    lib.check_status()
    # oracle chain, fed with the GPU's own bf16 inputs at every layer (isolates each call)
    prev = to_np64(x0)
    for i in range(layers):
        ref = nf4.quantize(to_np32(synthetic.weight(n, n, device="cuda", seed=3000 + i).cpu()), n, n)
        wd = nf4.dequantize(ref["codes"], ref["q"], ref["step"], ref["mu"], n, n)
        yr, _ = linear.lora_forward(prev, wd, to_np64(loras[i][0]), to_np64(loras[i][1]), 32.0, 16)
        assert_close(to_np64(outs[i]), yr, GEMM_TOL, "layer %d" % i)
        prev = to_np64(outs[i])
