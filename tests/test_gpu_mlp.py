"""GPU parity: SiLU * up glue and the Llama MLP block built from three QLoRA linears.

The glue (h = silu(g) * u) is not on the pages; it is checked against its plain
definition in the oracle.  The block: g = fwd(X, Wg), u = fwd(X, Wu),
h = silu(g) u, y = fwd(h, Wd); backward in reverse with dX accumulated over
the gate and up branches (QLORA_ACCUM_DX).  Every output is compared in full
(whole tensor and every row), at a reduced size and at the Llama-7B shape.
"""

import numpy as np
import pytest
import torch

import synthetic
from oracle import linear, nf4
from tests._helpers import GEMM_TOL, assert_close, to_np32, to_np64

pytestmark = pytest.mark.gpu


def test_silu_mul_elementwise(lib):
    g = torch.randn(4, 2048, generator=torch.Generator().manual_seed(0)).mul(3).to(torch.bfloat16)
    u = torch.randn(4, 2048, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    dh = torch.randn(4, 2048, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    h = lib.silu_mul_fwd(g.cuda(), u.cuda())
    dg, du = lib.silu_mul_bwd(dh.cuda(), g.cuda(), u.cuda())
    lib.check_status()
    href = linear.silu_mul_forward(to_np64(g), to_np64(u))
    dgr, dur = linear.silu_mul_backward(to_np64(dh), to_np64(g), to_np64(u))
    # float32 math then one bf16 rounding: within 2^-8 relative of the exact value
    for got, ref in ((h, href), (dg, dgr), (du, dur)):
        err = np.abs(to_np64(got) - ref)
        assert np.all(err <= np.abs(ref) * 2.0 ** -8 + 1e-6)


def _deq(w):
    n, k = w.shape
    rec = nf4.quantize(to_np32(w), n, k)
    return nf4.dequantize(rec["codes"], rec["q"], rec["step"], rec["mu"], n, k)


def _mlp_block(lib, hidden, inter, m, r, alpha, seeds, device):
    """Run the block on the GPU and in the float64 oracle; compare every output in full."""
    s0 = seeds
    wg = synthetic.weight(inter, hidden, device=device, seed=s0 + 1).cpu()
    wu = synthetic.weight(inter, hidden, device=device, seed=s0 + 2).cpu()
    wd = synthetic.weight(hidden, inter, device=device, seed=s0 + 3).cpu()
    ag, bg = (t.cpu() for t in synthetic.lora_pair(inter, hidden, r, device=device, seed=s0 + 10))
    au, bu = (t.cpu() for t in synthetic.lora_pair(inter, hidden, r, device=device, seed=s0 + 20))
    ad, bd = (t.cpu() for t in synthetic.lora_pair(hidden, inter, r, device=device, seed=s0 + 30))
    x = synthetic.activations(m, hidden, device=device, seed=s0 + 4).cpu()
    dy = synthetic.activations(m, hidden, device=device, seed=s0 + 5).cpu()

    c = lambda t: t.cuda()  # noqa: E731
    rg, ru, rd = lib.quantize(c(wg)), lib.quantize(c(wu)), lib.quantize(c(wd))
    g, tg = lib.linear_fwd(c(x), rg, c(ag), c(bg), alpha)
    u, tu = lib.linear_fwd(c(x), ru, c(au), c(bu), alpha)
    h = lib.silu_mul_fwd(g, u)
    y, td = lib.linear_fwd(h, rd, c(ad), c(bd), alpha)
    dh, dad, dbd = lib.linear_bwd(c(dy), h, rd, c(ad), c(bd), alpha, td)
    dg, du = lib.silu_mul_bwd(dh, g, u)
    dx, dag, dbg = lib.linear_bwd(dg, c(x), rg, c(ag), c(bg), alpha, tg)
    dx, dau, dbu = lib.linear_bwd(du, c(x), ru, c(au), c(bu), alpha, tu, dx=dx, flags=lib.ACCUM_DX)
    lib.check_status()

    # oracle, float64 end to end (glue exact, no bf16 rounding of g, u, h, dh)
    X, DY = to_np64(x), to_np64(dy)
    f = lambda t: to_np64(t)  # noqa: E731
    Wg, Wu, Wd = _deq(wg), _deq(wu), _deq(wd)
    G, Tg = linear.lora_forward(X, Wg, f(ag), f(bg), alpha, r)
    U, Tu = linear.lora_forward(X, Wu, f(au), f(bu), alpha, r)
    H = linear.silu_mul_forward(G, U)
    Y, Td = linear.lora_forward(H, Wd, f(ad), f(bd), alpha, r)
    DH, DAd, DBd, _ = linear.lora_backward(DY, H, Wd, f(ad), f(bd), alpha, r, Td)
    DG, DU = linear.silu_mul_backward(DH, G, U)
    DXg, DAg, DBg, _ = linear.lora_backward(DG, X, Wg, f(ag), f(bg), alpha, r, Tg)
    DXu, DAu, DBu, _ = linear.lora_backward(DU, X, Wu, f(au), f(bu), alpha, r, Tu)
    for name, got, ref in (("y", y, Y), ("dx", dx, DXg + DXu), ("dA down", dad, DAd), ("dB down", dbd, DBd),
                           ("dA gate", dag, DAg), ("dB gate", dbg, DBg), ("dA up", dau, DAu),
                           ("dB up", dbu, DBu)):
        assert_close(to_np64(got), ref, GEMM_TOL, name)


def test_mlp_block_small(lib):
    """Reduced sizes (512 / 1408, 160 tokens): the small-token GEMMs."""
    _mlp_block(lib, 512, 1408, 160, 16, 32.0, 0, "cpu")


def test_mlp_block_llama7b_shape(lib):
    """The Llama-7B MLP block the bench times: gate / up 11008 x 4096, down 4096 x 11008,
    2048 tokens, r=16, alpha=32, on the CTA-pair GEMMs; every row of Y and dX."""
    _mlp_block(lib, 4096, 11008, 2048, 16, 32.0, 100, "cuda")
