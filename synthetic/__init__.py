"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module draws random tensors only; it holds none of the method's
arithmetic (no quantisation, no level table, no matmul).  Both the oracle side
and the CUDA side are fed from here.

Shapes and distributions follow the five workload descriptions of the QLoRA
linear (Llama-7B / 65B shaped):

* weights ~ N(0, 0.02^2), drawn in float32, rounded to bfloat16 unless the
  workload keeps float32 (the tiny case);
* activations and upstream gradients ~ N(0, 1) in bfloat16;
* LoRA ``A``: N(0, 1/K) for the tiny case, Kaiming-uniform U(-1/sqrt(K),
  1/sqrt(K)) otherwise; LoRA ``B`` ~ N(0, 0.01^2) (non-zero on purpose).

Seeds: the tiny case uses one CPU generator with seed 0 drawn in the order
W, X, A, B, dY.  The larger cases draw tensor ``i`` from its own generator
seeded ``base + i`` (W=0, X=1, A=2, B=3, dY=4; stack matrices 1000 + 7*layer +
matrix), on the device the tensors are made on.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

W_STD = 0.02
B_STD = 0.01


@dataclass
class LinearCase:
    """One QLoRA linear problem: Y = X W^T + (alpha/r) (X A^T) B^T."""

    w: torch.Tensor      # [N, K] float32 or bfloat16
    x: torch.Tensor      # [M, K] bfloat16
    a: torch.Tensor      # [r, K] bfloat16
    b: torch.Tensor      # [N, r] bfloat16
    dy: torch.Tensor     # [M, N] bfloat16
    alpha: float
    r: int

    @property
    def m(self) -> int:
        return self.x.shape[0]

    @property
    def n(self) -> int:
        return self.w.shape[0]

    @property
    def k(self) -> int:
        return self.w.shape[1]


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, gen, device, dtype=torch.bfloat16):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std
    return t.to(dtype)


def _kaiming_uniform(shape, fan_in, gen, device):
    bound = 1.0 / math.sqrt(fan_in)
    t = (torch.rand(shape, generator=gen, device=device, dtype=torch.float32) * 2.0 - 1.0) * bound
    return t.to(torch.bfloat16)


def tiny_case() -> LinearCase:
    """W 256x256 float32, X 16x256, r=8, alpha=16, A ~ N(0, 1/256), seed 0 (CPU)."""
    g = _gen("cpu", 0)
    n = k = 256
    m, r = 16, 8
    w = torch.randn((n, k), generator=g, dtype=torch.float32) * W_STD
    x = torch.randn((m, k), generator=g, dtype=torch.float32).to(torch.bfloat16)
    a = (torch.randn((r, k), generator=g, dtype=torch.float32) / 16.0).to(torch.bfloat16)
    b = (torch.randn((n, r), generator=g, dtype=torch.float32) * B_STD).to(torch.bfloat16)
    dy = torch.randn((m, n), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return LinearCase(w, x, a, b, dy, 16.0, r)


def linear_case(n: int, k: int, m: int, r: int, alpha: float, device="cpu", base_seed: int = 0,
                w_dtype=torch.bfloat16, a_init: str = "kaiming") -> LinearCase:
    """A [N, K] weight with M tokens; each tensor from its own seeded generator."""
    w = _normal((n, k), W_STD, _gen(device, base_seed + 0), device, w_dtype)
    x = _normal((m, k), 1.0, _gen(device, base_seed + 1), device)
    if a_init == "kaiming":
        a = _kaiming_uniform((r, k), k, _gen(device, base_seed + 2), device)
    else:
        a = _normal((r, k), 1.0 / math.sqrt(k), _gen(device, base_seed + 2), device)
    b = _normal((n, r), B_STD, _gen(device, base_seed + 3), device)
    dy = _normal((m, n), 1.0, _gen(device, base_seed + 4), device)
    return LinearCase(w, x, a, b, dy, float(alpha), r)


def structured_weight(n: int, k: int, rank: int = 8, device="cpu", seed: int = 0, dtype=torch.float32):
    """N(0, 0.02^2) plus a rank-``rank`` part of about the same Frobenius norm, with
    geometrically decaying strengths (a weight whose spectrum has a few large
    directions on top of a noise floor, as pretrained projections do): the
    workload of the LoftQ initialisation."""
    g = _gen(device, seed)
    noise = torch.randn((n, k), generator=g, device=device, dtype=torch.float32) * W_STD
    u = torch.randn((n, rank), generator=g, device=device, dtype=torch.float32) / math.sqrt(n)
    v = torch.randn((rank, k), generator=g, device=device, dtype=torch.float32) / math.sqrt(k)
    strength = W_STD * math.sqrt(n * k) * torch.tensor([0.7 ** i for i in range(rank)], device=device)
    strength = strength / float(torch.sqrt((strength ** 2).sum() / (W_STD ** 2 * n * k)))
    return (noise + (u * strength[None, :]) @ v).to(dtype)


def weight(n: int, k: int, device="cpu", seed: int = 0, dtype=torch.bfloat16) -> torch.Tensor:
    """A single N(0, 0.02^2) weight [n, k]."""
    return _normal((n, k), W_STD, _gen(device, seed), device, dtype)


def activations(m: int, k: int, device="cpu", seed: int = 1) -> torch.Tensor:
    """N(0, 1) bfloat16 activations [m, k]."""
    return _normal((m, k), 1.0, _gen(device, seed), device)


def lora_pair(n: int, k: int, r: int, device="cpu", seed: int = 2):
    """(A [r, K] Kaiming-uniform, B [N, r] N(0, 0.01^2)), both bfloat16."""
    a = _kaiming_uniform((r, k), k, _gen(device, seed), device)
    b = _normal((n, r), B_STD, _gen(device, seed + 1), device)
    return a, b


# Llama-7B layer: q, k, v, o (4096 x 4096); gate, up (11008 x 4096); down (4096 x 11008)
LLAMA7B_LAYER = [(4096, 4096)] * 4 + [(11008, 4096)] * 2 + [(4096, 11008)]
# Llama-65B layer: q, k, v, o (8192 x 8192); gate, up (22016 x 8192); down (8192 x 22016)
LLAMA65B_LAYER = [(8192, 8192)] * 4 + [(22016, 8192)] * 2 + [(8192, 22016)]


def stack_seed(layer: int, matrix: int) -> int:
    """Seed of matrix ``matrix`` (0..6) of layer ``layer`` in a layer stack."""
    return 1000 + 7 * layer + matrix
