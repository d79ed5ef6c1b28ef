"""GPU parity: AdamW on the LoRA matrices (qlora_adamw_step), bit-exact against the oracle.

Three consecutive steps on a list of tensors in device memory (one launch per
step, sizes that split into several work items, a tensor of one element, an
empty tensor), then the same with the state in managed ("paged") memory from
cudaMallocManaged with the prefetch flag (glossary "QLoRA", "How QLoRA works":
paged optimizer state in unified memory).  A last test trains A and B for a few
steps through the whole path (forward, backward, AdamW) and checks the loss of
the LoRA branch goes down.
"""

import ctypes

import numpy as np
import pytest
import torch

import synthetic
from oracle import adamw

pytestmark = pytest.mark.gpu

HP = dict(lr=2e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
SIZES = [16 * 4096, 4096 * 16, 1, 0, 8192 * 3 + 5]


def _u32(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def test_adamw_device_tensors_three_steps(lib):
    rng = np.random.default_rng(0)
    host = [dict(p=rng.standard_normal(n).astype(np.float32), m=np.zeros(n, np.float32), v=np.zeros(n, np.float32))
            for n in SIZES]
    dev = [dict(master=torch.tensor(h["p"], device="cuda"), param=torch.empty(len(h["p"]), dtype=torch.bfloat16,
                                                                                device="cuda"),
                exp_avg=torch.zeros(len(h["p"]), device="cuda"), exp_avg_sq=torch.zeros(len(h["p"]), device="cuda"))
           for h in host]
    for step in (1, 2, 3):
        grads = [(rng.standard_normal(n) * 0.05).astype(np.float32) for n in SIZES]
        for d, g in zip(dev, grads):
            d["grad"] = torch.tensor(g, device="cuda")
        lib.adamw_step(dev, step=step, **HP)
        lib.check_status()
        for h, d, g in zip(host, dev, grads):
            h["p"], h["m"], h["v"], bits = adamw.adamw_step(h["p"], g, h["m"], h["v"], step=step, **HP)
            assert np.array_equal(_u32(d["master"].cpu().numpy()), _u32(h["p"]))
            assert np.array_equal(_u32(d["exp_avg"].cpu().numpy()), _u32(h["m"]))
            assert np.array_equal(_u32(d["exp_avg_sq"].cpu().numpy()), _u32(h["v"]))
            assert np.array_equal(d["param"].view(torch.int16).cpu().numpy().view(np.uint16), bits)


def test_adamw_paged_state(lib):
    """Master weights and moments in cudaMallocManaged memory (the host writes them, the GPU
    updates them after the prefetch, the host reads them back), gradients on the device."""
    n = 16 * 4096 + 3
    rng = np.random.default_rng(1)
    bufs = {k: lib.ManagedBuffer(4 * n) for k in ("master", "exp_avg", "exp_avg_sq")}
    views = {k: b.host_view(ctypes.c_float, n) for k, b in bufs.items()}
    p = rng.standard_normal(n).astype(np.float32)
    views["master"][:] = p
    views["exp_avg"][:] = 0
    views["exp_avg_sq"][:] = 0
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    try:
        for step in (1, 2):
            g = (rng.standard_normal(n) * 0.05).astype(np.float32)
            gd = torch.tensor(g, device="cuda")
            t = dict(master=bufs["master"], param=None, grad=gd, exp_avg=bufs["exp_avg"],
                     exp_avg_sq=bufs["exp_avg_sq"], numel=n)
            lib.adamw_step([t], step=step, prefetch=True, **HP)
            lib.check_status()
            torch.cuda.synchronize()
            p, m, v, _ = adamw.adamw_step(p, g, m, v, step=step, **HP)
            assert np.array_equal(_u32(views["master"]), _u32(p))
            assert np.array_equal(_u32(views["exp_avg"]), _u32(m))
            assert np.array_equal(_u32(views["exp_avg_sq"]), _u32(v))
    finally:
        torch.cuda.synchronize()
        for b in bufs.values():
            b.free()


def test_lora_training_steps_reduce_the_loss(lib):
    """Fit the LoRA branch to a target output through forward, backward and AdamW: the loss
    0.5 ||Y - Y*||^2 falls steadily (the LoRA matrices are the only trained parameters)."""
    n, k, m, r, alpha = 256, 512, 128, 8, 16.0
    case = synthetic.linear_case(n, k, m, r, alpha, device="cuda", base_seed=3)
    rec = lib.quantize(case.w)
    x = case.x
    target = lib.linear_fwd(x, rec, case.a, (case.b.float() * 30).to(torch.bfloat16), alpha)[0].float()
    a32, b32 = case.a.float().clone(), case.b.float().clone()
    a16, b16 = case.a.clone(), case.b.clone()
    state = [dict(master=a32, param=a16, exp_avg=torch.zeros_like(a32), exp_avg_sq=torch.zeros_like(a32)),
             dict(master=b32, param=b16, exp_avg=torch.zeros_like(b32), exp_avg_sq=torch.zeros_like(b32))]
    losses = []
    for step in range(1, 31):
        y, t = lib.linear_fwd(x, rec, a16, b16, alpha)
        dy = (y.float() - target)
        losses.append(0.5 * float((dy * dy).sum()))
        _, da, db = lib.linear_bwd(dy.to(torch.bfloat16), x, rec, a16, b16, alpha, t)
        state[0]["grad"], state[1]["grad"] = da, db
        lib.adamw_step(state, lr=5e-3, step=step)
    lib.check_status()
    assert losses[-1] < 0.3 * losses[0], losses
