"""Data-parallel LoRA gradient exchange on two gloo ranks (CPU, no GPU).

Each rank takes its token shard of one problem, computes its dA/dB with the
float64 oracle, and the exchange must give exactly the single-process
gradients of the whole batch (backprop is a sum over tokens).
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from bit_quantized_fine_nf4_b300.dp import allreduce_lora_grads, shard_tokens


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _problem():
    rng = np.random.default_rng(0)
    m, n, k, r = 37, 48, 64, 8
    x = rng.standard_normal((m, k))
    w = rng.standard_normal((n, k)) * 0.02
    a = rng.standard_normal((r, k)) / 8
    b = rng.standard_normal((n, r)) * 0.01
    dy = rng.standard_normal((m, n))
    return x, w, a, b, dy, 16.0, r


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import linear
    x, w, a, b, dy, alpha, r = _problem()
    sl = shard_tokens(x.shape[0], rank, world)
    _, da, db, _ = linear.lora_backward(dy[sl], x[sl], w, a, b, alpha, r)
    tda, tdb = torch.from_numpy(da.copy()), torch.from_numpy(db.copy())
    allreduce_lora_grads(tda, tdb)
    out[rank] = (tda.numpy(), tdb.numpy())
    dist.destroy_process_group()


def test_shard_tokens_covers_all():
    for m in (1, 7, 37, 2048):
        for world in (1, 2, 3, 8):
            idx = []
            for rk in range(world):
                s = shard_tokens(m, rk, world)
                idx.extend(range(s.start, s.stop))
            assert idx == list(range(m))


@pytest.mark.timeout(120)
def test_two_rank_allreduce_matches_single_process():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    from oracle import linear
    x, w, a, b, dy, alpha, r = _problem()
    _, da, db, _ = linear.lora_backward(dy, x, w, a, b, alpha, r)
    for rank in range(world):
        gda, gdb = out[rank]
        assert np.allclose(gda, da, rtol=1e-12, atol=1e-14)
        assert np.allclose(gdb, db, rtol=1e-12, atol=1e-14)
