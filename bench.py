#!/usr/bin/env python
"""Benchmark of the QLoRA NF4 linear hot path on one B300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--quick] [--full]

Headline (one JSON line on stdout, rank 0): fused forward + backward of the
Llama-7B attention projection -- W 4096x4096 NF4 + double quant, 2048 tokens,
LoRA r=16, alpha=32 -- in TFLOP/s (4MNK + 6Mr(N+K) algorithmic flops per
step), inputs resident in HBM, L2 flushed between steps, CUDA events on the
launching stream, max over ranks.  Also on the line:

* ``roofline``: the dominant kernel of the step, timed live with events
  around each of its launches, against the measured bf16 peak;
* ``e2e``: the same step through the public API with the inputs copied from
  pinned host memory and the LoRA gradients read back every step;
* ``cpu_baseline``: the float64 CPU oracle on a bounded sample of the workload;
* ``secondary``: the 32-layer Llama-7B decode sweep (weight GB/s at 1, 4, 16
  tokens; ``decode_per_layer`` is the decoder's dependency order, four calls a
  layer), dequantise and quantise GB/s, the Llama-7B MLP block fwd+bwd
  (``mlp_block``) and the 65B-shaped quantise stream + up-projection step
  (``llama65b``), each with its fraction of the measured roofline; the
  merge / export rate, the headline step with LoRA dropout p = 0.05, and one
  AdamW step over the LoRA matrices of a 32-layer 7B stack.

``--gpus N`` without a torchrun environment re-launches this script under
``torch.distributed.run`` with N ranks on 127.0.0.1 (one replica per GPU); under
torchrun, ``WORLD_SIZE`` must equal N.

``--impl reference`` times the CPU oracle (the reference for this build) on a
bounded sample of the same workload and prints the same line with
``"impl": "reference"``.

``--only quant [--shape NxK]`` / ``--only decode [--decode-layers L]
[--decode-tokens 1,4,16]`` / ``--only merge`` / ``--only smalltok [--tokens M]``
/ ``--only mlp`` / ``--only upproj65b`` run just that secondary measurement
(quantise + dequantise of one bf16 weight; the decode sweep; the merge of the
4096^2 projection; fwd+bwd at M <= 256 tokens; the Llama-7B MLP block; the
65B up-projection fwd+bwd without the 80-layer quantise) and print its figures
-- small, repeatable workloads for profilers, not bench lines.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "QLoRA NF4 linear fwd+bwd TFLOP/s; NF4 GEMV weight GB/s; % of roofline"
N_, K_, M_, R_, ALPHA_ = 4096, 4096, 2048, 16, 32.0
WORKLOAD = "Llama-7B attention projection: W 4096x4096 NF4+DQ, 2048 tokens (4 x 512), LoRA r=16 alpha=32, fwd+bwd"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def step_flops(m, n, k, r):
    return 4.0 * m * n * k + 6.0 * m * r * (n + k)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i] and "Not" not in r[5 + i]})
        loaded = [v for v in sm if mx and v > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ distributed
def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle leg
def oracle_sample(rows: int, seed_rows: int = 0):
    """Build the oracle inputs for a bounded sample of the headline workload (host only)."""
    import numpy as np

    import synthetic
    from oracle import nf4
    case = synthetic.linear_case(N_, K_, M_, R_, ALPHA_, device="cpu", base_seed=0)
    idx = np.random.default_rng(seed_rows).choice(M_, rows, replace=False)
    f = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
    rec = nf4.quantize(case.w.float().numpy(), N_, K_)
    return {"rec": rec, "x": f(case.x)[idx], "a": f(case.a), "b": f(case.b), "dy": f(case.dy)[idx]}


def oracle_step(s):
    """One oracle fwd+bwd on the sampled rows: dequantise W, forward, backward."""
    from oracle import linear, nf4
    rec = s["rec"]
    wd = nf4.dequantize(rec["codes"], rec["q"], rec["step"], rec["mu"], N_, K_)
    _, t = linear.lora_forward(s["x"], wd, s["a"], s["b"], ALPHA_, R_)
    linear.lora_backward(s["dy"], s["x"], wd, s["a"], s["b"], ALPHA_, R_, t)


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(budget_s: float = 12.0, rows: int = 256):
    s = oracle_sample(rows)
    flops = step_flops(rows, N_, K_, R_)
    oracle_step(s)  # warm
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle_step(s)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = (time.perf_counter() - t0) / n
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "sample": "float64 oracle fwd+bwd (dequantise the 4096x4096 NF4 record + LoRA linear forward and "
                      "backward) on %d of the 2048 token rows, %d repetitions, %.2f s each" % (rows, n, dt)}


def run_reference(args, world, rank):
    if rank != 0:
        return
    rows = args.ref_rows
    s = oracle_sample(rows)
    flops = step_flops(rows, N_, K_, R_)
    for _ in range(args.warmup):
        oracle_step(s)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(s)
    dt = (time.perf_counter() - t0) / args.steps
    val = flops / dt / 1e12
    cores = blas_threads()
    line = {"metric": METRIC, "value": val, "unit": "TFLOP/s", "impl": "reference", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "n": N_, "k": K_, "m": M_, "r": R_, "alpha": ALPHA_,
                       "sample_rows": rows},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": "float64 oracle fwd+bwd on %d of the 2048 token rows per step" % rows},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU legs
def time_events(torch, fn, steps, flush=None):
    """Per-step device time (ms) with events around fn only (flush outside)."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s, e in evs:
        if flush is not None:
            flush()
        s.record()
        fn()
        e.record()
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


def decode_sweep(q, torch, layers: int = 32, tokens=(1, 4, 16), passes: int = 10):
    """Weight GB/s of the Llama-7B decode stack at 1, 4 and 16 tokens.

    One pass = Y = X deq(W)^T + s (X A^T) B^T for all 7 x `layers` matrices, r=16, alpha=32.
    * ``grouped``: the whole stack as one qlora_linear_fwd_grouped call (independent inputs per matrix);
    * ``per_layer``: the dependency order of a decoder layer -- q,k,v | o | gate,up | down -- as four
      grouped calls per layer (128 calls per pass), captured in one CUDA graph;
    * ``per_matrix``: one qlora_linear_fwd call per matrix (224 calls), captured in one CUDA graph.
    """
    import synthetic
    shapes = synthetic.LLAMA7B_LAYER
    recs, loras = [], []
    for layer in range(layers):
        for mi, (n, k) in enumerate(shapes):
            w = synthetic.weight(n, k, device="cuda", seed=synthetic.stack_seed(layer, mi))
            recs.append(q.quantize(w))
            del w
            loras.append(synthetic.lora_pair(n, k, 16, device="cuda", seed=50_000 + 2 * (7 * layer + mi)))
    q.check_status()
    weight_bytes = sum(r.nbytes() for r in recs)
    lora_bytes = sum(a.numel() * 2 + b.numel() * 2 for a, b in loras)
    out = {"matrices": len(recs), "weight_bytes_per_pass": weight_bytes, "lora_bytes_per_pass": lora_bytes}
    stages = [(0, 3), (3, 4), (4, 6), (6, 7)]  # q,k,v | o | gate,up | down
    for t in tokens:
        xs = [synthetic.activations(t, r.k, device="cuda", seed=90_000 + i) for i, r in enumerate(recs)]
        ys = [torch.empty((t, r.n), dtype=torch.bfloat16, device="cuda") for r in recs]
        probs = [(xs[i], recs[i], loras[i][0], loras[i][1], 32.0, ys[i], None) for i in range(len(recs))]
        io_bytes = sum(x.numel() * 2 for x in xs) + sum(y.numel() * 2 for y in ys)
        res = {}
        # grouped: one call for the whole stack
        g_all = q.GroupedForward(probs)
        g_all.run()
        torch.cuda.synchronize()
        for _ in range(3):
            g_all.run()
        ms = statistics.median(time_events(torch, g_all.run, passes))
        res["grouped"] = {"ms_per_pass": ms, "weight_gbs": (weight_bytes + lora_bytes) / ms / 1e6, "launches": 2}
        # per layer: 4 dependent groups per layer
        groups = [q.GroupedForward(probs[7 * L + a:7 * L + b]) for L in range(layers) for (a, b) in stages]

        def per_layer():
            for g in groups:
                g.run()

        per_layer()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            per_layer()
        for _ in range(3):
            graph.replay()
        ms = statistics.median(time_events(torch, graph.replay, passes))
        res["per_layer"] = {"ms_per_pass": ms, "weight_gbs": (weight_bytes + lora_bytes) / ms / 1e6,
                            "launches": 2 * len(groups)}
        del graph
        # per matrix: one single-problem call each
        ts = [torch.empty((t, 16), dtype=torch.float32, device="cuda") for r in recs]
        wsb = max(q.fwd_workspace_bytes(t, r.n, r.k, 16) for r in recs)
        ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")

        def one_pass():
            for i, r in enumerate(recs):
                q.linear_fwd(xs[i], r, loras[i][0], loras[i][1], 32.0, y=ys[i], t_save=ts[i], workspace=ws)

        one_pass()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            one_pass()
        for _ in range(3):
            graph.replay()
        ms = statistics.median(time_events(torch, graph.replay, passes))
        res["per_matrix"] = {"ms_per_pass": ms, "weight_gbs": (weight_bytes + lora_bytes) / ms / 1e6}
        q.check_status()
        res["io_bytes_per_pass"] = io_bytes
        out["t%d" % t] = res
        del graph, xs, ys, ts, ws, g_all, groups
    del recs, loras
    torch.cuda.empty_cache()
    return out


def dequant_quant_rates(q, torch, flush, n=22016, k=8192):
    """Quantise / dequantise rates on one 22016x8192 matrix (the Llama-65B up-projection shape:
    360 MB of bf16 per call, so the per-launch overhead of a few microseconds does not dominate)."""
    import synthetic
    w = synthetic.weight(n, k, device="cuda", seed=2201)
    rec = q.quantize(w)
    q.check_status()
    out_b = torch.empty((n, k), dtype=torch.bfloat16, device="cuda")
    for _ in range(3):
        q.dequantize(rec, out=out_b)
    ms = statistics.median(time_events(torch, lambda: q.dequantize(rec, out=out_b), 10, flush))
    deq_bytes = rec.nbytes() + n * k * 2
    wsq = torch.empty(q.quantize_workspace_bytes(n, k), dtype=torch.uint8, device="cuda")
    rec2 = q.NF4Weight.empty(n, k)
    for _ in range(3):
        q.quantize(w, out=rec2, workspace=wsq)
    msq = statistics.median(time_events(torch, lambda: q.quantize(w, out=rec2, workspace=wsq), 10, flush))
    q.check_status()
    quant_bytes = n * k * 2 + rec.nbytes()
    del w, rec, rec2, out_b, wsq
    torch.cuda.empty_cache()
    return {"dequant": {"shape": [n, k], "ms": ms, "gbs": deq_bytes / ms / 1e6, "bytes": deq_bytes},
            "quantize": {"shape": [n, k], "ms": msq, "gbs": quant_bytes / msq / 1e6, "bytes": quant_bytes,
                         "kernels": 3}}


def mlp_block(q, torch, steps, flush, hidden=4096, inter=11008, m=2048, r=16, alpha=32.0):
    """Llama-7B MLP block fwd+bwd: gate/up [inter, hidden], down [hidden, inter], SiLU*up between
    (the gate and up forwards on two streams)."""
    import synthetic
    dev = "cuda"
    recs = [q.quantize(synthetic.weight(n, k, device=dev, seed=s)) for (n, k, s) in
            ((inter, hidden, 11), (inter, hidden, 12), (hidden, inter, 13))]
    loras = [synthetic.lora_pair(inter, hidden, r, device=dev, seed=21), synthetic.lora_pair(inter, hidden, r, device=dev, seed=23),
             synthetic.lora_pair(hidden, inter, r, device=dev, seed=25)]
    x = synthetic.activations(m, hidden, device=dev, seed=31)
    dy = synthetic.activations(m, hidden, device=dev, seed=32)
    bf = lambda *sh: torch.empty(sh, dtype=torch.bfloat16, device=dev)  # noqa: E731
    g, u, h, yv, dh, dg, du, dx = bf(m, inter), bf(m, inter), bf(m, inter), bf(m, hidden), bf(m, inter), bf(m, inter), \
        bf(m, inter), bf(m, hidden)
    ts = [torch.empty((m, r), dtype=torch.float32, device=dev) for _ in range(3)]
    das = [torch.empty((r, rec.k), dtype=torch.float32, device=dev) for rec in recs]
    dbs = [torch.empty((rec.n, r), dtype=torch.float32, device=dev) for rec in recs]
    wsf = torch.empty(max(q.fwd_workspace_bytes(m, rec.n, rec.k, r) for rec in recs) + 256, dtype=torch.uint8, device=dev)
    wsb = torch.empty(max(q.bwd_workspace_bytes(m, rec.n, rec.k, r) for rec in recs) + 256, dtype=torch.uint8, device=dev)
    # gate and up read the same X and are independent: the up forward runs on a second stream
    # (its own workspace), so its CTAs take the SMs the gate GEMM's last partial wave leaves idle
    s_up = torch.cuda.Stream()
    wsf_up = torch.empty_like(wsf)

    def fwd_bwd():
        main = torch.cuda.current_stream()
        s_up.wait_stream(main)
        q.linear_fwd(x, recs[0], *loras[0], alpha, y=g, t_save=ts[0], workspace=wsf)
        with torch.cuda.stream(s_up):
            q.linear_fwd(x, recs[1], *loras[1], alpha, y=u, t_save=ts[1], workspace=wsf_up)
        main.wait_stream(s_up)
        q.silu_mul_fwd(g, u, h)
        q.linear_fwd(h, recs[2], *loras[2], alpha, y=yv, t_save=ts[2], workspace=wsf)
        q.linear_bwd(dy, h, recs[2], *loras[2], alpha, ts[2], dx=dh, da=das[2], db=dbs[2], workspace=wsb)
        q.silu_mul_bwd(dh, g, u, dg, du)
        q.linear_bwd(dg, x, recs[0], *loras[0], alpha, ts[0], dx=dx, da=das[0], db=dbs[0], workspace=wsb)
        q.linear_bwd(du, x, recs[1], *loras[1], alpha, ts[1], dx=dx, da=das[1], db=dbs[1], workspace=wsb,
                     flags=q.ACCUM_DX)

    fwd_bwd()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fwd_bwd()
    for _ in range(3):
        if flush is not None:
            flush()
        graph.replay()
    ms = statistics.median(time_events(torch, graph.replay, steps, flush))
    q.check_status()
    flops = step_flops(m, inter, hidden, r) * 3
    return {"workload": "Llama-7B MLP block: gate/up 11008x4096, down 4096x11008, 2048 tokens, r=16, SiLU*up",
            "ms_per_step": ms, "tflops": flops / (ms / 1e3) / 1e12, "flops_per_step": flops}


def llama65b(q, torch, steps, flush, layers=80, m=4096, r=64, alpha=16.0):
    """Stream-quantise 80 Llama-65B-shaped layers (bf16 N(0, 0.02^2) made one matrix at a time), then
    fwd+bwd of one 22016x8192 up-projection at 4096 tokens, r=64."""
    import synthetic
    # the records (33 GB resident) and one workspace are allocated before the stream, so the
    # events bracket the quantiser's launches only, not the caching allocator's cudaMalloc calls
    shapes = [(n, k) for _ in range(layers) for (n, k) in synthetic.LLAMA65B_LAYER]
    recs = [q.NF4Weight.empty(n, k) for (n, k) in shapes]
    ws = torch.empty(max(q.quantize_workspace_bytes(n, k) for (n, k) in set(shapes)), dtype=torch.uint8,
                     device="cuda")
    wbuf = torch.empty(max(n * k for (n, k) in shapes), dtype=torch.bfloat16, device="cuda")
    qms = 0.0
    params = 0
    gen_ms = 0.0
    for i, (n, k) in enumerate(shapes):
        layer, mi = divmod(i, len(synthetic.LLAMA65B_LAYER))
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record()
        w = wbuf[: n * k].view(n, k)
        w.copy_(synthetic.weight(n, k, device="cuda", seed=synthetic.stack_seed(layer, mi)))
        e1.record()
        q.quantize(w, out=recs[i], workspace=ws)
        e2.record()
        e2.synchronize()
        gen_ms += e0.elapsed_time(e1)
        qms += e1.elapsed_time(e2)
        params += n * k
    del wbuf, ws
    q.check_status()
    resident = sum(rc.nbytes() for rc in recs)
    qbytes = 2 * params + resident
    out = {"layers": layers, "matrices": len(recs), "params": params, "resident_gb": resident / 1e9,
           "quantize_ms": qms, "quantize_gbs": qbytes / qms / 1e6, "weight_generation_ms_not_counted": gen_ms,
           "upproj_fwd_bwd": upproj_step(q, torch, steps, flush, recs[4], m=m, r=r, alpha=alpha)}
    del recs
    torch.cuda.empty_cache()
    return out


def upproj_step(q, torch, steps, flush, up=None, m=4096, r=64, alpha=16.0):
    """fwd+bwd of a Llama-65B up-projection (22016x8192 NF4 record `up`, quantised here when None)
    at m tokens, rank r, captured once in a CUDA graph and replayed."""
    import synthetic
    if up is None:
        up = q.quantize(synthetic.weight(22016, 8192, device="cuda", seed=synthetic.stack_seed(0, 4)))
    a, b = synthetic.lora_pair(up.n, up.k, r, device="cuda", seed=77)
    x = synthetic.activations(m, up.k, device="cuda", seed=78)
    dy = synthetic.activations(m, up.n, device="cuda", seed=79)
    y = torch.empty((m, up.n), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty((m, up.k), dtype=torch.bfloat16, device="cuda")
    t = torch.empty((m, r), dtype=torch.float32, device="cuda")
    da = torch.empty((r, up.k), dtype=torch.float32, device="cuda")
    db = torch.empty((up.n, r), dtype=torch.float32, device="cuda")
    wsf = torch.empty(q.fwd_workspace_bytes(m, up.n, up.k, r) + 256, dtype=torch.uint8, device="cuda")
    wsb = torch.empty(q.bwd_workspace_bytes(m, up.n, up.k, r) + 256, dtype=torch.uint8, device="cuda")

    def fwd_bwd():
        q.linear_fwd(x, up, a, b, alpha, y=y, t_save=t, workspace=wsf)
        q.linear_bwd(dy, x, up, a, b, alpha, t, dx=dx, da=da, db=db, workspace=wsb)

    fwd_bwd()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fwd_bwd()
    for _ in range(3):
        if flush is not None:
            flush()
        graph.replay()
    ms = statistics.median(time_events(torch, graph.replay, steps, flush))
    q.check_status()
    flops = step_flops(m, up.n, up.k, r)
    return {"n": up.n, "k": up.k, "m": m, "r": r, "alpha": alpha, "ms_per_step": ms,
            "tflops": flops / (ms / 1e3) / 1e12, "flops_per_step": flops}


def merge_rate(q, torch, flush, n=4096, k=4096, r=16, alpha=32.0):
    """Merge / export of the 4096^2 attention projection: bf16(deq(W) + s B A), GB/s of the weight
    record read and the bf16 weight written (HBM-bound; r float32 FMAs per weight on the CUDA cores)."""
    import synthetic
    case = synthetic.linear_case(n, k, 1, r, alpha, device="cuda", base_seed=4)
    rec = q.quantize(case.w)
    out = torch.empty((n, k), dtype=torch.bfloat16, device="cuda")
    for _ in range(3):
        q.merge(rec, case.a, case.b, alpha, out=out)
    ms = statistics.median(time_events(torch, lambda: q.merge(rec, case.a, case.b, alpha, out=out), 10, flush))
    q.check_status()
    byts = rec.nbytes() + n * k * 2 + case.a.numel() * 2 + case.b.numel() * 2
    return {"shape": [n, k], "r": r, "ms": ms, "gbs": byts / ms / 1e6, "bytes": byts}


def dropout_step(q, torch, steps, flush, p=0.05):
    """The headline fwd+bwd with LoRA dropout p = 0.05 on the branch input (mask drawn every step)."""
    import synthetic
    case = synthetic.linear_case(N_, K_, M_, R_, ALPHA_, device="cuda", base_seed=0)
    rec = q.quantize(case.w)
    x, a, b, dy = case.x, case.a, case.b, case.dy
    mask = torch.empty((M_, K_ // 8), dtype=torch.uint8, device="cuda")
    y = torch.empty((M_, N_), dtype=torch.bfloat16, device="cuda")
    xd = torch.empty_like(x)
    t = torch.empty((M_, R_), dtype=torch.float32, device="cuda")
    dx = torch.empty((M_, K_), dtype=torch.bfloat16, device="cuda")
    da = torch.empty((R_, K_), dtype=torch.float32, device="cuda")
    db = torch.empty((N_, R_), dtype=torch.float32, device="cuda")
    wsf = torch.empty(max(q.fwd_workspace_bytes(M_, N_, K_, R_), 256), dtype=torch.uint8, device="cuda")
    wsb = torch.empty(max(q.bwd_workspace_bytes(M_, N_, K_, R_), 256), dtype=torch.uint8, device="cuda")

    def fwd_bwd():
        q.dropout_mask(7, 11, M_, K_, p, out=mask)
        q.linear_fwd_dropout(x, rec, a, b, ALPHA_, mask, p, y=y, t_save=t, x_drop=xd, workspace=wsf)
        q.linear_bwd_dropout(dy, xd, rec, a, b, ALPHA_, mask, p, t, dx=dx, da=da, db=db, workspace=wsb)

    fwd_bwd()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fwd_bwd()
    for _ in range(3):
        if flush is not None:
            flush()
        graph.replay()
    ms = statistics.median(time_events(torch, graph.replay, steps, flush))
    q.check_status()
    flops = step_flops(M_, N_, K_, R_)
    return {"p": p, "ms_per_step": ms, "tflops": flops / (ms / 1e3) / 1e12}


def adamw_rate(q, torch, layers=32, r=16):
    """One AdamW step over the LoRA A and B of every linear of a 32-layer Llama-7B stack
    (448 tensors, 40 M parameters; one launch per 240 tensors)."""
    import synthetic
    ts = []
    for _ in range(layers):
        for (n, k) in synthetic.LLAMA7B_LAYER:
            for shape in ((r, k), (n, r)):
                nel = shape[0] * shape[1]
                ts.append({"master": torch.randn(nel, device="cuda"), "param": torch.empty(nel, dtype=torch.bfloat16,
                                                                                           device="cuda"),
                           "grad": torch.randn(nel, device="cuda") * 1e-3, "exp_avg": torch.zeros(nel, device="cuda"),
                           "exp_avg_sq": torch.zeros(nel, device="cuda")})
    params = sum(t["grad"].numel() for t in ts)
    step = [1]
    prepared = q.AdamwStep(ts)  # the tensor list is built once, as a training loop would

    def one():
        prepared.run(lr=1e-4, step=step[0])
        step[0] += 1

    for _ in range(3):
        one()
    ms = statistics.median(time_events(torch, one, 10))
    q.check_status()
    byts = params * (4 * 4 + 3 * 4 + 2)  # read master, grad, m, v; write master, m, v, bf16 param
    return {"tensors": len(ts), "params": params, "ms": ms, "gbs": byts / ms / 1e6}


def small_token_step(q, torch, m=128, n=4096, k=4096, r=16, alpha=32.0, steps=10):
    """fwd+bwd of the 4096^2 projection at m <= 256 tokens: the small-token GEMMs (k_qgemm_wa,
    k_qgemm_wb).  Returns ms per step and TFLOP/s (a profiler workload)."""
    import synthetic
    case = synthetic.linear_case(n, k, m, r, alpha, device="cuda", base_seed=6)
    rec = q.quantize(case.w)

    def step():
        y, t = q.linear_fwd(case.x, rec, case.a, case.b, alpha)
        q.linear_bwd(case.dy, case.x, rec, case.a, case.b, alpha, t)

    for _ in range(3):
        step()
    ms = statistics.median(time_events(torch, step, steps))
    q.check_status()
    return {"m": m, "n": n, "k": k, "r": r, "ms_per_step": ms,
            "tflops": step_flops(m, n, k, r) / (ms / 1e3) / 1e12}


def traffic_for(kernel: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if it matches the current source."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    import hashlib
    src = hashlib.sha1(open(os.path.join(ROOT, "bit_quantized_fine_nf4_b300", "csrc", "qgemm_pair.cu"), "rb").read())
    cur = src.hexdigest()[:12]
    for ln in open(p):
        parts = ln.split()
        if len(parts) >= 3 and parts[0] == kernel and parts[2] == cur:
            return float(parts[1])
    return None


def run_ours(args, world, rank, local):
    import torch

    import bit_quantized_fine_nf4_b300 as q
    import synthetic

    q.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks, peak_src = load_peaks()
    # -------------------------------------------------------------- workload (resident in HBM)
    case = synthetic.linear_case(N_, K_, M_, R_, ALPHA_, device="cuda", base_seed=0)
    rec = q.quantize(case.w)
    q.check_status()
    x, a, b, dy = case.x, case.a, case.b, case.dy
    y = torch.empty((M_, N_), dtype=torch.bfloat16, device=dev)
    t_save = torch.empty((M_, R_), dtype=torch.float32, device=dev)
    dx = torch.empty((M_, K_), dtype=torch.bfloat16, device=dev)
    da = torch.empty((R_, K_), dtype=torch.float32, device=dev)
    db = torch.empty((N_, R_), dtype=torch.float32, device=dev)
    ws_f = torch.empty(max(q.fwd_workspace_bytes(M_, N_, K_, R_), 256), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(max(q.bwd_workspace_bytes(M_, N_, K_, R_), 256), dtype=torch.uint8, device=dev)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # > 126 MB L2

    def flush():
        flush_buf.zero_()

    def allreduce_grads():
        if world > 1:
            from bit_quantized_fine_nf4_b300.dp import allreduce_lora_grads
            allreduce_lora_grads(da, db)

    def fwd_bwd():
        q.linear_fwd(x, rec, a, b, ALPHA_, y=y, t_save=t_save, workspace=ws_f)
        q.linear_bwd(dy, x, rec, a, b, ALPHA_, t_save, dx=dx, da=da, db=db, workspace=ws_b)

    def eager_step():
        fwd_bwd()
        allreduce_grads()

    flops = step_flops(M_, N_, K_, R_)
    for _ in range(args.warmup):
        flush()
        eager_step()
    torch.cuda.synchronize()
    q.check_status()

    # One fwd+bwd captured in a CUDA graph: the same library calls, replayed
    # without per-call host work.  The dA/dB all-reduce (N > 1) stays eager.
    l0 = q.launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fwd_bwd()
    kernels_per_step = q.launch_count() - l0

    def graph_step():
        graph.replay()
        allreduce_grads()

    step = graph_step if not args.eager else eager_step
    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    q.check_status()

    # -------------------------------------------------------------- headline timed region
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    l0 = q.launch_count()
    ms = time_events(torch, step, args.steps, flush)
    launches = (q.launch_count() - l0) if args.eager else kernels_per_step * args.steps
    barrier(world)
    clk = clocks.stop()
    q.check_status()
    ms_step = allreduce_max(sum(ms) / len(ms), world)
    value = flops * world / (ms_step / 1e3) / 1e12

    # eager calls (host launch work in the loop), for reference
    eager_ms = time_events(torch, eager_step, args.steps, flush)
    eager_ms_step = allreduce_max(sum(eager_ms) / len(eager_ms), world)

    # -------------------------------------------------------------- roofline of the dominant kernel
    # eager launches, each bracketed by events; a GPU sleep before each step lets
    # the host queue the whole step first so no submission latency lands inside.
    def padded_flush():
        flush()
        torch.cuda._sleep(2_000_000)

    q.profile_reset()
    q.profile_enable(True)
    time_events(torch, eager_step, args.steps, padded_flush)
    q.profile_enable(False)
    prof = q.profile_read()
    q.check_status()
    kflops = {
        "fwd_gemm": 2.0 * M_ * N_ * K_ + 2.0 * M_ * R_ * N_,
        "bwd_dx_gemm": 2.0 * M_ * N_ * K_ + 2.0 * M_ * R_ * K_,
    }
    # the dominant kernel is the larger GEMM (the LoRA side kernels run beside the GEMMs on the
    # SMs they leave idle, so their isolated time is not on the step's critical path)
    gemms = {k: v for k, v in prof.items() if k in kflops}
    dominant = max(gemms.items(), key=lambda kv: kv[1][0])[0] if gemms else None
    roof = None
    if dominant in kflops:
        tot_ms, calls = prof[dominant]
        avg = tot_ms / calls
        ach = kflops[dominant] / (avg / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": dominant, "achieved": ach, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"], "traffic": traffic_for(dominant),
                "peak_source": peak_src + " bf16 burst (kernel timed inside a sub-millisecond step)",
                "avg_launch_ms": avg, "flops_per_launch": kflops[dominant]}
    shares = {k: {"ms_per_step": v[0] / args.steps, "share": v[0] / sum(t for t, _ in prof.values())}
              for k, v in prof.items()} if prof else {}
    for k, kf in kflops.items():
        if k in prof:
            tot, c = prof[k]
            shares[k]["tflops"] = kf / (tot / c / 1e3) / 1e12

    # -------------------------------------------------------------- end to end (host buffers)
    x_h = x.cpu().pin_memory()
    dy_h = dy.cpu().pin_memory()
    da_h = torch.empty(da.shape, dtype=da.dtype).pin_memory()
    db_h = torch.empty(db.shape, dtype=db.dtype).pin_memory()

    def e2e_step():
        # the library's copy call: each copy cut into >= 2 MB pieces over four copy streams
        q.copy_many([(x, x_h), (dy, dy_h)])
        step()
        q.copy_many([(da_h, da), (db_h, db)])

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = time_events(torch, e2e_step, args.steps, flush)
    e2e_step_ms = allreduce_max(sum(e2e_ms) / len(e2e_ms), world)
    e2e = {"value": flops * world / (e2e_step_ms / 1e3) / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": x.numel() * 2 + dy.numel() * 2, "d2h_bytes_per_step": da.numel() * 4 + db.numel() * 4,
           "ms_per_step": e2e_step_ms}

    # -------------------------------------------------------------- secondary figures
    secondary = {"kernel_shares": shares,
                 "eager_calls": {"ms_per_step": eager_ms_step,
                                 "tflops": flops * world / (eager_ms_step / 1e3) / 1e12},
                 "kernels_per_step": kernels_per_step}
    if not args.quick:
        secondary.update(dequant_quant_rates(q, torch, flush))
        del y, dx
        torch.cuda.empty_cache()
        sweep = decode_sweep(q, torch, layers=args.decode_layers)
        for t in (1, 4, 16):
            for mode in ("grouped", "per_layer", "per_matrix"):
                d = sweep.get("t%d" % t, {}).get(mode)
                if d:
                    d["frac_of_hbm"] = d["weight_gbs"] / peaks["hbm_gbs"]
        secondary["decode_sweep"] = sweep
        secondary["dequant"]["frac_of_hbm"] = secondary["dequant"]["gbs"] / peaks["hbm_gbs"]
        secondary["quantize"]["frac_of_hbm"] = secondary["quantize"]["gbs"] / peaks["hbm_gbs"]
    if not args.quick:
        secondary["decode_per_layer"] = {
            "t%d" % t: {"weight_gbs": sweep["t%d" % t]["per_layer"]["weight_gbs"],
                        "frac_of_hbm": sweep["t%d" % t]["per_layer"]["frac_of_hbm"],
                        "ms_per_pass": sweep["t%d" % t]["per_layer"]["ms_per_pass"]}
            for t in (1, 4, 16) if "t%d" % t in sweep}
        secondary["merge"] = merge_rate(q, torch, flush)
        secondary["merge"]["frac_of_hbm"] = secondary["merge"]["gbs"] / peaks["hbm_gbs"]
        secondary["dropout_step"] = dropout_step(q, torch, args.steps, flush)
        secondary["adamw"] = adamw_rate(q, torch)
        cs = ClockSampler(local)
        cs.start()
        secondary["mlp_block"] = mlp_block(q, torch, args.steps, flush)
        secondary["mlp_block"]["clocks"] = cs.stop()
        secondary["mlp_block"]["frac_of_bf16_peak"] = secondary["mlp_block"]["tflops"] / peaks["bf16_tflops"]
        cs = ClockSampler(local)
        cs.start()
        secondary["llama65b"] = llama65b(q, torch, max(3, args.steps // 4), flush)
        secondary["llama65b"]["clocks"] = cs.stop()
        secondary["llama65b"]["quantize_frac_of_hbm"] = secondary["llama65b"]["quantize_gbs"] / peaks["hbm_gbs"]
        secondary["llama65b"]["upproj_fwd_bwd"]["frac_of_bf16_peak"] = (
            secondary["llama65b"]["upproj_fwd_bwd"]["tflops"] / peaks["bf16_tflops"])

    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "n": N_, "k": K_, "m": M_, "r": R_, "alpha": ALPHA_,
                       "weights": "nf4 + double-quant (block 64, dq group 256)",
                       "launch": "eager library calls" if args.eager else
                                 "library calls captured once in a CUDA graph, replayed per step",
                       "l2": "flushed between steps (256 MB write outside the timed events)",
                       "parallelism": "dp%d (replica per GPU, all-reduce of dA/dB)" % world},
            "roofline": roof, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
            "frac_of_bf16_peak": value / world / peaks["bf16_tflops"], "secondary": secondary}
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)


def relaunch_under_torchrun(n: int, argv) -> int:
    """Run this script as n ranks (one per GPU) under torch.distributed.run on 127.0.0.1."""
    import socket
    sk = socket.socket()
    sk.bind(("127.0.0.1", 0))
    port = sk.getsockname()[1]
    sk.close()
    args = list(sys.argv[1:] if argv is None else argv)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(n),
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *args]
    return subprocess.call(cmd)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--quick", action="store_true", help="headline only (no decode sweep / dequant rates)")
    ap.add_argument("--eager", action="store_true", help="time eager library calls instead of the graph replay")
    ap.add_argument("--full", action="store_true", help="(kept for old command lines: the MLP block and the 65B "
                                                        "leg are part of the default run)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=128)
    ap.add_argument("--decode-layers", type=int, default=32)
    ap.add_argument("--decode-tokens", default="1", help="token counts of --only decode, e.g. 1,4,16")
    ap.add_argument("--tokens", type=int, default=128, help="tokens of --only smalltok (<= 256: small-token GEMMs)")
    ap.add_argument("--only", choices=("quant", "decode", "merge", "smalltok", "adamw", "dropout", "mlp", "upproj65b"),
                    default=None,
                    help="run one secondary measurement alone (a workload for profilers)")
    ap.add_argument("--shape", default="22016x8192", help="weight shape for --only quant")
    args = ap.parse_args(argv)
    if args.only:
        import torch
        import bit_quantized_fine_nf4_b300 as q
        q.load()
        if args.only == "quant":
            n, k = (int(v) for v in args.shape.lower().split("x"))
            print(json.dumps(dequant_quant_rates(q, torch, None, n=n, k=k)), flush=True)
        elif args.only == "merge":
            print(json.dumps(merge_rate(q, torch, None)), flush=True)
        elif args.only == "adamw":
            print(json.dumps(adamw_rate(q, torch)), flush=True)
        elif args.only == "dropout":
            print(json.dumps(dropout_step(q, torch, args.steps, None)), flush=True)
        elif args.only == "smalltok":
            print(json.dumps(small_token_step(q, torch, m=args.tokens)), flush=True)
        elif args.only == "mlp":
            print(json.dumps(mlp_block(q, torch, args.steps, None)), flush=True)
        elif args.only == "upproj65b":
            print(json.dumps(upproj_step(q, torch, args.steps, None)), flush=True)
        else:
            toks = tuple(int(t) for t in args.decode_tokens.split(","))
            print(json.dumps(decode_sweep(q, torch, layers=args.decode_layers, tokens=toks)), flush=True)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return
    env_world = os.environ.get("WORLD_SIZE")
    if env_world is None and args.gpus > 1:
        sys.exit(relaunch_under_torchrun(args.gpus, argv))
    if env_world is not None and int(env_world) != args.gpus:
        sys.stderr.write("bench.py: --gpus %d but WORLD_SIZE=%s\n" % (args.gpus, env_world))
        sys.exit(2)
    world, rank, local = dist_setup(args)
    run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
