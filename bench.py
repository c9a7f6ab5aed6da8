"""Throughput of the fused top-K forward-KL loss (forward + backward) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config I] [--chunk C]
                    [--impl fused|reference] [--no-cpu-baseline] [--no-e2e]

One step = fkl_forward + fkl_backward over one batch of synthetic tokens of the
chosen workload (default: the gpt-oss-20b-like long-context loss, N=32768,
d=2880, V=201088, K=100, T=1).  Inputs are resident in HBM before the timed
region; W (1.16 GB) alone is larger than L2, so no flush is needed.  Under
torchrun (N > 1) every rank runs an independent replica of the same workload on
its own GPU: the loss has no exchange step on one GPU per problem, so the job's
value is the tokens of all ranks over the slowest rank's time.

`--impl reference` times the plain C++ fp64 CPU oracle instead, on a bounded row
sample of the same workload per step (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused top-K KL fwd+bwd tokens/s at V=201088; % of bf16 tensor peak; peak GB"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}

# DRAM bytes (read + write) per launch of the dominant kernel at the default
# gpt-oss-20b-like workload: dram__bytes_read.sum + dram__bytes_write.sum from a
# one-pass ncu capture of the same kernel on a two-chunk case with V = 32768,
# averaged over its store and reduce-add launches as a full step mixes them and
# scaled to V = 201088 by the vocabulary rows processed.  Keyed by the digest of
# the kernel sources the capture ran; after any change of them the figure is
# stale and the line reports null.
TRAFFIC = {("bwd_gemm_dw", "1c905e1d5c98"): 5.92e9}


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except OSError:
        return FALLBACK_PEAKS, "fallback"


def kernel_digest():
    """Hash of the GEMM kernels' code (gemm_tc.cu, ptx.cuh, fkl_internal.h) with
    comments and blank lines removed, so that only a change of code retires
    counters taken on an earlier build."""
    import re
    m = hashlib.sha256()
    for f in ("gemm_tc.cu", "ptx.cuh", "fkl_internal.h"):
        with open(os.path.join(ROOT, "lm_head_kl_fkl_b300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        m.update("\n".join(l.strip() for l in src.splitlines() if l.strip()).encode())
    return m.hexdigest()[:12]


def slowest_ms(ms, world, device):
    """The slowest rank's time: each rank's number max-reduced (identity on one rank)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank, world, steps, ms):
    """Whole-job tokens/s: the tokens of every replica over the slowest rank's time."""
    return tokens_per_rank * world * steps / (ms / 1e3)


def per_kernel(prof, steps):
    """{kernel: ms per step, TFLOP/s where the kernel does tensor work} from profile_read()."""
    out = {}
    for k, (ms, n, fl) in prof.items():
        out[k] = {"ms_per_step": ms / steps, "launches": n}
        if fl > 0:
            out[k]["tflops"] = fl / (ms / 1e3) / 1e12
    return out


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "power_w": statistics.median(pw) if pw else None, "reasons": sorted(reasons)}


def threads_used():
    """Threads the C++ oracle runs on (it splits rows / vocabulary rows over them)."""
    from oracle import cpp
    return cpp.threads()


def oracle_step_on_sample(x, rows, Wf):
    """One forward + backward of the plain C++ fp64 oracle (as it stands, all host
    cores) over a row sample: the sampled rows form the batch, every row with the
    full vocabulary and hidden size."""
    from oracle import cpp
    from lm_head_kl_fkl_b300 import synth
    orc = cpp.load()
    hs = synth.bf16_bits_to_f64(x["h"][rows])
    f = orc.forward(hs, Wf, x["idx"][rows], x["t"][rows], x["mask"][rows], x["T"])
    g = orc.backward(hs, Wf, x["idx"][rows], x["t"][rows], x["mask"][rows], x["T"])
    return f, g


def cpu_baseline(x, budget_s=12.0, max_rows=1024):
    """Oracle tokens/s on a bounded sample of the workload's rows (fp64, host cores)."""
    from lm_head_kl_fkl_b300 import synth
    Wf = synth.bf16_bits_to_f64(x["W"])
    rng = np.random.default_rng(1)
    probe = min(x["N"], max(8, threads_used()))  # one row per worker thread
    rows = np.sort(rng.choice(x["N"], probe, replace=False))
    t0 = time.perf_counter()
    oracle_step_on_sample(x, rows, Wf)
    per_row = (time.perf_counter() - t0) / len(rows)
    n = int(min(max_rows, x["N"], max(probe, budget_s / max(per_row, 1e-6))))
    rows = np.sort(rng.choice(x["N"], n, replace=False))
    t0 = time.perf_counter()
    oracle_step_on_sample(x, rows, Wf)
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "tokens/s", "cores": threads_used(), "kind": "oracle",
            "sample": f"{n} seeded rows of the {x['name']} workload (full d and V) as one batch, "
                      f"plain C++ fp64 oracle forward + backward, {dt:.1f} s"}


def workload(cfg, shape=None):
    """Inputs of a named workload, or of a custom (N, d, V, K) with that workload's generators."""
    import dataclasses
    from lm_head_kl_fkl_b300 import synth
    c = synth.CONFIGS[cfg]
    if shape is None:
        return synth.config_inputs(cfg), c
    N, d, V, K = shape
    c = dataclasses.replace(c, name=f"{c.name}-shape-N{N}-d{d}-V{V}-K{K}", N=N, d=d, V=V, K=K)
    x = synth.make_inputs(N, d, V, K, c.T, c.pad_frac, c.index, synth.config_seed(cfg))
    x["name"] = c.name
    return x, c


def config_dict(c, chunk, world):
    return {"workload": f"{c.name} fused top-K KL loss", "N": c.N, "d": c.d, "V": c.V, "K": c.K,
            "T": c.T, "pad_frac": c.pad_frac, "teacher_ids": c.index, "chunk": chunk or "default",
            "global_batch": c.N * world, "l2": "no flush: W (bf16 V x d) alone exceeds the 126 MB L2",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def memory_stress(api, dev, stream, chunk, steps):
    """Forward + backward of the gpt-oss-120b-like memory-stress workload (N = 131072,
    d = 2880, V = 201088, K = 100): time per step and peak device memory, against
    what the inputs and the gradients alone occupy."""
    import torch
    from lm_head_kl_fkl_b300 import synth
    c = synth.CONFIGS[4]
    x = synth.config_inputs(4)
    N, d, V, K, T = c.N, c.d, c.V, c.K, c.T
    torch.cuda.reset_peak_memory_stats(dev)
    base0 = torch.cuda.memory_allocated(dev)
    h = torch.from_numpy(x["h"].view(np.int16)).view(torch.bfloat16).to(dev)
    W = torch.from_numpy(x["W"].view(np.int16)).view(torch.bfloat16).to(dev)
    idx, t, mask = (torch.from_numpy(x[k]).to(dev) for k in ("idx", "t", "mask"))
    del x
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    dh = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    dW = torch.empty((V, d), dtype=torch.float32, device=dev)
    io = torch.cuda.memory_allocated(dev) - base0
    ws = api.alloc_workspace(N, d, V, K, chunk, dev)

    def step():
        api.forward(h, W, idx, t, mask, T, chunk, ws=ws, loss=loss, lse=lse)
        api.backward(h, W, idx, t, mask, T, lse, chunk=chunk, ws=ws, dh=dh, dW=dW)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    peak = torch.cuda.max_memory_allocated(dev) - base0
    status = api.get_status(ws)
    out = {"workload": f"{c.name} fused top-K KL loss", "N": N, "d": d, "V": V, "K": K, "steps": steps,
           "ms_per_step": ms, "value": N / (ms / 1e3), "unit": "tokens/s",
           "tflops": 8.0 * N * d * V / (ms / 1e3) / 1e12,
           "peak_mem_gb": peak / 1e9, "inputs_and_grads_gb": io / 1e9, "workspace_gb": ws.numel() / 1e9,
           "peak_beyond_inputs_and_grads_gb": (peak - io) / 1e9, "device_status": status}
    del h, W, idx, t, mask, loss, lse, dh, dW, ws
    torch.cuda.empty_cache()
    return out


def dominant_roofline(prof, peaks, peaks_kind):
    """The tensor-core kernel with the largest share of the recorded time: its
    algorithmic FLOP per launch over its mean CUDA-event launch time, against the
    sustained measured bf16 peak (the kernels run inside a long power-capped step)."""
    gemms = {k: v for k, v in prof.items() if v[2] > 0}
    if not gemms:
        return None
    dom = max(gemms, key=lambda k: gemms[k][0])
    tot_ms, n_l, fl = gemms[dom]
    achieved = fl / (tot_ms / 1e3) / 1e12
    peak = peaks["bf16_tflops_sustained"]
    return {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "peak_kind": f"bf16 dense, sustained, {peaks_kind}",
            "flop_per_launch": fl / n_l, "launch_ms": tot_ms / n_l, "launches": n_l}


def kernel_table(prof):
    total = max(1e-9, sum(p[0] for p in prof.values()))
    return {k: {"ms_total": v[0], "launches": v[1], "share": v[0] / total,
                **({"tflops": v[2] / (v[0] / 1e3) / 1e12} if v[2] > 0 else {})}
            for k, v in prof.items()}


def config_leg(api, cfg, dev, stream, chunk, steps, warmup, peaks, peaks_kind, with_cpu):
    """fkl_forward + fkl_backward on another named workload (inputs resident in HBM,
    L2 flushed before each step): mean time per step, tokens/s, TFLOP/s (8 N d V),
    the per-kernel list and its dominant kernel's roofline, next to the C++ oracle on
    a bounded row sample."""
    import torch
    from lm_head_kl_fkl_b300 import synth
    c = synth.CONFIGS[cfg]
    x = synth.config_inputs(cfg)
    N, d, V, K, T = c.N, c.d, c.V, c.K, c.T
    h = torch.from_numpy(x["h"].view(np.int16)).view(torch.bfloat16).to(dev)
    W = torch.from_numpy(x["W"].view(np.int16)).view(torch.bfloat16).to(dev)
    idx, t, mask = (torch.from_numpy(x[k]).to(dev) for k in ("idx", "t", "mask"))
    ws = api.alloc_workspace(N, d, V, K, chunk, dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    dh = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    dW = torch.empty((V, d), dtype=torch.float32, device=dev)

    def step():
        api.forward(h, W, idx, t, mask, T, chunk, ws=ws, loss=loss, lse=lse)
        api.backward(h, W, idx, t, mask, T, lse, chunk=chunk, ws=ws, dh=dh, dW=dW)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    # each step timed on its own, after a 256 MB write that evicts the 126 MB L2 (the
    # smaller workloads' inputs would otherwise stay L2-resident between steps)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    api.profile_reset()
    with ClockSampler(dev.index or 0) as clk:
        for e0, e1 in events:
            flush.zero_()
            api.profile_enable(True)
            e0.record(stream)
            step()
            e1.record(stream)
            api.profile_enable(False)
        torch.cuda.synchronize()
    prof = api.profile_read()
    ms = sum(e0.elapsed_time(e1) for e0, e1 in events) / steps
    del flush
    tflops = 8.0 * N * d * V / (ms / 1e3) / 1e12
    out = {"workload": f"{c.name} fused top-K KL loss", "N": N, "d": d, "V": V, "K": K, "T": T,
           "chunk": chunk or "default", "steps": steps, "warmup": warmup, "ms_per_step": ms,
           "value": N / (ms / 1e3), "unit": "tokens/s", "tflops": tflops,
           "frac_of_bf16_peak": {"burst": tflops / peaks["bf16_tflops"],
                                 "sustained": tflops / peaks["bf16_tflops_sustained"], "kind": peaks_kind},
           "roofline": dominant_roofline(prof, peaks, peaks_kind), "kernels": kernel_table(prof),
           "clocks": clk.summary(), "device_status": api.get_status(ws),
           "l2": "inputs resident in HBM; L2 flushed (256 MB write) before each timed step, outside its events"}
    del h, W, idx, t, mask, ws, loss, lse, dh, dW
    torch.cuda.empty_cache()
    if with_cpu:
        out["cpu_baseline"] = cpu_baseline(x, budget_s=6.0)
    return out


def dense_kl_step(h, W, idx, tlogit, mask, T):
    """The dense method the pages compare the fused loss with: the full N x V logits
    materialised (bf16 matmul, fp32 softmax over the vocabulary), the same top-K
    forward KL, and autograd's backward through it.  A measurement baseline in plain
    torch ops, not the library's path.  Returns (loss, dh, dW)."""
    import torch
    hh = h.detach().requires_grad_(True)
    WW = W.detach().requires_grad_(True)
    logq = torch.log_softmax((hh @ WW.t()).float() / T, dim=1)          # [N, V]
    u = tlogit / T
    finite = torch.isfinite(u)
    logp = torch.log_softmax(torch.where(finite, u, torch.full_like(u, -float("inf"))), dim=1)
    p = torch.where(finite, logp.exp(), torch.zeros_like(u))
    plogp = torch.where(p > 0, p * logp, torch.zeros_like(u))
    kl = (plogp - p * logq.gather(1, idx.long())).sum(dim=1)
    valid = finite.any(dim=1)
    if mask is not None:
        valid = valid & (mask != 0)
    n_valid = valid.sum()
    loss = (T * T) * torch.where(valid, kl, torch.zeros_like(kl)).sum() / n_valid.clamp(min=1)
    loss.backward()
    return loss.detach(), hh.grad, WW.grad


def dense_baseline(cfg, dev, steps=2):
    """Peak device memory and time per step of dense_kl_step on a named workload."""
    import torch
    from lm_head_kl_fkl_b300 import synth
    c = synth.CONFIGS[cfg]
    x = synth.config_inputs(cfg)
    h = torch.from_numpy(x["h"].view(np.int16)).view(torch.bfloat16).to(dev)
    W = torch.from_numpy(x["W"].view(np.int16)).view(torch.bfloat16).to(dev)
    idx, t, mask = (torch.from_numpy(x[k]).to(dev) for k in ("idx", "t", "mask"))
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    try:
        dense_kl_step(h, W, idx, t, mask, c.T)  # warm-up (cuBLAS workspaces, allocator)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            loss, dh, dW = dense_kl_step(h, W, idx, t, mask, c.T)
            del dh, dW
        e1.record()
        torch.cuda.synchronize()
        out = {"workload": c.name, "N": c.N, "V": c.V, "d": c.d, "ms_per_step": e0.elapsed_time(e1) / steps,
               "tokens_per_s": c.N / (e0.elapsed_time(e1) / steps / 1e3), "loss": float(loss.item()),
               "peak_beyond_inputs_gb": (torch.cuda.max_memory_allocated(dev) - base) / 1e9}
    except torch.cuda.OutOfMemoryError as e:
        out = {"workload": c.name, "N": c.N, "V": c.V, "d": c.d, "out_of_memory": str(e).splitlines()[0]}
    del h, W, idx, t, mask
    torch.cuda.empty_cache()
    return out


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    x, c = workload(args.config, args.shape)
    from lm_head_kl_fkl_b300 import synth
    Wf = synth.bf16_bits_to_f64(x["W"])
    rng = np.random.default_rng(2)
    n = args.ref_rows
    times = []
    for i in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(x["N"], n, replace=False))
        t0 = time.perf_counter()
        oracle_step_on_sample(x, rows, Wf)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    sec = sum(times) / len(times)
    value = n / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(c, args.chunk, 1),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads_used(),
                             "kind": "oracle",
                             "sample": f"{n} seeded rows per step of the {c.name} workload (full d and V) as "
                                       f"one batch, plain C++ fp64 oracle forward + backward"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_fused(args):
    import torch
    import torch.distributed as dist
    from lm_head_kl_fkl_b300 import api

    rank, local_rank, world = dist_env()
    if world > 1:
        torch.cuda.set_device(local_rank)  # bind the rank's GPU before NCCL comes up
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    x, c = workload(args.config, args.shape)
    N, d, V, K, T = c.N, c.d, c.V, c.K, c.T
    stream = torch.cuda.current_stream(dev)

    def dev_tensor(a, dtype=None):
        t = torch.from_numpy(a)
        return (t.view(dtype) if dtype is not None else t).to(dev)

    h = dev_tensor(x["h"].view(np.int16), torch.bfloat16)
    W = dev_tensor(x["W"].view(np.int16), torch.bfloat16)
    idx, t, mask = dev_tensor(x["idx"]), dev_tensor(x["t"]), dev_tensor(x["mask"])
    ws = api.alloc_workspace(N, d, V, K, args.chunk, dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    dh = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    dW = torch.empty((V, d), dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    base_mem = torch.cuda.memory_allocated(dev)

    def step():
        api.forward(h, W, idx, t, mask, T, args.chunk, ws=ws, loss=loss, lse=lse)
        api.backward(h, W, idx, t, mask, T, lse, chunk=args.chunk, ws=ws, dh=dh, dW=dW)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if api.get_status(ws) != 0:
        raise RuntimeError(f"device status {api.get_status(ws)} after warm-up")

    # ---- timed region: device-resident inputs
    api.profile_reset()
    api.profile_enable(True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = api.launch_count()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    api.profile_enable(False)
    launches = api.launch_count() - launches0
    ms = ev0.elapsed_time(ev1)
    prof = api.profile_read()
    ms = slowest_ms(ms, world, dev)
    peak_mem = torch.cuda.max_memory_allocated(dev)
    status = api.get_status(ws)
    ms_per_step = ms / args.steps
    tokens = N * world * args.steps
    value = job_throughput(N, world, args.steps, ms)
    flop_step = 8.0 * N * d * V
    tflops = flop_step / (ms_per_step / 1e3) / 1e12

    peaks, peaks_kind = load_peaks()
    roofline = dominant_roofline(prof, peaks, peaks_kind)
    if roofline:
        roofline["traffic"] = (TRAFFIC.get((roofline["kernel"], kernel_digest()))
                               if args.config == 3 and args.shape is None and not args.chunk else None)
    kernels = kernel_table(prof)

    # ---- the same step through fkl_forward_backward (one call, logits kept per chunk)
    variants = None
    if not args.no_variants:
        def step_fb():
            api.forward_backward(h, W, idx, t, mask, T, chunk=args.chunk, ws=ws, loss=loss, lse=lse, dh=dh, dW=dW)

        for _ in range(args.warmup):
            step_fb()
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        api.profile_reset()
        api.profile_enable(True)
        f0.record(stream)
        for _ in range(args.steps):
            step_fb()
        f1.record(stream)
        torch.cuda.synchronize()
        api.profile_enable(False)
        fb_kernels = per_kernel(api.profile_read(), args.steps)
        fms = slowest_ms(f0.elapsed_time(f1), world, dev)
        fstep = fms / args.steps
        variants = {"forward_backward_one_call": {
            "value": job_throughput(N, world, args.steps, fms), "unit": "tokens/s", "ms_per_step": fstep,
            "tflops_8NdV": flop_step / (fstep / 1e3) / 1e12,
            "tensor_tflops_6NdV": 0.75 * flop_step / (fstep / 1e3) / 1e12,
            "what": "fkl_forward_backward: each chunk's logits kept in fp16 between its loss and gradient "
                    "passes instead of recomputed (6 N d V tensor FLOP)",
            "kernels": fb_kernels, "device_status": api.get_status(ws)}}

        # the KL + hard-label cross-entropy mixture (alpha = 0.5) through its own entry points
        label = torch.from_numpy(np.random.default_rng(11).integers(0, V, N).astype(np.int32)).to(dev)

        def step_mix():
            _, ls, l1 = api.mix_forward(h, W, idx, t, mask, label, T, 0.5, chunk=args.chunk, ws=ws)
            api.mix_backward(h, W, idx, t, mask, label, T, 0.5, ls, l1, chunk=args.chunk, ws=ws)

        for _ in range(2):
            step_mix()
        torch.cuda.synchronize()
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        m0.record(stream)
        for _ in range(args.steps):
            step_mix()
        m1.record(stream)
        torch.cuda.synchronize()
        mstep = m0.elapsed_time(m1) / args.steps
        variants["kl_ce_mixture"] = {
            "value": N / (mstep / 1e3), "unit": "tokens/s (this rank)", "ms_per_step": mstep,
            "tflops_8NdV": flop_step / (mstep / 1e3) / 1e12, "alpha": 0.5,
            "what": "fkl_mix_forward + fkl_mix_backward: alpha T^2 KL + (1 - alpha) CE on a hard label",
            "device_status": api.get_status(ws)}

    # ---- the teacher top-K cache producer on the same shapes (h, W standing in for the teacher's)
    topk = None
    if not args.no_variants:
        tk_ws = torch.empty(api.topk_workspace_size(N, d, V, K), dtype=torch.uint8, device=dev)
        for _ in range(2):
            api.teacher_topk(h, W, K, ws=tk_ws)
        torch.cuda.synchronize()
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        api.profile_reset()
        api.profile_enable(True)
        k0.record(stream)
        for _ in range(args.steps):
            api.teacher_topk(h, W, K, ws=tk_ws)
        k1.record(stream)
        torch.cuda.synchronize()
        api.profile_enable(False)
        tk_kernels = per_kernel(api.profile_read(), args.steps)
        kstep = k0.elapsed_time(k1) / args.steps
        topk = {"value": N / (kstep / 1e3), "unit": "tokens/s", "ms_per_step": kstep,
                "tflops_2NdV": 2.0 * N * d * V / (kstep / 1e3) / 1e12, "K": K,
                "workspace_gb": tk_ws.numel() / 1e9, "kernels": tk_kernels,
                "what": "fkl_teacher_topk: one tensor-core pass over z = h W^T keeping each row's top eight "
                        "per vocabulary tile, candidates >= the K-th largest tile max gathered from them (a second "
                        "pass only for rows with eight or more in one tile), top-K selection per row",
                "device_status": api.get_status(tk_ws)}
        del tk_ws

    # ---- e2e: the public API with host buffers (pinned), copies inside the timed region.
    # Each step's inputs are copied host -> device on a copy stream into one of two
    # buffers while the previous step computes (as a training loop prefetches its next
    # batch); each step's loss is read back on the host before the next step starts.
    e2e = None
    if not args.no_e2e:
        hp = torch.from_numpy(x["h"].view(np.int16)).view(torch.bfloat16).pin_memory()
        ip, tp, mp = (torch.from_numpy(x[k]).pin_memory() for k in ("idx", "t", "mask"))
        host_in = (hp, ip, tp, mp)
        lossp = torch.empty(1, dtype=torch.float32).pin_memory()
        bufs = [tuple(torch.empty_like(a, device=dev) for a in host_in) for _ in range(2)]
        copy_stream = torch.cuda.Stream(dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        used = [torch.cuda.Event() for _ in range(2)]

        def enqueue_copy(slot, after=None):
            with torch.cuda.stream(copy_stream):
                if after is not None:
                    copy_stream.wait_event(after)
                copy_stream.wait_event(used[slot])  # the step that last read this buffer is done
                for dst, src in zip(bufs[slot], host_in):
                    dst.copy_(src, non_blocking=True)
                copied[slot].record(copy_stream)

        def enqueue_step(slot):
            stream.wait_event(copied[slot])
            h_in, idx_in, t_in, m_in = bufs[slot]
            api.forward(h_in, W, idx_in, t_in, m_in, T, args.chunk, ws=ws, loss=loss, lse=lse)
            api.backward(h_in, W, idx_in, t_in, m_in, T, lse, chunk=args.chunk, ws=ws, dh=dh, dW=dW)
            lossp.copy_(loss, non_blocking=True)
            used[slot].record(stream)

        def run_e2e(steps, start=None):
            enqueue_copy(0, after=start)
            for i in range(steps):
                if i + 1 < steps:
                    enqueue_copy((i + 1) % 2)
                enqueue_step(i % 2)
                stream.synchronize()  # the loss is read on the host every step
                float(lossp.item())

        run_e2e(2)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        e0.record(stream)
        run_e2e(args.steps, start=e0)
        e1.record(stream)
        torch.cuda.synchronize()
        ems = slowest_ms(e0.elapsed_time(e1), world, dev)
        bi = sum(a.numel() * a.element_size() for a in host_in)
        e2e = {"value": job_throughput(N, world, args.steps, ems), "unit": "tokens/s", "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": 4, "ms_per_step": ems / args.steps,
               "resident": "W (model weight) stays on the device; h, teacher ids/logits and mask are copied "
                           "per step from pinned host memory, overlapped with the previous step"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(x)

    # ---- the smaller workloads (tiny, small LM head, Llama-8B->3.2B-like head) on the same call pair
    legs = {}
    if not args.no_config_legs and args.config == 3 and args.shape is None and world == 1:
        del x
        for cfg in (0, 1, 2):
            legs[f"config_{cfg}"] = config_leg(api, cfg, dev, stream, args.chunk, args.steps, args.warmup, peaks,
                                               peaks_kind, with_cpu=not args.no_cpu_baseline)

    # ---- the dense method (full N x V logits in plain torch) on the same workloads: its
    # peak memory beside the fused path's (the pages' dense-versus-fused comparison)
    dense = None
    if not args.no_dense and args.config == 3 and args.shape is None and world == 1:
        dense = {"what": "dense_kl_step: the N x V logits materialised (bf16 matmul, fp32 log-softmax), "
                         "the same top-K forward KL, autograd backward; plain torch, a comparison baseline",
                 "fused_config_3_peak_beyond_inputs_gb":
                     (peak_mem - sum(a.numel() * a.element_size() for a in (h, W, idx, t, mask))) / 1e9,
                 "fused_config_3_what": "the fused two-call path at the same workload: workspace, lse, loss, "
                                        "dh (bf16) and dW (fp32)"}
        for cfg in (1, 2, 3):
            dense[f"config_{cfg}"] = dense_baseline(cfg, dev)

    # ---- the memory-stress workload (N = 131072): peak device memory of the same call pair
    mem = None
    ws_gb = ws.numel() / 1e9
    if not args.no_memory_stress and args.config == 3 and args.shape is None and world == 1:
        del h, W, idx, t, mask, ws, loss, lse, dh, dW
        if not args.no_e2e:
            del bufs
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        mem = memory_stress(api, dev, stream, args.chunk, min(args.steps, 3))

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": config_dict(c, args.chunk, world),
                "tflops": tflops,
                "frac_of_bf16_peak": {"burst": tflops / peaks["bf16_tflops"],
                                      "sustained": tflops / peaks["bf16_tflops_sustained"],
                                      "kind": peaks_kind},
                "peak_mem_gb": peak_mem / 1e9,
                "workspace_gb": ws_gb,
                "resident_gb": base_mem / 1e9,
                "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
                "variants": variants, "teacher_topk": topk, "memory_stress": mem, **legs,
                "dense_baseline": dense,
                "clocks": clk.summary(), "gpu_launches": launches, "device_status": status,
                "kernel_digest": kernel_digest()}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0 if status == 0 else 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--chunk", type=int, default=0)
    ap.add_argument("--impl", choices=["fused", "reference"], default="fused")
    ap.add_argument("--ref-rows", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-variants", action="store_true", help="skip the one-call forward+backward timing")
    ap.add_argument("--no-memory-stress", action="store_true", help="skip the N=131072 peak-memory leg")
    ap.add_argument("--no-dense", action="store_true",
                    help="skip the dense (materialised N x V logits) comparison baseline")
    ap.add_argument("--no-config-legs", action="store_true",
                    help="skip the tiny, small LM head and Llama-like head workloads (config_0..2 keys)")
    ap.add_argument("--shape", type=lambda s: tuple(int(v) for v in s.split(",")), default=None,
                    help="N,d,V,K: a smaller case of the chosen workload (profiling captures)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "fused":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    return run_fused(args)


if __name__ == "__main__":
    sys.exit(main())
