#!/usr/bin/env python3
"""Benchmark of the fused chunked top-K KL loss (forward + backward).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config 3] [--chunk 0]

One step is one kd_topk_kl_fwd_bwd call over one batch of synthetic inputs:
teacher preparation, and per token chunk the logsumexp pass, the gradient tile
and both gradient GEMMs (every row of the hot path).  The default workload is
the large-vocabulary long-context case: N = 32,768 tokens, d = 2880,
V = 201,088, K = 100 teacher entries, T = 1, bf16 h and W.  Throughput is
tokens/s of the whole job; TFLOP/s counts 6 N d V per step (forward logits,
grad_h and grad_W products).  Inputs are larger than L2 (W alone is 1.16 GB),
so no flush is needed between steps.

Under torchrun (N > 1) every rank runs its own token shard of the same size
(weak scaling) as one data-parallel step (fwd_bwd_dp): the ranks' valid-token
counts are all-reduced before the loss is divided, and loss and grad_W are
all-reduced after it, inside the timed region; the barrier and max-over-ranks
time use torch.distributed.  `--impl reference` times the fp64 CPU oracle on a
bounded sample of the same workload (rank 0 only).

Other modes, one JSON line each, same timing rules:
  --fwd            the loss alone (kd_topk_kl_fwd), 2 N d V flops per step;
  --builder        the teacher top-K cache (kd_topk_cache_build) of N positions;
  --full-teacher   the full-vocabulary loss (kd_full_kl_fwd_bwd);
  --mem-scaling    device memory of the fused call at N = 8K ... 256K tokens;
  --dense-context  plain-PyTorch dense and forward-chunked KL beside the fused
                   call: peak memory and time at N = 8K ... 128K tokens.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused KL fwd+bwd tokens/s and TFLOP/s (% of B300 bf16 peak); peak GiB"
FWD_METRIC = "fused KL fwd (loss only) tokens/s and TFLOP/s (% of B300 bf16 peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# Kernel sources whose DRAM traffic a committed ncu capture describes; the
# capture applies only while these files are unchanged.
TRAFFIC_SOURCES = ["top_kl_loss_token_b300/csrc/kd_tc_gemm.cu",
                   "top_kl_loss_token_b300/csrc/kd_ptx.cuh",
                   "top_kl_loss_token_b300/csrc/kd_internal.h",
                   "top_kl_loss_token_b300/csrc/kd_api.cu"]
TRAFFIC_PROFILE = "profiles/dram_traffic_vocab201k-32k.md"


def kernel_source_hash() -> str:
    """SHA-256 of the kernel sources' code: comments removed and whitespace
    collapsed, so that only a change of the code itself retires a capture."""
    import hashlib
    import re
    h = hashlib.sha256()
    for rel in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


def measured_traffic(kernel: str, workload: str, chunk: int):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when it was taken on other sources or another workload."""
    import re
    path = os.path.join(ROOT, TRAFFIC_PROFILE)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"^source-sha256: ([0-9a-f]{64})$", text, re.M)
    w = re.search(r"^workload: (.+)$", text, re.M)
    b = re.search(r"^%s: ([0-9]+) bytes per launch" % re.escape(kernel), text, re.M)
    if not (m and w and b) or m.group(1) != kernel_source_hash():
        return None
    if w.group(1).strip() != f"{workload}; chunk {chunk}":
        return None
    return int(b.group(1))


def hbm_kernel_bytes(x, chunk: int, valid: int, grads: bool = True) -> dict:
    """Algorithmic DRAM bytes per launch of the bandwidth-bound kernels (each
    input read once, each output written once)."""
    N, d, V, K = x.N, x.d, x.V, x.K
    n_pb = -(-V // 128)
    ldg = -(-V // 256) * 256
    c = min(chunk, valid) if valid else 0
    n_chunks = max(1, -(-valid // chunk)) if valid else 1
    c_avg = valid / n_chunks if valid else 0
    elem = 2 if x.dtype == "bf16" else 4
    return {
        # topk_idx and topk_logit read, sorted (index, p) lists written
        "teacher_prep": 16.0 * N * K,
        # fp32 path: u read and G written, per-(row, block) alpha and offsets, sorted lists
        "grad_tile": c_avg * (2.0 * elem * ldg + 6.0 * n_pb + 8.0 * K),
        # bf16 path: the chunk's h row read and written, the sorted lists read,
        # one stored value read and written per teacher entry, three row factors
        "grad_prepare": c_avg * (2.0 * elem * d + 8.0 * K + 4.0 * K + 12.0),
        # three per-(row, block) statistics read, alpha written
        "lse_combine": c_avg * 16.0 * n_pb,
        # sorted indices read, per-(row, block) offsets written
        "bucket_offsets": c_avg * (4.0 * K + 2.0 * (n_pb + 1)),
        # the chunk's h rows read and written contiguously
        # (bf16 with gradients: also the W row of the teacher's top entry, for
        # the row's exponential reference)
        "gather_rows": c_avg * (2.0 * elem * d + (elem * d if grads and elem == 2 else 0.0)),
    }


def workload_name(x) -> str:
    mask = f", {x.masked_fraction() * 100:.1f}% masked" if x.mask is not None else ""
    return (f"{x.name}: N={x.N} tokens, d={x.d}, V={x.V}, K={x.K}, T={x.T:g}, "
            f"{x.dtype} h/W, fp32 teacher top-K{mask}")


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
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
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_oracle_time(x, rows: int, grads: bool = True):
    """Times the fp64 oracle (fwd+bwd, or the loss alone) on the first `rows`
    tokens of x."""
    import oracle
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] or [os.cpu_count()])
    except Exception:
        cores = os.cpu_count()
    h = x.h_f32()[:rows].astype(np.float64)
    W = x.W_f32().astype(np.float64)
    m = None if x.mask is None else x.mask[:rows]
    t0 = time.perf_counter()
    if grads:
        oracle.fwd_bwd(h, W, x.idx[:rows], x.logit[:rows], m, x.T)
    else:
        oracle.fwd(h, W, x.idx[:rows], x.logit[:rows], m, x.T)
    dt = time.perf_counter() - t0
    return dt, cores


def run_reference(args, x):
    """The oracle as the reference arm: each step is a bounded sample of the workload."""
    rows = args.ref_rows
    for _ in range(args.warmup):
        cpu_oracle_time(x, rows)
    times, cores = [], 1
    for _ in range(args.steps):
        dt, cores = cpu_oracle_time(x, rows)
        times.append(dt)
    total = sum(times)
    value = rows * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(x), "sample": f"first {rows} tokens per step"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"fwd+bwd of the first {rows} of {x.N} tokens, per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def shard_seed(seed: int, rank: int, world: int) -> int:
    """Seed of this rank's token shard: every rank draws its own tokens of the
    same sizes (weak scaling); a single process keeps the workload's seed."""
    return seed if world <= 1 else seed + 1000 * rank


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time (the whole job ends when the last rank does)."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


BUILDER_METRIC = "teacher top-K cache build tokens/s and TFLOP/s (% of B300 bf16 peak)"


def run_builder(args):
    """The offline teacher top-K cache (kd_topk_cache_build) on one GPU: the
    workload's h as teacher final hidden states, its W as the teacher LM head
    (d = 2880, V = 201,088 by default: a gpt-oss-120b-class teacher head), K
    entries per position.  One step builds the cache of all N positions.  The
    metric counts the logits' 2 N d V flops; the kernels execute more: the
    first pass computes the logits of the sampled blocks again, and a row whose
    candidates overflow is collected a third time (include/kd_topk_cache.h).
    The roofline is taken on the all-logits candidate pass, 2 c d V per launch."""
    import torch
    import top_kl_loss_token_b300 as kd
    from top_kl_loss_token_b300 import synth
    kd.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    c = dict(synth.CONFIGS[args.config])
    if args.tokens:
        c["N"] = args.tokens
    c["mask"] = None
    c.pop("mask_frac_range", None)
    x = synth.make_inputs(**c)
    N, d, V, K = x.N, x.d, x.V, x.K
    h_pin = torch.from_numpy(x.h.view(np.int16)).view(torch.bfloat16).pin_memory()
    W = torch.from_numpy(x.W.view(np.int16)).view(torch.bfloat16).to(dev)
    h = h_pin.to(dev)
    chunk = args.chunk or int(kd.load_library().kd_topk_cache_default_chunk(N, V, K))
    idx = torch.empty((N, K), dtype=torch.int32, device=dev)
    val = torch.empty((N, K), dtype=torch.float32, device=dev)
    ws = torch.empty(kd.topk_cache_workspace_bytes(N, d, V, K, chunk), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kd.topk_cache_build(h, W, K, chunk, topk_idx=idx, topk_logit=val, workspace=ws,
                            err_flags=err, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flags {int(err.item())}")
    kd.timing_enable(True)
    kd.timing_collect()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    kd.timing_enable(False)
    kernels = kd.timing_collect()
    ms = ev0.elapsed_time(ev1)
    value = N * args.steps / (ms / 1000.0)
    peaks, peaks_src = load_peaks()
    tflops = 2.0 * N * d * V * args.steps / (ms / 1000.0) / 1e12
    n_pb = -(-V // 128)
    n_s = min(n_pb, -(-max(K, -(-n_pb // 8)) // 2) * 2)  # the sampled blocks (kd_topk_cache.cu)
    v_s = min(V, n_s * 128)
    dom = "topk_candidates"
    launches, tot_ms = kernels[dom]
    flops_per_launch = 2.0 * N * d * V * args.steps / launches
    redo_launches, redo_ms = kernels.get("topk_redo", (0, 0.0))
    achieved = flops_per_launch / (tot_ms / launches / 1000.0) / 1e12
    roof = {"kernel": dom, "bound": "tensor", "achieved": achieved,
            "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_tflops_sustained"], "traffic": None,
            "peak_source": f"{peaks_src} bf16 sustained (kernel timed inside a long step)",
            "flops_per_launch": flops_per_launch, "avg_launch_ms": tot_ms / launches}
    # end to end: teacher hidden states in from pinned memory, the cache out
    idx_host = torch.empty((N, K), dtype=torch.int32).pin_memory()
    val_host = torch.empty((N, K), dtype=torch.float32).pin_memory()
    e_steps = max(1, min(args.steps, 5))
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e_steps):
        h.copy_(h_pin, non_blocking=True)
        step()
        idx_host.copy_(idx, non_blocking=True)
        val_host.copy_(val, non_blocking=True)
        stream.synchronize()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e_value = N * e_steps / (e0.elapsed_time(e1) / 1000.0)
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        rows = min(512, N)  # about 12 s on 16 host cores at V = 201,088
        hh = x.h_f32()[:rows].astype(np.float64)
        WW = x.W_f32().astype(np.float64)
        t0 = time.perf_counter()
        oracle.topk_cache(hh, WW, K, block_rows=min(rows, 128))
        dtc = time.perf_counter() - t0
        cpu = {"value": rows / dtc, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"fp64 oracle top-{K} cache of the first {rows} of {N} positions "
                         f"({dtc:.1f} s)"}
    line = {
        "metric": BUILDER_METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"teacher top-{K} cache: N={N} positions, d={d}, V={V}, bf16 "
                               f"hidden states and LM head", "chunk": chunk,
                   "l2": "inputs larger than L2 (W alone 1.16 GB), no flush"},
        "tflops_per_gpu": tflops, "tflops_executed_per_gpu": tflops * (1.0 + v_s / V),
        "sampled_columns": v_s, "redo_launches": redo_launches, "redo_ms": redo_ms,
        "pct_of_bf16_peak": {"burst": tflops / peaks["bf16_tflops"],
                             "sustained": tflops / peaks["bf16_tflops_sustained"],
                             "source": peaks_src},
        "workspace_gib": ws.numel() / 2 ** 30,
        "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": e_value, "unit": "tokens/s", "h2d_bytes_per_step": h_pin.numel() * 2,
                "d2h_bytes_per_step": N * K * 8},
        "gpu_launches": sum(v[0] for v in kernels.values()),
        "kernels": {k: {"launches": v[0], "ms": v[1]} for k, v in kernels.items()},
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


FULL_METRIC = "full-vocabulary KL fwd+bwd tokens/s and TFLOP/s (% of B300 bf16 peak)"


def run_full_teacher(args):
    """The full-vocabulary loss (kd_full_kl_fwd_bwd): the workload's student
    (h, W) against a teacher of the same hidden size whose hidden states and
    LM head are drawn like the student's from their own seed.  One step is one
    fused fwd+bwd over all N tokens; it executes 2 N d_t V (teacher logits) +
    6 N d_s V (student logits, grad_h, grad_W) flops."""
    import torch
    import top_kl_loss_token_b300 as kd
    from top_kl_loss_token_b300 import synth
    kd.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    c = dict(synth.CONFIGS[args.config])
    if args.tokens:
        c["N"] = args.tokens
        if c.get("mask") == "packed":
            c["mask_frac_range"] = None
    xs = synth.make_inputs(**c)
    xt = synth.make_inputs(**synth.full_teacher_config(c))
    N, d, V = xs.N, xs.d, xs.V

    def bf(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    hs_pin, ht_pin = bf(xs.h).pin_memory(), bf(xt.h).pin_memory()
    m_pin = None if xs.mask is None else torch.from_numpy(xs.mask).pin_memory()
    Ws, Wt = bf(xs.W).to(dev), bf(xt.W).to(dev)
    hs, ht = hs_pin.to(dev), ht_pin.to(dev)
    mask = None if m_pin is None else m_pin.to(dev)
    chunk = args.chunk or int(kd.load_library().kd_full_kl_default_chunk(N, d, xt.d, V))
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    gh = torch.empty((N, d), dtype=torch.float32, device=dev)
    gW = torch.empty((V, d), dtype=torch.float32, device=dev)
    ws = torch.empty(kd.full_kl_workspace_bytes(N, d, d, V, chunk), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kd.full_kl_fwd_bwd(hs, Ws, ht, Wt, mask, xs.T, chunk, loss=loss, grad_h=gh, grad_W=gW,
                           workspace=ws, err_flags=err, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flags {int(err.item())}")
    kd.timing_enable(True)
    kd.timing_collect()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    kd.timing_enable(False)
    kernels = kd.timing_collect()
    ms = ev0.elapsed_time(ev1)
    value = N * args.steps / (ms / 1000.0)
    valid = N if xs.mask is None else int(xs.mask.sum())
    flops_step = 8.0 * N * d * V
    tflops = flops_step * args.steps / (ms / 1000.0) / 1e12
    peaks, peaks_src = load_peaks()
    per_token = {"full_pass1_gemm": 4.0 * d * V, "bwd_gemm": 4.0 * d * V}
    dom = max(kernels.items(), key=lambda kv: kv[1][1])[0]
    roof = None
    if dom in per_token:
        launches, tot_ms = kernels[dom]
        fpl = per_token[dom] * valid * args.steps / launches
        ach = fpl / (tot_ms / launches / 1000.0) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach,
                "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16_tflops_sustained"], "traffic": None,
                "peak_source": f"{peaks_src} bf16 sustained (kernel timed inside a long step)",
                "flops_per_launch": fpl, "avg_launch_ms": tot_ms / launches}
    loss_host = torch.empty(1, dtype=torch.float32).pin_memory()
    h2d = 2 * hs_pin.numel() * 2 + (0 if m_pin is None else m_pin.numel())
    e_steps = max(1, min(args.steps, 5))
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e_steps):
        hs.copy_(hs_pin, non_blocking=True)
        ht.copy_(ht_pin, non_blocking=True)
        if m_pin is not None:
            mask.copy_(m_pin, non_blocking=True)
        step()
        loss_host.copy_(loss, non_blocking=True)
        stream.synchronize()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e_value = N * e_steps / (e0.elapsed_time(e1) / 1000.0)
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        rows = min(768, N)
        t0 = time.perf_counter()
        oracle.full_kl_fwd_bwd(xs.h_f32()[:rows], xs.W_f32(), xt.h_f32()[:rows], xt.W_f32(),
                               None if xs.mask is None else xs.mask[:rows], xs.T,
                               block_rows=min(rows, 256))
        dtc = time.perf_counter() - t0
        cpu = {"value": rows / dtc, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"fp64 oracle fwd+bwd of the first {rows} of {N} tokens ({dtc:.1f} s)"}
    line = {
        "metric": FULL_METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": (f"{xs.name} student: N={N} tokens, d={d}, V={V}, T={xs.T:g}, "
                                f"bf16 h/W" + (f", {xs.masked_fraction() * 100:.1f}% masked"
                                               if xs.mask is not None else "")
                                + f"; full-vocabulary teacher d={d} computed in the same pass"),
                   "chunk": chunk, "l2": "inputs larger than L2 (W alone 1.16 GB), no flush"},
        "tflops_per_gpu": tflops,
        "pct_of_bf16_peak": {"burst": tflops / peaks["bf16_tflops"],
                             "sustained": tflops / peaks["bf16_tflops_sustained"],
                             "source": peaks_src},
        "workspace_gib": ws.numel() / 2 ** 30,
        "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": 4},
        "gpu_launches": sum(v[0] for v in kernels.values()),
        "kernels": {k: {"launches": v[0], "ms": v[1]} for k, v in kernels.items()},
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def run_mem_scaling(args):
    """Device memory of one fused fwd+bwd at the 201,088-vocabulary shapes for
    N = 8K, 32K, 128K and 256K tokens at a fixed 8192-token chunk.  Extra memory (the
    workspace) must grow as O(chunk V + N K), not O(N V).  Values of the inputs
    do not matter here, so they are drawn on the device."""
    import torch
    import top_kl_loss_token_b300 as kd
    kd.load_library()
    dev = torch.device("cuda", 0)
    d, V, K, chunk = 2880, 201088, 100, args.chunk or 8192
    g = torch.Generator(device=dev).manual_seed(0)
    W = (torch.randn(V, d, device=dev, generator=g) * 0.02).to(torch.bfloat16)
    out = []
    for N in (8192, 32768, 131072, 262144):
        h = torch.randn(N, d, device=dev, generator=g).to(torch.bfloat16)
        idx = torch.randint(0, V, (N, K), device=dev, generator=g, dtype=torch.int32)
        lg = torch.randn(N, K, device=dev, generator=g)
        loss = torch.empty(1, device=dev)
        gh = torch.empty(N, d, device=dev)
        gW = torch.empty(V, d, device=dev)
        torch.cuda.synchronize(dev)
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        ws = kd.allocate_workspace(N, d, V, K, chunk, kd.KD_BF16, dev)
        kd.fwd_bwd(h, W, idx, lg, None, 1.0, chunk, loss=loss, grad_h=gh, grad_W=gW, workspace=ws)
        torch.cuda.synchronize(dev)
        peak = torch.cuda.max_memory_allocated(dev)
        out.append({"N": N, "chunk": chunk, "workspace_gib": ws.numel() / 2 ** 30,
                    "peak_extra_gib": (peak - base) / 2 ** 30,
                    "inputs_outputs_gib": base / 2 ** 30,
                    "dense_bf16_logits_gib": N * V * 2 / 2 ** 30})
        del h, idx, lg, loss, gh, gW, ws
        torch.cuda.empty_cache()
    print(json.dumps({"mem_scaling": out, "d": d, "V": V, "K": K}), flush=True)


def _torch_kl_sum(h, W, idx, lg, T):
    """Sum over rows of KL(p || q) in plain PyTorch: q the softmax of the
    student logits h W^T / T over the whole vocabulary, p the teacher's top-K
    logits renormalised; the N x V logit grid is built and kept for autograd."""
    import torch
    logq = torch.log_softmax((h @ W.t()).float() / T, dim=-1)
    logp = torch.log_softmax(lg / T, dim=-1)
    return (logp.exp() * (logp - logq.gather(1, idx.long()))).sum()


def torch_kl_arm(h, W, idx, lg, T, chunk=0):
    """One of the pages' two plain-PyTorch baselines for the memory comparison:
    the dense KL (chunk <= 0: the whole N x V logit grid built at once and kept
    for autograd) or the forward-chunked KL (the grid built chunk by chunk in
    the forward, every chunk's grid still kept for the one backward).  Returns
    (loss = mean over the rows, grad_h, grad_W) from autograd."""
    h = h.detach().requires_grad_(True)
    W = W.detach().requires_grad_(True)
    N = h.shape[0]
    if chunk <= 0:
        tot = _torch_kl_sum(h, W, idx, lg, T)
    else:
        tot = sum(_torch_kl_sum(h[r:r + chunk], W, idx[r:r + chunk], lg[r:r + chunk], T)
                  for r in range(0, N, chunk))
    loss = tot / N
    loss.backward()
    return loss.detach(), h.grad, W.grad


def run_dense_context(args):
    """Context for the pages' peak-memory comparison (dense KL, forward-chunked
    KL, fused chunked KL): peak device memory and time of one fwd+bwd of the
    distillation loss at the d, V and K of --config (default: the
    201,088-vocabulary shapes) for N = 8K, 32K, 64K and 128K tokens.  The dense and forward-chunked arms are plain PyTorch (bf16 matmul,
    fp32 log-softmax, autograd; the forward-chunked arm loops over 8192-token
    chunks in the forward and runs one backward); the fused arm is this
    library's kd_topk_kl_fwd_bwd.  An arm that runs out of device memory is
    recorded as such.  Values of the inputs do not matter for memory, so they
    are drawn on the device."""
    import torch
    import top_kl_loss_token_b300 as kd
    kd.load_library()
    from top_kl_loss_token_b300 import synth
    dev = torch.device("cuda", 0)
    cfg = synth.CONFIGS[args.config]
    d, V, K, T, chunk = cfg["d"], cfg["V"], cfg["K"], 1.0, args.chunk or 8192
    g = torch.Generator(device=dev).manual_seed(0)
    W0 = (torch.randn(V, d, device=dev, generator=g) * 0.02).to(torch.bfloat16)
    reps = max(1, min(args.steps, 3))

    def timed(fn):
        fn()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b))
        return float(np.median(ts))

    rows = []
    for N in (8192, 32768, 65536, 131072):
        h0 = torch.randn(N, d, device=dev, generator=g).to(torch.bfloat16)
        idx = torch.randint(0, V, (N, K), device=dev, generator=g, dtype=torch.int32)
        lg = torch.randn(N, K, device=dev, generator=g) * 2.0
        for arm in ("dense", "forward_chunked", "fused_chunked"):
            torch.cuda.synchronize(dev)
            torch.cuda.empty_cache()
            base = torch.cuda.memory_allocated(dev)
            torch.cuda.reset_peak_memory_stats(dev)
            rec = {"N": N, "arm": arm}
            try:
                if arm == "fused_chunked":
                    loss = torch.empty(1, device=dev)
                    gh = torch.empty(N, d, device=dev)
                    gW = torch.empty(V, d, device=dev)
                    ws = kd.allocate_workspace(N, d, V, K, chunk, kd.KD_BF16, dev)

                    def fn():
                        kd.fwd_bwd(h0, W0, idx, lg, None, T, chunk, loss=loss, grad_h=gh,
                                   grad_W=gW, workspace=ws)
                    rec["grad_dtype"] = "fp32"
                else:
                    out = {}

                    def fn():
                        out.clear()
                        out["loss"], out["gh"], out["gW"] = torch_kl_arm(
                            h0, W0, idx, lg, T, 0 if arm == "dense" else chunk)
                    rec["grad_dtype"] = "bf16"
                rec["ms"] = timed(fn)
                torch.cuda.synchronize(dev)
                rec["peak_gib"] = torch.cuda.max_memory_allocated(dev) / 2 ** 30
                rec["peak_over_inputs_gib"] = (torch.cuda.max_memory_allocated(dev) - base) / 2 ** 30
                rec["loss"] = float((loss if arm == "fused_chunked" else out["loss"]).item())
            except torch.cuda.OutOfMemoryError:
                rec["outcome"] = "out of device memory"
            rec["inputs_gib"] = base / 2 ** 30
            rows.append(rec)
            loss = gh = gW = ws = out = fn = None  # release this arm's buffers
            torch.cuda.synchronize(dev)
            torch.cuda.empty_cache()
        del h0, idx, lg
        torch.cuda.empty_cache()
    print(json.dumps({"dense_context": rows, "d": d, "V": V, "K": K, "T": T, "chunk": chunk,
                      "device_gib": torch.cuda.get_device_properties(dev).total_memory / 2 ** 30}),
          flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--chunk", type=int, default=0)
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the token count (smaller cases for profiling)")
    ap.add_argument("--cpu-rows", type=int, default=1536,
                    help="tokens in the CPU-oracle baseline sample (about 15 s of fp64 "
                         "fwd+bwd on 16 host cores at the default workload)")
    ap.add_argument("--ref-rows", type=int, default=64,
                    help="tokens per step of the reference (oracle) arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fwd", action="store_true",
                    help="time the loss alone (kd_topk_kl_fwd: no gradients) on the same workload")
    ap.add_argument("--builder", action="store_true",
                    help="time the teacher top-K cache builder on the workload's teacher-side "
                         "shapes instead of the loss")
    ap.add_argument("--full-teacher", action="store_true",
                    help="time the full-vocabulary loss with the teacher computed in the same "
                         "pass (teacher hidden size = the student's) instead of the top-K loss")
    ap.add_argument("--mem-scaling", action="store_true",
                    help="report device memory at N = 8K, 32K, 128K, 256K tokens (fixed chunk) "
                         "and exit")
    ap.add_argument("--dense-context", action="store_true",
                    help="peak memory and time of plain-PyTorch dense and forward-chunked KL "
                         "against the fused call at N = 8K, 32K, 64K, 128K tokens, and exit")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup

    from top_kl_loss_token_b300 import synth

    if args.impl == "reference":
        if rank != 0:
            return
        x = synth.make_config(args.config, **({"N": args.tokens} if args.tokens else {}))
        run_reference(args, x)
        return

    import torch
    import torch.distributed as dist
    import top_kl_loss_token_b300 as kd

    if args.mem_scaling:
        run_mem_scaling(args)
        return
    if args.dense_context:
        run_dense_context(args)
        return
    if args.builder:
        run_builder(args)
        return
    if args.full_teacher:
        run_full_teacher(args)
        return

    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank if world > 1 else 0)
    torch.cuda.set_device(dev)
    kd.load_library()

    c = dict(synth.CONFIGS[args.config])
    if args.tokens:
        c["N"] = args.tokens
        if c.get("mask") == "packed":
            c["mask_frac_range"] = None
    c["seed"] = shard_seed(c["seed"], rank, world)
    x = synth.make_inputs(**c)
    N, d, V, K = x.N, x.d, x.V, x.K
    dt_code = kd.KD_BF16 if x.dtype == "bf16" else kd.KD_FP32
    chunk = args.chunk if args.chunk > 0 else kd.default_chunk(N, d, V, dt_code)

    # host copies (pinned) and resident device inputs
    if x.dtype == "bf16":
        h_host = torch.from_numpy(x.h.view(np.int16)).view(torch.bfloat16)
        W_host = torch.from_numpy(x.W.view(np.int16)).view(torch.bfloat16)
    else:
        h_host, W_host = torch.from_numpy(x.h), torch.from_numpy(x.W)
    idx_host = torch.from_numpy(x.idx)
    lg_host = torch.from_numpy(x.logit)
    m_host = None if x.mask is None else torch.from_numpy(x.mask)
    h_pin, idx_pin, lg_pin = h_host.pin_memory(), idx_host.pin_memory(), lg_host.pin_memory()
    m_pin = None if m_host is None else m_host.pin_memory()
    W = W_host.to(dev)
    h, idx, lg = h_pin.to(dev), idx_pin.to(dev), lg_pin.to(dev)
    mask = None if m_pin is None else m_pin.to(dev)
    base_alloc = torch.cuda.memory_allocated(dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    grad_h = torch.empty((N, d), dtype=torch.float32, device=dev)
    grad_W = torch.empty((V, d), dtype=torch.float32, device=dev)
    ws_bytes = kd.workspace_bytes(N, d, V, K, chunk, dt_code)
    torch.cuda.reset_peak_memory_stats(dev)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        if args.fwd:
            kd.fwd(h, W, idx, lg, mask, x.T, chunk, loss=loss, workspace=ws, err_flags=err,
                   stream=stream)
            return
        if world > 1:
            # the data-parallel step: counts, loss and grad_W all-reduced
            kd.fwd_bwd_dp(h, W, idx, lg, mask, x.T, chunk, loss=loss, grad_h=grad_h,
                          grad_W=grad_W, workspace=ws, err_flags=err, stream=stream)
            return
        kd.fwd_bwd(h, W, idx, lg, mask, x.T, chunk, loss=loss, grad_h=grad_h, grad_W=grad_W,
                   workspace=ws, err_flags=err, stream=stream)

    def check_flags(where):
        if int(err.item()) != 0:
            raise RuntimeError(f"device error flags {int(err.item())} after {where}")

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    check_flags("the warm-up steps")
    peak_extra = (torch.cuda.max_memory_allocated(dev) - base_alloc) / 2 ** 30

    # ---------------- timed region: inputs resident in HBM
    kd.timing_enable(True)
    kd.timing_collect()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    kd.timing_enable(False)
    kernels = kd.timing_collect()
    check_flags("the timed steps")
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    tokens_total = N * args.steps * world
    value = tokens_total / (ms / 1000.0)
    flops_per_token = (2.0 if args.fwd else 6.0) * d * V  # logits (+ grad_h, grad_W)
    flops_step = flops_per_token * N
    tflops = flops_step * args.steps * world / (ms / 1000.0) / 1e12 / world  # per GPU

    # ---------------- end to end: H2D of the step's inputs, D2H of the loss
    loss_host = torch.empty(1, dtype=torch.float32).pin_memory()
    h2d = h_pin.numel() * h_pin.element_size() + idx_pin.numel() * 4 + lg_pin.numel() * 4
    if m_pin is not None:
        h2d += m_pin.numel()
    e_steps = max(1, min(args.steps, 5))
    barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as e_clk:
        e0.record(stream)
        for _ in range(e_steps):
            h.copy_(h_pin, non_blocking=True)
            idx.copy_(idx_pin, non_blocking=True)
            lg.copy_(lg_pin, non_blocking=True)
            if m_pin is not None:
                mask.copy_(m_pin, non_blocking=True)
            step()
            loss_host.copy_(loss, non_blocking=True)
            stream.synchronize()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    check_flags("the end-to-end steps")
    barrier()
    e_value = N * e_steps * world / (max_over_ranks(e0.elapsed_time(e1), world, dev) / 1000.0)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    # ---------------- roofline of the dominant kernel
    peaks, peaks_src = load_peaks()
    n_chunks = -(-N // chunk)
    valid_tokens = N if x.mask is None else int(x.mask.sum())
    # algorithmic flops per token of each tensor-core kernel
    per_token = {"pass1_gemm": 2.0 * d * V, "bwd_gemm": 4.0 * d * V}
    dom = max(kernels.items(), key=lambda kv: kv[1][1])[0] if kernels else None
    roof = None
    if dom in per_token:
        launches, tot_ms = kernels[dom]
        flops_per_launch = per_token[dom] * valid_tokens * args.steps / launches
        achieved = flops_per_launch / (tot_ms / launches / 1000.0) / 1e12
        peak = peaks["bf16_tflops_sustained"]
        traffic = None
        if not args.tokens and args.config == 3 and not args.fwd:
            # the capture is of the fwd+bwd launches (pass 1 storing its exponentials)
            traffic = measured_traffic(dom, x.name, chunk)
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peaks_src} bf16 sustained (kernel timed inside a long step)",
                "flops_per_launch": flops_per_launch,
                "avg_launch_ms": tot_ms / launches}
    launches_total = sum(v[0] for v in kernels.values())
    hbm = {}
    for name, nbytes in hbm_kernel_bytes(x, chunk, valid_tokens, grads=not args.fwd).items():
        if name not in kernels:
            continue
        launches, tot_ms = kernels[name]
        gbs = nbytes / (tot_ms / launches / 1000.0) / 1e9
        hbm[name] = {"bytes_per_launch": nbytes, "ms_per_launch": tot_ms / launches,
                     "achieved_gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"]}

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        # the loss alone costs the oracle about a third of fwd+bwd
        rows = min(args.cpu_rows * (3 if args.fwd else 1), N)
        dtc, cores = cpu_oracle_time(x, rows, grads=not args.fwd)
        what = "fwd" if args.fwd else "fwd+bwd"
        cpu = {"value": rows / dtc, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"fp64 oracle {what} of the first {rows} of {N} tokens ({dtc:.1f} s)"}

    line = {
        "metric": FWD_METRIC if args.fwd else METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": x.dtype,
        "data": "synthetic",
        "config": {"workload": workload_name(x), "chunk": chunk, "n_chunks": n_chunks,
                   "l2": "inputs larger than L2 (W alone 1.16 GB), no flush",
                   "parallelism": (f"token shards x{world}, counts, loss and grad_W "
                                   "all-reduced per step") if world > 1 else "1 GPU"},
        "tflops_per_gpu": tflops,
        "pct_of_bf16_peak": {"burst": tflops / peaks["bf16_tflops"],
                             "sustained": tflops / peaks["bf16_tflops_sustained"],
                             "source": peaks_src},
        "tflops_valid_tokens_per_gpu": flops_per_token * valid_tokens * args.steps / (ms / 1000.0) / 1e12,
        "hbm_kernels": hbm,
        "peak_extra_gib": peak_extra,
        "workspace_gib": ws_bytes / 2 ** 30,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": 4, "steps": e_steps,
                # each step waits for its copies and its loss, so the GPU idles
                # briefly between steps; under the power cap the SM clock then
                # runs higher than in the back-to-back timed region
                "clocks": e_clk.summary()},
        "gpu_launches": launches_total,
        "kernels": {k: {"launches": v[0], "ms": v[1]} for k, v in kernels.items()},
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
