#!/usr/bin/env python
"""Benchmark of the paged MLA decode path on GB300.

One step = one mla_decode_fwd call on one batch through the C ABI: the
split-KV decode kernel and the combine kernel.  The plan (mla_get_metadata, the
tile scheduler) is built once per decode step and shared by every layer, so it
is built before the timed region and its own duration is reported beside the
step (kernel_ms.sched); the e2e figure includes it.  The headline
workload is the memory-bound decode (batch 64, s_q 1, h_q 16, every sequence
4096 tokens, 64-token pages permuted at random, bf16); metric and unit follow
the benchmark's definition (TFLOP/s and HBM GB/s of algorithmic work, as a
fraction of the measured BF16 / HBM peaks).

Timing (rank-local, then max over ranks):
  * timed region (`value`): K back-to-back steps, each exactly the call a
    user makes, launched as CUDA graphs of 8 consecutive calls (as a model's
    layers issue them; programmatic launch overlaps each call with the one
    before, inside a graph), bracketed by a barrier and a device
    synchronisation; CUDA events on the replay stream.  No L2 flush between
    steps: the inputs (~300 MB of KV pages) exceed the 129 MB L2;
  * flushed step: up to 2000 replays of a graph of one step, each preceded by a
    write of twice the L2 size outside the events, so that every step starts
    with a cold L2 (`step_l2_flushed`);
  * kernel region: K steps (at most 2000) with the three kernels launched as
    separate graphs and CUDA events between them, giving each kernel's average
    duration; the decode kernel's inputs exceed L2 (the KV pages alone are
    ~300 MB against a 129 MB L2), and an L2-sized buffer is written before
    every decode launch, outside its events;
  * e2e: the same step through the public Python API from pinned host buffers,
    with the host->device copies of the inputs and the device->host copy of
    out/lse inside the timed region.
  * clocks: nvidia-smi sampled during the timed and kernel regions.
The CPU baseline (and the --impl reference arm) is the fp64 oracle timed on
this host's cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADLINE = "memory_bound"
METRIC = "MLA decode TFLOP/s & HBM GB/s at 1 GB300, % of BF16/HBM roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024


# --------------------------------------------------------------------- helpers
def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--kernel", choices=["auto", "single", "tq", "duo"], default="auto",
                    help="decode kernel: auto (default: tq for s_q*h_q <= 32, duo for >= 128, "
                         "else single), single CTA, Q in TMEM, or a CTA pair")
    ap.add_argument("--sparse-only", action="store_true",
                    help="time only the sparse-decode workload (steps/warmup as given) and "
                         "print its line; for profiling")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(x, dist=None):
    """The slowest rank's value, on every rank (the timing rule for N > 1)."""
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_workload(W_mod, name, rank):
    """Weak scaling: every rank decodes its own seeded batch of the workload."""
    return W_mod.CONFIGS[name](seed_offset=1000 * rank)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


KERNEL_SOURCES = {"single": ("decode_kernel", "decode_attention_paged_gb300/csrc/mla_decode.cu"),
                  "tq": ("decode_tq_kernel", "decode_attention_paged_gb300/csrc/mla_decode_tq.cu"),
                  "duo": ("decode_duo_kernel", "decode_attention_paged_gb300/csrc/mla_decode_duo.cu")}


def kernel_source_hash(kernel="single"):
    h = hashlib.sha256()
    for rel in (KERNEL_SOURCES[kernel][1], "decode_attention_paged_gb300/csrc/sm103_ptx.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profile_traffic(workload, kernel="single"):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"{KERNEL_SOURCES[kernel][0]}_{workload}_ncu.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_hash") != kernel_source_hash(kernel):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_indices):
        self.gpus = set(gpu_indices)
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()

    def summary(self):
        rows = []
        try:
            with open(self.file.name) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        idx = int(parts[0])
                    except ValueError:
                        continue
                    if self.gpus and idx not in self.gpus:
                        continue
                    rows.append(parts)
        finally:
            os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = sorted(v for v in (num(r[1]) for r in rows) if v is not None)
        smax = max(v for v in (num(r[2]) for r in rows) if v is not None) if sm else None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": smax,
                "reasons": reasons, "samples": len(rows)}


def kernel_of(kind, w):
    """Name of the decode kernel a dense call on workload w launches."""
    if kind != "auto":
        return kind
    R = w.s_q * w.h_q
    return "tq" if R <= 32 else ("duo" if R >= 128 else "single")


def sparse_kernel_of(kind, h_q):
    """Name of the decode kernel a sparse call with h_q query heads launches
    (lists of h_q rows: the CTA pair where a dense call would take it, else
    the single-CTA kernel)."""
    return "duo" if (kind == "duo" or (kind == "auto" and h_q >= 128)) else "single"


def sparse_line(w, r, kname, peaks, kx):
    """Sparse-decode entry: step throughput, fractions of the peaks and the
    DRAM traffic of the committed ncu summary when it matches the source."""
    hbm_peak, bf16_peak = peaks[0], peaks[1]
    t_s = r["ms_per_step"] * 1e-3
    traffic = profile_traffic("sparse", kname)
    return {
        "workload": w.name, "kernel": KERNEL_SOURCES[kname][0] + " (row gather)",
        "ms_per_step": r["ms_per_step"],
        "step_tflops": r["flops"] / t_s / 1e12, "step_gbs": r["bytes"] / t_s / 1e9,
        "frac_bf16_peak": r["flops"] / t_s / 1e12 / bf16_peak,
        "frac_hbm_peak": r["bytes"] / t_s / 1e9 / hbm_peak,
        "algorithmic_bytes": r["bytes"], "algorithmic_flops": r["flops"],
        "traffic": traffic, "pieces": r["pieces"], "steps": kx,
    }


def roofline_of(res, workload, kname, peaks):
    """Roofline object of the decode kernel of one workload: bound by the
    side of the ridge its arithmetic intensity falls on; achieved algorithmic
    bytes (or FLOPs) per launch over the kernel's mean CUDA-event duration."""
    hbm_peak, bf16_peak, _, peak_src = peaks
    dec_s = res["ms_decode"] * 1e-3
    tensor = res["flops"] / res["bytes"] > bf16_peak * 1e12 / (hbm_peak * 1e9)
    gbs = res["bytes"] / dec_s / 1e9
    tfl = res["flops"] / dec_s / 1e12
    r = {"bound": "tensor" if tensor else "hbm",
         "achieved": tfl if tensor else gbs, "peak": bf16_peak if tensor else hbm_peak,
         "unit": "TFLOP/s" if tensor else "GB/s",
         "frac": tfl / bf16_peak if tensor else gbs / hbm_peak,
         "traffic": profile_traffic(workload, kname),
         "kernel": KERNEL_SOURCES[kname][0] + " (split-KV)", "peak_source": peak_src,
         "algorithmic_bytes": res["bytes"], "algorithmic_flops": res["flops"],
         "hbm_frac": gbs / hbm_peak, "tensor_frac_of_bf16_peak": tfl / bf16_peak,
         "ms_per_launch": res["ms_decode"], "launches_timed": res["kernel_steps"]}
    return r


# ------------------------------------------------------------------ GPU arm
def build_step(w, torch, api):
    """Device buffers and the three per-kernel callables of one step."""
    g = w.to("cuda")
    meta, ns = api.mla_get_metadata(g.cache_seqlens, w.h_q, w.s_q)
    call = api.DecodeCall(g.q, g.k_cache, g.block_table, g.cache_seqlens, w.softmax_scale,
                          w.causal, meta, ns)

    def sched():
        api.mla_get_metadata(g.cache_seqlens, w.h_q, w.s_q, meta=meta, num_splits=ns)

    return g, meta, ns, call, sched


def capture(torch, fn):
    gr = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm the allocator/stream state once outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(gr):
        fn()
    torch.cuda.synchronize()
    return gr


CALLS_PER_GRAPH = 8


def time_calls(torch, fn, K, W, dist=None):
    """Time exactly K calls of fn (one step each), launched as CUDA graphs of
    CALLS_PER_GRAPH consecutive calls -- the way a model's layers issue them
    back to back, so that programmatic launch overlaps each call with the
    previous one -- plus one graph of the remainder.  At least W calls of
    warm-up.  Returns (ms for the K calls, wall-clock window)."""
    G = max(1, min(CALLS_PER_GRAPH, K))

    def calls(n):
        def run():
            for _ in range(n):
                fn()
        return run

    gr = capture(torch, calls(G))
    rem = K - (K // G) * G
    gr_rem = capture(torch, calls(rem)) if rem else None
    for _ in range((W + G - 1) // G):
        gr.replay()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record()
    for _ in range(K // G):
        gr.replay()
    if gr_rem is not None:
        gr_rem.replay()
    e1.record()
    torch.cuda.synchronize()
    t1 = time.time()
    if dist is not None:
        dist.barrier()
    del gr, gr_rem
    return e0.elapsed_time(e1), (t0, t1)


def time_steps_flushed(torch, graph, K, flush_buf):
    """Average duration (ms) of one replay of `graph` when L2 is cold: each
    replay is preceded by a write of flush_buf, outside the events."""
    K = max(1, min(K, 2000))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush_buf.add_(1)
        ev[i][0].record()
        graph.replay()
        ev[i][1].record()
    torch.cuda.synchronize()
    return sum(e[0].elapsed_time(e[1]) for e in ev) / K


def time_kernels(torch, g_sched, g_split, g_comb, K, flush_buf):
    """Average duration (ms) of each kernel over K steps, from events placed
    between separately launched single-kernel graphs."""
    K = max(1, min(K, 2000))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    t0 = time.time()
    for i in range(K):
        flush_buf.add_(1)  # evict L2 before the step, outside the events
        ev[i][0].record()
        g_sched.replay()
        ev[i][1].record()
        g_split.replay()
        ev[i][2].record()
        g_comb.replay()
        ev[i][3].record()
    torch.cuda.synchronize()
    t1 = time.time()
    sums = [0.0, 0.0, 0.0]
    for i in range(K):
        for k in range(3):
            sums[k] += ev[i][k].elapsed_time(ev[i][k + 1])
    return [s / K for s in sums], K, (t0, t1)


def measure_workload(w, torch, api, W_mod, K, Wup, dist=None):
    g, meta, ns, call, sched = build_step(w, torch, api)

    # One step = mla_decode_fwd (split-KV decode + combine).  The plan from
    # mla_get_metadata is built once per decode step and reused by every
    # layer, so it stays outside the timed step and is timed on its own.
    def full_step():
        call.fwd()

    gr_full = capture(torch, full_step)
    gr_sched = capture(torch, sched)
    gr_split = capture(torch, call.splitkv)
    gr_comb = capture(torch, call.combine)
    assert api.mla_last_device_error() == 0
    ms_total, win1 = time_calls(torch, full_step, K, Wup, dist)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    flush.zero_()
    kt, k_used, win2 = time_kernels(torch, gr_sched, gr_split, gr_comb, K, flush)
    ms_flushed = time_steps_flushed(torch, gr_full, K, flush)
    code = api.mla_last_device_error()
    assert code == 0, f"device error {code}"
    seqlens = w.cache_seqlens.tolist()
    res = {
        "ms_total": ms_total, "ms_per_step": ms_total / K, "ms_per_step_flushed": ms_flushed,
        "ms_sched": kt[0], "ms_decode": kt[1], "ms_combine": kt[2], "kernel_steps": k_used,
        "flops": W_mod.flops(seqlens, w.s_q, w.h_q, w.causal),
        "bytes": W_mod.hbm_bytes(seqlens, w.s_q, w.h_q),
        "pieces": int(ns[-1].item()), "windows": [win1, win2],
    }
    del gr_full, gr_sched, gr_split, gr_comb, flush
    return res, (g, call)


def measure_sparse(w, torch, api, W_mod, K, Wup):
    """Sparse decode (per-token key lists): mla_decode_sparse_fwd steps in a
    CUDA graph; the plan is built once, outside the timed steps."""
    g = w.to("cuda")
    meta, ns = api.mla_get_metadata_sparse(w.topk, w.b, w.h_q, w.s_q)
    call = api.SparseDecodeCall(g.q, g.k_cache, g.indices, w.softmax_scale, meta, ns)
    ms_total, _ = time_calls(torch, call.fwd, K, Wup)
    code = api.mla_last_device_error()
    assert code == 0, f"device error {code}"
    res = {"ms_per_step": ms_total / K, "flops": W_mod.sparse_flops(w.indices, w.h_q),
           "bytes": W_mod.sparse_hbm_bytes(w.indices, w.h_q), "pieces": int(ns[-1].item())}
    del call, g
    return res


def measure_fp8(w, torch, api, W_mod, K, Wup):
    """Decode over the FP8-layout cache: mla_decode_fp8_fwd steps in a CUDA
    graph; the plan is built once, outside the timed steps."""
    g = w.to("cuda")
    meta, ns = api.mla_get_metadata(g.cache_seqlens, w.h_q, w.s_q)
    call = api.Fp8DecodeCall(g.q, g.k_cache, g.block_table, g.cache_seqlens, w.softmax_scale,
                             w.causal, meta, ns)
    ms_total, _ = time_calls(torch, call.fwd, K, Wup)
    code = api.mla_last_device_error()
    assert code == 0, f"device error {code}"
    sl = w.cache_seqlens.tolist()
    res = {"ms_per_step": ms_total / K, "flops": W_mod.flops(sl, w.s_q, w.h_q, w.causal),
           "bytes": W_mod.fp8_hbm_bytes(sl, w.s_q, w.h_q), "tokens": sum(sl)}
    del call, g
    return res


def e2e_measure(w, torch, api, steps):
    """Public API from pinned host buffers, copies inside the timed region."""
    host = {
        "q": w.q.pin_memory(), "k_cache": w.k_cache.pin_memory(),
        "block_table": w.block_table.pin_memory(), "cache_seqlens": w.cache_seqlens.pin_memory(),
    }
    dev = {k: torch.empty_like(v, device="cuda") for k, v in host.items()}
    out_h = torch.empty(w.b, w.s_q, w.h_q, 512, dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty(w.b, w.h_q, w.s_q, dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()

    def step():
        for k in host:
            dev[k].copy_(host[k], non_blocking=True)
        meta, ns = api.mla_get_metadata(dev["cache_seqlens"], w.h_q, w.s_q)
        out, lse = api.mla_decode_fwd(dev["q"], dev["k_cache"], dev["block_table"],
                                      dev["cache_seqlens"], w.softmax_scale, w.causal, meta, ns)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return ms, h2d, d2h


# --------------------------------------------------------------- CPU oracle
def oracle_throughput(w, seconds, W_mod, max_units=None):
    """Time the fp64 oracle on this host over a bounded row sample; return
    (GB/s of algorithmic bytes, TFLOP/s, cores, sample description)."""
    import numpy as np

    import oracle

    cores = os.cpu_count() or 1
    p = oracle.Problem(oracle.bf16_bits(w.q), oracle.bf16_bits(w.k_cache), w.block_table.numpy(),
                       w.cache_seqlens.numpy(), w.softmax_scale, w.causal)
    R = w.s_q * w.h_q
    total_units = w.b * R
    order = np.random.default_rng(0).permutation(total_units)
    units_all = np.stack([order // R, order % R], axis=1).astype(np.int32)
    # calibrate on one unit per core
    n = min(total_units, cores)
    t0 = time.time()
    oracle.mla_decode_rows(p, units_all[:n], nthreads=cores)
    dt = max(time.time() - t0, 1e-6)
    n_target = int(n * seconds / dt)
    if max_units:
        n_target = min(n_target, max_units)
    n_run = max(n, min(total_units, n_target))
    t0 = time.time()
    oracle.mla_decode_rows(p, units_all[:n_run], nthreads=cores)
    dt = time.time() - t0
    nbytes, nflops = W_mod.unit_work(w.cache_seqlens.tolist(), w.s_q, w.h_q, w.causal,
                                     units_all[:n_run])
    gbs = nbytes / dt / 1e9
    tfl = nflops / dt / 1e12
    sample = (f"{n_run} of {total_units} (request, row) units in a seeded random order, "
              f"{dt:.1f} s; bytes and FLOPs of exactly those rows")
    return gbs, tfl, cores, sample, dt


def reference_arm(args, rank, world):
    """--impl reference: the oracle on the host cores, bounded sample per step."""
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    from decode_attention_paged_gb300 import workloads as W_mod

    w = W_mod.CONFIGS[args.workload]()
    cores = os.cpu_count() or 1
    p = oracle.Problem(oracle.bf16_bits(w.q), oracle.bf16_bits(w.k_cache), w.block_table.numpy(),
                       w.cache_seqlens.numpy(), w.softmax_scale, w.causal)
    R = w.s_q * w.h_q
    total_units = w.b * R
    # the seeded random order of oracle_throughput: every step's rows are a
    # representative mix of the workload's requests, and the work counted is
    # that of exactly the rows computed
    order = np.random.default_rng(0).permutation(total_units)
    units_all = np.stack([order // R, order % R], axis=1).astype(np.int32)
    seqlens = w.cache_seqlens.tolist()
    t0 = time.time()
    oracle.mla_decode_rows(p, units_all[:cores], nthreads=cores)
    t_batch = max(time.time() - t0, 1e-6)
    budget = 150.0  # seconds for warmup + timed steps together
    per_step = budget / max(1, args.steps + args.warmup)
    batches = max(1, int(per_step / t_batch))
    n_step = min(total_units, cores * batches)
    for i in range(args.warmup):
        oracle.mla_decode_rows(p, units_all[:n_step], nthreads=cores)
    nbytes = nflops = 0.0
    t_run = 0.0
    for i in range(args.steps):
        s = (i * n_step) % total_units
        idx = np.arange(s, s + n_step) % total_units
        t0 = time.time()
        oracle.mla_decode_rows(p, units_all[idx], nthreads=cores)
        t_run += time.time() - t0
        b_i, f_i = W_mod.unit_work(seqlens, w.s_q, w.h_q, w.causal, units_all[idx])
        nbytes += b_i
        nflops += f_i
    dt = t_run
    gbs = nbytes / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.b, "s_q": w.s_q, "h_q": w.h_q,
                   "page": 64, "parallelism": "host cores"},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n_step} of {total_units} (request, row) units per step, "
                                   "seeded random order; bytes and FLOPs of those rows"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "tflops": nflops / dt / 1e12,
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------- main
def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return reference_arm(args, rank, world)

    import torch

    from decode_attention_paged_gb300 import _build

    dist = None
    if world > 1:
        import torch.distributed as td

        td.init_process_group("gloo")
        dist = td
        if rank == 0:
            _build.build()
        td.barrier()  # rank 0 builds; the others then find the library up to date
    _build.build()
    torch.cuda.set_device(local)
    from decode_attention_paged_gb300 import api
    from decode_attention_paged_gb300 import workloads as W_mod

    api.set_decode_kernel({"auto": api.KERNEL_AUTO, "single": api.KERNEL_SINGLE,
                           "tq": api.KERNEL_TQ, "duo": api.KERNEL_DUO}[args.kernel])
    hbm_peak, bf16_peak, bf16_sust, peak_src = load_peaks()
    if args.sparse_only:
        if rank == 0:
            ws = W_mod.sparse()
            r = measure_sparse(ws, torch, api, W_mod, args.steps, args.warmup)
            print(json.dumps({"sparse": sparse_line(ws, r, sparse_kernel_of(args.kernel, ws.h_q),
                                                    (hbm_peak, bf16_peak), args.steps)}),
                  flush=True)
        if dist is not None:
            dist.barrier()
        return 0
    # weak scaling: every rank decodes its own batch of requests (replicas).
    w = replica_workload(W_mod, args.workload, rank)
    sampler = ClockSampler(list(range(world)) if world > 1 else [local]) if rank == 0 else None
    if sampler:
        sampler.start()
    res, (g, call) = measure_workload(w, torch, api, W_mod, args.steps, args.warmup, dist)
    if sampler:
        sampler.stop()

    ms_total = max_over_ranks(res["ms_total"], dist)
    ms_step = ms_total / args.steps
    gbs = res["bytes"] * world / (ms_step * 1e-3) / 1e9
    tflops = res["flops"] * world / (ms_step * 1e-3) / 1e12

    e2e = None
    if not args.no_e2e:
        ms_e2e, h2d, d2h = e2e_measure(w, torch, api, steps=max(3, min(args.steps, 20)))
        e2e = {"value": res["bytes"] * world / (ms_e2e * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e}
    del g, call
    torch.cuda.empty_cache()

    if rank != 0:
        if dist is not None:
            dist.barrier()
        return 0

    clocks = sampler.summary() if sampler else None
    peaks = (hbm_peak, bf16_peak, bf16_sust, peak_src)
    roofline = roofline_of(res, args.workload, kernel_of(args.kernel, w), peaks)
    flushed = {"ms_per_step": res["ms_per_step_flushed"],
               "value": res["bytes"] / (res["ms_per_step_flushed"] * 1e-3) / 1e9, "unit": "GB/s",
               "what": "mean of up to 2000 replays of the step graph, each after a 2x L2 write "
                       "outside the events (rank 0)"}

    cpu = None
    if world == 1 and not args.no_cpu:
        c_gbs, c_tfl, cores, sample, _ = oracle_throughput(W_mod.CONFIGS[args.workload](),
                                                           args.cpu_seconds, W_mod)
        cpu = {"value": c_gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": sample, "tflops": c_tfl}

    extra = {}
    if not args.no_extra:
        for name in ("compute_bound", "mtp", "long_ragged"):
            if name == args.workload:
                continue
            wx = W_mod.CONFIGS[name]()
            kx = max(50, min(args.steps, 1000))
            r, (gx, cx) = measure_workload(wx, torch, api, W_mod, kx, 5)
            extra[name] = {
                "workload": wx.name,
                "ms_per_step": r["ms_per_step"], "ms_per_step_flushed": r["ms_per_step_flushed"],
                "ms_decode": r["ms_decode"],
                "ms_combine": r["ms_combine"], "ms_sched": r["ms_sched"],
                "decode_tflops": r["flops"] / (r["ms_decode"] * 1e-3) / 1e12,
                "decode_gbs": r["bytes"] / (r["ms_decode"] * 1e-3) / 1e9,
                "step_tflops": r["flops"] / (r["ms_per_step"] * 1e-3) / 1e12,
                "frac_bf16_peak": r["flops"] / (r["ms_decode"] * 1e-3) / 1e12 / bf16_peak,
                "frac_hbm_peak": r["bytes"] / (r["ms_decode"] * 1e-3) / 1e9 / hbm_peak,
                "pieces": r["pieces"], "steps": kx,
                "roofline": roofline_of(r, name, kernel_of(args.kernel, wx), peaks),
            }
            del gx, cx
            torch.cuda.empty_cache()
        wf = W_mod.memory_bound_fp8()
        kx = max(50, min(args.steps, 1000))
        r = measure_fp8(wf, torch, api, W_mod, kx, 5)
        t_s = r["ms_per_step"] * 1e-3
        extra["memory_bound_fp8"] = {
            "workload": wf.name, "ms_per_step": r["ms_per_step"],
            "step_gbs": r["bytes"] / t_s / 1e9, "step_tflops": r["flops"] / t_s / 1e12,
            "frac_hbm_peak": r["bytes"] / t_s / 1e9 / hbm_peak,
            "tokens_per_s": r["tokens"] / t_s, "steps": kx,
        }
        del wf
        torch.cuda.empty_cache()
        wh = W_mod.gqa()
        kx = max(50, min(args.steps, 1000))
        gh = wh.to("cuda")
        meta_h, ns_h = api.mla_get_metadata(gh.cache_seqlens, wh.h_q, wh.s_q, wh.h_kv)
        call_h = api.DecodeCall(gh.q, gh.k_cache, gh.block_table, gh.cache_seqlens,
                                wh.softmax_scale, wh.causal, meta_h, ns_h)
        ms_h, _ = time_calls(torch, call_h.fwd, kx, 5)
        assert api.mla_last_device_error() == 0
        t_s = ms_h / kx * 1e-3
        sl = wh.cache_seqlens.tolist()
        bytes_h = W_mod.heads_hbm_bytes(sl, wh.s_q, wh.h_q, wh.h_kv)
        flops_h = W_mod.flops(sl, wh.s_q, wh.h_q, wh.causal)
        extra["gqa"] = {
            "workload": wh.name, "ms_per_step": ms_h / kx,
            "step_gbs": bytes_h / t_s / 1e9, "step_tflops": flops_h / t_s / 1e12,
            "frac_hbm_peak": bytes_h / t_s / 1e9 / hbm_peak, "steps": kx,
        }
        del call_h, gh, wh
        torch.cuda.empty_cache()
        ws = W_mod.sparse()
        kx = max(50, min(args.steps, 1000))
        r = measure_sparse(ws, torch, api, W_mod, kx, 5)
        extra["sparse"] = sparse_line(ws, r, sparse_kernel_of(args.kernel, ws.h_q), peaks, kx)
        del ws
        torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.b, "s_q": w.s_q, "h_q": w.h_q,
                   "seqlen": int(w.cache_seqlens.max()), "page": 64, "d_qk": 576, "d_v": 512,
                   "causal": w.causal, "parallelism": f"replicas x{world}",
                   "l2": "value: back-to-back steps, inputs larger than L2 (KV 302 MB "
                         "vs 129 MB); step_l2_flushed and roofline: L2 flushed before each "
                         "step / launch",
                   "launch": f"steps as CUDA graphs of {CALLS_PER_GRAPH} consecutive calls"},
        "tflops": tflops, "frac_hbm_peak_step": gbs / world / hbm_peak,
        "step_l2_flushed": flushed,
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": 2 * args.steps, "clocks": clocks,
        "kernel_ms": {"sched": res["ms_sched"], "decode": res["ms_decode"],
                      "combine": res["ms_combine"]},
        "pieces": res["pieces"], "other_workloads": extra,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
    return 0


if __name__ == "__main__":
    sys.exit(main())
