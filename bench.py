#!/usr/bin/env python3
"""Benchmark of the fused INT4 dequant-GEMV on one GB300 (or N replicas).

Workload (one "step"): the decode MLP GEMV pair at M = 1 -- the up projection
N=15360, K=3840 followed by the down projection N=3840, K=15360, INT4
asymmetric weights with FP16 scale/zero per 128 codes, BF16 activations and
outputs (Gemma4-12B-shaped linears; synthetic seeded data), two GEMV launches
chained by programmatic dependent launch.  Eight rotating weight sets (about
500 MB) keep every step's weights out of the 129 MB L2.

Metric: whole-job HBM throughput in GB/s over the algorithmic bytes (packed
weights + scales + zeros + activations + outputs).  Also reported: the
roofline of the GEMV kernel, the same metric end to end through the C ABI
with host buffers, per-configuration kernel timings, GPU clocks during the
timed region, and the CPU oracle timed on a bounded sample.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Multi-GPU: launched under torchrun, one process per GPU; every rank runs an
independent replica (the path needs no exchange), rank 0 prints the line.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused INT4 dequant-GEMV HBM GB/s (% of peak) at M=1; TFLOPS at M=128"
WORKLOAD = ("decode MLP GEMV pair, M=1: up N=15360 K=3840 then down N=3840 K=15360, "
            "INT4 group-128 asymmetric, FP16 scale/zero, BF16 x and y")
UP = (15360, 3840)
DOWN = (3840, 15360)
L2_SETS = 8
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def gemv_bytes(N, K, group=128):
    """Algorithmic bytes of one M=1 GEMV: packed W + s + z + x + y."""
    G = K // group
    return N * K // 2 + 2 * N * G * 2 + 2 * K + 2 * N


STEP_BYTES = gemv_bytes(*UP) + gemv_bytes(*DOWN)


def kernel_sources_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gemm_w4a16_gemv_gb300", "csrc")
    for name in ("gemv_kernel.cuh", "gemv_common.cuh", "common.cuh", "gemv_int4.cu"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def read_traffic(digest):
    """DRAM bytes per launch of the GEMV kernel from the committed ncu summary,
    or None when the summary was taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", "gemv_int4_decode_mlp_pair.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_sources_sha256_16") != digest:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_setup():
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def dist_max(value, device=None):
    """Max of a float over ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# --------------------------------------------------------------- CPU oracle

def oracle_rows_per_second(oracle, synth, N, K, rows):
    p = synth.int4_problem(rows, K, seed=11)
    t0 = time.perf_counter()
    oracle.gemv_int4(p["x"], p["qw"], p["s"], p["z"], K=K)
    return rows / (time.perf_counter() - t0)


def host_cpu():
    """(usable cores, CPU model name) of this host."""
    try:
        cores = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        cores = os.cpu_count() or 1
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return cores, model or "unknown"


def oracle_step_sample(oracle, synth, seconds, threads=1):
    """A bounded sample of one step for the CPU oracle: the same fraction of
    the up and the down projection rows, sized to take about `seconds` with
    `threads` threads.  Returns (callable running the sample, algorithmic
    bytes of the sample, description)."""
    oracle.set_threads(threads)
    oracle_rows_per_second(oracle, synth, UP[0], UP[1], 2)  # load the library first
    up_rps = oracle_rows_per_second(oracle, synth, UP[0], UP[1], 64 * threads)
    dn_rps = oracle_rows_per_second(oracle, synth, DOWN[0], DOWN[1], 16 * threads)
    # fraction f of both projections: f*UP[0]/up_rps + f*DOWN[0]/dn_rps = seconds
    f = seconds / (UP[0] / up_rps + DOWN[0] / dn_rps)
    f = max(min(f, 1.0), 1e-4)
    n_up = max(2, int(UP[0] * f))
    n_dn = max(2, int(DOWN[0] * f))
    pu = synth.int4_problem(n_up, UP[1], seed=0)
    pd = synth.int4_problem(n_dn, DOWN[1], seed=1)

    def run():
        oracle.gemv_int4(pu["x"], pu["qw"], pu["s"], pu["z"], K=UP[1])
        oracle.gemv_int4(pd["x"], pd["qw"], pd["s"], pd["z"], K=DOWN[1])

    sample_bytes = (n_up * (UP[1] // 2 + 4 * (UP[1] // 128)) + 2 * UP[1] + 2 * n_up
                    + n_dn * (DOWN[1] // 2 + 4 * (DOWN[1] // 128)) + 2 * DOWN[1] + 2 * n_dn)
    desc = "%d of %d up rows + %d of %d down rows per step, %d thread%s" % (
        n_up, UP[0], n_dn, DOWN[0], threads, "" if threads == 1 else "s (OpenMP over output rows)")
    return run, sample_bytes, desc


def cpu_baseline(seconds=10.0):
    """The oracle timed on this host: on all its cores (the reported value)
    and on one core; each leg a bounded sample of the step."""
    import oracle
    import synth
    cores, model = host_cpu()

    def leg(threads, secs):
        run, nbytes, desc = oracle_step_sample(oracle, synth, secs / 2, threads)
        t0 = time.perf_counter()
        n = 0
        while True:
            run()
            n += 1
            if time.perf_counter() - t0 >= secs / 2:
                break
        dt = time.perf_counter() - t0
        return nbytes * n / dt / 1e9, desc + ", %d repetitions in %.1f s" % (n, dt)

    try:
        v_all, d_all = leg(cores, seconds)
        v_one, d_one = leg(1, seconds / 2)
    finally:
        oracle.set_threads(1)
    return {"value": round(v_all, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": d_all,
            "cpu_model": model, "single_thread": {"value": round(v_one, 4), "unit": "GB/s", "sample": d_one}}


def run_reference(args):
    """The CPU oracle as the reference arm: K timed steps, each a bounded
    sample of the workload, on the host cores (rank 0 only)."""
    world, rank, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return 0
    import oracle
    import synth
    cores, model = host_cpu()
    per_step = max(0.05, 100.0 / max(1, args.steps + args.warmup))
    run, nbytes, desc = oracle_step_sample(oracle, synth, per_step, cores)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    oracle.set_threads(1)
    value = nbytes * args.steps / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": desc},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": desc, "cpu_model": model},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm

def make_gemv_sets(torch, synth, dev, N, K, seed, nsets):
    """Seeded host problem; `nsets` device copies of its weights (distinct
    addresses, so rotating through them streams from HBM, not L2)."""
    p = synth.int4_problem(N, K, seed=seed)
    base = {"qw": torch.from_numpy(p["qw"]).to(dev),
            "s": torch.from_numpy(p["s"]).view(torch.float16).to(dev),
            "z": torch.from_numpy(p["z"]).view(torch.float16).to(dev)}
    sets = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(nsets - 1)]
    x_host = torch.from_numpy(p["x"].reshape(-1)).view(torch.bfloat16)
    return sets, x_host


def time_each(torch, fn, n, stream):
    """Device time of each of n launches, bracketed one by one by CUDA events
    (an event between launches also ends any overlap of consecutive
    kernels): (p10, median, p90) in seconds."""
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    torch.cuda._sleep(int(5e7))
    ev[0].record(stream)
    for i in range(n):
        fn(i)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    d = sorted(ev[i].elapsed_time(ev[i + 1]) * 1e-3 for i in range(n))
    pick = lambda q: d[min(n - 1, max(0, int(round(q * (n - 1)))))]
    return pick(0.1), pick(0.5), pick(0.9)


def spread(torch, fn, n, stream, scale=1e6):
    """p10 / median / p90 of individually bracketed launches, in us."""
    p10, p50, p90 = time_each(torch, fn, n, stream)
    return {"p10_us": round(p10 * scale, 2), "median_us": round(p50 * scale, 2), "p90_us": round(p90 * scale, 2)}


def l2_sets(nbytes, l2_bytes=129e6, cap=24):
    """Weight copies to rotate through so that their total is at least twice
    the L2 (each launch then streams its weights from HBM)."""
    return max(1, min(cap, int(2 * l2_bytes // nbytes) + 1))


def time_launches(torch, fn, n, stream):
    """Average device time of n back-to-back launches (CUDA events)."""
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    torch.cuda._sleep(int(5e7))  # queue the launches behind a short spin
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e-3 / n


# The pages' 48-layer decode step (Gemma4-12B: hidden 3840, 16 query heads and
# 8 key/value heads of 256, MLP 15360, vocabulary 262144): 40 sliding-window
# layers of 7 linears (q, k, v, o, gate, up, down) and 8 global layers of 6
# (keys and values shared: no v), 328 linears, then the vocabulary GEMV.
STEP_H, STEP_Q, STEP_KV, STEP_F, STEP_V = 3840, 4096, 2048, 15360, 262144
STEP_SLIDING, STEP_GLOBAL = 40, 8


def decode_step_ops(torch, synth, dev, fused=False):
    """The step's INT4 linears as (x, qw, s, z, y) tuples, each with its own
    weight copy (6.2 GB in all, so every step streams from HBM).  Scales are
    drawn so that a linear keeps the activations' magnitude (mean scale
    1 / (6.5 sqrt(K)), 6.5 being the spread of q - z).  Data flow through
    activation buffers: q, k, v, gate, up read the hidden state h; o reads q
    (the attention is not on this path) and writes h; down reads up and
    writes h; the vocabulary GEMV reads h."""
    protos = {}

    def weights(N, K):
        if (N, K) not in protos:
            m = 1.0 / (6.5 * K ** 0.5)
            p = synth.int4_problem(N, K, seed=N + K, s_range=(0.5 * m, 1.5 * m))
            protos[(N, K)] = (torch.from_numpy(p["qw"]).to(dev),
                              torch.from_numpy(p["s"]).view(torch.float16).to(dev),
                              torch.from_numpy(p["z"]).view(torch.float16).to(dev))
        return tuple(t.clone() for t in protos[(N, K)])

    views = decode_step_views(fused)
    store = {}
    for base, off, n in views.values():
        store[base] = max(store.get(base, 0), off + n)
    store = {k: torch.zeros(n, dtype=torch.bfloat16, device=dev) for k, n in store.items()}
    h = torch.from_numpy(synth.normal_bf16(synth.Stream(5), (STEP_H,))).view(torch.bfloat16)
    store["h"].copy_(h)

    def view(name, n):
        base, off, _ = views[name]
        return store[base][off:off + n]

    ops = [(view(src, K), *weights(N, K), view(dst, N)) for src, dst, N, K in decode_step_linears(fused)]
    protos.clear()
    return ops


def decode_step_linears(fused=False):
    """(source, destination, N, K) of the step's linears in launch order.
    fused: the linears that read the same input stored as one weight tensor
    (q|k|v and gate|up, a layout choice of the model: the same weights and
    bytes), so that one launch covers each group: 48 x 4 + 1 launches."""
    H, Q, KV, F = STEP_H, STEP_Q, STEP_KV, STEP_F
    out = []
    for layer in range(STEP_SLIDING + STEP_GLOBAL):
        sliding = layer < STEP_SLIDING
        if fused:
            out += [("h", "qkv", Q + (2 if sliding else 1) * KV, H), ("q", "h", H, Q),
                    ("h", "gateup", 2 * F, H), ("up", "h", H, F)]
            continue
        out += [("h", "q", Q, H), ("h", "k", KV, H)]
        if sliding:
            out.append(("h", "v", KV, H))
        out += [("q", "h", H, Q), ("h", "gate", F, H), ("h", "up", F, H), ("up", "h", H, F)]
    out.append(("h", "logits", STEP_V, H))
    return out


def decode_step_views(fused=False):
    """Activation buffer name -> (storage, offset, length).  In the fused
    layout q and up are the leading part of the q|k|v output and the
    trailing part of the gate|up output."""
    H, Q, KV, F = STEP_H, STEP_Q, STEP_KV, STEP_F
    v = {"h": ("h", 0, H), "logits": ("logits", 0, STEP_V)}
    if fused:
        v.update({"qkv": ("qkv", 0, Q + 2 * KV), "q": ("qkv", 0, Q),
                  "gateup": ("gateup", 0, 2 * F), "up": ("gateup", F, F)})
    else:
        v.update({"q": ("q", 0, Q), "k": ("k", 0, KV), "v": ("v", 0, KV), "gate": ("gate", 0, F),
                  "up": ("up", 0, F)})
    return v


def decode_step(torch, w4, synth, dev, stream, hbm_peak, fused=False):
    """The decode step replayed from one CUDA graph, against the same launches
    made one by one from the host (w4a16_linear_sequence)."""
    ops = decode_step_ops(torch, synth, dev, fused)
    nbytes = sum(gemv_bytes(op[1].shape[0], 2 * op[1].shape[1]) for op in ops)
    arr = w4.w4a16_linear_array(ops)
    g = w4.w4a16_graph_create(ops)
    try:
        t_graph = time_launches(torch, lambda i: g.launch(), 20, stream)
        t_seq = time_launches(torch, lambda i: w4.w4a16_linear_sequence(arr, count=len(ops)), 20, stream)
        # host time of one call of each (what a decode loop pays per step)
        torch.cuda.synchronize()
        h0 = time.perf_counter()
        for _ in range(5):
            w4.w4a16_linear_sequence(arr, count=len(ops))
        h1 = time.perf_counter()
        for _ in range(5):
            g.launch()
        h2 = time.perf_counter()
        torch.cuda.synchronize()
        status = w4.w4a16_check_device_error()
    finally:
        g.destroy()
    gbs = nbytes / t_graph / 1e9
    return {"linears": len(ops), "weights_GB": round(nbytes / 1e9, 3), "us": round(t_graph * 1e6, 1),
            "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm_peak, 3),
            "host_launched_us": round(t_seq * 1e6, 1),
            "host_us_per_step": {"sequence_call": round((h1 - h0) / 5 * 1e6, 1),
                                 "graph_launch": round((h2 - h1) / 5 * 1e6, 1)},
            "device_status": status}


def decode_step_chain(torch, w4, synth, dev, stream, hbm_peak, fused=False):
    """The decode step as chains of linears (w4a16_linear_chain: at most 192
    linears per persistent launch, two launches for the 329), timed per step,
    against the same step's per-linear launches from one graph."""
    ops = decode_step_ops(torch, synth, dev, fused)
    nbytes = sum(gemv_bytes(op[1].shape[0], 2 * op[1].shape[1]) for op in ops)
    arr = w4.w4a16_linear_array(ops)
    scratch = w4.chain_scratch(len(ops), dev)
    t = time_launches(torch, lambda i: w4.w4a16_linear_chain(arr, scratch, count=len(ops)), 20, stream)
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    for _ in range(5):
        w4.w4a16_linear_chain(arr, scratch, count=len(ops))
    h1 = time.perf_counter()
    torch.cuda.synchronize()
    status = w4.w4a16_check_device_error()
    gbs = nbytes / t / 1e9
    return {"linears": len(ops), "launches": (len(ops) + 191) // 192, "weights_GB": round(nbytes / 1e9, 3),
            "us": round(t * 1e6, 1), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm_peak, 3),
            "host_us_per_call": round((h1 - h0) / 5 * 1e6, 1), "device_status": status}


def per_config(torch, w4, synth, dev, stream, hbm_peak, tf_peak):
    """Kernel-only timings of every configuration (launches back to back)."""
    out = {}
    for name, (N, K) in {"gemv_3840x3840": (3840, 3840), "gemv_up_15360x3840": UP,
                         "gemv_down_3840x15360": DOWN, "gemv_vocab_262144x3840": (262144, 3840)}.items():
        nsets = l2_sets(gemv_bytes(N, K))
        sets, xh = make_gemv_sets(torch, synth, dev, N, K, seed=0, nsets=nsets)
        x = xh.to(dev)
        y = torch.empty(N, dtype=torch.bfloat16, device=dev)
        fn = lambda i: w4.w4a16_gemv(x, sets[i % nsets]["qw"], sets[i % nsets]["s"], sets[i % nsets]["z"], y)
        t = time_launches(torch, fn, 40, stream)
        gbs = gemv_bytes(N, K) / t / 1e9
        out[name] = {"us": round(t * 1e6, 2), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm_peak, 3),
                     "weight_sets": nsets, "each": spread(torch, fn, 100, stream)}
        del sets
        torch.cuda.empty_cache()
    # decode-sized batches through w4a16_gemm: the M rows share one pass over
    # the weights (bytes: weights + scales/zeros once, M activations/outputs)
    N, K = UP
    nsets = l2_sets(gemv_bytes(N, K))
    sets, _ = make_gemv_sets(torch, synth, dev, N, K, seed=0, nsets=nsets)
    for M in (2, 4, 8):
        X = torch.randn(M, K, device=dev).to(torch.bfloat16)
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        t = time_launches(torch, lambda i: w4.w4a16_gemm(X, sets[i % nsets]["qw"], sets[i % nsets]["s"],
                                                          sets[i % nsets]["z"], Y), 40, stream)
        nb = gemv_bytes(N, K) + (M - 1) * (2 * K + 2 * N)
        m1 = out["gemv_up_15360x3840"]["us"]
        out["decode_batch_m%d_15360x3840" % M] = {"us": round(t * 1e6, 2), "GB/s": round(nb / t / 1e9, 1),
                                                  "frac_hbm": round(nb / t / 1e9 / hbm_peak, 3),
                                                  "vs_m_single_launches": round(t * 1e6 / (M * m1), 2)}
    del sets
    torch.cuda.empty_cache()
    # MoE FP4: 64 experts resident (~1 GB), 6 selected per launch
    E, N, K, topk = 64, 4096, 7168, 6
    m = synth.fp4_moe_problem(E, N, K, topk, seed=0)
    qw = torch.from_numpy(m["qw"]).to(dev)
    s = torch.from_numpy(m["s"]).view(torch.float16).to(dev)
    x = torch.from_numpy(m["x"]).view(torch.bfloat16).to(dev)
    ids = [torch.from_numpy(synth.sample_experts(synth.Stream(100 + i), E, topk)).to(dev) for i in range(16)]
    y = torch.empty(topk, N, dtype=torch.bfloat16, device=dev)
    fn = lambda i: w4.fp4_moe_gemv(x, qw, s, ids[i % 16], y)
    t = time_launches(torch, fn, 40, stream)
    mb = topk * (N * K // 2 + 2 * N * (K // 32)) + 2 * K + 2 * topk * N + 4 * topk
    out["moe_fp4_64x4096x7168_top6"] = {"us": round(t * 1e6, 2), "GB/s": round(mb / t / 1e9, 1),
                                        "frac_hbm": round(mb / t / 1e9 / hbm_peak, 3),
                                        "each": spread(torch, fn, 100, stream)}
    # the same resident experts for M tokens routed 6 ways (fp4_moe_gemm):
    # bytes = the weights of every expert used (once) + tokens and outputs
    for M in (16, 128):
        g = synth.Stream(200 + M)
        idm = torch.stack([torch.from_numpy(synth.sample_experts(g, E, topk)) for _ in range(M)]).to(dev)
        X = torch.randn(M, K, device=dev).to(torch.bfloat16)
        Y = torch.empty(M, topk, N, dtype=torch.bfloat16, device=dev)
        scr = torch.empty(w4.fp4_moe_gemm_scratch_bytes(M, topk, E, K), dtype=torch.uint8, device=dev)
        fn = lambda i: w4.fp4_moe_gemm(X, qw, s, idm, Y, scr)
        t = time_launches(torch, fn, 20, stream)
        used = int(torch.unique(idm).numel())
        gb = used * (N * K // 2 + 2 * N * (K // 32)) + 2 * M * K + 2 * M * topk * N + 4 * M * topk
        tf = 2.0 * M * topk * N * K / t / 1e12
        out["moe_fp4_gemm_m%d_64x4096x7168_top6" % M] = {
            "us": round(t * 1e6, 2), "experts_used": used, "GB/s": round(gb / t / 1e9, 1),
            "frac_hbm": round(gb / t / 1e9 / hbm_peak, 3), "TFLOP/s": round(tf, 1),
            "frac_bf16": round(tf / tf_peak, 4), "launches_per_call": 3}
    del qw, s
    torch.cuda.empty_cache()
    # prefill GEMM through the tensor cores
    for M in (128, 2048):
        name = "gemm_m%d_15360x3840" % M
        try:
            N, K = 15360, 3840
            ns = l2_sets(gemv_bytes(N, K))
            sets, _ = make_gemv_sets(torch, synth, dev, N, K, seed=0, nsets=ns)
            X = torch.randn(M, K, device=dev).to(torch.bfloat16)
            Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            fn = lambda i: w4.w4a16_gemm(X, sets[i % ns]["qw"], sets[i % ns]["s"], sets[i % ns]["z"], Y)
            t = time_launches(torch, fn, 20, stream)
            tf = 2.0 * M * N * K / t / 1e12
            out[name] = {"us": round(t * 1e6, 2), "TFLOP/s": round(tf, 1), "frac_bf16": round(tf / tf_peak, 3),
                         "weight_sets": ns, "each": spread(torch, fn, 50, stream)}
            # the binary16-operand variant (w4a16_gemm_f16: pre-pass + GEMM, and at
            # M = 2048 the reduction of the K-split tiles past the last full wave)
            fn16 = lambda i: w4.w4a16_gemm_f16(X, sets[i % ns]["qw"], sets[i % ns]["s"], sets[i % ns]["z"], Y)
            t16 = time_launches(torch, fn16, 20, stream)
            tf16 = 2.0 * M * N * K / t16 / 1e12
            out["gemm_f16_m%d_15360x3840" % M] = {"us": round(t16 * 1e6, 2), "TFLOP/s": round(tf16, 1),
                                                  "frac_bf16": round(tf16 / tf_peak, 3), "weight_sets": ns,
                                                  "launches_per_call": 3 if M >= 2048 else 2}
            del sets
        except Exception as e:  # the tensor-core GEMM may be unavailable on this device
            out[name] = {"unavailable": str(e).splitlines()[0][:120]}
        torch.cuda.empty_cache()
    # the unfused two-pass ablation: dequantise to BF16 weights in HBM, then
    # the dense BF16 GEMM (both this library's kernels), at the same shapes
    for M in (128, 2048):
        name = "two_pass_m%d_15360x3840" % M
        try:
            N, K = 15360, 3840
            ns = l2_sets(gemv_bytes(N, K))
            sets, _ = make_gemv_sets(torch, synth, dev, N, K, seed=0, nsets=ns)
            nw = l2_sets(2 * N * K)  # BF16 weight matrices, 118 MB each
            Wb = [torch.empty(N, K, dtype=torch.bfloat16, device=dev) for _ in range(nw)]
            X = torch.randn(M, K, device=dev).to(torch.bfloat16)
            Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)

            def deq(i):
                w4.w4a16_dequant(w4.FMT_INT4, sets[i % ns]["qw"], sets[i % ns]["s"], sets[i % ns]["z"],
                                 out=Wb[i % nw], out_dtype=w4.OUT_BF16)

            t_deq = time_launches(torch, deq, 20, stream)
            t_mm = time_launches(torch, lambda i: w4.w4a16_bf16_gemm(X, Wb[i % nw], Y), 20, stream)
            t_two = time_launches(torch, lambda i: (deq(i), w4.w4a16_bf16_gemm(X, Wb[i % nw], Y)), 20, stream)
            fused = out.get("gemm_m%d_15360x3840" % M, {}).get("us")
            fused16 = out.get("gemm_f16_m%d_15360x3840" % M, {}).get("us")
            out[name] = {"us": round(t_two * 1e6, 2), "dequant_us": round(t_deq * 1e6, 2),
                         "bf16_gemm_us": round(t_mm * 1e6, 2),
                         "bf16_gemm_TFLOP/s": round(2.0 * M * N * K / t_mm / 1e12, 1),
                         "fused_speedup": round(t_two * 1e6 / fused, 2) if fused else None,
                         "fused_f16_speedup": round(t_two * 1e6 / fused16, 2) if fused16 else None}
            del sets, Wb
        except Exception as e:
            out[name] = {"unavailable": str(e).splitlines()[0][:120]}
        torch.cuda.empty_cache()
    # the whole decode step (328 linears and the vocabulary GEMV) as one graph;
    # then the same weights with q|k|v and gate|up each stored as one tensor
    for name, fused in (("decode_step_328_linears_vocab", False), ("decode_step_fused_qkv_gateup", True)):
        try:
            out[name] = decode_step(torch, w4, synth, dev, stream, hbm_peak, fused)
        except Exception as e:
            out[name] = {"unavailable": str(e).splitlines()[0][:120]}
        torch.cuda.empty_cache()
        try:
            out[name + "_chain"] = decode_step_chain(torch, w4, synth, dev, stream, hbm_peak, fused)
        except Exception as e:
            out[name + "_chain"] = {"unavailable": str(e).splitlines()[0][:120]}
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    import gemm_w4a16_gemv_gb300 as w4
    import synth

    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (use --impl reference for the CPU oracle)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    hbm_peak, tf_peak, tf_sust, peak_src = read_peaks()

    up_sets, xu_h = make_gemv_sets(torch, synth, dev, *UP, seed=0, nsets=L2_SETS)
    dn_sets, xd_h = make_gemv_sets(torch, synth, dev, *DOWN, seed=1, nsets=L2_SETS)
    xu, xd = xu_h.to(dev), xd_h.to(dev)
    # both outputs in one buffer (the end-to-end step reads them back in one copy)
    y_all = torch.empty(UP[0] + DOWN[0], dtype=torch.bfloat16, device=dev)
    yu, yd = y_all[:UP[0]], y_all[UP[0]:]

    # one op array per weight set: the pair as a chain (the two linears are
    # independent, so the chain streams them back to back in one launch)
    scratch = w4.chain_scratch(2, dev)

    def pair_ops(i, x_up, x_dn, y_up, y_dn):
        a, b = up_sets[i % L2_SETS], dn_sets[i % L2_SETS]
        return w4.w4a16_linear_array([(x_up, a["qw"], a["s"], a["z"], y_up), (x_dn, b["qw"], b["s"], b["z"], y_dn)])

    arrays = [pair_ops(i, xu, xd, yu, yd) for i in range(L2_SETS)]

    def step(i, x_up=xu, x_dn=xd):
        a, b = up_sets[i % L2_SETS], dn_sets[i % L2_SETS]
        w4.w4a16_gemv(x_up, a["qw"], a["s"], a["z"], yu)
        w4.w4a16_gemv(x_dn, b["qw"], b["s"], b["z"], yd)

    def step_chain(i):
        w4.w4a16_linear_chain(arrays[i % L2_SETS], scratch, count=2)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if w4.w4a16_check_device_error() != 0:
        raise SystemExit("device status set during warm-up")

    # CUDA graphs: one holding a step for each of the L2_SETS weight sets back
    # to back (so consecutive launches chain inside the graph), and one
    # holding the remaining steps % L2_SETS steps, likewise chained; the timed
    # loop runs exactly args.steps steps.
    graphs = None
    if not args.no_graph:
        try:
            whole = torch.cuda.CUDAGraph()
            with torch.cuda.graph(whole):
                for i in range(L2_SETS):
                    step(i)
            rest = None
            if args.steps % L2_SETS:
                rest = torch.cuda.CUDAGraph()
                with torch.cuda.graph(rest):
                    for i in range(args.steps % L2_SETS):
                        step(i)
            whole.replay()
            if rest is not None:
                rest.replay()
            torch.cuda.synchronize()
            graphs = (whole, rest)
        except Exception:
            graphs = None
            torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    dist_barrier()
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e7))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    if graphs is not None:
        whole, rest = graphs
        for _ in range(args.steps // L2_SETS):
            whole.replay()
        if rest is not None:
            rest.replay()
    else:
        for i in range(args.steps):
            step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    dist_barrier()
    clk = clocks.stop()
    elapsed = e0.elapsed_time(e1) * 1e-3
    status = w4.w4a16_check_device_error()
    elapsed_max = dist_max(elapsed, dev if torch.distributed.is_initialized() and
                           torch.distributed.get_backend() == "nccl" else None)
    value = STEP_BYTES * args.steps * world / elapsed_max / 1e9

    # roofline of the GEMV kernel: the step is two launches of it
    launch_s = elapsed / (2 * args.steps)
    achieved = (STEP_BYTES / 2) / launch_s / 1e9
    digest = kernel_sources_digest()
    traffic = read_traffic(digest)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs: copy bandwidth)" if peak_src == "measured"
                else "fallback 6.8 TB/s", "kernel": "gemv_stream_kernel<INT4>",
                "bytes_per_launch": STEP_BYTES // 2, "launch_us": round(launch_s * 1e6, 3)}

    # end to end through the C ABI with host buffers: H2D x, two GEMVs, D2H y
    # one pinned host buffer and one copy each way per step: both activation
    # vectors in, both output vectors out
    x_pin = torch.cat([xu_h.reshape(-1), xd_h.reshape(-1)]).pin_memory()
    y_pin = torch.empty(UP[0] + DOWN[0], dtype=torch.bfloat16).pin_memory()
    x_d = torch.empty(x_pin.numel(), dtype=torch.bfloat16, device=dev)
    xu_d, xd_d = x_d[:UP[1]], x_d[UP[1]:]
    e2e_steps = min(args.steps, 300)

    def e2e_body(i):
        w4.w4a16_copy(x_d, x_pin)
        step(i, xu_d, xd_d)
        w4.w4a16_copy(y_pin, y_all)

    # As a decode loop runs it: the step -- the activations copied in from
    # pinned host memory, the two library calls, the outputs copied out to
    # pinned host memory, the copies by the library's copy kernel (reading
    # and writing the mapped host buffers) so that all four launches chain
    # by programmatic dependent launch -- captured once per weight set into a
    # CUDA graph, replayed once per step, and the host waits for each step's
    # result.  The copies read and write the host buffers at every replay.
    e2e_graphs = None
    if not args.no_graph:
        try:
            e2e_graphs = []
            for i in range(L2_SETS):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    e2e_body(i)
                e2e_graphs.append(g)
            torch.cuda.synchronize()
        except Exception:
            e2e_graphs = None

    def e2e_step(i):
        if e2e_graphs is not None:
            e2e_graphs[i % L2_SETS].replay()
        else:
            e2e_body(i)
        torch.cuda.current_stream().synchronize()

    for i in range(3):
        e2e_step(i)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    e2e_dt = time.perf_counter() - t0
    e2e_dt = dist_max(e2e_dt, dev if torch.distributed.is_initialized() and
                      torch.distributed.get_backend() == "nccl" else None)
    h2d = 2 * (UP[1] + DOWN[1])
    d2h = 2 * (UP[0] + DOWN[0])
    e2e = {"value": round(STEP_BYTES * e2e_steps * world / e2e_dt / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "sync_per_step": True,
           "launch": ("one CUDA graph per step (w4a16_copy of the pinned activations in, the two library "
                      "calls, w4a16_copy of the outputs out to pinned memory)"
                      if e2e_graphs is not None else "eager (copies and library calls per step)")}

    extra = {}
    if rank == 0 and not args.no_configs:
        t2 = time_launches(torch, step_chain, 400, stream)
        extra["gemv_pair_one_chain_launch"] = {"us": round(t2 * 1e6, 2), "GB/s": round(STEP_BYTES / t2 / 1e9, 1),
                                               "frac_hbm": round(STEP_BYTES / t2 / 1e9 / hbm_peak, 3)}
        extra.update(per_config(torch, w4, synth, dev, stream, hbm_peak, tf_peak))
    base = None
    if rank == 0 and not args.no_cpu:
        try:
            base = cpu_baseline(args.cpu_seconds)
        except Exception as e:
            base = {"unavailable": str(e)[:120]}
    if rank != 0:
        return 0
    line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed_max / args.steps * 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "s32+f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "bytes_per_step": STEP_BYTES,
                       "arithmetic": ("u4 codes times s16 fixed-point activations (one power-of-two scale per "
                                      "128-element group; the largest values of each 64-element half group above "
                                      "its third-largest binade enter exactly in f32) in exact s32 dot products; "
                                      "f32 scale, zero point and accumulation; bf16 output"),
                       "l2": "%d rotating weight sets of %.1f MB each (inputs larger than the 129 MB L2)"
                             % (L2_SETS, STEP_BYTES / 1e6),
                       "launch": ("CUDA graph of %d steps (programmatic dependent launch between kernels)" % L2_SETS)
                       if graphs is not None else "eager (programmatic dependent launch between kernels)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": roofline, "cpu_baseline": base, "e2e": e2e,
            "gpu_launches": 2 * args.steps, "clocks": clk, "device_status": status,
            "per_config": extra}
    print(json.dumps(line), flush=True)
    return 0


def profile_cases(torch, w4, dev):
    """One workload each, for a profiler to capture: name -> (setup, run).
    Random weights and activations of the workload's shape (torch.randint /
    randn: quick to make at full size)."""

    def gemv(N, K):
        def setup():
            qw = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=dev)
            s = (torch.rand(N, K // 128, device=dev) * 0.02 + 0.001).half()
            z = torch.randint(0, 16, (N, K // 128), device=dev).half()
            x = torch.randn(K, device=dev).bfloat16()
            y = torch.empty(N, dtype=torch.bfloat16, device=dev)
            return lambda: w4.w4a16_gemv(x, qw, s, z, y)
        return setup

    def gemm(M, N, K, f16=False):
        def setup():
            qw = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=dev)
            s = (torch.rand(N, K // 128, device=dev) * 0.02 + 0.001).half()
            z = torch.randint(0, 16, (N, K // 128), device=dev).half()
            X = torch.randn(M, K, device=dev).bfloat16()
            Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            fn = w4.w4a16_gemm_f16 if f16 else w4.w4a16_gemm
            return lambda: fn(X, qw, s, z, Y)
        return setup

    def moe(M):
        def setup():
            E, N, K, topk = 64, 4096, 7168, 6
            qw = torch.randint(0, 256, (E, N, K // 2), dtype=torch.uint8, device=dev)
            s = (torch.rand(E, N, K // 32, device=dev) * 0.09 + 0.01).half()
            g = torch.Generator().manual_seed(M)
            ids = torch.stack([torch.randperm(E, generator=g)[:topk] for _ in range(M)]).int().to(dev)
            X = torch.randn(M, K, device=dev).bfloat16()
            if M == 1:
                y = torch.empty(topk, N, dtype=torch.bfloat16, device=dev)
                return lambda: w4.fp4_moe_gemv(X[0], qw, s, ids[0], y)
            Y = torch.empty(M, topk, N, dtype=torch.bfloat16, device=dev)
            scratch = torch.empty(w4.fp4_moe_gemm_scratch_bytes(M, topk, E, K), dtype=torch.uint8, device=dev)
            return lambda: w4.fp4_moe_gemm(X, qw, s, ids, Y, scratch)
        return setup

    return {"gemv_3840x3840": gemv(3840, 3840), "gemv_up_15360x3840": gemv(*UP),
            "gemv_down_3840x15360": gemv(*DOWN), "gemv_vocab_262144x3840": gemv(262144, 3840),
            "gemm_m16_15360x3840": gemm(16, 15360, 3840),
            "gemm_m128_15360x3840": gemm(128, 15360, 3840), "gemm_m2048_15360x3840": gemm(2048, 15360, 3840),
            "gemm_f16_m128_15360x3840": gemm(128, 15360, 3840, True),
            "gemm_f16_m2048_15360x3840": gemm(2048, 15360, 3840, True),
            "moe_fp4_64x4096x7168_top6": moe(1), "moe_fp4_gemm_m16_64x4096x7168_top6": moe(16),
            "moe_fp4_gemm_m128_64x4096x7168_top6": moe(128)}


def run_case(args):
    """Run one workload --reps times, untimed (the command a profiler wraps)."""
    import torch
    import gemm_w4a16_gemv_gb300 as w4
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cases = profile_cases(torch, w4, dev)
    if args.case not in cases:
        raise SystemExit("unknown --case %s; one of: %s" % (args.case, ", ".join(sorted(cases))))
    run = cases[args.case]()
    for _ in range(args.reps):
        run()
    torch.cuda.synchronize()
    status = w4.w4a16_check_device_error()
    print(json.dumps({"case": args.case, "reps": args.reps, "device_status": status}))
    return 0 if status == 0 else 1


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-graph", action="store_true", help="launch steps eagerly")
    ap.add_argument("--no-configs", action="store_true", help="skip per-configuration timings")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--case", help="run one workload --reps times, untimed (for a profiler)")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args(argv)
    if args.case:
        return run_case(args)
    if args.steps < 1 or args.warmup < 0:
        ap.error("--steps must be >= 1 and --warmup >= 0")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
