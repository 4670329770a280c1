#!/usr/bin/env python3
"""Benchmark of paged sliding-window attention on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one pass of the whole hot path over the batch-decode workload: 64
requests with kv_len ~ U[256, 4096], 32 query / 8 KV heads, head_dim 128, page 16,
once for each window_left in {-1, 0, 31, 127, 1023} (plans made beforehand; each
run = one decode kernel, which also merges split-KV partials when a plan splits). The metric is the algorithmic KV
bytes read (visible rows x 2 x H_kv x d x 2 B) per second. The line also carries
the prefill (TFLOP/s) and long-context decode (GB/s) workloads under "workloads",
including the extend prefill and both decodes over 8-bit (E4M3) K/V caches, whose
GB/s count one byte per cached element.

L2 is flushed between timed steps, outside the timed events: a 512 MiB write, then a
256 MiB read of the same buffer (so the flush leaves no dirty line to write back).
Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_sliding_gb300 import inputs as wl  # noqa: E402
from paged_kv_sliding_gb300 import workcount  # noqa: E402

METRIC = "prefill TFLOP/s + decode KV GB/s, paged SWA attn, 1 GB300, % of roofline"
UNIT = "GB/s"
WORKLOAD = ("batch decode: 64 requests, kv_len U[256,4096], 32q/8kv heads, d 128, page 16, "
            "window_left in {-1,0,31,127,1023}, bf16, lse")


def _max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """The largest of the ranks' values, returned on every rank (the slowest rank's
    time is the job's time)."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput: the units all ranks processed over the job's time."""
    return world * units_per_rank / seconds


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def _profiled_traffic(kernel: str, workload: str, source: str):
    """dram bytes per launch recorded by an ncu capture under profiles/, if the
    recorded source hash still matches the kernel's source."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    src = os.path.join(ROOT, "paged_kv_sliding_gb300", "csrc", source)
    if not os.path.exists(path) or not os.path.exists(src):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    if not m or not h:
        return None
    cur = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return float(m.group(1)) if cur.startswith(h.group(1)) else None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.idx = device_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _cudart():
    import ctypes
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    return None


class RawEvent:
    """A cudaEvent_t created through the CUDA runtime, for the library's timing hook."""
    _rt = None

    def __init__(self):
        import ctypes
        if RawEvent._rt is None:
            RawEvent._rt = _cudart()
        self.h = ctypes.c_void_p()
        assert RawEvent._rt.cudaEventCreate(ctypes.byref(self.h)) == 0

    def elapsed_ms(self, later: "RawEvent") -> float:
        import ctypes
        ms = ctypes.c_float()
        assert RawEvent._rt.cudaEventElapsedTime(ctypes.byref(ms), self.h, later.h) == 0
        return ms.value


def _flush_l2(buf):
    """Write the whole buffer (larger than L2), then read its first half: L2 then
    holds none of the inputs and only clean lines, so no write-back of the flush's
    own dirty lines lands inside the next timed region."""
    buf.zero_()
    buf[: buf.numel() // 2].max()


# ------------------------------------------------------------------------------- ours

def _timed_runs(runs, steps, warmup, flush):
    """runs: list of (plan, args) executed back to back as one step. Returns
    (per-step device ms list, main-kernel ms per run index summed over steps)."""
    stream = torch.cuda.current_stream()
    evs = [(RawEvent(), RawEvent()) for _ in runs]
    for (plan, _), (b, e) in zip(runs, evs):
        plan.set_timing_events(b.h.value, e.h.value)
    for _ in range(warmup):
        for plan, a in runs:
            plan.run(*a)
    torch.cuda.synchronize()
    step_ms = []
    kern_ms = [0.0] * len(runs)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(steps):
        flush()
        start.record(stream)
        for plan, a in runs:
            plan.run(*a)
        end.record(stream)
        end.synchronize()
        step_ms.append(start.elapsed_time(end))
        for i, (b, e) in enumerate(evs):
            kern_ms[i] += b.elapsed_ms(e)
    for plan, _ in runs:
        plan.set_timing_events(None, None)
    return step_ms, kern_ms


def bench_decode_windows(pkv, w_base, windows, steps, warmup, flush):
    plans, runs, bytes_per = [], [], []
    out = torch.empty_like(w_base.q)
    lse = torch.empty(w_base.q.shape[0], w_base.q.shape[1], dtype=torch.float32, device="cuda")
    launches = 0
    for W in windows:
        w = w_base.with_window(W)
        plan = pkv.plan_for(w)
        plans.append(plan)
        runs.append((plan, (w.q, w.k_cache, w.v_cache, out, lse)))
        bytes_per.append(workcount.decode_kv_bytes(w))
        launches += plan.info["kernels_per_run"]
    step_ms, kern_ms = _timed_runs(runs, steps, warmup, flush)
    return plans, runs, bytes_per, step_ms, kern_ms, launches


def graph_step_ms(runs, steps, warmup, flush):
    """Capture the step's launches (timing hooks off) into one CUDA graph and time
    its replays with CUDA events, flushing L2 between replays outside the events.
    Returns the per-step device times."""
    for plan, _ in runs:
        plan.set_timing_events(None, None)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(warmup):
            for plan, a in runs:
                plan.run(*a)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for plan, a in runs:
            plan.run(*a)
    torch.cuda.synchronize()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out = []
    for _ in range(steps):
        flush()
        start.record(stream)
        graph.replay()
        end.record(stream)
        end.synchronize()
        out.append(start.elapsed_time(end))
    del graph
    return out


def bench_prefill(pkv, w, steps, warmup, flush):
    plan = pkv.plan_for(w)
    out = torch.empty_like(w.q)
    lse = torch.empty(w.q.shape[0], w.q.shape[1], dtype=torch.float32, device="cuda")
    step_ms, kern_ms = _timed_runs([(plan, (w.q, w.k_cache, w.v_cache, out, lse))], steps, warmup, flush)
    flops = workcount.attention_flops(w)
    t = sum(kern_ms) / steps
    return {"tflops": flops / (t * 1e-3) / 1e12, "kernel_ms": t, "algorithmic_gflop": flops / 1e9,
            "work_items": plan.info["num_work_items"]}


def e2e_decode(pkv, w_dev, windows, steps, warmup):
    """Same step through the public API from pinned HOST buffers: H2D of q, the
    paged K/V pool and the page ids, the five runs, D2H of out and lse."""
    host = {k: getattr(w_dev, k).cpu().pin_memory() for k in ("q", "k_cache", "v_cache")}
    idx_host = torch.as_tensor(w_dev.kv_indices, dtype=torch.int32).pin_memory()
    dev = {k: torch.empty_like(getattr(w_dev, k)) for k in ("q", "k_cache", "v_cache")}
    idx_dev = torch.empty_like(idx_host, device="cuda")
    plans = [pkv.plan_for(w_dev.with_window(W), kv_indices=idx_dev) for W in windows]
    outs = [torch.empty_like(w_dev.q) for _ in windows]
    lses = [torch.empty(w_dev.q.shape[:2], dtype=torch.float32, device="cuda") for _ in windows]
    out_host = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    lse_host = [torch.empty(l.shape, dtype=l.dtype).pin_memory() for l in lses]
    h2d = sum(t.numel() * t.element_size() for t in host.values()) + idx_host.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in out_host + lse_host)

    def step():
        for k in host:
            dev[k].copy_(host[k], non_blocking=True)
        idx_dev.copy_(idx_host, non_blocking=True)
        for p, o, l in zip(plans, outs, lses):
            p.run(dev["q"], dev["k_cache"], dev["v_cache"], o, l)
        for o, l, oh, lh in zip(outs, lses, out_host, lse_host):
            oh.copy_(o, non_blocking=True)
            lh.copy_(l, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    return (time.perf_counter() - t0) / steps, h2d, d2h


def run_ours(args, rank, world):
    from paged_kv_sliding_gb300 import build, pkv
    build.build()
    pkv.load_library()
    dev_index = torch.cuda.current_device()
    peaks = _peaks()
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    flush = lambda: _flush_l2(flush_buf)  # noqa: E731

    w = wl.batch_decode(-1, device="cuda")
    windows = wl.BATCH_DECODE_WINDOWS

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # Per-kernel breakdown (CUDA events around each decode kernel, eager launches).
    plans, runs, bytes_per, eager_ms, kern_ms, launches = bench_decode_windows(
        pkv, w, windows, args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # The timed steps: the five runs replayed as one captured CUDA graph.
    with ClockSampler(dev_index) as clk:
        step_ms = graph_step_ms(runs, args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = _max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    step_bytes = sum(bytes_per)
    value = _job_rate(step_bytes, world, ms_per_step * 1e-3) / 1e9

    # dominant kernel: the decode kernel's window_left = -1 launch (the largest
    # share of the step), averaged over the timed steps
    i_full = list(windows).index(-1)
    kern_full = kern_ms[i_full] / args.steps
    achieved = bytes_per[i_full] / (kern_full * 1e-3) / 1e9
    per_window = {str(W): {"kv_mb": b / 1e6, "kernel_us": 1e3 * k / args.steps,
                           "gbs": b / (k / args.steps * 1e-3) / 1e9,
                           "frac_hbm": b / (k / args.steps * 1e-3) / 1e9 / peaks["hbm_gbs"],
                           "splits": p.info["num_partials"], "ctas": p.info["num_work_items"]}
                  for W, b, k, p in zip(windows, bytes_per, kern_ms, plans)}
    traffic = _profiled_traffic("decode", "batch_decode", "pkv_decode_kernel.cuh")

    e2e_s, h2d, d2h = e2e_decode(pkv, w, windows, max(3, args.steps // 4), 2)
    e2e_s = _max_over_ranks(e2e_s, world)
    del plans, runs
    torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "flushed between steps (512 MiB write, then a 256 MiB read)",
                   "timing": "step = the five runs captured in one CUDA graph, CUDA-event timed "
                             "replays; per_window = CUDA events around each decode kernel",
                   "eager_ms_per_step": round(sum(eager_ms) / len(eager_ms), 5),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": traffic, "kernel": "pkv decode_kernel<128>, window_left -1 launch",
                     "algorithmic_bytes": bytes_per[i_full], "kernel_us": round(1e3 * kern_full, 2),
                     "peak_source": peaks["source"]},
        "e2e": {"value": round(_job_rate(step_bytes, world, e2e_s) / 1e9, 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches * args.steps,
        "per_window": per_window,
    }
    clocks = clk.summary()
    if clocks:
        line["clocks"] = clocks

    oracle_mod, cores = None, None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle as oracle_mod
        oracle_mod.build()
        cores = oracle_mod.set_threads(0)
    if not args.no_extra:
        line["workloads"] = extra_workloads(pkv, args, peaks, flush, oracle=oracle_mod, cores=cores)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
        line["host"] = _host_info()
    return line


EXTRA = ("swa_prefill_p1", "swa_prefill_p16", "extend_prefix", "extend_ragged", "long_decode",
         "batch_decode_fp8", "long_decode_fp8", "extend_prefix_fp8")


# --------------------------------------------------------------- oracle beside each workload

def _host_info():
    return {"nproc": os.cpu_count(), "OMP_NUM_THREADS": os.environ.get("OMP_NUM_THREADS")}


def _oracle_args(w, **over):
    a = dict(qo_indptr=w.qo_indptr, kv_indptr=w.kv_indptr, kv_indices=w.kv_indices,
             kv_last_page_len=w.kv_last_page_len, num_qo_heads=w.num_qo_heads,
             num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, page_size=w.page_size,
             window_left=w.window_left, causal=w.causal, sm_scale=w.sm_scale, q=w.q.cpu(),
             k_cache=w.k_cache.cpu(), v_cache=w.v_cache.cpu(), q_start=w.q_start, num_pages=w.num_pages)
    a.update(over)
    return a


def extend_sample_rows(w, seed=9):
    """The seeded row sample of the extend parity tests: every request's first and
    last 64 rows plus 64 random rows."""
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(w.batch):
        lo, hi = int(w.qo_indptr[b]), int(w.qo_indptr[b + 1])
        sel = set(range(lo, min(hi, lo + 64))) | set(range(max(lo, hi - 64), hi))
        sel |= set(rng.integers(lo, hi, size=64).tolist())
        rows.extend(sorted(sel))
    return np.array(rows)


def oracle_prefill(oracle, cores, w, rows=None, note=""):
    """The oracle on a prefill workload (its device tensors copied to the host), in
    full or on a row sample; TFLOP/s of algorithmic work, and for a sample the full
    workload's time extrapolated from that rate."""
    args = _oracle_args(w)
    t0 = time.perf_counter()
    oracle.attention(rows=rows, **args)
    el = time.perf_counter() - t0
    full = workcount.attention_flops(w)
    flops = full if rows is None else workcount.attention_flops_rows(w, rows)
    r = {"value": round(flops / el / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
         "seconds": round(el, 3), "sample": "the full workload" if rows is None else
         f"{len(rows)} of {int(w.qo_indptr[-1])} query rows (every request's first and last 64 rows "
         f"and 64 seeded random rows), all heads"}
    if rows is not None:
        r["extrapolated_full_s"] = round(full / (flops / el), 3)
        r["extrapolated"] = True
    if note:
        r["note"] = note
    return r


def oracle_decode(oracle, cores, w, n_req=None, seed=44):
    """The oracle on a decode workload, in full or on n_req seeded requests (their
    pages gathered on the device and copied to the host); GB/s of visible KV."""
    import dataclasses
    if n_req is None or n_req >= w.batch:
        sub, label = w, "the full workload"
    else:
        rng = np.random.default_rng(seed)
        sel = np.sort(rng.choice(w.batch, size=n_req, replace=False))
        pages = np.concatenate([w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]] for b in sel])
        pidx = torch.as_tensor(pages.astype(np.int64), device=w.k_cache.device)
        kv_indptr = np.zeros(len(sel) + 1, dtype=np.int32)
        kv_indptr[1:] = np.cumsum(np.diff(w.kv_indptr)[sel])
        tsel = torch.as_tensor(sel, device=w.q.device)
        sub = dataclasses.replace(
            w, qo_indptr=np.arange(len(sel) + 1, dtype=np.int32), kv_indptr=kv_indptr,
            kv_indices=np.arange(len(pages), dtype=np.int32), kv_last_page_len=w.kv_last_page_len[sel],
            num_pages=len(pages), q=w.q[tsel].cpu(), k_cache=w.k_cache[pidx].cpu(),
            v_cache=w.v_cache[pidx].cpu(), q_start=None if w.q_start is None else w.q_start[sel])
        label = f"{n_req} of {w.batch} requests (seeded), every head and visible key"
    args = _oracle_args(sub)
    t0 = time.perf_counter()
    oracle.attention(**args)
    el = time.perf_counter() - t0
    nbytes = workcount.decode_kv_bytes(sub)
    r = {"value": round(nbytes / el / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
         "seconds": round(el, 3), "sample": label}
    if sub is not w:
        r["extrapolated_full_s"] = round(workcount.decode_kv_bytes(w) / (nbytes / el), 3)
        r["extrapolated"] = True
    return r


def bench_prefill_ragged(pkv, w, steps, warmup, flush):
    """The workload's K/V packed contiguously, request after request, through the
    ragged (non-paged) prefill path."""
    P = w.page_size
    idx = torch.as_tensor(w.kv_indices.astype(np.int64), device="cuda")
    kp = w.k_cache[idx].reshape(-1, w.num_kv_heads, w.head_dim)
    vp = w.v_cache[idx].reshape(-1, w.num_kv_heads, w.head_dim)
    lens = [int(x) for x in w.kv_lens]
    sel = torch.cat([torch.arange(int(w.kv_indptr[b]) * P, int(w.kv_indptr[b]) * P + lens[b])
                     for b in range(w.batch)]).to("cuda")
    k, v = kp[sel].contiguous(), vp[sel].contiguous()
    del kp, vp
    kv_indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    plan = pkv.Plan(kind="prefill_ragged", qo_indptr=w.qo_indptr, kv_indptr=kv_indptr,
                    num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                    window_left=w.window_left, causal=w.causal, sm_scale=w.sm_scale, q_start=w.q_start)
    out = torch.empty_like(w.q)
    lse = torch.empty(w.q.shape[0], w.q.shape[1], dtype=torch.float32, device="cuda")
    step_ms, kern_ms = _timed_runs([(plan, (w.q, k, v, out, lse))], steps, warmup, flush)
    flops = workcount.attention_flops(w)
    t = sum(kern_ms) / steps
    return {"tflops": flops / (t * 1e-3) / 1e12, "kernel_ms": t, "algorithmic_gflop": flops / 1e9,
            "work_items": plan.info["num_work_items"]}


def extra_workloads(pkv, args, peaks, flush, only=None, oracle=None, cores=None):
    """The prefill and long-decode workloads on the GPU; with `oracle` given, the
    float64 oracle is timed on the host beside each one (in full, or on the seeded
    sample of the parity tests with the full time extrapolated)."""
    res = {}
    steps = max(3, min(args.steps, 10))
    want = lambda n: only is None or only == n  # noqa: E731
    for P in (1, 16):
        if not want(f"swa_prefill_p{P}"):
            continue
        w = wl.swa_prefill(page_size=P, device="cuda")
        r = bench_prefill(pkv, w, steps, 3, flush)
        r["frac_bf16"] = r["tflops"] / peaks["bf16_tflops"]
        if oracle is not None:
            r["cpu_baseline"] = oracle_prefill(oracle, cores, w)
        res[f"swa_prefill_8x1500_d256_W511_p{P}"] = r
        del w
    if want("extend_prefix") or want("extend_ragged"):
        w = wl.extend_with_prefix(device="cuda")
        ext_cpu = oracle_prefill(oracle, cores, w, rows=extend_sample_rows(w)) if oracle is not None else None
        if want("extend_prefix"):
            r = bench_prefill(pkv, w, steps, 3, flush)
            r["frac_bf16"] = r["tflops"] / peaks["bf16_tflops"]
            r["traffic"] = _profiled_traffic("prefill", "extend_with_prefix", "pkv_prefill_kernel.cuh")
            if ext_cpu is not None:
                r["cpu_baseline"] = ext_cpu
            res["extend_prefix_16req_W4095"] = r
        if want("extend_ragged"):
            r = bench_prefill_ragged(pkv, w, steps, 3, flush)
            r["frac_bf16"] = r["tflops"] / peaks["bf16_tflops"]
            if ext_cpu is not None:
                r["cpu_baseline"] = dict(ext_cpu, note="the same oracle computation as the paged extend "
                                                       "(the oracle walks a page table; the ragged path "
                                                       "computes the same attention)")
            res["extend_prefix_16req_W4095_ragged_kv"] = r
        del w
        torch.cuda.empty_cache()
    if want("extend_prefix_fp8"):
        w = wl.to_kv8(wl.extend_with_prefix(device="cuda"), "e4m3")
        r = bench_prefill(pkv, w, steps, 3, flush)
        r["frac_bf16"] = r["tflops"] / peaks["bf16_tflops"]  # f16 MMAs run at the bf16 rate
        if oracle is not None:
            r["cpu_baseline"] = oracle_prefill(oracle, cores, w, rows=extend_sample_rows(w))
        res["extend_prefix_16req_W4095_e4m3"] = r
        del w
        torch.cuda.empty_cache()
    for W in (wl.LONG_DECODE_WINDOWS if want("long_decode") else ()):
        w = wl.long_decode(W, device="cuda", batch=args.long_requests)
        plans, runs, bytes_per, step_ms, kern_ms, _ = bench_decode_windows(pkv, w, [W], steps, 2, flush)
        k = kern_ms[0] / steps
        key = f"long_decode_{w.batch}x32768_W{W}"
        res[key] = {
            "gbs": bytes_per[0] / (k * 1e-3) / 1e9, "kernel_ms": k,
            "step_ms": statistics.mean(step_ms), "kv_gb": bytes_per[0] / 1e9,
            "frac_hbm": bytes_per[0] / (k * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "frac_note": "the peak is a copy's (read + write) rate; this kernel only reads",
            "splits": plans[0].info["num_partials"], "ctas": plans[0].info["num_work_items"]}
        del plans, runs
        if oracle is not None:
            res[key]["cpu_baseline"] = oracle_decode(oracle, cores, w, n_req=32)
        del w
        torch.cuda.empty_cache()
    # 8-bit KV caches (E4M3): the batch-decode windows and the long decode. GB/s counts
    # the bytes of the 8-bit cache a pass must read (half of bf16's per key).
    if want("batch_decode_fp8"):
        w = wl.to_kv8(wl.batch_decode(device="cuda"), "e4m3")
        plans, runs, bytes_per, step_ms, kern_ms, _ = bench_decode_windows(
            pkv, w, wl.BATCH_DECODE_WINDOWS, steps, 3, flush)
        for i, W in enumerate(wl.BATCH_DECODE_WINDOWS):
            k = kern_ms[i] / steps
            res[f"batch_decode_e4m3_W{W}"] = {
                "gbs": bytes_per[i] / (k * 1e-3) / 1e9, "kernel_us": k * 1e3, "kv_mb": bytes_per[i] / 1e6,
                "frac_hbm": bytes_per[i] / (k * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "keys_per_s": bytes_per[i] / (2 * w.num_kv_heads * w.head_dim) / (k * 1e-3),
                "kv_tile": plans[i].info["kv_tile"], "ctas": plans[i].info["num_work_items"]}
            if oracle is not None:
                res[f"batch_decode_e4m3_W{W}"]["cpu_baseline"] = oracle_decode(oracle, cores, w.with_window(W))
        res["batch_decode_e4m3_step_ms"] = statistics.mean(step_ms)
        del w, plans, runs
        torch.cuda.empty_cache()
    if want("long_decode_fp8"):
        base = wl.long_decode(-1, device="cuda")
        w = wl.to_kv8(base, "e4m3")
        del base
        torch.cuda.empty_cache()
        plans, runs, bytes_per, step_ms, kern_ms, _ = bench_decode_windows(pkv, w, [-1], steps, 2, flush)
        k = kern_ms[0] / steps
        res["long_decode_256x32768_W-1_e4m3"] = {
            "gbs": bytes_per[0] / (k * 1e-3) / 1e9, "kernel_ms": k, "kv_gb": bytes_per[0] / 1e9,
            "frac_hbm": bytes_per[0] / (k * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "frac_note": "the peak is a copy's (read + write) rate; this kernel only reads",
            "splits": plans[0].info["num_partials"], "ctas": plans[0].info["num_work_items"]}
        del plans, runs
        if oracle is not None:
            res["long_decode_256x32768_W-1_e4m3"]["cpu_baseline"] = oracle_decode(oracle, cores, w, n_req=32)
        del w
        torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------------------- oracle

def _oracle_decode_step(oracle, w, windows):
    for W in windows:
        oracle.attention(qo_indptr=w.qo_indptr, kv_indptr=w.kv_indptr, kv_indices=w.kv_indices,
                         kv_last_page_len=w.kv_last_page_len, num_qo_heads=w.num_qo_heads,
                         num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                         page_size=w.page_size, window_left=W, causal=w.causal,
                         sm_scale=w.sm_scale, q=w.q, k_cache=w.k_cache, v_cache=w.v_cache)


def cpu_baseline(args, budget_s: float = 12.0):
    """The float64 oracle, as it stands, on this host's cores: the same batch-decode
    step (all five windows, all 64 requests) repeated until about `budget_s`."""
    import oracle
    oracle.build()
    cores = oracle.set_threads(0)
    w = wl.batch_decode(-1)
    windows = wl.BATCH_DECODE_WINDOWS
    step_bytes = sum(workcount.decode_kv_bytes(w.with_window(W)) for W in windows)
    reps, t0 = 0, time.perf_counter()
    while True:
        _oracle_decode_step(oracle, w, windows)
        reps += 1
        el = time.perf_counter() - t0
        if el > budget_s or reps >= 20:
            break
    return {"value": round(reps * step_bytes / el / 1e9, 4), "unit": UNIT, "cores": cores,
            "kind": "oracle", "sample": f"{reps} full batch-decode step(s) (64 requests x 5 windows), "
                                        f"{el:.1f} s wall", "seconds": round(el, 2), **_host_info()}


def run_reference(args, rank, world):
    import oracle
    oracle.build()
    cores = oracle.set_threads(0)
    w = wl.batch_decode(-1)
    windows = wl.BATCH_DECODE_WINDOWS
    step_bytes = sum(workcount.decode_kv_bytes(w.with_window(W)) for W in windows)
    for _ in range(args.warmup):
        _oracle_decode_step(oracle, w, windows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_decode_step(oracle, w, windows)
    el = time.perf_counter() - t0
    value = step_bytes * args.steps / el / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * el / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": "host cores (OpenMP)"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} full batch-decode steps (64 requests x 5 windows)"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the prefill / long-decode workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=EXTRA, default=None,
                    help="run just one of the extra workloads (for profiling) and print its numbers")
    ap.add_argument("--long-requests", type=int, default=256,
                    help="requests of the long-context decode workload (256; fewer only for small profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        # the oracle runs on host cores; for N > 1 only rank 0 runs it
        line = run_reference(args, rank, world)
        print(json.dumps(line), flush=True)
        return

    if args.only:
        from paged_kv_sliding_gb300 import build, pkv
        build.build()
        buf = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
        res = extra_workloads(pkv, args, _peaks(), lambda: _flush_l2(buf), only=args.only)
        print(json.dumps({"only": args.only, "workloads": res}), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
