#!/usr/bin/env python
"""Benchmark of the fused inference attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one fia_decode call (split plan, split-KV attention, merge) over the
whole bf16 paged GQA decode workload: B 32, Nq 32, Nkv 8, D 128, query length 1,
KV lengths U[1, 4096] (seeded), blockSize 128, shuffled block table.  Inputs are
resident in HBM and rotated over 4 copies (4 x 268 MB of KV > the 126 MB L2), so
no step reads KV left in L2 by the previous one.

The JSON line reports the KV-read throughput (algorithmic bytes / time, GB/s)
as `value`, with queries/s and the fraction of the measured HBM copy bandwidth.
`roofline` is for the split-KV attention kernel, timed by CUDA events that the
library records around each of its launches (fia_trace_enable) during the timed
region.  `e2e` repeats the measurement through the public API with the per-step
inputs (query, block table, lengths) copied from pinned host memory and the
results (out, softmax max/sum) copied back inside the timed region; the KV cache
stays resident, as it does across decode steps.  `cpu_baseline` times the fp64
oracle on the host cores over a bounded sample of the same workload.

Under torchrun each rank runs its own copy of the workload on its own GPU
(weak scaling; decode batches are independent, so no data is exchanged); the
time is the max over ranks.  --impl reference times the oracle alone (rank 0).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import fia_workloads as W  # noqa: E402

METRIC = "paged decode attn KV-read GB/s (% HBM peak), queries/s; prefill TFLOP/s"
COPIES = 4


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------------------- workload arithmetic
def decode_bytes(case: W.DecodeCase) -> dict:
    """Algorithmic bytes of one decode step: every visible K/V element once, q, out,
    the block-table entries in use, the lengths, antiquant params, sink and max/sum."""
    L = case.lengths.astype(np.int64)
    kv = int(L.sum()) * 2 * case.Nkv * case.D * case.kv_elem_bytes
    qo = 2 * case.B * case.Nq * case.D * 2
    bt = int(((L + case.block_size - 1) // case.block_size).sum()) * 4
    aux = case.B * 8 + 2 * case.B * case.Nq * 4
    if case.aq_scale is not None:
        aux += 2 * case.aq_scale.size * 4
    if case.sink is not None:
        aux += case.Nq * 4
    return {"kv": kv, "total": kv + qo + bt + aux}


def max_over_ranks(x: float, dist, device) -> float:
    """The largest x over all ranks (each rank's timed duration: the job is as slow as its
    slowest rank); x itself when there is one rank (dist None)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def e2e_pipeline(torch, stream, call, dev_in, pin_in, outs, warmup, steps, barrier):
    """Times `steps` end-to-end steps: step i copies its inputs host -> device (pin_in[j] ->
    dev_in[j], j = i mod len(dev_in)) on a copy stream, runs call(i, j, o) on the compute
    stream, and copies its results device -> host (outs[o], o = i mod 2) on a second copy
    stream; events keep every buffer's copies and use in order, so one step's copies overlap
    its neighbours' compute.  Groups of 8 len(dev_in) steps are captured once in a CUDA graph
    and replayed (issuing a step's copies, events and launches from Python costs about as
    much host time as the GPU spends on it; a replay starts by joining the copy streams, so
    one input copy per replay is not overlapped, hence long groups); the remaining steps are a
    second graph.  Returns the milliseconds from the first copy to the last result in host
    memory (CUDA events on the compute stream)."""
    nin = len(dev_in)
    group = 8 * nin
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()

    def steps_on(comp, first, n):
        """Issues steps first .. first + n - 1 with `comp` as the compute stream (the copy
        streams wait for comp before, and comp for them after)."""
        in_free, out_free = [None] * nin, [None, None]
        h2d.wait_stream(comp)
        d2h.wait_stream(comp)
        for i in range(first, first + n):
            j, o = i % nin, i % 2
            with torch.cuda.stream(h2d):
                if in_free[j] is not None:
                    h2d.wait_event(in_free[j])
                dev_in[j].copy_(pin_in[j], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(h2d)
            comp.wait_event(ready)
            if out_free[o] is not None:
                comp.wait_event(out_free[o])
            with torch.cuda.stream(comp):
                call(i, j, o)
            done = torch.cuda.Event()
            done.record(comp)
            in_free[j] = done
            with torch.cuda.stream(d2h):
                d2h.wait_event(done)
                outs[o][1].copy_(outs[o][0], non_blocking=True)
                freed = torch.cuda.Event()
                freed.record(d2h)
                out_free[o] = freed
        comp.wait_stream(h2d)
        comp.wait_stream(d2h)

    steps_on(stream, 0, min(warmup, 2 * nin))  # uncaptured warm-up (the library's set-up happens here)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        steps_on(cap, 0, group)
    rest = None
    if steps % group:
        rest = torch.cuda.CUDAGraph()
        with torch.cuda.graph(rest, stream=cap):
            steps_on(cap, 0, steps % group)
    graph.replay()
    if rest is not None:
        rest.replay()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps // group):
        graph.replay()
    if rest is not None:
        rest.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    return e0.elapsed_time(e1)


def staged(tensors, dev, torch):
    """One device buffer holding copies of `tensors` (each at a 256-byte aligned offset) and a
    pinned host buffer of the same bytes; returns (device buffer, host buffer, views of the
    device buffer shaped and typed as the tensors)."""
    offs, n = [], 0
    for t in tensors:
        offs.append(n)
        n += (t.numel() * t.element_size() + 255) // 256 * 256
    d = torch.zeros(n, dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(tensors, offs):
        nb = t.numel() * t.element_size()
        v = d[o:o + nb].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    h = torch.empty(n, dtype=torch.uint8).pin_memory()
    h.copy_(d)
    return d, h, tuple(views)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []  # (host time, sm, max, power, reasons)
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            reasons = [n for n, v in zip(names, parts[3:7]) if v.lower().startswith("active")]
            self.samples.append((time.time(), sm, mx, parts[2], reasons))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1, pad=1.0):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed region"
        if len(inside) < 3:
            inside = [s for s in self.samples if t0 - pad <= s[0] <= t1 + 0.2]
            window = "timed region and the last second of warm-up"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "none sampled"}
        reasons = sorted({r for s in inside for r in s[4]})
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# ----------------------------------------------------------------------------- oracle timing
def oracle_decode_sample(case: W.DecodeCase, groups):
    """Run the oracle on every query head of the (b, kv-head) groups given; returns
    (seconds, algorithmic bytes of that sample, threads)."""
    import oracle
    G = case.Nq // case.Nkv
    rows = np.array([b * case.Nq + hk * G + g for (b, hk) in groups for g in range(G)], np.int64)
    code = {W.BF16: oracle.BF16, W.FP16: oracle.F16}
    kvc = oracle.I8 if case.kv_dtype == W.INT8 else code[case.kv_dtype]
    t = time.perf_counter()
    oracle.decode(case.q, case.k_cache, case.v_cache, case.lengths, Nq=case.Nq, Nkv=case.Nkv, D=case.D,
                  scale=case.scale, q_dtype=code[case.dtype], kv_dtype=kvc, block_table=case.block_table,
                  block_size=case.block_size, aq_scale=case.aq_scale, aq_offset=case.aq_offset, sink=case.sink,
                  rows=rows)
    dt = time.perf_counter() - t
    kvb = sum(int(case.lengths[b]) for (b, _) in groups) * 2 * case.D * case.kv_elem_bytes
    nbytes = kvb + len(rows) * case.D * 2 * 2 + len(rows) * 8
    return dt, nbytes, oracle.max_threads()


def cpu_baseline(case: W.DecodeCase, budget_s: float = 15.0, seed: int = 0):
    rng = np.random.default_rng(seed)
    all_groups = [(b, h) for b in range(case.B) for h in range(case.Nkv)]
    order = rng.permutation(len(all_groups))
    probe = [all_groups[i] for i in order[:4]]
    dt, nb, cores = oracle_decode_sample(case, probe)
    per_group = max(dt / len(probe), 1e-4)
    n = int(min(len(all_groups), max(4, budget_s / per_group)))
    groups = [all_groups[i] for i in order[:n]]
    # whole passes are repeated (up to 20) until the budget is spent, for a stable figure
    dt, nb, passes = 0.0, 0, 0
    while passes < 20 and (passes == 0 or (n == len(all_groups) and dt < budget_s)):
        t, b, cores = oracle_decode_sample(case, groups)
        dt, nb, passes = dt + t, nb + b, passes + 1
    what = "the whole workload" if n == len(all_groups) else f"{n} of {len(all_groups)} (batch, kv-head) groups"
    return {"value": nb / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{what} x {passes} pass(es), all {case.Nq // case.Nkv} query heads per group; "
                      f"{dt:.1f} s of fp64 CPU work", "seconds": round(dt, 2)}


# ----------------------------------------------------------------------------- our implementation
def run_ours(args, rank, world, local_rank):
    import torch
    import attention_ifa_fia_gb300 as F
    from fia_workloads import DeviceDecode

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    case = W.WORKLOADS[args.workload]()  # every rank runs the same workload (independent replicas)
    nbytes = decode_bytes(case)
    copies = [DeviceDecode(case, dev) for _ in range(COPIES)]
    num_splits = W.LONG_CTX_CHUNKS if args.workload == "long_ctx_sink_decode" else 0
    ws_bytes = F.fia_decode_workspace_size(case.B, case.Nq, case.Nkv, case.D, case.max_len, case.block_size,
                                           num_splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((case.B, case.Nq, case.D), dtype=copies[0].q.dtype, device=dev)
    mx = torch.empty((case.B, case.Nq), dtype=torch.float32, device=dev)
    sm = torch.empty_like(mx)

    def step(i):
        c = copies[i % COPIES]
        F.fia_decode(c.q, c.k, c.v, c.bt, c.lens, max_kv_len=case.max_len, num_heads=case.Nq,
                     num_kv_heads=case.Nkv, scale=case.scale, antiquant_scale=c.aq_scale,
                     antiquant_offset=c.aq_offset, sink=c.sink, out=out, softmax_max=mx, softmax_sum=sm,
                     num_splits=num_splits, workspace=ws)

    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()

    sampler = ClockSampler(local_rank)
    sampler.start()
    # warm-up: at least W steps and at least one second of load
    t_w = time.time()
    i = 0
    while i < args.warmup or time.time() - t_w < args.min_warmup_s:
        step(i)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    F.fia_device_status()

    # ---- timed region: exactly K steps
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # The headline time is taken with the launch tracer off: its events between
    # the kernels would stop a dependent launch from starting before the kernel
    # ahead of it ends.
    barrier()
    torch.cuda.synchronize()
    h0 = time.time()
    e0.record(stream)
    for k in range(args.steps):
        step(k)
    e1.record(stream)
    host_s = time.time() - h0  # host time to issue the K steps (asynchronous launches)
    torch.cuda.synchronize()
    h1 = time.time()
    barrier()
    ms = e0.elapsed_time(e1)
    # Per-kernel durations and launch counts: the same K steps again, traced.
    kern_ids = (("plan", F.KERNEL_DECODE_PLAN), ("attention", F.KERNEL_DECODE_ATTENTION),
                ("merge", F.KERNEL_DECODE_MERGE))
    F.fia_trace_enable(True)
    for _, kid in kern_ids:
        F.fia_trace_collect(kid)
    e0.record(stream)
    for k in range(args.steps):
        step(k)
    e1.record(stream)
    torch.cuda.synchronize()
    F.fia_trace_enable(False)
    ms_traced = e0.elapsed_time(e1)
    kern = {name: F.fia_trace_collect(kid) for name, kid in kern_ids}
    status = F.fia_device_status()
    ms = max_over_ranks(ms, dist, dev)

    # ---- end to end through the public API with host buffers: per step the query, block
    # table and lengths go host -> device in one copy (one pinned staging buffer, one device
    # buffer whose views are the call's inputs), and out, max and sum come back in one copy
    in_views = [(c.q, c.bt, c.lens) for c in copies]
    dev_in, pin_in, e2e_in = [], [], []
    for views in in_views:
        d, h, v = staged(views, dev, torch)
        dev_in.append(d)
        pin_in.append(h)
        e2e_in.append(v)
    outs = [staged((out, mx, sm), dev, torch) for _ in range(2)]  # results double-buffered
    h2d = dev_in[0].numel()
    d2h = outs[0][0].numel()

    def e2e_call(i, j, o):
        c = copies[j]
        q_e, bt_e, len_e = e2e_in[j]
        o_e, mx_e, sm_e = outs[o][2]
        F.fia_decode(q_e, c.k, c.v, bt_e, len_e, max_kv_len=case.max_len, num_heads=case.Nq,
                     num_kv_heads=case.Nkv, scale=case.scale, antiquant_scale=c.aq_scale,
                     antiquant_offset=c.aq_offset, sink=c.sink, out=o_e, softmax_max=mx_e, softmax_sum=sm_e,
                     num_splits=num_splits, workspace=ws)

    ms_e2e = e2e_pipeline(torch, stream, e2e_call, dev_in, pin_in, outs, args.warmup, args.steps, barrier)
    ms_e2e = max_over_ranks(ms_e2e, dist, dev)
    sampler.stop()

    if rank != 0:
        return None
    hbm, tf_burst, tf_sus, src = peaks()
    steps = args.steps
    gbs = world * nbytes["total"] * steps / (ms / 1e3) / 1e9
    att_ms, att_n = kern["attention"]
    achieved = nbytes["total"] / (att_ms / att_n / 1e3) / 1e9 if att_n else None
    traffic = load_traffic(args.workload)
    line = {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(ms / steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if case.dtype == W.BF16 else "f16",
        "data": "synthetic",
        "config": {"workload": args.workload, "B": case.B, "Nq": case.Nq, "Nkv": case.Nkv, "D": case.D,
                   "block_size": case.block_size, "kv_dtype": case.kv_dtype,
                   "kv_lengths": f"seeded (sum {int(case.lengths.sum())}, max {case.max_len})",
                   "kv_bytes_per_step": nbytes["kv"], "algorithmic_bytes_per_step": nbytes["total"],
                   "l2": f"inputs rotated over {COPIES} device copies ({COPIES} x {nbytes['kv'] / 1e6:.0f} MB of KV > L2)",
                   "parallelism": f"independent replicas x{world}" if world > 1 else "single GPU"},
        "hbm_frac_of_measured": round(gbs / world / hbm, 4),
        "queries_per_s": round(world * case.B * steps / (ms / 1e3), 1),
        "head_queries_per_s": round(world * case.B * case.Nq * steps / (ms / 1e3), 1),
        "kernels_ms_per_launch": {k: round(v[0] / v[1], 5) if v[1] else None for k, v in kern.items()},
        "kernel_timing": "per-kernel CUDA events in a second pass of the same K steps "
                         f"(ms_per_step {ms_traced / steps:.5f} with the events in place); "
                         "value and ms_per_step come from the untraced pass",
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1) if achieved else None, "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4) if achieved else None,
                     "traffic": traffic, "kernel": "decode_tc (tcgen05 split-KV attention)" if case.kv_dtype != W.INT8
                     else "decode_i8tc (tcgen05 split-KV attention over int8 codes)",
                     "peak_source": f"{src} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" if src == "measured"
                     else "fallback 6.8 TB/s"},
        "e2e": {"value": round(world * nbytes["total"] * steps / (ms_e2e / 1e3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "per step: q, block table and lengths host->device in one copy; out, max and sum "
                        "device->host in one copy; copies on their own streams, overlapping neighbouring "
                        "steps' compute (inputs over 4 buffers, results over 2); each group of 32 steps one "
                        "CUDA graph launch; KV cache resident"},
        "gpu_launches": sum(v[1] for v in kern.values()),
        "host_us_per_step": round(host_s / steps * 1e6, 2),
        "device_status": status,
        "clocks": sampler.summary(h0, h1),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case)
    return line


def prefill_flops(case: W.PrefillCase, causal=True) -> int:
    """Algorithmic FLOPs of one prefill: 4 * D per visible (query, key) pair and query head
    (2 for the score, 2 for the value product); masked pairs are not counted."""
    pairs = 0
    for Lq, Lk in zip(case.lengths_q.tolist(), case.lengths_kv.tolist()):
        if not causal:
            pairs += Lq * Lk
            continue
        i = np.arange(Lq, dtype=np.int64)
        pairs += int(np.clip(i + (Lk - Lq) + 1, 0, Lk).sum())
    return 4 * case.D * case.Nq * pairs


def run_prefill_bench(args, rank, world, local_rank):
    import torch
    import attention_ifa_fia_gb300 as F
    from fia_workloads import DevicePrefill

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    case = W.WORKLOADS[args.workload]()  # every rank runs the same workload (independent replicas)
    flops = prefill_flops(case)
    copies = [DevicePrefill(case, dev) for _ in range(COPIES)]
    msq, mskv = int(case.lengths_q.max()), int(case.lengths_kv.max())
    ws = torch.empty(F.fia_prefill_workspace_size(case.B, case.Nq, case.Nkv, case.D, msq), dtype=torch.uint8,
                     device=dev)
    out = torch.empty((case.T, case.Nq, case.D), dtype=copies[0].q.dtype, device=dev)
    mx = torch.empty((case.T, case.Nq), dtype=torch.float32, device=dev)
    sm = torch.empty_like(mx)

    def step(i):
        c = copies[i % COPIES]
        F.fia_prefill(c.q, c.k, c.v, c.cu_q, c.cu_kv, max_seqlen_q=msq, max_seqlen_kv=mskv, num_heads=case.Nq,
                      num_kv_heads=case.Nkv, scale=case.scale, mask=3, out=out, softmax_max=mx, softmax_sum=sm,
                      workspace=ws)

    dist = None
    if world > 1:
        import torch.distributed as dist
    sampler = ClockSampler(local_rank)
    sampler.start()
    t_w = time.time()
    i = 0
    while i < args.warmup or time.time() - t_w < args.min_warmup_s:
        step(i)
        i += 1
        if i % 32 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    F.fia_device_status()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # The headline time is taken with the launch tracer off (its events between calls stop
    # a dependent launch from starting before the kernel ahead of it ends); the plan and
    # attention kernels are then timed together on the same steps, traced.
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    h0 = time.time()
    e0.record(stream)
    for k in range(args.steps):
        step(k)
    e1.record(stream)
    torch.cuda.synchronize()
    h1 = time.time()
    if dist is not None:
        dist.barrier()
    ms = e0.elapsed_time(e1)
    F.fia_trace_enable(True)
    F.fia_trace_collect(F.KERNEL_PREFILL)
    for k in range(args.steps):
        step(k)
    torch.cuda.synchronize()
    F.fia_trace_enable(False)
    pf_ms, pf_n = F.fia_trace_collect(F.KERNEL_PREFILL)
    status = F.fia_device_status()
    ms = max_over_ranks(ms, dist, dev)
    # end to end: q, k, v and both cumulative lengths host -> device in one copy (one pinned
    # staging buffer, one device buffer whose views are the call's inputs); out, max and sum
    # device -> host in one copy
    dev_in, pin_in, e2e_in = [], [], []
    for c in copies:
        d, h, v = staged((c.q, c.k, c.v, c.cu_q, c.cu_kv), dev, torch)
        dev_in.append(d)
        pin_in.append(h)
        e2e_in.append(v)
    outs = [staged((out, mx, sm), dev, torch) for _ in range(2)]  # results double-buffered
    h2d = dev_in[0].numel()
    d2h = outs[0][0].numel()

    def e2e_call(i, j, o):
        q_e, k_e, v_e, cuq_e, cukv_e = e2e_in[j]
        o_e, mx_e, sm_e = outs[o][2]
        F.fia_prefill(q_e, k_e, v_e, cuq_e, cukv_e, max_seqlen_q=msq, max_seqlen_kv=mskv, num_heads=case.Nq,
                      num_kv_heads=case.Nkv, scale=case.scale, mask=3, out=o_e, softmax_max=mx_e, softmax_sum=sm_e,
                      workspace=ws)

    ms_e2e = e2e_pipeline(torch, stream, e2e_call, dev_in, pin_in, outs, args.warmup, args.steps,
                          (lambda: dist.barrier()) if dist is not None else (lambda: None))
    ms_e2e = max_over_ranks(ms_e2e, dist, dev)
    sampler.stop()
    if rank != 0:
        return None
    hbm, tf_burst, tf_sus, src = peaks()
    tflops = world * flops * args.steps / (ms / 1e3) / 1e12
    # The roofline numerator is the untraced step: one step is exactly the plan and the attention
    # kernel back to back (the tracer's events between calls would stop the next call's plan from
    # starting under the attention kernel's tail, and the traced pass runs a few percent slower).
    achieved = flops / (ms / args.steps / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "B": case.B, "T": case.T, "Nq": case.Nq, "Nkv": case.Nkv,
                   "D": case.D, "lengths": case.lengths_q.tolist(), "causal_flops_per_step": flops,
                   "l2": f"inputs rotated over {COPIES} device copies",
                   "parallelism": f"independent replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2) if achieved else None, "peak": tf_burst,
                     "unit": "TFLOP/s", "frac": round(achieved / tf_burst, 4) if achieved else None,
                     "traffic": load_traffic("causal_prefill_tnd"),
                     "kernel": "prefill_pair (tcgen05 head-pair attention; plan + attention per untraced step)",
                     "traced_plan_attention_ms": round(pf_ms / pf_n, 5) if pf_n else None,
                     "peak_source": f"{src} bf16 dense burst (MEASURED_PEAKS.json bf16_tflops)"},
        "e2e": {"value": round(world * flops * args.steps / (ms_e2e / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "per step: q, k, v and cumulative lengths host->device in one copy; out, max and sum "
                        "device->host in one copy; copies on their own streams, overlapping neighbouring "
                        "steps' compute (inputs over 4 buffers, results over 2); each group of 32 steps one "
                        "CUDA graph launch"},
        "gpu_launches": 2 * pf_n, "device_status": status, "clocks": sampler.summary(h0, h1),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_prefill(case)
    return line


def cpu_baseline_prefill(case: W.PrefillCase, budget_s: float = 15.0, seed: int = 0):
    """The oracle on a sample of (token, head) rows, in algorithmic TFLOP/s of that sample."""
    import oracle
    rng = np.random.default_rng(seed)
    total = case.T * case.Nq
    n = 256
    while True:
        rows = rng.choice(total, size=min(n, total), replace=False).astype(np.int64)
        t = time.perf_counter()
        oracle.prefill(case.q, case.k, case.v, case.cu_q, case.cu_kv, Nq=case.Nq, Nkv=case.Nkv, D=case.D,
                       scale=case.scale, causal=True, dtype=oracle.BF16, rows=rows)
        dt = time.perf_counter() - t
        if dt > budget_s / 4 or n >= total:
            break
        n = min(total, int(n * max(2.0, budget_s / max(dt, 1e-3) * 0.8)))
    tok = rows // case.Nq
    b = np.searchsorted(case.cu_q, tok, side="right") - 1
    qi = tok - case.cu_q[b]
    Lq = case.lengths_q[b]
    Lk = case.lengths_kv[b]
    vis = np.clip(qi + (Lk - Lq) + 1, 0, Lk)
    fl = 4 * case.D * int(vis.sum())
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{len(rows)} of {total} (token, head) rows; {dt:.1f} s of fp64 CPU work",
            "seconds": round(dt, 2)}


def run_ring_bench(args, rank, world, local_rank):
    """The context-parallel ring (attention_ifa_fia_gb300.ring) on one GPU: the long-context
    workload's KV cache split into --ring-shards shards, one per simulated rank (a CUDA
    stream); a step is fia_decode over every shard, then the ring of partial exchanges
    (device copies) and RingAttentionUpdate merges, every rank ending with the full result.
    value = the workload's algorithmic bytes / step time."""
    import torch
    import attention_ifa_fia_gb300 as F
    from attention_ifa_fia_gb300.ring import RingDecodeGraph
    from fia_workloads import DeviceDecode

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    case = W.long_ctx_sink_decode()
    nbytes = decode_bytes(case)
    ncopies = 2  # 2 x 1.07 GB of KV > L2
    copies = [DeviceDecode(case, dev) for _ in range(ncopies)]
    shards = args.ring_shards
    # one CUDA graph per input copy: a step is one graph launch (the ring's few hundred
    # operations issued from Python would otherwise bound it)
    graphs = [RingDecodeGraph(c.q, c.k, c.v, c.bt, c.lens, world=shards, max_kv_len=case.max_len,
                              num_heads=case.Nq, num_kv_heads=case.Nkv, scale=case.scale, sink=c.sink)
              for c in copies]

    def step(i):
        return graphs[i % ncopies].replay()

    dist = None
    if world > 1:
        import torch.distributed as dist
    sampler = ClockSampler(local_rank)
    sampler.start()
    t_w = time.time()
    i = 0
    while i < args.warmup or time.time() - t_w < args.min_warmup_s:
        step(i)
        i += 1
        if i % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    F.fia_device_status()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    h0 = time.time()
    e0.record(stream)
    for k in range(args.steps):
        step(k)
    e1.record(stream)
    torch.cuda.synchronize()
    h1 = time.time()
    if dist is not None:
        dist.barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    # kernels of one step: per shard the decode's plan, attention and merge, then one merge
    # (ring_attention_update) per rank and ring step
    launches = 3 * shards + shards * (shards - 1)
    status = F.fia_device_status()
    sampler.stop()
    if rank != 0:
        return None
    hbm, _, _, src = peaks()
    gbs = world * nbytes["total"] * args.steps / (ms / 1e3) / 1e9
    return {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "long_ctx_sink_ring", "B": case.B, "Nq": case.Nq, "Nkv": case.Nkv, "D": case.D,
                   "block_size": case.block_size, "kv_lengths": "131072 each", "ring_shards": shards,
                   "algorithmic_bytes_per_step": nbytes["total"],
                   "l2": f"inputs rotated over {ncopies} device copies ({ncopies} x {nbytes['kv'] / 1e6:.0f} MB of KV > L2)",
                   "parallelism": f"{shards} ranks simulated as CUDA streams of one GPU"
                                  + (f", independent replicas x{world}" if world > 1 else "")},
        "hbm_frac_of_measured": round(gbs / world / hbm, 4),
        "roofline": {"bound": "hbm", "achieved": round(gbs / world, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gbs / world / hbm, 4), "traffic": None,
                     "kernel": "whole ring step (attention on every shard, exchanges and merges)",
                     "peak_source": f"{src} HBM copy bandwidth"},
        "gpu_launches": launches * args.steps, "device_status": status, "clocks": sampler.summary(h0, h1),
        "graph": "each step one CUDA graph launch of the captured ring",
    }


# Sources of the kernel whose DRAM traffic bench.py reports, per workload; a recorded
# figure is used only while the sha1 of these files matches the one taken with it.
TRAFFIC_SOURCES = {
    "bf16_gqa_decode": ("decode_tc.cu", "decode.cu", "decode_common.cuh", "fia_device.cuh", "fia_internal.h"),
    "long_ctx_sink_decode": ("decode_tc.cu", "decode.cu", "decode_common.cuh", "fia_device.cuh", "fia_internal.h"),
    "int8_antiquant_decode": ("decode_i8tc.cu", "decode_i8.cuh", "decode.cu", "decode_common.cuh", "fia_device.cuh",
                              "fia_internal.h"),
    "causal_prefill_tnd": ("prefill.cu", "decode_common.cuh", "fia_device.cuh", "fia_internal.h"),
    "causal_prefill_tnd_t8k": ("prefill.cu", "decode_common.cuh", "fia_device.cuh", "fia_internal.h"),
}


def traffic_sha(workload):
    import hashlib
    csrc = os.path.join(ROOT, "attention_ifa_fia_gb300", "csrc")
    h = hashlib.sha1()
    for name in TRAFFIC_SOURCES[workload]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def load_traffic(workload):
    """DRAM bytes (read + write) per launch of the dominant kernel from the committed ncu summary
    (profiles/kernel_traffic.json), or None if the kernel's sources changed since it was taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "kernel_traffic.json")) as f:
            entry = json.load(f).get(workload)
        if not entry or entry.get("sources_sha1") != traffic_sha(workload):
            return None
        return entry.get("bytes_per_launch")
    except Exception:
        return None


# ----------------------------------------------------------------------------- reference arm: the oracle
def run_reference_prefill(args):
    """The oracle's prefill on a bounded sample of (token, head) rows per step."""
    import oracle
    case = W.WORKLOADS[args.workload]()
    rng = np.random.default_rng(0)
    total = case.T * case.Nq
    t = time.perf_counter()
    oracle.prefill(case.q, case.k, case.v, case.cu_q, case.cu_kv, Nq=case.Nq, Nkv=case.Nkv, D=case.D,
                   scale=case.scale, causal=True, dtype=oracle.BF16, rows=np.arange(64, dtype=np.int64))
    per_row = max((time.perf_counter() - t) / 64, 1e-5)
    n = int(min(total, max(16, 120.0 / max(args.steps + args.warmup, 1) / per_row)))
    tot_t, tot_f = 0.0, 0
    for k in range(args.warmup + args.steps):
        rows = rng.choice(total, size=n, replace=False).astype(np.int64)
        t = time.perf_counter()
        oracle.prefill(case.q, case.k, case.v, case.cu_q, case.cu_kv, Nq=case.Nq, Nkv=case.Nkv, D=case.D,
                       scale=case.scale, causal=True, dtype=oracle.BF16, rows=rows)
        dt = time.perf_counter() - t
        tok = rows // case.Nq
        b = np.searchsorted(case.cu_q, tok, side="right") - 1
        qi = tok - case.cu_q[b]
        vis = np.clip(qi + (case.lengths_kv[b] - case.lengths_q[b]) + 1, 0, case.lengths_kv[b])
        if k >= args.warmup:
            tot_t += dt
            tot_f += 4 * case.D * int(vis.sum())
    value = tot_f / tot_t / 1e12
    sample = f"each step: {n} of {total} (token, head) rows of {args.workload}"
    return {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload}, "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.max_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    if args.workload.startswith("causal_prefill_tnd"):
        return run_reference_prefill(args)
    case = W.WORKLOADS["long_ctx_sink_decode" if args.workload == "long_ctx_sink_ring" else args.workload]()
    rng = np.random.default_rng(0)
    all_groups = [(b, h) for b in range(case.B) for h in range(case.Nkv)]
    probe = [all_groups[i] for i in rng.permutation(len(all_groups))[:2]]
    dt, _, _ = oracle_decode_sample(case, probe)
    per_group = max(dt / len(probe), 1e-4)
    budget = 120.0 / max(args.steps + args.warmup, 1)
    n = int(min(len(all_groups), max(1, budget / per_group)))
    tot_t, tot_b, cores = 0.0, 0, 1
    for k in range(args.warmup + args.steps):
        idx = rng.permutation(len(all_groups))[:n]
        dt, nb, cores = oracle_decode_sample(case, [all_groups[i] for i in idx])
        if k >= args.warmup:
            tot_t += dt
            tot_b += nb
    value = tot_b / tot_t / 1e9
    sample = f"each step: {n} of {len(all_groups)} (batch, kv-head) groups of {args.workload}, all query heads"
    return {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload}, "impl": "reference",
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="bf16_gqa_decode",
                    choices=["bf16_gqa_decode", "int8_antiquant_decode", "long_ctx_sink_decode", "tiny_decode",
                             "causal_prefill_tnd", "causal_prefill_tnd_t8k", "long_ctx_sink_ring"])
    ap.add_argument("--ring-shards", type=int, default=8,
                    help="long_ctx_sink_ring: KV shards (ranks simulated as CUDA streams of one GPU)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--min-warmup-s", type=float, default=1.0,
                    help="keep warming up for at least this long (clocks settle, the sampler sees load)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        if args.workload.startswith("causal_prefill_tnd"):
            line = run_prefill_bench(args, rank, world, local_rank)
        elif args.workload == "long_ctx_sink_ring":
            line = run_ring_bench(args, rank, world, local_rank)
        else:
            line = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
