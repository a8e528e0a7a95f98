#!/usr/bin/env python
"""Benchmark of the paged GQA attention hot path on one GB300 (or N replicas).

Metric: decode KV GB/s (algorithmic bytes / time) on the bf16 GQA decode workload
(batch 64, 24 q / 4 kv heads, head_dim 512, page_size 64, kv_len uniform in [1024, 8192],
shuffled pages, split-K), with the causal bf16 prefill workload (lengths 2048 / 3000 /
4096 / 6272, 24 / 4 heads, head_dim 512) reported beside it in TFLOP/s.  Each figure is
also given as a fraction of the measured GB300 roofline (MEASURED_PEAKS.json).

A step is one call of the C ABI (all kernels of the phase) on inputs already resident in
HBM; "e2e" repeats the metric with host buffers (pinned host -> device copies of every
input and the device -> host read of the output inside the timed region).

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference] [--all]
"""

from __future__ import annotations

import argparse
import hashlib
import json
import random
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synth  # noqa: E402

MAIN = "gqa_decode_bf16"
PREFILL = "causal_prefill_bf16"
# the configurations the numbers are quoted on (synth.WORKLOADS holds their recipes)
DESCRIBE = {
    "tiny_mqa_decode": "tiny decode: batch 2, MQA 8 q / 1 kv heads, head_dim 512, bf16, page_size 16, "
                       "kv_len 37 and 64, shuffled pages, no window",
    "gqa_decode_bf16": "bf16 GQA decode: batch 64, 24 q / 4 kv heads, head_dim 512, page_size 64, "
                       "kv_len uniform in [1024, 8192], shuffled pages, split-K",
    "fp8_decode": "FP8 KV decode: batch 128, 12 q / 4 kv heads, head_dim 512, e4m3 KV with per-tensor fp32 "
                  "scales, page_size 16, kv_len 32768, bf16 q and output",
    "causal_prefill_bf16": "causal paged prefill bf16: new-token lengths 2048 / 3000 / 4096 / 6272, no cached "
                           "prefix, 24 q / 4 kv heads, head_dim 512, page_size 64, shuffled pages",
    "nvfp4_asym_prefill": "asymmetric NVFP4 causal prefill: qk 512 / vo 256, 16 q / 2 kv heads, 8 x 1024 "
                          "tokens, NVFP4 KV (e2m1, e4m3 scale per 16, fp32 global), page_size 32",
    "sliding_decode_d256": "sliding-window decode: head_dim 256, window_left 1023, 32 q / 16 kv heads, "
                           "batch 256, kv_len 8192, bf16 KV, page_size 16",
    "prefill_extend_bf16": "extend prefill: 4 x 32 new tokens over 16384 cached keys, 24 q / 4 kv heads, "
                           "head_dim 512, page_size 64, bf16",
}


def rank_world():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))


def bench_case(name, device="cuda"):
    """This rank's shard of the global batch (the whole workload on one GPU)."""
    rank, world = rank_world()
    return synth.workload_shard(name, rank, world, device=device)


def prefill_launches(variant: str) -> int:
    """Kernels one prefill call launches: the preparation (planner, with the FP8 / NVFP4
    page conversion or the small-page padding in the same launch) and the prefill kernel,
    plus the split-KV merge when the variant names it."""
    return 2 + ("_splitkv" in variant)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DECODE_SOURCES = ("decode_impl.cuh", "common.cuh", "decode_inst.cuh", "kernel_params.h")
PREFILL_SOURCES = ("prefill_impl.cuh", "common.cuh", "tc_helpers.cuh", "kernel_params.h")
APPEND_SOURCES = ("append.cu", "common.cuh", "kernel_params.h")


# ------------------------------------------------------------------------- work counts
def _beta_x2(kv_dtype):
    return {synth.KV_BF16: 4, synth.KV_FP8: 2, synth.KV_NVFP4: 1}[kv_dtype]


def decode_bytes(c) -> int:
    """Algorithmic bytes of one decode call: visible (in-window) K and V of every kv head,
    NVFP4 block scales, q, out and lse."""
    tokens = 0
    for L in c.kv_lens:
        tokens += min(L, c.window_left + 1) if c.window_left >= 0 else L
    per_tok = c.Hkv * (c.d_qk + c.d_vo) * _beta_x2(c.kv_dtype) // 2
    if c.kv_dtype == synth.KV_NVFP4:
        per_tok += c.Hkv * (c.d_qk + c.d_vo) // 16
    rows = c.total_q * c.Hq
    return tokens * per_tok + rows * (c.d_qk * 2 + c.d_vo * 2 + 4)


def prefill_flops(c) -> float:
    """Unmasked (query, key) pairs x (2 d_qk + 2 d_vo) x query heads."""
    pairs = 0
    for L, Q in zip(c.kv_lens, c.qo_lens):
        for i in range(Q):
            pos = L - Q + i
            hi = pos if c.causal else L - 1
            lo = max(0, pos - c.window_left) if c.window_left >= 0 else 0
            pairs += max(0, hi - lo + 1)
    return float(pairs) * c.Hq * (2 * c.d_qk + 2 * c.d_vo)


def prefill_kv_bytes(c) -> int:
    return sum(c.kv_lens) * c.Hkv * (c.d_qk + c.d_vo) * _beta_x2(c.kv_dtype) // 2


# ------------------------------------------------------------------------- environment
def peaks():
    p = dict(FALLBACK_PEAKS)
    src = "fallback"
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        for k in FALLBACK_PEAKS:
            if k in m:
                p[k] = float(m[k])
        src = "measured"
    return p, src


def code_tokens(text: str) -> str:
    """C / CUDA source without comments, whitespace runs collapsed: what the compiler sees.
    String and character literals are kept as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def sources_digest(names, read=None) -> str:
    """Digest of the kernel sources' code (comments and layout do not count), used to tell
    whether a recorded ncu capture was taken on the current kernel."""
    h = hashlib.sha256()
    for n in names:
        path = os.path.join(ROOT, "paged_gqa_attention_hd512_gb300", "csrc", n)
        text = read(n) if read else (open(path).read() if os.path.exists(path) else None)
        if text is not None:
            h.update(code_tokens(text).encode())
    return h.hexdigest()[:16]


def traffic_record(kernel: str, workload: str, digest: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current
    kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path)).get(f"{kernel}:{workload}")
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_digest") != digest:
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------- timing
def max_over_ranks(x: float, device="cuda") -> float:
    """The largest x over all ranks of the default process group (x itself when there is
    no group): the step time every rank reports is the slowest rank's."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(units_per_rank: float, world: int, ms: float, scale: float = 1e9) -> float:
    """Whole-job throughput: every rank processes the same workload (weak scaling), so the
    job processes `world` times the units of one rank in the slowest rank's time."""
    return units_per_rank * world / (ms * 1e-3) / scale


def time_region(fn, steps, warmup, barrier=None):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return e0.elapsed_time(e1)


def oracle_sample_rate(host_case, budget_s: float, kind: str):
    """Time the fp64 oracle on a bounded sample of the workload and return (rate in the
    metric's unit, seconds, description, threads).

    Decode samples (sequence, kv head) units, all query heads of the group each; prefill
    samples (query token, kv head) units, strided across every sequence so that short and
    long causal rows are both represented.  The sample cycles through the units (repeating
    them when the workload has fewer than the budget needs) and grows until it takes
    roughly ``budget_s`` seconds."""
    import numpy as np

    import oracle

    threads = oracle.default_threads()
    c = host_case
    g = c.group
    qo = c.qo_indptr.tolist()
    if kind == "decode":
        units = [(b, k, qo[b]) for b in range(c.batch) for k in range(c.Hkv) if qo[b + 1] > qo[b]]
    else:
        units = [(b, k, t) for b in range(c.batch) for t in range(qo[b], qo[b + 1]) for k in range(c.Hkv)]
        units = units[::max(1, len(units) // 4096)]
    # a fixed shuffle, so that any prefix of the sample spans the whole batch
    random.Random(0).shuffle(units)

    def work_of(sel):
        if kind == "decode":
            tok = 0
            for b, _, _ in sel:
                L = c.kv_lens[b]
                tok += min(L, c.window_left + 1) if c.window_left >= 0 else L
            return tok * (c.d_qk + c.d_vo) * _beta_x2(c.kv_dtype) // 2 + len(sel) * g * (2 * c.d_qk + 2 * c.d_vo + 4)
        pairs = 0
        for b, _, t in sel:
            L, Q = c.kv_lens[b], c.qo_lens[b]
            pos = L - Q + (t - qo[b])
            lo = max(0, pos - c.window_left) if c.window_left >= 0 else 0
            pairs += max(0, (pos if c.causal else L - 1) - lo + 1)
        return pairs * g * (2 * c.d_qk + 2 * c.d_vo)

    def run(n):
        sel = [units[i % len(units)] for i in range(n)]
        tok = np.repeat(np.array([t for _, _, t in sel], dtype=np.int64), g)
        head = np.concatenate([np.arange(k * g, (k + 1) * g) for _, k, _ in sel])
        t0 = time.perf_counter()
        oracle.rows(c, tok, head, threads=threads)
        return time.perf_counter() - t0, sel

    n = threads
    dt, sel = run(n)
    while dt < budget_s * 0.5:
        n = max(n + 1, int(n * min(64.0, budget_s * 0.8 / max(dt, 1e-3))))
        dt, sel = run(n)
    rate = work_of(sel) / dt / (1e9 if kind == "decode" else 1e12)
    distinct = len({u for u in sel})
    seqs = len({b for b, _, _ in sel})
    what = "(sequence, kv head)" if kind == "decode" else "(query token, kv head)"
    desc = (f"{len(sel)} {what} units ({distinct} distinct, from {seqs} sequences), all {g} query heads each, "
            f"{dt:.1f} s of oracle time")
    return rate, dt, desc, threads


# ------------------------------------------------------------------------- our arm
def bench_decode(name, steps, warmup, barrier, gpu_index, pk, with_e2e=True, with_cpu=True):
    import paged_gqa_attention_hd512_gb300 as pa

    c = bench_case(name)
    kw = pa.case_args(c)
    out = torch.empty(c.batch, c.Hq, c.d_vo, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(c.batch, c.Hq, dtype=torch.float32, device="cuda")

    def step():
        pa.paged_attn_decode(c.q, c.kv_cache, c.kv_indptr, c.kv_indices, c.kv_last_page_len, out=out, lse=lse,
                             **kw)

    step()
    torch.cuda.synchronize()
    if pa.paged_attn_check_device_error() != 0:
        raise RuntimeError("device error word set after the first decode call")
    nbytes = decode_bytes(c)
    with ClockSampler(gpu_index) as clk:
        # the steps as a user makes them; then the same steps again with the library's
        # events around the decode kernel for its own duration (an event between the
        # planner and the kernel keeps the kernel from starting under the planner's tail,
        # so those steps are not the ones the value reports)
        ms = time_region(step, steps, warmup, barrier)
        pa.paged_attn_profile_begin(steps)
        time_region(step, steps, 0, barrier)
        n_k, k_ms = pa.paged_attn_profile_end()
    clocks = clk.summary()
    variant = pa.paged_attn_last_variant()
    # planner, decode kernel and merge; the decode kernel alone on the single-launch path
    launches = (1 if variant.endswith("_direct") else 3) * steps
    res = {"workload": name, "config": {"workload": DESCRIBE.get(name, name), "name": name},
           "ms_per_step": ms / steps, "value": nbytes / (ms / steps * 1e-3) / 1e9,
           "unit": "GB/s", "bytes_per_step": nbytes, "steps": steps, "clocks": clocks, "variant": variant,
           "gpu_launches": launches}
    kern_ms = k_ms / max(1, n_k)
    achieved = nbytes / (kern_ms * 1e-3) / 1e9
    digest = sources_digest(DECODE_SOURCES)
    res["roofline"] = {"bound": "hbm", "achieved": achieved, "peak": pk[0]["hbm_gbs"], "unit": "GB/s",
                       "frac": achieved / pk[0]["hbm_gbs"], "traffic": traffic_record("decode_kernel", name, digest),
                       "kernel": "decode_kernel", "kernel_ms": kern_ms, "launches_timed": n_k,
                       "peak_source": f"{pk[1]} hbm_gbs", "source_digest": digest}
    if with_e2e:
        res["e2e"] = decode_e2e(c, kw, max(3, min(steps, 10)), nbytes)
    if with_cpu:
        host = c.to("cpu")
        rate, dt, desc, threads = oracle_sample_rate(host, 15.0, "decode")
        res["cpu_baseline"] = {"value": rate, "unit": "GB/s", "cores": threads, "kind": "oracle",
                               "sample": desc, "seconds": dt}
    del c
    torch.cuda.empty_cache()
    return res


def decode_e2e(c, kw, steps, nbytes):
    """Same metric through the C ABI from pinned host buffers, copies in the timed region."""
    import paged_gqa_attention_hd512_gb300 as pa

    names = ("q", "kv_cache", "kv_indptr", "kv_indices", "kv_last_page_len")
    host = {n: getattr(c, n).cpu().pin_memory() for n in names}
    dev = {n: torch.empty_like(getattr(c, n)) for n in names}
    out_h = torch.empty(c.batch, c.Hq, c.d_vo, dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty(c.batch, c.Hq, dtype=torch.float32).pin_memory()
    out = torch.empty(c.batch, c.Hq, c.d_vo, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(c.batch, c.Hq, dtype=torch.float32, device="cuda")
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * 2 + lse_h.numel() * 4

    def step():
        for n in names:
            dev[n].copy_(host[n], non_blocking=True)
        pa.paged_attn_decode(dev["q"], dev["kv_cache"], dev["kv_indptr"], dev["kv_indices"],
                             dev["kv_last_page_len"], out=out, lse=lse, **kw)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    ms = time_region(step, steps, 2)
    res = {"value": nbytes / (ms / steps * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": ms / steps}
    del dev, host
    return res


def bench_prefill(name, steps, warmup, gpu_index, pk, with_cpu=False, split_kv=True, with_e2e=False):
    import paged_gqa_attention_hd512_gb300 as pa

    pa.paged_attn_set_prefill_split_kv(-1 if split_kv else 0)
    try:
        res = _bench_prefill(pa, name, steps, warmup, gpu_index, pk, with_cpu, with_e2e)
    finally:
        pa.paged_attn_set_prefill_split_kv(-1)
    if not split_kv:
        res["workload"] = name + " (split KV off)"
    return res


def prefill_e2e(c, kw, steps, flops):
    """Same metric through the C ABI from pinned host buffers: q, the page table and the
    cache copied in, out and lse copied back, inside the timed region."""
    import paged_gqa_attention_hd512_gb300 as pa

    names = ["q", "qo_indptr", "kv_cache", "kv_indptr", "kv_indices", "kv_last_page_len"]
    if c.sf is not None:
        names.append("sf")
    host = {n: getattr(c, n).cpu().pin_memory() for n in names}
    dev = {n: torch.empty_like(getattr(c, n)) for n in names}
    kw = dict(kw)
    out_h = torch.empty(c.total_q, c.Hq, c.d_vo, dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty(c.total_q, c.Hq, dtype=torch.float32).pin_memory()
    out = torch.empty(c.total_q, c.Hq, c.d_vo, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(c.total_q, c.Hq, dtype=torch.float32, device="cuda")
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    if "sf" in dev:
        kw["sf"] = dev["sf"]

    def step():
        for n in names:
            dev[n].copy_(host[n], non_blocking=True)
        pa.paged_attn_prefill(dev["q"], dev["qo_indptr"], dev["kv_cache"], dev["kv_indptr"], dev["kv_indices"],
                              dev["kv_last_page_len"], causal=bool(c.causal), out=out, lse=lse, **kw)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    ms = time_region(step, steps, 2)
    res = {"value": flops / (ms / steps * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": ms / steps}
    del dev, host
    return res


def _bench_prefill(pa, name, steps, warmup, gpu_index, pk, with_cpu, with_e2e):
    c = bench_case(name)
    kw = pa.case_args(c)
    out = torch.empty(c.total_q, c.Hq, c.d_vo, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(c.total_q, c.Hq, dtype=torch.float32, device="cuda")

    def step():
        pa.paged_attn_prefill(c.q, c.qo_indptr, c.kv_cache, c.kv_indptr, c.kv_indices, c.kv_last_page_len,
                              causal=bool(c.causal), out=out, lse=lse, **kw)

    try:
        step()
    except pa.PagedAttnError as e:
        return {"workload": name, "unavailable": str(e)}
    torch.cuda.synchronize()
    if pa.paged_attn_check_device_error() != 0:
        raise RuntimeError("device error word set after the first prefill call")
    flops = prefill_flops(c)
    # the KV of this workload (~126 MB) is about the size of L2: flush L2 between steps
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    with ClockSampler(gpu_index) as clk:
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()

        def timed_steps():
            tot = 0.0
            for _ in range(steps):
                flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                step()
                e1.record(s)
                e1.synchronize()
                tot += e0.elapsed_time(e1)
            return tot

        # the calls as a user makes them, then again with the library's events around the
        # prefill kernel for its own duration (an event between the preparation kernel and
        # the prefill kernel keeps the latter from starting under the former's tail)
        tot = timed_steps()
        pa.paged_attn_profile_begin(steps)
        timed_steps()
        n_k, k_ms = pa.paged_attn_profile_end()
    ms = tot / steps
    kern_ms = k_ms / max(1, n_k)
    achieved = flops / (kern_ms * 1e-3) / 1e12
    digest = sources_digest(PREFILL_SOURCES)
    variant = pa.paged_attn_last_variant()
    res = {"workload": name, "config": {"workload": DESCRIBE.get(name, name), "name": name},
           "ms_per_step": ms, "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
           "flops_per_step": flops, "steps": steps, "variant": variant, "clocks": clk.summary(),
           "l2": "flushed between steps (256 MiB write)", "gpu_launches": prefill_launches(variant) * steps,
           "roofline": {"bound": "tensor", "achieved": achieved, "peak": pk[0]["bf16_tflops"], "unit": "TFLOP/s",
                        "frac": achieved / pk[0]["bf16_tflops"],
                        "traffic": traffic_record("prefill_kernel", name, digest), "kernel": "prefill_kernel",
                        "kernel_ms": kern_ms, "launches_timed": n_k, "peak_source": f"{pk[1]} bf16_tflops (burst)",
                        "source_digest": digest}}
    if with_e2e:
        res["e2e"] = prefill_e2e(c, kw, max(3, min(steps, 10)), flops)
    if with_cpu:
        rate, dt, desc, threads = oracle_sample_rate(c.to("cpu"), 15.0, "prefill")
        res["cpu_baseline"] = {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                               "sample": desc, "seconds": dt}
    del c, flush
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------------- append
APPEND_WORKLOADS = {
    # name: (kv dtype, sequences, new tokens each, kv heads, d_qk, d_vo, page_size)
    "append_nvfp4_asym": (synth.KV_NVFP4, 64, 1024, 2, 512, 256, 32),
    "append_fp8_gqa": (synth.KV_FP8, 128, 512, 4, 512, 512, 16),
}


def append_bytes(kv_dtype, total, hkv, dqk, dvo) -> int:
    """bf16 rows read + converted rows (and NVFP4 block scales) written."""
    elems = total * hkv * (dqk + dvo)
    out = elems * _beta_x2(kv_dtype) // 2 + (elems // 16 if kv_dtype == synth.KV_NVFP4 else 0)
    return elems * 2 + out


def bench_append(name, steps, warmup, gpu_index, pk):
    """paged_attn_append_kv writing whole sequences of new tokens into an empty cache."""
    import numpy as np
    import paged_gqa_attention_hd512_gb300 as pa

    kvt, nseq, ntok, hkv, dqk, dvo, ps = APPEND_WORKLOADS[name]
    total = nseq * ntok
    pages_per = -(-ntok // ps)
    num_pages = nseq * pages_per
    dev = "cuda"
    perm = torch.from_numpy(np.random.default_rng(4242).permutation(num_pages).astype(np.int32))
    kv_indices = perm.to(dev)
    kv_indptr = torch.arange(0, num_pages + 1, pages_per, dtype=torch.int32, device=dev)
    last = torch.full((nseq,), (ntok - 1) % ps + 1, dtype=torch.int32, device=dev)
    append_indptr = torch.arange(0, total + 1, ntok, dtype=torch.int32, device=dev)
    k_new = synth.normal_bf16(4242, 1, 0, total * hkv * dqk, dev).view(total, hkv, dqk)
    v_new = synth.normal_bf16(4242, 2, 0, total * hkv * dvo, dev).view(total, hkv, dvo)
    page_bytes = hkv * ps * (dqk + dvo) * _beta_x2(kvt) // 2
    cache = torch.zeros(num_pages * page_bytes, dtype=torch.uint8, device=dev)
    sf = torch.zeros(num_pages * hkv * ps * (dqk + dvo) // 16, dtype=torch.uint8, device=dev) \
        if kvt == synth.KV_NVFP4 else None
    ks = torch.tensor([2.0 ** -8 if kvt == synth.KV_NVFP4 else 0.02], dtype=torch.float32, device=dev)
    vs = ks.clone()

    def step():
        pa.paged_attn_append_kv(k_new, v_new, append_indptr, cache, kv_indptr, kv_indices, last, page_size=ps,
                                kv_dtype=kvt, k_scale=ks, v_scale=vs, sf=sf, num_pages=num_pages)

    step()
    torch.cuda.synchronize()
    if pa.paged_attn_check_device_error() != 0:
        raise RuntimeError("device error word set after the first append call")
    nbytes = append_bytes(kvt, total, hkv, dqk, dvo)
    with ClockSampler(gpu_index) as clk:
        pa.paged_attn_profile_begin(steps)
        ms = time_region(step, steps, warmup)
        n_k, k_ms = pa.paged_attn_profile_end()
    kern_ms = k_ms / max(1, n_k)
    achieved = nbytes / (kern_ms * 1e-3) / 1e9
    digest = sources_digest(APPEND_SOURCES)
    res = {"workload": name, "ms_per_step": ms / steps, "value": nbytes / (ms / steps * 1e-3) / 1e9, "unit": "GB/s",
           "bytes_per_step": nbytes, "variant": pa.paged_attn_last_variant(), "clocks": clk.summary(),
           "l2": f"{nbytes / 1e6:.0f} MB per step, larger than L2", "gpu_launches": steps,
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk[0]["hbm_gbs"], "unit": "GB/s",
                        "frac": achieved / pk[0]["hbm_gbs"],
                        "traffic": traffic_record("append_kv_kernel", name, digest), "kernel": "append_kv_kernel",
                        "kernel_ms": kern_ms, "launches_timed": n_k, "peak_source": f"{pk[1]} hbm_gbs",
                        "source_digest": digest}}
    del k_new, v_new, cache, sf
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--all", action="store_true", help="also time every other workload")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle cpu_baseline leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer e2e legs")
    ap.add_argument("--no-secondary", action="store_true", help="time only the main decode and prefill lines")
    ap.add_argument("--workload", default=MAIN, help="decode workload of the main line")
    ap.add_argument("--prefill-only", action="store_true", help="time only the prefill workload (profiling)")
    ap.add_argument("--prefill-workload", default=PREFILL, help="prefill workload of --prefill-only")
    ap.add_argument("--append-only", choices=sorted(APPEND_WORKLOADS), default=None,
                    help="time only this append workload (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    barrier = None
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference" and rank != 0:
            return 0
        if args.impl == "ours":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
            barrier = dist.barrier

    if args.impl == "reference":
        return reference_arm(args, world)

    from paged_gqa_attention_hd512_gb300 import build as pa_build
    if rank == 0 or world == 1:
        pa_build.build()
    if barrier:
        barrier()
    torch.cuda.set_device(local)
    pk = peaks()
    psteps = max(5, min(50, args.steps // 2))
    if args.prefill_only:
        res = bench_prefill(args.prefill_workload, psteps, args.warmup, local, pk)
        if rank == 0:
            print(json.dumps({"prefill": res}), flush=True)
        return 0
    if args.append_only:
        res = bench_append(args.append_only, max(3, args.steps // 10), args.warmup, local, pk)
        if rank == 0:
            print(json.dumps({"append": res}), flush=True)
        return 0
    main_res = bench_decode(args.workload, args.steps, args.warmup, barrier, local, pk,
                            with_e2e=not args.no_e2e, with_cpu=(rank == 0 and not args.no_cpu))
    ms = max_over_ranks(main_res["ms_per_step"])
    value = weak_scaling_value(main_res["bytes_per_step"], world, ms)
    line = {
        "metric": "decode KV GB/s and prefill TFLOPS at hd512, % of GB300 roofline",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Irwin-Hall(4) standard-normal draws; seeded random page order)",
        "config": {"workload": DESCRIBE.get(args.workload, args.workload),
                   "name": args.workload, "l2": "inputs (2.6 GB of KV) larger than L2, no flush",
                   "parallelism": (f"global batch of {world} x the workload's batch, split by sequence over "
                                   f"{world} rank(s) (one shard each), no collective")},
        "e2e": main_res.get("e2e"), "roofline": main_res["roofline"], "cpu_baseline": main_res.get("cpu_baseline"),
        "clocks": main_res["clocks"], "gpu_launches": main_res["gpu_launches"], "variant": main_res["variant"],
    }
    if not args.no_prefill:
        line["prefill"] = bench_prefill(PREFILL, psteps, 3, local, pk, with_cpu=(rank == 0 and not args.no_cpu),
                                        with_e2e=not args.no_e2e)
    if not args.no_secondary:
        # the other configurations the metric covers; --all adds the extend prefill and
        # the append kernel
        extra = []
        for name in ("tiny_mqa_decode", "fp8_decode", "sliding_decode_d256"):
            extra.append(bench_decode(name, args.steps, args.warmup, barrier, local, pk, with_e2e=False,
                                      with_cpu=False))
        if not args.no_prefill:
            extra.append(bench_prefill("nvfp4_asym_prefill", psteps, 3, local, pk))
        if args.all:
            for split_kv in (True, False):
                extra.append(bench_prefill("prefill_extend_bf16", psteps, 3, local, pk, split_kv=split_kv))
            for name in APPEND_WORKLOADS:
                extra.append(bench_append(name, max(3, args.steps // 10), args.warmup, local, pk))
        line["secondary"] = extra
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def reference_arm(args, world):
    """The oracle (fp64, host cores) as the reference arm: each step is a bounded sample of
    the same workload, sized so the whole run ends within a few minutes."""
    import numpy as np

    import oracle

    oracle.build()
    c = synth.workload(MAIN, device="cuda" if torch.cuda.is_available() else "cpu").to("cpu")
    threads = oracle.default_threads()
    g = c.group
    budget = 120.0 / (args.steps + args.warmup)
    # calibrate: one (sequence, kv head) unit per thread
    units = [(b, k) for b in range(c.batch) for k in range(c.Hkv)]

    def rows_of(sel):
        tok, head = [], []
        for b, k in sel:
            tok += [b] * g
            head += list(range(k * g, (k + 1) * g))
        return np.array(tok), np.array(head)

    def unit_bytes(sel):
        return sum(c.kv_lens[b] for b, _ in sel) * (c.d_qk + c.d_vo) * 2 + len(sel) * g * (2 * c.d_qk + 2 * c.d_vo + 4)

    t0 = time.perf_counter()
    oracle.rows(c, *rows_of(units[:1]), threads=1)
    per_unit = time.perf_counter() - t0
    n = max(1, min(len(units), int(budget / max(per_unit, 1e-6) * min(threads, 8))))
    cursor = [0]

    def one_step():
        sel = [units[(cursor[0] + i) % len(units)] for i in range(n)]
        cursor[0] += n
        t = time.perf_counter()
        oracle.rows(c, *rows_of(sel), threads=threads)
        return time.perf_counter() - t, unit_bytes(sel)

    for _ in range(args.warmup):
        one_step()
    tot_t, tot_b = 0.0, 0
    for _ in range(args.steps):
        dt, nb = one_step()
        tot_t += dt
        tot_b += nb
    value = tot_b / tot_t / 1e9
    sample = f"{n} (sequence, kv head) unit(s) per step, all {g} query heads each, cycling through the batch"
    line = {"impl": "reference", "metric": "decode KV GB/s and prefill TFLOPS at hd512, % of GB300 roofline",
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": DESCRIBE[MAIN], "name": MAIN},
            "cpu_baseline": {"kind": "oracle", "cores": threads, "sample": sample, "value": value, "unit": "GB/s"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
