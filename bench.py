"""Benchmark of the paged varlen relative-bias attention forward on GB300.

One step = one rel_attn_paged_varlen call over the whole workload: the split
heuristic, the main kernel and (when splits > 1) the LSE combine.  Inputs are
seeded and synthetic (paged_attention_relative_gb300.workloads) and resident
in HBM before timing; the attention inputs (KV cache >= 512 MiB for the
decode workloads, 2.55 GB per chunked-prefill step) are larger than the
129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

The default run prints the long-decode headline (`value`) and, under
"workloads", a complete record for each of the other measured workloads:
batched decode, chunked prefill, mixed varlen with a window, and the paged
KV-cache append of the chunked-prefill tokens.  Every record times its own
steps after at least one second of back-to-back steps, with nvidia-smi
sampling clocks over that whole busy period.  `--workload NAME` prints that
workload's record alone.

Prints one JSON line on rank 0.  Under torchrun every rank runs its own
replica of the workload on its own GPU (the work shards by request and kv
head with no exchange), so scaling is weak.  The library is a one-GPU
library and its prefill kernel loads K/V tiles with cluster multicast:
multi-rank runs refuse the prefill workloads and leave them out of the
default record.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode HBM TB/s & % roofline; prefill TFLOP/s & % bf16 peak (1×GB300)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {"decode": ["decode.cu", "common.cuh"], "prefill": ["prefill.cu", "common.cuh"],
                  "prefill_pair": ["prefill_pair.cu", "common.cuh"],
                  "append": ["append.cu", "common.cuh"]}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_hash(kind: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        p = os.path.join(ROOT, "paged_attention_relative_gb300", "csrc", name)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kind: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_hash(kind)
    for line in open(path):
        parts = line.split("#")[0].split()
        if len(parts) >= 4 and parts[0] == workload and parts[1] == kind and parts[2] == want:
            return int(float(parts[3]))
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's):
    an all-reduce on `device` (a CUDA device under NCCL, CPU under gloo)."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, work_per_replica: float, ms: float) -> float:
    """Whole-job throughput in work units per second x 1e-12: every rank runs
    one replica of the workload, so the job did world x the work in the
    slowest rank's time."""
    return world * work_per_replica / (ms * 1e-3) / 1e12


def make_workload(name: str):
    from paged_attention_relative_gb300 import workloads as W
    return W.WORKLOADS[name](0)


def heuristic_splits(case, lib_splits):
    d = case.dims
    sk = case.cache_seqlens.tolist()
    return lib_splits(case.window_left >= 0 or case.window_right >= 0, d["B"], max(case.seqlens_q), d["H"],
                      d["Hk"], max(sk) if sk else 0)


PREFILL_MULTI_RANK = ("1-GPU library: the prefill kernel loads K/V tiles with cluster multicast, which runs on "
                      "one GPU only; multi-rank runs time the decode workloads and the append")


def uses_prefill(case) -> bool:
    """The library picks the tcgen05 prefill kernel above 64 GQA-packed rows."""
    d = case.dims
    return case.max_seqlen_q * (d["H"] // d["Hk"]) > 64


def soak_then_time(step, steps: int, soak_s: float, stream, dev, world):
    """Run `step` back to back for about soak_s seconds (untimed), then time
    exactly `steps` steps with CUDA events on `stream`, bracketed by a barrier
    and a device synchronize; nvidia-smi samples clocks over the whole busy
    period (so the samples see the GPU under load).  Returns (ms per step,
    max over ranks; the clock summary; the soak's step count)."""
    import torch
    barrier = (lambda: torch.distributed.barrier()) if world > 1 else (lambda: None)
    with ClockSampler(dev.index) as clocks:
        t0 = time.perf_counter()
        n_soak = 0
        while True:
            for _ in range(8):
                step()
            n_soak += 8
            torch.cuda.synchronize()
            if time.perf_counter() - t0 >= soak_s:
                break
        barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world, dev)
    summ = clocks.summary()
    summ["window"] = f"{soak_s:g} s of back-to-back steps ({n_soak}) ending with the timed steps"
    return ms, summ, n_soak


def run_ours(args, rank, world, workload=None, steps=None, soak_s=1.0):
    """One attention workload: device step time, the main kernel's time from
    library-recorded events, end to end through the public API, roofline."""
    import ctypes

    import torch

    import paged_attention_relative_gb300 as pa
    from paged_attention_relative_gb300 import _lib
    from paged_attention_relative_gb300.roofline import algorithmic_bytes, algorithmic_flops

    workload = workload or args.workload
    steps = steps or args.steps
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    case = make_workload(workload)
    if world > 1 and uses_prefill(case):
        raise SystemExit(f"bench.py: {workload} refused with {world} ranks: {PREFILL_MULTI_RANK}")
    if args.splits is not None and workload == args.workload:
        splits = args.splits
    elif workload == "long_decode":
        splits = case.num_splits                  # the workload's own split count (16)
    else:
        splits = heuristic_splits(case, pa.rel_attn_num_splits)
    g = {k: getattr(case, k).to(dev) for k in ("q", "key_cache", "value_cache", "block_table", "cache_seqlens",
                                               "cu_seqlens_q", "rel_logits")}
    out = torch.empty_like(g["q"])
    stream = torch.cuda.current_stream(dev)

    # Pre-built descriptors: the timed loop is the bare C-ABI call.
    D = [_lib.describe(g[k]) for k in ("q", "key_cache", "value_cache", "block_table", "cache_seqlens",
                                       "cu_seqlens_q")]
    rel = _lib.describe(g["rel_logits"]) if case.rel_extent > 0 else None
    od = _lib.describe(out)
    refs = [ctypes.byref(d) for d in D]
    rref = ctypes.byref(rel) if rel is not None else None
    oref = ctypes.byref(od)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    call_args = (*refs, case.max_seqlen_q, ctypes.c_float(case.softmax_scale), int(case.causal),
                 case.window_left, case.window_right, case.rel_extent, rref, splits, oref, sptr)
    fn = _lib.lib.rel_attn_paged_varlen

    def step():
        st = fn(*call_args)
        if st != 0:
            raise RuntimeError(_lib.lib.rel_attn_last_error().decode())

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize()
    info = pa.last_launch()
    kind = info["kernel"]

    # Whole-step timing after a soak of back-to-back steps.
    ms_step, clocks, n_soak = soak_then_time(step, steps, soak_s, stream, dev, world)

    # Main-kernel timing with events recorded by the library around the launch.
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for b, e in evs:          # torch creates the CUDA event on first record
        b.record(stream)
        e.record(stream)
    for b, e in evs:
        pa.set_kernel_events(b, e)
        step()
    pa.set_kernel_events(None, None)
    torch.cuda.synchronize()
    kern_ms = [b.elapsed_time(e) for b, e in evs]
    kern_avg = max_over_ranks(sum(kern_ms) / len(kern_ms), world, dev)

    # End to end through the public API: pinned host inputs -> device, call,
    # result -> pinned host, every step.  The paged KV cache stays resident.
    # The step's inputs live packed in one pinned host buffer (each at a
    # 256-byte aligned offset) and move in one copy; the device views are
    # what the call receives.
    names_in = ("q", "rel_logits", "block_table", "cache_seqlens", "cu_seqlens_q")
    srcs = {k: getattr(case, k).contiguous() for k in names_in}
    offs, total = {}, 0
    for k in names_in:
        offs[k] = total
        total += (srcs[k].numel() * srcs[k].element_size() + 255) // 256 * 256
    host_buf = torch.empty(max(total, 256), dtype=torch.uint8, pin_memory=True)
    dev_buf = torch.empty_like(host_buf, device=dev)

    def views(buf):
        return {k: buf[offs[k]:offs[k] + srcs[k].numel() * srcs[k].element_size()].view(srcs[k].dtype)
                .view(srcs[k].shape) for k in names_in}

    for k, v in views(host_buf).items():
        v.copy_(srcs[k])
    dev_in = views(dev_buf)
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in srcs.values())
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step():
        dev_buf.copy_(host_buf, non_blocking=True)
        pa.rel_attn_paged_varlen(dev_in["q"], g["key_cache"], g["value_cache"], dev_in["block_table"],
                                 dev_in["cache_seqlens"], dev_in["cu_seqlens_q"], case.max_seqlen_q,
                                 case.softmax_scale, case.causal, case.window_left, case.window_right,
                                 case.rel_extent, dev_in["rel_logits"], splits, out=out)
        host_out.copy_(out, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(steps):
        e2e_step()
    a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a0.elapsed_time(a1) / steps, world, dev)

    nbytes = algorithmic_bytes(case)
    flops = algorithmic_flops(case)
    pk, pk_src = peaks()
    decode = kind == "decode"
    if decode:
        value = job_rate(world, nbytes, ms_step)
        unit = "TB/s"
        e2e_value = job_rate(world, nbytes, e2e_ms)
        ach = nbytes / (kern_avg * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / pk["hbm_gbs"], 4), "traffic": recorded_traffic(workload, kind),
                "peak_source": f"{pk_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if pk_src == "measured" else "fallback 6.8 TB/s",
                "nominal_frac_8tbs": round(ach / 8000.0, 4)}
    else:
        value = job_rate(world, flops, ms_step)
        unit = "TFLOP/s"
        e2e_value = job_rate(world, flops, e2e_ms)
        ach = flops / (kern_avg * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(ach / pk["bf16_tflops"], 4), "traffic": recorded_traffic(workload, kind),
                "peak_source": f"{pk_src} cuBLAS bf16 burst (MEASURED_PEAKS.json bf16_tflops)",
                "frac_of_sustained": round(ach / pk.get("bf16_tflops_sustained", pk["bf16_tflops"]), 4)}
    d = case.dims
    res = {
        "metric": METRIC, "value": round(value, 4), "unit": unit, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, shuffled page pool)",
        "config": {"workload": workload, "batch": d["B"], "tokens": d["T"], "num_heads": d["H"],
                   "num_kv_heads": d["Hk"], "head_dim": d["D"], "block_size": d["BS"], "rel_extent": d["R"],
                   "max_kv_len": int(case.cache_seqlens.max()), "num_splits": splits,
                   "window": [case.window_left, case.window_right], "causal": case.causal,
                   "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2 (paged KV > 129 MB)" if decode
                   else "inputs larger than L2 (K/V, q and rel_logits > 129 MB)",
                   "algorithmic_bytes": nbytes, "algorithmic_flops": flops},
        "kernel": {"name": kind, "avg_ms": round(kern_avg, 5), "launches_per_step": info["launches"],
                   "grid": info["grid"], "block": info["block"], "smem_bytes": info["smem_bytes"]},
        "roofline": roof,
        "tokens_per_s": round(world * d["T"] / (ms_step * 1e-3), 1),
        "e2e": {"value": round(e2e_value, 4), "unit": unit, "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "pinned host q, rel_logits, block_table, cache_seqlens, cu_seqlens_q in (one packed copy); out back; paged KV resident"},
        "gpu_launches": steps * info["launches"],
        "clocks": clocks,
    }
    del g, out, host_buf, dev_buf, host_out
    torch.cuda.empty_cache()
    return res, case


def run_append(args, rank, world, steps=None, soak_s=1.0):
    """The paged KV-cache append for the chunked-prefill workload's new tokens
    (4 x 4096 tokens, 8 kv heads, head_dim 128): HBM-bound, so `value` is
    algorithmic bytes (key and value rows read once and written once) per
    kernel second; L2 is flushed (a 256 MB buffer read) before every launch since the
    rows (67 MB) fit in L2."""
    import torch

    import paged_attention_relative_gb300 as pa

    steps = steps or args.steps
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    case = make_workload("chunked_prefill")
    d = case.dims
    gen = torch.Generator().manual_seed(0)
    key = torch.randn(d["T"], d["Hk"], d["D"], generator=gen).to(torch.bfloat16)
    value = torch.randn(d["T"], d["Hk"], d["D"], generator=gen).to(torch.bfloat16)
    g = {k: getattr(case, k).to(dev) for k in ("key_cache", "value_cache", "block_table", "cache_seqlens",
                                               "cu_seqlens_q")}
    kd, vd = key.to(dev), value.to(dev)
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)  # 256 MB, read (clean lines) before each launch
    stream = torch.cuda.current_stream(dev)

    def call(k, v):
        pa.rel_attn_cache_append(k, v, g["key_cache"], g["value_cache"], g["block_table"], g["cache_seqlens"],
                                 g["cu_seqlens_q"])

    for _ in range(max(args.warmup, 3)):
        call(kd, vd)
    torch.cuda.synchronize()
    # Events recorded by the library right around the launch (no host work
    # inside), after a soak of flush + append steps under the clock sampler.
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for b, e in evs:          # torch creates the CUDA event on first record
        b.record(stream)
        e.record(stream)
    with ClockSampler(dev.index) as clocks:
        t0 = time.perf_counter()
        n_soak = 0
        while time.perf_counter() - t0 < soak_s:
            for _ in range(8):
                flush.sum()
                call(kd, vd)
            n_soak += 8
            torch.cuda.synchronize()
        for b, e in evs:
            flush.sum()
            pa.set_kernel_events(b, e)
            call(kd, vd)
        pa.set_kernel_events(None, None)
        torch.cuda.synchronize()
    kern_ms = max_over_ranks(sum(b.elapsed_time(e) for b, e in evs) / steps, world, dev)
    rows = 2 * d["T"] * d["Hk"] * d["D"] * 2
    nbytes = 2 * rows + (d["B"] + 1) * 4 + d["B"] * 4 + d["T"] * 4  # rows in and out, lengths, a table entry per token
    pk, pk_src = peaks()
    ach = nbytes / (kern_ms * 1e-3) / 1e9

    # End to end: pinned host key/value copied in, then the append, every step.
    hk, hv = key.pin_memory(), value.pin_memory()

    def e2e_step():
        kd.copy_(hk, non_blocking=True)
        vd.copy_(hv, non_blocking=True)
        call(kd, vd)

    e2e_step()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(steps):
        e2e_step()
    a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a0.elapsed_time(a1) / steps, world, dev)
    summ = clocks.summary()
    summ["window"] = f"{soak_s:g} s of back-to-back flush + append steps ({n_soak}) ending with the timed launches"
    res = {
        "metric": "paged KV-cache append bandwidth", "value": round(job_rate(world, nbytes, kern_ms), 4),
        "unit": "TB/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": round(kern_ms, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 rows, shuffled page pool)",
        "config": {"workload": "append_chunked_prefill", "batch": d["B"], "tokens": d["T"],
                   "num_kv_heads": d["Hk"], "head_dim": d["D"], "block_size": d["BS"],
                   "l2": "flushed (a 256 MB buffer read) before every launch", "algorithmic_bytes": nbytes},
        "kernel": {"name": "append", "avg_ms": round(kern_ms, 5), "launches_per_step": 1},
        "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(ach / pk["hbm_gbs"], 4),
                     "traffic": recorded_traffic("append_chunked_prefill", "append"),
                     "peak_source": f"{pk_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"},
        "e2e": {"value": round(job_rate(world, nbytes, e2e_ms), 4), "unit": "TB/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": rows, "d2h_bytes_per_step": 0,
                "note": "pinned host key/value in, append; the product is the device cache (nothing read back)"},
        "gpu_launches": steps,
        "clocks": summ,
    }
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import reference as ref
        t0 = time.perf_counter()
        ref.cache_append(case, key, value)
        s = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": round(nbytes / s / 1e12, 6), "unit": "TB/s", "cores": 1, "kind": "oracle",
                               "sample": "the whole write (every token), once", "seconds_per_step": round(s, 3)}
    del g, kd, vd, flush
    torch.cuda.empty_cache()
    return res


def time_oracle(case, budget_s: float, cores: int | None = None):
    """The fp64 oracle on the host cores (all of them unless `cores` is given),
    on a bounded sample of the workload's output rows; returns (seconds per
    full workload, sample description, cores)."""
    import numpy as np

    from oracle import reference as ref
    cores = cores or ref.default_threads()
    d = case.dims
    T, H = d["T"], d["H"]
    n_rows = T * H
    rng = np.random.default_rng(0)
    # Rows in a random order, timed in growing chunks until the budget is
    # spent (or every row is done); the time scales by the rows processed.
    order = rng.permutation(n_rows)
    done, spent, chunk = 0, 0.0, max(4 * cores, 16)
    while done < n_rows and spent < budget_s:
        idx = order[done:done + chunk]
        t0 = time.perf_counter()
        ref.forward_rows(case, idx // H, idx % H, num_threads=cores)
        spent += time.perf_counter() - t0
        done += idx.size
        rate = spent / done  # seconds per row
        chunk = int(min(2 * chunk, 65536, max(cores, (budget_s - spent) / max(rate, 1e-9))))
    full = spent * n_rows / done
    return full, f"{done} of {n_rows} (token, head) output rows in a random order (seed 0), scaled to the whole workload", cores


def add_cpu_baseline(res, case, budget_s: float, single_core_s: float = 0.0):
    full_s, sample, cores = time_oracle(case, budget_s)
    unit_work = res["config"]["algorithmic_bytes"] if res["unit"] == "TB/s" else res["config"]["algorithmic_flops"]
    res["cpu_baseline"] = {"value": round(unit_work / full_s / 1e12, 6), "unit": res["unit"], "cores": cores,
                           "kind": "oracle", "sample": sample, "seconds_per_step": round(full_s, 3)}
    if single_core_s > 0:
        one_s, one_sample, _ = time_oracle(case, single_core_s, cores=1)
        res["cpu_baseline"]["single_core"] = {"value": round(unit_work / one_s / 1e12, 6), "cores": 1,
                                              "sample": one_sample, "seconds_per_step": round(one_s, 3)}


SUB_WORKLOADS = ("batched_decode", "chunked_prefill", "mixed_window", "append_chunked_prefill")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long_decode")
    ap.add_argument("--splits", type=int, default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--sub-cpu-budget", type=float, default=4.0,
                    help="seconds of oracle work for each sub-record's cpu_baseline")
    ap.add_argument("--soak-s", type=float, default=1.0,
                    help="seconds of back-to-back steps (clock-sampled) before each timed region")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub-workloads", action="store_true",
                    help="print the headline workload's record only")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    if world > 1 and args.workload in ("chunked_prefill", "mixed_window"):
        if rank == 0:
            print(f"bench.py: --workload {args.workload} refused with {world} ranks: {PREFILL_MULTI_RANK}",
                  file=sys.stderr, flush=True)
        sys.exit(2)

    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    if args.workload == "append_chunked_prefill":
        res = run_append(args, rank, world, soak_s=args.soak_s)
    else:
        res, case = run_ours(args, rank, world, soak_s=args.soak_s)
        if rank == 0 and not args.no_cpu_baseline:
            add_cpu_baseline(res, case, args.cpu_budget, min(4.0, args.cpu_budget))
    default_run = args.workload == "long_decode" and not args.no_sub_workloads and args.splits is None
    if default_run:
        subs, skipped = {}, {}
        for name in SUB_WORKLOADS:
            if name == "append_chunked_prefill":
                subs[name] = run_append(args, rank, world, soak_s=args.soak_s)
                continue
            if world > 1 and name in ("chunked_prefill", "mixed_window"):
                skipped[name] = PREFILL_MULTI_RANK
                continue
            sub, sub_case = run_ours(args, rank, world, workload=name, soak_s=args.soak_s)
            if rank == 0 and not args.no_cpu_baseline:
                add_cpu_baseline(sub, sub_case, args.sub_cpu_budget)
            subs[name] = sub
        res["workloads"] = subs
        if skipped:
            res["workloads_skipped"] = skipped
        res["gpu_launches_all_records"] = res["gpu_launches"] + sum(r["gpu_launches"] for r in subs.values())
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores, per step a bounded sample."""
    if rank != 0:
        return
    from paged_attention_relative_gb300.roofline import algorithmic_bytes, algorithmic_flops
    case = make_workload(args.workload)
    decode = case.max_seqlen_q * (case.dims["H"] // case.dims["Hk"]) <= 64
    work = algorithmic_bytes(case) if decode else algorithmic_flops(case)
    unit = "TB/s" if decode else "TFLOP/s"
    budget = max(1.0, 120.0 / max(args.steps + args.warmup, 1))
    for _ in range(args.warmup):
        time_oracle(case, min(budget, 2.0))
    times = []
    sample = cores = None
    for _ in range(args.steps):
        full_s, sample, cores = time_oracle(case, budget)
        times.append(full_s)
    s = statistics.mean(times)
    value = work / s / 1e12
    d = case.dims
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit, "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(s * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) bf16)",
           "config": {"workload": args.workload, "batch": d["B"], "tokens": d["T"], "num_heads": d["H"],
                      "num_kv_heads": d["Hk"], "head_dim": d["D"], "rel_extent": d["R"]},
           "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": cores, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
