#!/usr/bin/env python
"""Benchmark of the exact attention forward pass on GB300: prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one call of the fused kernel (every step of the hot path: tile
scheduling, TMA loads, QK^T, online softmax, rescale, PV, epilogue) over one
batch of the workload.  ``value`` is attention-forward TFLOPS counted on the
algorithmic work, 4*D FLOP per unmasked (query, key) pair summed over all
heads and rows, over the max-over-ranks device time of K steps, with the
inputs resident in HBM and L2 flushed between steps.  ``e2e`` is the same
metric through the public API with the step's inputs copied from pinned host
memory and its outputs copied back inside the timed region.

Under torchrun each rank runs its own copy of the workload on its own GPU
(independent problems, no collective on the data path: weak scaling).
``--impl reference`` times the fp64 CPU oracle, as it stands, on a bounded
sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from attention_forward_06_gb300.inputs import (WORKLOADS, Workload, bf16_bits, block_mask_blocks,  # noqa: E402
                                               draw_workload, sample_rows)

METRIC = "attn fwd TFLOPS (bf16, 1×GB300) and % of dense-BF16 tensor peak; geomean"
PERF_WORKLOADS = ["train", "gqa", "chunked128", "chunked64", "long"]
L2_FLUSH_BYTES = 256 << 20  # > 129 MB L2
# Dense bf16 tensor-core work one SM completes per clock: one 128 x 256 x 16 tcgen05 MMA (1 048 576 FLOP) per 128
# cycles, as the MMA-rate probe (attn_probe_mma_rate, tests/test_probe.py) measures on GB300.
BF16_FLOP_PER_CLK_PER_SM = 8192
KERNEL_SOURCES = ["attention_forward_06_gb300/csrc/attn_fwd.cu", "attention_forward_06_gb300/csrc/ptx.cuh"]


# ----------------------------------------------------------------------------- work accounting
def allowed_pairs(w: Workload) -> int:
    """Unmasked (query row, key) pairs of one (batch, head)."""
    if w.causal == 0:
        return w.Sq * w.Sk
    i = np.arange(w.Sq, dtype=np.int64)
    last = i + (w.Sk - w.Sq if w.causal == 1 else 0)
    return int(np.clip(last + 1, 0, w.Sk).sum())


def alg_flops(w: Workload) -> float:
    return 4.0 * w.D * w.B * w.Hq * allowed_pairs(w)


def conv_flops(w: Workload) -> float:
    return 4.0 * w.B * w.Hq * w.Sq * w.Sk * w.D * (0.5 if w.causal else 1.0)


def min_hbm_bytes(w: Workload) -> int:
    """Bytes of Q, K, V, O (bf16) and LSE (fp32), each moved once."""
    return 2 * (2 * w.B * w.Hq * w.Sq * w.D + 2 * w.B * w.Hkv * w.Sk * w.D) + 4 * w.B * w.Hq * w.Sq


def blocksparse_pairs(w: Workload, blocks: np.ndarray, block: int = 128) -> int:
    """Unmasked (row, key) pairs under a block mask [B, Hm, QB, KB] and the workload's causal rule, summed over
    every (batch, head)."""
    i = np.arange(w.Sq)
    last = np.full(w.Sq, w.Sk - 1) if w.causal == 0 else np.minimum(i + (w.Sk - w.Sq if w.causal == 1 else 0), w.Sk - 1)
    total = 0
    KB = blocks.shape[3]
    for qb in range(blocks.shape[2]):
        rows = last[qb * block:(qb + 1) * block]
        # keys of key block kb visible to each row of the query block: clip(last + 1 - kb*block, 0, block)
        per_kb = np.clip(rows[None, :] + 1 - (np.arange(KB) * block)[:, None], 0, block)
        per_kb = np.minimum(per_kb, (w.Sk - np.arange(KB) * block)[:, None])
        counts = per_kb.sum(axis=1)  # [KB]
        marked = blocks[:, :, qb, :].astype(np.int64)  # [B, Hm, KB]
        total += int((marked * counts).sum()) * (w.Hq // blocks.shape[1])
    return total


def row_flops(w: Workload, rows: np.ndarray) -> float:
    i = rows % w.Sq
    if w.causal == 0:
        n = np.full(i.shape, w.Sk)
    else:
        n = np.clip(i + (w.Sk - w.Sq if w.causal == 1 else 0) + 1, 0, w.Sk)
    return float(4.0 * w.D * n.sum())


# ----------------------------------------------------------------------------- peaks, clocks
def measured_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- multi-rank
def reduce_max(x: float, dist, device) -> float:
    """Max of a per-rank float over all ranks (identity without a process group)."""
    if dist is None:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flop_per_rank_step: float, world: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput: every rank's work over the slowest rank's time."""
    return world * flop_per_rank_step * steps / (max_ms * 1e-3) / 1e12


# ----------------------------------------------------------------------------- timing
def time_kernel(fn, steps: int, warmup: int, flush: torch.Tensor, stream) -> list[float]:
    """Per-step kernel time (ms) with CUDA events on the launching stream; L2 flushed before each step."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def kernel_code_sha256(sources=None) -> str:
    """sha256 of the forward kernel's sources with comments and blank lines removed: the key of the DRAM traffic
    record, which a change to the code invalidates and a change to a comment does not."""
    h = hashlib.sha256()
    for src in sources or [os.path.join(ROOT, s) for s in KERNEL_SOURCES]:
        with open(src) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(line.rstrip() for line in text.splitlines() if line.strip()).encode())
        h.update(b"\0")
    return h.hexdigest()


def traffic_for(workload: str):
    """DRAM bytes per launch from a committed ncu capture, or None if absent or the kernel changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(workload)
    if not entry or entry.get("kernel_sha256") != kernel_code_sha256():
        return None
    return entry.get("dram_bytes_per_launch")


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or 'unknown'."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_rows(w: Workload, budget_s: float, seed: int):
    """The oracle, as it stands, on rows drawn uniformly per (batch, head) in rounds of doubling size for about
    budget_s seconds: (rows, o [n, D], lse [n], FLOP, seconds)."""
    import oracle  # test infrastructure: timed here as the CPU baseline only

    q, k, v = draw_workload(w)
    qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    flops, elapsed, chunk = 0.0, 0.0, 1
    rows_all, o_all, l_all = [], [], []
    while elapsed < budget_s:
        rows = sample_rows(w.B, w.Hq, w.Sq, chunk, seed=seed)
        seed += 1
        t0 = time.perf_counter()
        o, lse = oracle.attention(qb, kb, vb, w.causal, w.scale, rows=rows)
        dt = time.perf_counter() - t0
        elapsed += dt
        flops += row_flops(w, rows)
        rows_all.append(rows)
        o_all.append(o)
        l_all.append(lse)
        if dt < budget_s / 8:
            chunk = min(chunk * 2, w.Sq)
    return np.concatenate(rows_all), np.concatenate(o_all), np.concatenate(l_all), flops, elapsed


def sampled_parity(o_gpu: np.ndarray, lse_gpu: np.ndarray, o_ref: np.ndarray, lse_ref: np.ndarray) -> dict:
    """The parity rule of the tests on sampled rows: |dO| <= 1e-2 where |O_ref| < 4 (some bf16 value lies within
    2^-7 there), the excess over the bf16 rounding floor <= 1e-2 from 4 upwards, |dLSE| <= 1e-3."""
    d = np.abs(o_gpu - o_ref)
    small = np.abs(o_ref) < 4.0
    _, ex = np.frexp(np.abs(o_ref[~small]))  # the exact result rounded to bf16 (8 significant bits)
    spacing = np.ldexp(1.0, ex - 8)
    floor = np.abs(np.round(np.abs(o_ref[~small]) / spacing) * spacing - np.abs(o_ref[~small]))
    excess = d[~small] - floor
    live = np.isfinite(lse_ref)
    dl = np.abs(lse_gpu[live] - lse_ref[live])
    out = {"rows": int(o_ref.shape[0]), "max_abs_dO": float(d.max()) if d.size else 0.0,
           "max_abs_dO_below_4": float(d[small].max()) if small.any() else 0.0,
           "max_excess_dO_from_4": float(excess.max()) if excess.size else 0.0,
           "max_abs_dLSE": float(dl.max()) if dl.size else 0.0}
    out["plain_dO_within_1e-2"] = out["max_abs_dO_below_4"] <= 1e-2
    out["within_tolerance"] = (out["plain_dO_within_1e-2"] and out["max_excess_dO_from_4"] <= 1e-2
                               and out["max_abs_dLSE"] <= 1e-3)
    return out


def cpu_baseline(w: Workload, outputs: dict, budget_s: float = 8.0, other_budget_s: float = 3.0) -> dict:
    """The oracle, as it stands, on the machine's host cores: the headline workload for about budget_s seconds and
    every other workload whose GPU output is in `outputs` for about other_budget_s seconds.  Each gives the
    oracle's rate, the seconds the whole workload would take at that rate (extrapolated) and, where the GPU's
    output rows are at hand, the parity of those rows under the tests' rule."""
    import oracle

    per = {}
    names = [w.name] + [n for n in outputs if n != w.name]
    for name in names:
        wx = WORKLOADS[name]
        rows, o_ref, l_ref, flops, secs = oracle_rows(wx, budget_s if name == w.name else other_budget_s,
                                                      wx.seed + 2000)
        entry = {"tflops": flops / secs / 1e12, "rows": int(rows.size), "seconds": secs,
                 "full_config_s_extrapolated": alg_flops(wx) / (flops / secs)}
        if name in outputs:
            o_gpu, l_gpu = outputs[name]  # host copies of the GPU's outputs, [B, Hq, Sq, D] bf16 and [B, Hq, Sq]
            idx = torch.from_numpy(rows)
            entry["parity"] = sampled_parity(o_gpu.reshape(-1, wx.D)[idx].double().numpy(),
                                             l_gpu.reshape(-1)[idx].double().numpy(), o_ref, l_ref)
        per[name] = entry
    head = per[w.name]
    return {"value": head["tflops"], "unit": "TFLOPS", "cores": oracle.num_threads(), "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{head['rows']} query rows in total, drawn uniformly per (batch, head) in rounds, of the "
                      f"{w.name} workload ({head['seconds']:.1f} s, fp64); the other workloads for about "
                      f"{other_budget_s:g} s each; full_config_s_extrapolated = the workload's algorithmic FLOP at "
                      f"the measured rate",
            "per_workload": per}


# ----------------------------------------------------------------------------- arms
def run_reference(args, w: Workload, rank: int, world: int):
    if rank != 0:
        return None
    import oracle

    q, k, v = draw_workload(w)
    qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    per_head = max(1, 4096 // (w.B * w.Hq))  # bounded sample per step
    times, flops = [], []
    for step in range(args.warmup + args.steps):
        rows = sample_rows(w.B, w.Hq, w.Sq, per_head, seed=w.seed + 3000 + step)
        t0 = time.perf_counter()
        oracle.attention(qb, kb, vb, w.causal, w.scale, rows=rows)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            flops.append(row_flops(w, rows))
    value = sum(flops) / sum(times) / 1e12
    sample = f"{per_head} query rows per (batch, head) per step, {w.name} workload, fp64 oracle"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.label(), "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_ours(args, w: Workload, rank: int, world: int, dist):
    from attention_forward_06_gb300 import ops

    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream(dev)
    q, k, v = draw_workload(w)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    qd, kd, vd = qh.to(dev), kh.to(dev), vh.to(dev)
    od = torch.empty_like(qd)
    lsed = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    oh = torch.empty(od.shape, dtype=od.dtype, pin_memory=True)
    lseh = torch.empty(lsed.shape, dtype=lsed.dtype, pin_memory=True)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        ops.attn_fwd(qd, kd, vd, causal=w.causal, scale=w.scale, o=od, lse=lsed, stream=stream)

    sampler = ClockSampler(dev.index) if rank == 0 else None
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    times = time_kernel(step, args.steps, 0, flush, stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    st, site = ops.debug_status(stream)
    if st != ops.ATTN_OK:
        raise RuntimeError(f"kernel wait ran out (site {site})")
    total_ms = reduce_max(sum(times), dist, dev)
    ms_per_step = total_ms / args.steps
    flops = alg_flops(w)
    value = job_tflops(flops, world, args.steps, total_ms)

    # end to end through the public API: pinned host inputs -> HBM -> kernel -> host outputs, every step.  Steps
    # are pipelined over two device buffer sets: the copies in on one stream, the kernel on the compute stream, the
    # copies out on a third, so step i's copies overlap step i-1's kernel and copies out (whole-job throughput; the
    # host link bounds it: spreading the copies in over three streams measured the same).
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bufs = [(qd, kd, vd, od, lsed)] + [(torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd),
                                        torch.empty_like(od), torch.empty_like(lsed))]
    ev_in = [torch.cuda.Event() for _ in bufs]
    ev_done = [torch.cuda.Event() for _ in bufs]
    ev_out = [torch.cuda.Event() for _ in bufs]
    used = [False] * len(bufs)

    def e2e_step(i):
        b = i % len(bufs)
        qb, kb, vb, ob, lb = bufs[b]
        if used[b]:
            s_in.wait_event(ev_out[b])  # this set's previous outputs have been copied out
        with torch.cuda.stream(s_in):
            qb.copy_(qh, non_blocking=True)
            kb.copy_(kh, non_blocking=True)
            vb.copy_(vh, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        ops.attn_fwd(qb, kb, vb, causal=w.causal, scale=w.scale, o=ob, lse=lb, stream=stream)
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            oh.copy_(ob, non_blocking=True)
            lseh.copy_(lb, non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    e2e_steps = max(3, min(args.steps, 50))
    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_out)  # after the last copy out, which follows every earlier step's work
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1), dist, dev)
    e2e_value = job_tflops(flops, world, e2e_steps, e2e_ms)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = oh.numel() * oh.element_size() + lseh.numel() * lseh.element_size()

    if rank != 0:
        return None
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["bf16_tflops"])
    achieved = flops / (statistics.mean(times) * 1e-3) / 1e12
    # the tensor cores' own rate: SMs x dense bf16 FLOP per clock per SM x clock, at the maximum SM clock and at
    # the median SM clock sampled during the timed region
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    hw = {}
    for key, mhz in (("at_max_clock", (clocks or {}).get("sm_max_mhz")), ("at_median_clock", (clocks or {}).get("sm_mhz"))):
        if mhz:
            hw[key] = {"sm_mhz": mhz, "peak_tflops": sms * BF16_FLOP_PER_CLK_PER_SM * mhz * 1e6 / 1e12}
            hw[key]["frac"] = achieved / hw[key]["peak_tflops"]
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.label(), "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk, "D": w.D,
                   "causal": w.causal, "flop_count": "algorithmic: 4*D per unmasked (row, key) pair",
                   "alg_flop_per_step": flops, "conv_flop_per_step": conv_flops(w),
                   "tflops_conv": job_tflops(conv_flops(w), world, args.steps, total_ms),
                   "pct_of_peak": 100.0 * achieved / peak,
                   "headline": "the line's value is this training-prefill workload; geomean_tflops is the geomean "
                               "of the five performance workloads (train, gqa, chunked128, chunked64, long)",
                   "l2": f"flushed before every timed step ({L2_FLUSH_BYTES >> 20} MiB write, outside the events)"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "peak_source": f"{peak_kind} bf16_tflops: cuBLAS-achieved bf16 matmul (burst; the kernel is "
                                    f"timed alone), of measured",
                     "peak_hw": {"sms": sms, "bf16_flop_per_clk_per_sm": BF16_FLOP_PER_CLK_PER_SM, **hw},
                     "traffic": traffic_for(w.name), "alg_hbm_bytes": min_hbm_bytes(w)},
        "e2e": {"value": e2e_value, "unit": "TFLOPS", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    outputs = {w.name: (od.cpu(), lsed.cpu())}  # host copies of the GPU's outputs, for the sampled parity check
    if not args.skip_workloads:
        per, detail = {}, {}
        for name in ["tiny"] + PERF_WORKLOADS:
            wx = WORKLOADS[name]
            if name == w.name:
                ms = statistics.mean(times)
            else:
                qx, kx, vx = [t.to(dev) for t in draw_workload(wx)]
                ox = torch.empty_like(qx)
                lx = torch.empty((wx.B, wx.Hq, wx.Sq), dtype=torch.float32, device=dev)

                def fx():
                    ops.attn_fwd(qx, kx, vx, causal=wx.causal, scale=wx.scale, o=ox, lse=lx, stream=stream)

                ms = statistics.mean(time_kernel(fx, min(args.steps, 10), 3, flush, stream))
                if name in PERF_WORKLOADS:
                    outputs[name] = (ox.cpu(), lx.cpu())
                del qx, kx, vx, ox, lx
            alg = alg_flops(wx) / (ms * 1e-3) / 1e12
            if name in PERF_WORKLOADS:
                per[name] = alg
            # both FLOP conventions (they differ for the bottom-right chunked shapes), and the algorithmic HBM
            # bytes (Q, K, V, O, LSE once) over the launch time
            detail[name] = {"ms": ms, "tflops_alg": alg, "tflops_conv": conv_flops(wx) / (ms * 1e-3) / 1e12,
                            "pct_of_peak_alg": 100.0 * alg / peak,
                            "alg_hbm_gbs": min_hbm_bytes(wx) / (ms * 1e-3) / 1e9}
            # DRAM bytes of one launch from the committed ncu capture (null once the kernel has changed since), and
            # the HBM throughput they make at this launch time
            traffic = traffic_for(name)
            detail[name]["traffic"] = traffic
            detail[name]["dram_gbs"] = traffic / (ms * 1e-3) / 1e9 if traffic else None
        line["per_workload_tflops"] = per
        line["per_workload"] = detail
        line["tiny_latency_us"] = 1e3 * detail["tiny"]["ms"]
        line["geomean_tflops"] = math.exp(sum(math.log(x) for x in per.values()) / len(per))
        line["geomean_pct_of_peak"] = 100.0 * line["geomean_tflops"] / peak
        with_tiny = list(per.values()) + [detail["tiny"]["tflops_alg"]]
        line["geomean_tflops_with_tiny"] = math.exp(sum(math.log(x) for x in with_tiny) / len(with_tiny))
        line["blocksparse"] = bench_blocksparse(stream, flush, dev, min(args.steps, 10))
        line["backward"] = bench_backward(stream, flush, dev, min(args.steps, 10))
        line["splitkv"] = bench_splitkv(stream, flush, dev, min(args.steps, 10))
        line["ordered"] = bench_ordered(stream, flush, dev, min(args.steps, 10))
    if world == 1 and not args.skip_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, outputs)
    return line


def bench_blocksparse(stream, flush, dev, steps: int, density: float = 0.25) -> dict:
    """Block-sparse forward on the gqa shape with a quarter of the 128 x 128 blocks marked (the diagonal always),
    per-head masks, against the dense kernel on the same inputs: once with every query block drawn on its own, once
    with pairs of query blocks (one 256-row work item) sharing their key blocks."""
    from attention_forward_06_gb300 import ops

    w = WORKLOADS["gqa"]
    qx, kx, vx = [t.to(dev) for t in draw_workload(w)]
    ox = torch.empty_like(qx)
    lx = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)

    def fd():
        ops.attn_fwd(qx, kx, vx, causal=w.causal, scale=w.scale, o=ox, lse=lx, stream=stream)

    td = statistics.mean(time_kernel(fd, steps, 3, flush, stream))
    out = {"workload": f"{w.label()}, {density:.0%} of 128x128 blocks marked (diagonal always), per-head masks",
           "dense_ms": td}
    for name, group in (("independent_rows", 1), ("paired_rows", 2)):
        blocks = block_mask_blocks(w.B, w.Hq, w.Sq, w.Sk, density, seed=w.seed + 4000, row_group=group)
        words = ops.pack_block_mask(torch.from_numpy(blocks).to(dev))

        def fs():
            ops.attn_fwd_blocksparse(qx, kx, vx, words, causal=w.causal, scale=w.scale, o=ox, lse=lx, stream=stream)

        ts = statistics.mean(time_kernel(fs, steps, 3, flush, stream))
        flops = 4.0 * w.D * blocksparse_pairs(w, blocks)
        out[name] = {"tflops": flops / (ts * 1e-3) / 1e12, "ms": ts, "speedup_vs_dense": td / ts,
                     "marked_fraction": float(blocks.mean())}
    return out


def bench_ordered(stream, flush, dev, steps: int) -> dict:
    """Ordered forward on the gqa shape (sharply peaked rows): every 256-row query block visits its key tiles best
    first, ranked by the dot product of block means of Q and K (a training-free priority list built outside the
    timed region), and, as a check on the cost of the walk itself, in ascending order; both against the dense
    kernel on the same inputs.  The work is the same as dense (every tile is visited)."""
    from attention_forward_06_gb300 import ops

    w = WORKLOADS["gqa"]
    qx, kx, vx = [t.to(dev) for t in draw_workload(w)]
    ox = torch.empty_like(qx)
    lx = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    nqb, nkb = -(-w.Sq // ops.ORDER_ROWS), -(-w.Sk // ops.ORDER_KEYS)
    with torch.no_grad():
        qm = qx.float().reshape(w.B, w.Hq, nqb, ops.ORDER_ROWS, w.D).mean(3)
        km = kx.float().reshape(w.B, w.Hkv, nkb, ops.ORDER_KEYS, w.D).mean(3).repeat_interleave(w.Hq // w.Hkv, 1)
        ranked = torch.argsort(torch.einsum("bhqd,bhkd->bhqk", qm, km), dim=-1, descending=True)
        ranked = ranked.to(torch.int32).contiguous()
        ascending = torch.arange(nkb, dtype=torch.int32, device=dev).expand(w.B, 1, nqb, nkb).contiguous()
    torch.cuda.synchronize()

    def fd():
        ops.attn_fwd(qx, kx, vx, causal=w.causal, scale=w.scale, o=ox, lse=lx, stream=stream)

    td = statistics.mean(time_kernel(fd, steps, 3, flush, stream))
    out = {"workload": f"{w.label()}, key tiles visited in a given order per 256-row block", "dense_ms": td}
    for name, order in (("ranked", ranked), ("ascending", ascending)):
        def fo():
            ops.attn_fwd_ordered(qx, kx, vx, order, causal=w.causal, scale=w.scale, o=ox, lse=lx, stream=stream)

        to = statistics.mean(time_kernel(fo, steps, 3, flush, stream))
        out[name] = {"tflops": alg_flops(w) / (to * 1e-3) / 1e12, "ms": to, "vs_dense": td / to}
    return out


def bench_splitkv(stream, flush, dev, steps: int) -> dict:
    """Split-key forward on a shape with too few work items for the GPU -- one 512-row chunk of 32 query heads
    (8 kv heads) over 131072 keys, bottom-right causal, N(0,1) -- against the plain forward."""
    from attention_forward_06_gb300 import ops
    import dataclasses

    w = dataclasses.replace(WORKLOADS["chunked128"], name="splitkv_probe", B=1, Sq=512, Sk=131072, seed=6)
    qx, kx, vx = [t.to(dev) for t in draw_workload(w)]
    ox = torch.empty_like(qx)
    lx = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    n_splits = ops.splitkv_suggest(w.B, w.Hq, w.Sq, w.Sk, w.D, w.causal)
    ws = torch.empty(ops.splitkv_workspace_size(w.B, w.Hq, w.Sq, w.D, n_splits), dtype=torch.uint8, device=dev)

    def fp():
        ops.attn_fwd(qx, kx, vx, causal=w.causal, scale=w.scale, o=ox, lse=lx, stream=stream)

    def fs():
        ops.attn_fwd_splitkv(qx, kx, vx, causal=w.causal, scale=w.scale, n_splits=n_splits, workspace=ws, o=ox,
                             lse=lx, stream=stream)

    tp = statistics.mean(time_kernel(fp, steps, 3, flush, stream))
    ts = statistics.mean(time_kernel(fs, steps, 3, flush, stream))
    flops = alg_flops(w)
    out = {"workload": f"{w.label()} (a prefill chunk over a long context)", "n_splits": n_splits,
           "tflops": flops / (ts * 1e-3) / 1e12, "ms": ts, "plain_ms": tp,
           "plain_tflops": flops / (tp * 1e-3) / 1e12, "speedup_vs_plain": tp / ts}
    del qx, kx, vx, ox, lx, ws
    # the chunked workloads through the same entry point with its suggested split count (the last, partly
    # filled wave of 512 equal items is what a split of the keys evens out)
    for name in ("chunked128", "chunked64"):
        wc = WORKLOADS[name]
        qc, kc, vc = [t.to(dev) for t in draw_workload(wc)]
        oc = torch.empty_like(qc)
        lc = torch.empty((wc.B, wc.Hq, wc.Sq), dtype=torch.float32, device=dev)
        nc = ops.splitkv_suggest(wc.B, wc.Hq, wc.Sq, wc.Sk, wc.D, wc.causal)
        wsc = torch.empty(ops.splitkv_workspace_size(wc.B, wc.Hq, wc.Sq, wc.D, nc), dtype=torch.uint8, device=dev)

        def fc():
            ops.attn_fwd_splitkv(qc, kc, vc, causal=wc.causal, scale=wc.scale, n_splits=nc, workspace=wsc, o=oc,
                                 lse=lc, stream=stream)

        tc = statistics.mean(time_kernel(fc, steps, 3, flush, stream))
        out[name] = {"n_splits": nc, "ms": tc, "tflops": alg_flops(wc) / (tc * 1e-3) / 1e12}
        del qc, kc, vc, oc, lc, wsc
    return out


def bench_backward(stream, flush, dev, steps: int, names=("train", "gqa"), warmup: int = 3) -> dict:
    """Backward (dQ, dK, dV) of the train and gqa workloads.  FLOP convention: the five products of the
    backward, 10*D per unmasked (row, key) pair (2.5x the forward); the kernels recompute S and dP for dQ,
    which is extra work not counted."""
    from attention_forward_06_gb300 import ops

    peak = float(measured_peaks()[0]["bf16_tflops"])
    out = {"flop_count": "algorithmic: 10*D per unmasked (row, key) pair"}
    for name in names:
        w = WORKLOADS[name]
        q, k, v = [t.to(dev) for t in draw_workload(w)]
        do = torch.randn(q.shape, generator=torch.Generator().manual_seed(w.seed + 5000)).to(torch.bfloat16).to(dev)
        o, lse = ops.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, stream=stream)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(ops.bwd_workspace_size(w.B, w.Hq, w.Sq), dtype=torch.uint8, device=dev)

        def fb():
            ops.attn_bwd(q, k, v, o, lse, do, causal=w.causal, scale=w.scale, dq=dq, dk=dk, dv=dv, workspace=ws,
                         stream=stream)

        tb = statistics.mean(time_kernel(fb, steps, warmup, flush, stream))
        flops = 2.5 * alg_flops(w)
        out[name] = {"tflops": flops / (tb * 1e-3) / 1e12, "ms": tb, "pct_of_peak": 100.0 * flops / (tb * 1e-3) / 1e12 / peak}
        del q, k, v, do, o, lse, dq, dk, dv, ws
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="train", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-workloads", action="store_true", help="time only --workload, not the geomean set")
    ap.add_argument("--backward", action="store_true",
                    help="time only the backward (attn_bwd) of --workload and print its own JSON line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as tdist
        if args.impl == "reference" and rank != 0:
            return 0
        if args.impl == "ours":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            tdist.init_process_group("nccl")
            dist = tdist
    w = WORKLOADS[args.workload]
    if args.backward:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py --backward needs a GPU (the CUDA path has no CPU fallback)")
        dev = torch.device("cuda", torch.cuda.current_device())
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        res = bench_backward(torch.cuda.current_stream(dev), flush, dev, args.steps, names=(w.name,),
                             warmup=args.warmup)
        print(json.dumps({"metric": "attn bwd TFLOPS (bf16, 1xGB300), 10*D FLOP per unmasked pair",
                          "workload": w.label(), "steps": args.steps, "warmup": args.warmup, **res[w.name]}))
        return 0
    if args.impl == "reference":
        line = run_reference(args, w, rank, world)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a GPU for --impl ours (the CUDA path has no CPU fallback)")
        line = run_ours(args, w, rank, world, dist)
    if line is not None and rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
