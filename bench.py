#!/usr/bin/env python3
"""Benchmark of the GB300 per-token group-wise cast.

One step = one pass of the whole cast (load, group amax, scale, quantize,
store codes, store scales -- all in one kernel launch) over one batch: the
4096 x 7168 BF16 -> FP8 E4M3, group 128, UE8M0-packed workload by default.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c2]
    python bench.py --impl reference ...     # the CPU oracle as the baseline

Timing: W untimed warm-up steps, then exactly K timed steps between a
barrier + cuda synchronize on both sides, bracketed by one pair of CUDA
events on the launching stream; ms_per_step is the mean (max over ranks).
Inputs are larger than L2: the batch is held in enough copies (at least 3x
the L2 size together) that each step reads a copy that is not L2-resident.
A secondary figure times each launch alone between events after an L2
flush, next to a near-empty kernel timed the same way.  N > 1 runs one independent
replica of the workload per GPU (rows are independent: no collective on the
data path), so scaling is weak and value = bytes of all ranks / that time.

Prints ONE JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from precision_quantization_token_gb300.inputs import (WORKLOADS,  # noqa: E402
                                                       make_gain, make_input)

METRIC = "per-token cast GB/s (in+out bytes) and % of GB300 HBM peak at 4096x7168"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "per_token_cast_c2_traffic.txt")


# ------------------------------------------------------------------ utils

def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default="c2", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--per-config-steps", type=int, default=10000,
                    help="timed steps for each of the other workloads "
                         "(0 disables the per-config table)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--flushed-steps", type=int, default=2000,
                    help="steps of the secondary flushed per-launch timing")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU time budget of the oracle baseline sample")
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def reduce_max(value: float, world: int) -> float:
    """Max of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_step: int, mean_ms: float, world: int):
    """(whole-job GB/s, slowest rank's ms per step): every rank processes
    its own replica of the workload (weak scaling), so the job moves
    world x bytes_per_step per step in the slowest rank's time."""
    slowest = reduce_max(mean_ms, world)
    return bytes_per_step * world / (slowest * 1e-3) / 1e9, slowest


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def kernel_source_hash() -> str:
    """Hash of the sources the per-token cast kernel is built from (its
    translation unit, the shared device header, the public header)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "precision_quantization_token_gb300", "csrc")
    files = [os.path.join(csrc, f) for f in ("tk_cast.cu", "tk_device.cuh",
                                              "tk_internal.h")] + \
        sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))
    for p in files:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(workload: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source and the same workload (else None)."""
    try:
        fields = {}
        with open(PROFILE_TRAFFIC) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("source_sha256") != kernel_source_hash():
            return None
        if fields.get("workload") != workload:
            return None
        return int(fields["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}",
                 f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None,
                    "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------- GPU arm

class GpuWorkload:
    """Device buffers for one workload and a launcher through the C ABI.

    The batch is held in R copies (input and outputs), R chosen so that the
    copies together are at least 3x the L2 size: step i works on copy i % R,
    so its input was last touched R-1 steps earlier, with more than twice the
    L2 size of other traffic in between, and is never L2-resident.  When even
    32 copies cannot reach that (tiny workloads), R = 1 and the timing
    flushes the L2 before each step instead.
    """

    MAX_COPIES = 32

    def __init__(self, w, torch, tk, device, l2_bytes):
        self.w, self.torch, self.tk = w, torch, tk
        self.bytes = w.algorithmic_bytes()
        step = self.bytes["total"]
        copies = max(1, -(-3 * l2_bytes // step))
        self.rotating = copies <= self.MAX_COPIES
        self.copies = copies if self.rotating else 1
        bits = make_input(w)
        x0 = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(device)
        row_bytes = w.K if w.fmt == "e4m3" else w.K // 2
        if w.op in ("block", "block_dequant"):
            shape, dt = tk.block_scale_shape(w.M, w.K, w.scale)
        elif w.op == "channel_dequant":
            shape, dt = tk.channel_scale_shape(w.K, w.scale)
        elif w.op == "channel":
            shape, dt = tk.channel_scale_shape(w.K, w.scale)
            self.workspace = torch.zeros(tk.tk_per_channel_workspace_bytes(w.K),
                                         dtype=torch.uint8, device=device)
        else:
            shape, dt = tk.scale_shape(w.M, w.K, w.group, w.scale, w.layout)
        if w.op == "rmsnorm":
            g = make_gain(w)
            self.gain = torch.from_numpy(g.view(np.int16)).view(
                torch.bfloat16).to(device)
        if w.op.endswith("dequant"):
            # the codes and scales to dequantize come from one (untimed) cast
            if w.op == "block_dequant":
                c0, s0 = tk.per_block_cast(x0, w.fmt, w.scale)
            elif w.op == "channel_dequant":
                c0, s0 = tk.per_channel_cast(x0, w.fmt, w.scale)
            else:
                c0, s0 = tk.per_token_cast(x0, w.group, w.fmt, w.scale, w.layout)
            torch.cuda.synchronize()
            del x0
        self.sets = []
        for i in range(self.copies):
            if w.op.endswith("dequant"):
                codes = c0 if i == 0 else c0.clone()
                scales = s0 if i == 0 else s0.clone()
                y = torch.empty((w.M, w.K), dtype=torch.bfloat16, device=device)
                self.sets.append((codes, scales, y))
                continue
            x = x0 if i == 0 else x0.clone()
            if w.op == "cast_back":
                y = torch.empty((w.M, w.K), dtype=torch.bfloat16, device=device)
                self.sets.append((x, y, None))
                continue
            codes = torch.empty((w.M, row_bytes), dtype=torch.uint8, device=device)
            scales = torch.empty(shape, dtype=getattr(torch, dt), device=device)
            self.sets.append((x, codes, scales))
        self.entry = (tk.tk_swiglu_per_token_cast if w.swiglu
                      else tk.tk_per_token_cast)

    def launch(self, i, stream_handle):
        w, tk = self.w, self.tk
        a, b, c = self.sets[i % self.copies]
        if w.op == "dequant":
            tk.tk_per_token_dequant(a.data_ptr(), a.stride(0), b.data_ptr(),
                                    b.stride(0), w.M, w.K, w.group,
                                    tk.FMT[w.fmt], tk.SCALE[w.scale],
                                    tk.LAYOUT[w.layout], c.data_ptr(),
                                    c.stride(0), tk.OUT_DTYPE["bf16"],
                                    stream_handle)
        elif w.op == "cast_back":
            tk.tk_per_token_cast_back(a.data_ptr(), w.M, w.K, a.stride(0),
                                      w.group, tk.FMT[w.fmt],
                                      tk.SCALE[w.scale], b.data_ptr(),
                                      b.stride(0), stream_handle)
        elif w.op == "block_dequant":
            tk.tk_per_block_dequant(a.data_ptr(), a.stride(0), b.data_ptr(),
                                    b.stride(0), w.M, w.K, tk.FMT[w.fmt],
                                    tk.SCALE[w.scale], c.data_ptr(),
                                    c.stride(0), tk.OUT_DTYPE["bf16"],
                                    stream_handle)
        elif w.op == "channel_dequant":
            tk.tk_per_channel_dequant(a.data_ptr(), a.stride(0), b.data_ptr(),
                                      w.M, w.K, tk.FMT[w.fmt],
                                      tk.SCALE[w.scale], c.data_ptr(),
                                      c.stride(0), tk.OUT_DTYPE["bf16"],
                                      stream_handle)
        elif w.op == "rmsnorm":
            tk.tk_rmsnorm_per_token_cast(a.data_ptr(), self.gain.data_ptr(),
                                         w.M, w.K, a.stride(0), w.eps,
                                         w.group, tk.FMT[w.fmt],
                                         tk.SCALE[w.scale],
                                         tk.LAYOUT[w.layout], b.data_ptr(),
                                         b.stride(0), c.data_ptr(),
                                         c.stride(0), stream_handle)
        elif w.op == "block":
            tk.tk_per_block_cast(a.data_ptr(), w.M, w.K, a.stride(0),
                                 tk.FMT[w.fmt], tk.SCALE[w.scale],
                                 b.data_ptr(), b.stride(0), c.data_ptr(),
                                 c.stride(0), stream_handle)
        elif w.op == "channel":
            tk.tk_per_channel_cast(a.data_ptr(), w.M, w.K, a.stride(0),
                                   tk.FMT[w.fmt], tk.SCALE[w.scale],
                                   b.data_ptr(), b.stride(0), c.data_ptr(),
                                   self.workspace.data_ptr(),
                                   self.workspace.numel(), stream_handle)
        else:
            self.entry(a.data_ptr(), w.M, w.K, a.stride(0), w.group,
                       tk.FMT[w.fmt], tk.SCALE[w.scale], tk.LAYOUT[w.layout],
                       b.data_ptr(), b.stride(0), c.data_ptr(), c.stride(0),
                       stream_handle)

    def l2_note(self, l2_bytes):
        if self.rotating:
            mib = self.copies * self.bytes["total"] / 2 ** 20
            return (f"inputs larger than L2: {self.copies} copies of the batch "
                    f"({mib:.0f} MiB of inputs+outputs, L2 {l2_bytes >> 20} "
                    "MiB) cycled step by step, no step's input L2-resident")
        return (f"L2 flushed before every step by writing {2 * l2_bytes >> 20}"
                f" MiB then reading {l2_bytes >> 20} MiB (outside the timed "
                "events)")


def _flush(torch, fw, fr):
    fw.zero_()
    fr.sum(dtype=torch.float32)


def time_steps(torch, wl, steps, warmup, fw, fr, world):
    """Mean ms per step over exactly `steps` steps, events on the launching
    stream; returns (mean ms, wall seconds of the timed region)."""
    stream = torch.cuda.current_stream()
    handle = stream.cuda_stream
    for i in range(warmup):
        if not wl.rotating:
            _flush(torch, fw, fr)
        wl.launch(i, handle)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    if wl.rotating:
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(steps):
            wl.launch(warmup + i, handle)
        b.record(stream)
        torch.cuda.synchronize()
        total = a.elapsed_time(b)
    else:
        ev = [(torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i, (a, b) in enumerate(ev):
            _flush(torch, fw, fr)
            a.record(stream)
            wl.launch(warmup + i, handle)
            b.record(stream)
        torch.cuda.synchronize()
        total = sum(a.elapsed_time(b) for a, b in ev)
    barrier(world)
    return total / steps, time.perf_counter() - t0


def time_flushed(torch, wl, steps, fw, fr, launch=None):
    """Secondary figure: each launch alone between CUDA events, with the L2
    flushed (2x L2 written, then L2 read) before it."""
    stream = torch.cuda.current_stream()
    handle = stream.cuda_stream
    launch = launch or (lambda i: wl.launch(i, handle))
    for i in range(5):
        _flush(torch, fw, fr)
        launch(i)
    ev = [(torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i, (a, b) in enumerate(ev):
        _flush(torch, fw, fr)
        a.record(stream)
        launch(i)
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.fmean(a.elapsed_time(b) for a, b in ev)


def run_gpu(args):
    import torch

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    import precision_quantization_token_gb300 as tk
    tk.load()

    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    fw = torch.empty(2 * l2, dtype=torch.uint8, device=device)
    fr = torch.ones(l2 // 2, dtype=torch.bfloat16, device=device)

    w = WORKLOADS[args.workload]
    wl = GpuWorkload(w, torch, tk, device, l2)
    peak, peak_src = measured_peaks()

    clocks = ClockSampler(local_rank)
    clocks.start()
    mean_ms, wall = time_steps(torch, wl, args.steps, args.warmup, fw, fr,
                               world)
    clock_info = clocks.stop()

    value, mean_ms_all = job_throughput(wl.bytes["total"], mean_ms, world)
    achieved = wl.bytes["total"] / (mean_ms * 1e-3) / 1e9

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(mean_ms_all, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded numpy PCG64, BF16-rounded)",
        "config": {
            "workload": w.describe(), "name": w.name, "M": w.M, "K": w.K,
            "group": w.group, "fmt": w.fmt, "scale": w.scale,
            "layout": w.layout, "swiglu": w.swiglu, "seed": w.seed,
            "bytes_per_step": wl.bytes, "l2": wl.l2_note(l2),
            "timing": ("one CUDA event pair on the launching stream around "
                       "exactly K back-to-back steps (one kernel launch "
                       "each); mean per step; max over ranks"),
            "wall_s_timed_region": round(wall, 3),
            "parallelism": f"replicas x{world} (rows independent)"},
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 2),
            "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic(w.name), "peak_source": peak_src,
            "kernel": "per_token_cast_kernel"},
        "gpu_launches": args.steps,
        "clocks": clock_info,
    }

    if rank == 0 and args.flushed_steps > 0:
        f_ms = time_flushed(torch, wl, args.flushed_steps, fw, fr)
        e_ms = time_flushed(torch, wl, args.flushed_steps, fw, fr,
                            launch=lambda i: torch.cuda._sleep(1))
        result["flushed_per_launch"] = {
            "ms": round(f_ms, 6),
            "GB/s": round(wl.bytes["total"] / f_ms / 1e6, 1),
            "frac_of_peak": round(wl.bytes["total"] / f_ms / 1e6 / peak, 4),
            "empty_kernel_ms": round(e_ms, 6),
            "how": ("each launch alone between CUDA events after an L2 flush "
                    "(2x L2 written then L2 read); empty_kernel_ms is a "
                    "near-empty kernel timed the same way (event and launch "
                    "overhead included in both)")}

    if rank == 0 and args.per_config_steps > 0:
        table = {}
        for name in sorted(WORKLOADS):
            if name == w.name:
                continue
            other = GpuWorkload(WORKLOADS[name], torch, tk, device, l2)
            m, _ = time_steps(torch, other, args.per_config_steps,
                              max(3, args.warmup), fw, fr, 1)
            gbps = other.bytes["total"] / (m * 1e-3) / 1e9
            table[name] = {"workload": other.w.describe(),
                           "kernels_per_step": 2 if other.w.op == "channel" else 1,
                           "ms": round(m, 6), "GB/s": round(gbps, 1),
                           "frac_of_peak": round(gbps / peak, 4),
                           "bytes": other.bytes["total"],
                           "l2": other.l2_note(l2)}
            if not args.no_cpu_baseline:     # the oracle timed beside it
                table[name]["cpu_oracle"] = cpu_baseline(other.w, 1.0)
            del other
        result["per_config"] = table

    if args.e2e_steps > 0:
        result["e2e"] = run_e2e(torch, tk, w, args.e2e_steps, device, world)

    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)

    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def run_e2e(torch, tk, w, steps, device, world):
    """Same metric through the public API with host buffers: each step the
    library's host-buffer entry uploads the pinned host input to the device
    in chunks, casts them, and downloads codes and scales to pinned host
    memory (all inside the timed interval)."""
    bits = make_input(w)
    xh = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    xh = xh.pin_memory()
    row_bytes = w.K if w.fmt == "e4m3" else w.K // 2
    codes = torch.empty((w.M, row_bytes), dtype=torch.uint8, pin_memory=True)
    shape, dt = tk.scale_shape(w.M, w.K, w.group, w.scale, w.layout)
    scales = torch.empty(shape, dtype=getattr(torch, dt), pin_memory=True)
    fn = tk.swiglu_per_token_cast if w.swiglu else tk.per_token_cast
    for _ in range(3):
        fn(xh, w.group, w.fmt, w.scale, w.layout, codes=codes, scales=scales)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        fn(xh, w.group, w.fmt, w.scale, w.layout, codes=codes, scales=scales)
    torch.cuda.synchronize()
    barrier(world)
    dt_s = reduce_max((time.perf_counter() - t0) / steps, world)
    b = w.algorithmic_bytes()
    return {"value": round(b["total"] * world / dt_s / 1e9, 2), "unit": UNIT,
            "ms_per_step": round(dt_s * 1e3, 4),
            "h2d_bytes_per_step": int(xh.numel() * 2),
            "d2h_bytes_per_step": int(codes.numel() + scales.numel() * 4),
            "api": ("precision_quantization_token_gb300."
                    + ("swiglu_per_token_cast" if w.swiglu
                       else "per_token_cast") + " on pinned host tensors "
                    "(C entry tk_" + ("swiglu_" if w.swiglu else "")
                    + "per_token_cast_host)")}


# ------------------------------------------------------------- CPU arm

def _oracle_op(w, threads):
    """(prepare, run) for the oracle of a workload's op on a block of rows:
    prepare(bits) builds the op's inputs (for dequantization: the oracle's
    own codes and scales, outside the timed part), run(inputs) runs it."""
    import oracle
    fmt = oracle.FMT_E4M3 if w.fmt == "e4m3" else oracle.FMT_E2M1
    mode = {"fp32": oracle.SCALE_FP32, "pow2": oracle.SCALE_FP32_POW2,
            "ue8m0": oracle.SCALE_UE8M0}[w.scale]
    layout = (oracle.LAYOUT_ROW_MAJOR if w.layout == "row"
              else oracle.LAYOUT_TRANSPOSED)
    same = (lambda bits: bits)
    if w.op == "dequant":
        def prep(bits):
            return oracle.per_token_cast(bits, w.K, w.group, fmt, mode, layout,
                                         threads=threads)
        return prep, lambda cs: oracle.per_token_dequant(
            cs[0], cs[1], w.K, w.group, fmt, mode, layout, threads=threads)
    if w.op in ("block_dequant", "channel_dequant"):
        if w.op == "block_dequant":
            return (lambda bits: oracle.per_block_cast(bits, w.K, 128, fmt, mode,
                                                       threads=threads),
                    lambda cs: oracle.per_block_dequant(cs[0], cs[1], w.K, 128,
                                                        fmt, mode,
                                                        threads=threads))
        return (lambda bits: oracle.per_channel_cast(bits, w.K, fmt, mode,
                                                     threads=threads),
                lambda cs: oracle.per_channel_dequant(cs[0], cs[1], w.K, fmt,
                                                      mode, threads=threads))
    if w.op == "cast_back":
        return same, lambda b: oracle.per_token_cast_back(
            b, w.K, w.group, fmt, mode, threads=threads)
    if w.op == "block":
        return same, lambda b: oracle.per_block_cast(b, w.K, 128, fmt, mode,
                                                     threads=threads)
    if w.op == "channel":
        return same, lambda b: oracle.per_channel_cast(b, w.K, fmt, mode,
                                                       threads=threads)
    if w.op == "rmsnorm":
        gain = make_gain(w)
        return same, lambda b: oracle.rmsnorm_per_token_cast(
            b, gain, w.K, w.eps, w.group, fmt, mode, layout, threads=threads)
    fn = oracle.swiglu_per_token_cast if w.swiglu else oracle.per_token_cast
    return same, lambda b: fn(b, w.K, w.group, fmt, mode, layout,
                              threads=threads)


def cpu_baseline(w, seconds: float):
    """The oracle as it stands, on all host cores, over whole passes of the
    workload (or a leading block of rows when one pass would exceed the
    budget); GB/s over the same algorithmic bytes."""
    import oracle
    threads = oracle.host_threads()
    prep, run = _oracle_op(w, threads)
    # probe on a small block to size the sample
    probe_rows = max(threads, min(w.M, 256))
    bits = make_input(w, M=probe_rows) if probe_rows < w.M else make_input(w)
    probe = prep(bits[:probe_rows])
    t0 = time.perf_counter()
    run(probe)
    per_row = (time.perf_counter() - t0) / probe_rows
    rows = int(min(w.M, max(probe_rows, seconds / max(per_row, 1e-9))))
    sample = prep(make_input(w, M=rows) if rows < w.M else make_input(w))
    passes, elapsed = 0, 0.0
    t0 = time.perf_counter()
    while True:
        run(sample)
        passes += 1
        elapsed = time.perf_counter() - t0
        if elapsed >= min(seconds, 3.0) or passes >= 1000:
            break
    frac = rows / w.M
    gb = w.algorithmic_bytes()["total"] * frac * passes / 1e9
    return {"value": round(gb / elapsed, 3), "unit": UNIT, "cores": threads,
            "kind": "oracle",
            "sample": (f"{rows} of {w.M} rows of the workload, {passes} "
                       f"pass(es), {elapsed:.2f} s wall on {threads} threads")}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    import oracle
    threads = oracle.host_threads()
    fmt = oracle.FMT_E4M3 if w.fmt == "e4m3" else oracle.FMT_E2M1
    mode = {"fp32": oracle.SCALE_FP32, "pow2": oracle.SCALE_FP32_POW2,
            "ue8m0": oracle.SCALE_UE8M0}[w.scale]
    layout = (oracle.LAYOUT_ROW_MAJOR if w.layout == "row"
              else oracle.LAYOUT_TRANSPOSED)
    fn = oracle.swiglu_per_token_cast if w.swiglu else oracle.per_token_cast
    # each step is a bounded sample of rows sized so that the whole run
    # stays within a few minutes
    budget_s = 120.0 / max(1, args.steps + args.warmup)
    probe_rows = min(w.M, max(threads, 64))
    probe = make_input(w, M=probe_rows)
    t0 = time.perf_counter()
    fn(probe, w.K, w.group, fmt, mode, layout, threads=threads)
    per_row = (time.perf_counter() - t0) / probe_rows
    rows = int(min(w.M, max(1, budget_s / max(per_row, 1e-9))))
    sample = make_input(w, M=rows) if rows < w.M else make_input(w)
    for _ in range(args.warmup):
        fn(sample, w.K, w.group, fmt, mode, layout, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn(sample, w.K, w.group, fmt, mode, layout, threads=threads)
    dt_s = (time.perf_counter() - t0) / args.steps
    gb = w.algorithmic_bytes()["total"] * rows / w.M / 1e9
    value = round(gb / dt_s, 3)
    sample_desc = (f"{rows} of {w.M} rows per step, {threads} threads")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt_s * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded numpy PCG64, BF16-rounded)",
        "config": {"workload": w.describe(), "name": w.name, "M": w.M,
                   "K": w.K, "group": w.group},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample_desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
