#!/usr/bin/env python
"""Benchmark of the quantized GEMM library on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl qk|reference] [--formats default|none]

One step is one full GEMM call (operand staging, scale staging, contraction,
tile scheduling, fused epilogue, ragged edges) over one batch of synthetic
input, on the workload the metric is quoted on: the INT8 row/column-scaled
GEMM M=30000, N=21504, K=5376 with bf16 output (comfy-kitchen PR #174,
"Performance").  Rank 0 prints one JSON line.

Timing: W untimed warm-up calls, then K timed calls bracketed by a barrier and
a device synchronize on both sides, CUDA events on the launching stream, the
maximum over ranks.  The inputs (277 MB of int8 operands, 553 MB of f16
copies, 1.29 GB of output) are larger than the 129 MB L2, so no flush is
needed between headline steps; the secondary workloads, some of which fit in
L2, flush it before every timed call by reading a 256 MB buffer.

--impl reference times the CPU oracle on a bounded sample of the same
workload (the source pages hold no runnable code, so the oracle stands in as
the reference).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TOPS/TFLOPS (bf16 out) per format & shape; % of GB300 dense peak"
HEADLINE = {"M": 30000, "N": 21504, "K": 5376}
# comfy-kitchen PR #174, "Performance": 33.052 ms = 209.9 TOPS at this shape on an
# RX 9070 XT (gfx1201).  Another machine's number: context for vs_baseline only.
PAGES_INT8_TOPS = 209.9
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# nominal dense ratios to bf16 (2.25 PF bf16, 4.5 PF fp8, 13.5 PF fp4)
RATIO = {"bf16": 1.0, "f16": 1.0, "fp8": 2.0, "fp4": 6.0}
PROFILE_DIR = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "block_scaled_precision_tcgen05_gb300", "csrc")


# ----------------------------------------------------------------------------
# process topology and cross-rank aggregation
# ----------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x: float, dist, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Units all ranks processed per second of the slowest rank."""
    return units_per_rank * world / max_seconds


# ----------------------------------------------------------------------------
# peaks, clocks, source hash
# ----------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# the sources the headline INT8 GEMM (widening pass + f16-pipe kernel) is built from
HEADLINE_SOURCES = ("qk_api.cu", "qk_device.cuh", "qk_gemm_kernel.cuh", "qk_int8.cu", "qk_int8_exact.cuh",
                    "qk_internal.h", "qk_launch.cuh")


def _strip_comments(text: str) -> str:
    """C/C++ source without its comments, trailing blanks and empty lines
    (none of the hashed files has a comment marker inside a string literal)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.split("\n") if line.strip())


def kernel_source_hash() -> str:
    """Hash of the headline kernel's sources, comments left out: a committed
    DRAM-traffic figure counts only while the code it was captured on is
    unchanged."""
    h = hashlib.sha1()
    for path in [os.path.join(CSRC, n) for n in HEADLINE_SOURCES]:
        with open(path, encoding="utf-8") as f:
            h.update(os.path.basename(path).encode())
            h.update(_strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current kernel sources."""
    path = os.path.join(PROFILE_DIR, f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha1") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str, interval_ms: int = 100):
        self.gpu_index = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="qk_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", str(self.interval_ms)],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 5.0 and os.path.getsize(self.path) == 0:
            time.sleep(0.02)

    def stop(self, t_begin: float, t_end: float):
        if self.proc is None:
            return None
        time.sleep(self.interval_ms / 1000.0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S")) + \
                    float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:8]))
            except Exception:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        inside = [r for r in rows if t_begin - 0.15 <= r[0] <= t_end + 0.15] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def gpu_index_for(local_rank: int) -> str:
    """nvidia-smi -i id of this rank's GPU (index or UUID from CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


def _to_dev(x, dev):
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev)


def _bias_dev(bits, dev):
    import numpy as np
    import torch
    return None if bits is None else _to_dev(bits.view(np.int16), dev).view(torch.bfloat16)


def time_headline(qk, p, steps, warmup, dev, dist, sampler):
    """K timed INT8 calls with inputs resident in HBM."""
    import torch
    A, B, sa, sb = (_to_dev(x, dev) for x in (p.A, p.B, p.sa, p.sb))
    bias = _bias_dev(p.bias, dev)
    out = torch.empty((p.M, p.N), dtype=torch.bfloat16, device=dev)
    for _ in range(warmup):
        qk.gemm_int8_rowwise(A, B, sa, sb, bias, out)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    barrier(dist)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.start()
    qk.profile_read(reset=True)
    qk.profile_enable(True)
    l0 = qk.launch_count()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_begin = time.time()
    e0.record(stream)
    for _ in range(steps):
        qk.gemm_int8_rowwise(A, B, sa, sb, bias, out)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    barrier(dist)
    torch.cuda.synchronize(dev)
    launches = qk.launch_count() - l0
    qk.profile_enable(False)
    kstats = qk.profile_read(reset=True)
    clocks = sampler.stop(t_begin, t_end) if sampler else None
    del A, B, sa, sb, bias, out
    torch.cuda.empty_cache()
    return e0.elapsed_time(e1), launches, kstats, clocks, t_end - t_begin


def time_e2e(qk, p, steps, dev):
    """The same calls through host buffers: each step copies its inputs from pinned host memory and
    its result back to pinned host memory inside the timed region.  Three streams overlap step i's
    GEMM with step i+1's input copies and step i-1's output copy (device buffers double-buffered)."""
    import numpy as np
    import torch
    pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    hA, hB, hsa, hsb = pin(p.A), pin(p.B), pin(p.sa), pin(p.sb)
    hbias = None if p.bias is None else pin(p.bias.view(np.int16)).view(torch.bfloat16)
    hout = [torch.empty((p.M, p.N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dA = [torch.empty_like(hA, device=dev) for _ in range(2)]
    dB = [torch.empty_like(hB, device=dev) for _ in range(2)]
    dsa = [torch.empty_like(hsa, device=dev) for _ in range(2)]
    dsb = [torch.empty_like(hsb, device=dev) for _ in range(2)]
    dbias = [None if hbias is None else torch.empty_like(hbias, device=dev) for _ in range(2)]
    dout = [torch.empty((p.M, p.N), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()

    def run(n):
        in_done, comp_done, out_done = [], [], []
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[i - 2])      # buffer b's inputs consumed by GEMM i-2
                dA[b].copy_(hA, non_blocking=True)
                dB[b].copy_(hB, non_blocking=True)
                dsa[b].copy_(hsa, non_blocking=True)
                dsb[b].copy_(hsb, non_blocking=True)
                if hbias is not None:
                    dbias[b].copy_(hbias, non_blocking=True)
                e = ev(); e.record(s_in); in_done.append(e)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(in_done[i])
                if i >= 2:
                    s_comp.wait_event(out_done[i - 2])     # output b read back by step i-2
                qk.gemm_int8_rowwise(dA[b], dB[b], dsa[b], dsb[b], dbias[b], dout[b])
                e = ev(); e.record(s_comp); comp_done.append(e)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i])
                hout[b].copy_(dout[b], non_blocking=True)
                e = ev(); e.record(s_out); out_done.append(e)
        return out_done

    run(2)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_comp.wait_event(e0)
    s_out.wait_event(e0)
    out_done = run(steps)
    s_out.wait_event(out_done[-1])
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    h2d = hA.numel() + hB.numel() + 4 * (hsa.numel() + hsb.numel()) + (0 if hbias is None else 2 * hbias.numel())
    d2h = 2 * hout[0].numel()
    ms = e0.elapsed_time(e1)
    del dA, dB, dsa, dsb, dbias, dout, hA, hB, hout
    torch.cuda.empty_cache()
    return ms, h2d, d2h


def time_calls(fn, iters, warmup, dev, flush):
    """Median call time over `iters` calls, each after an L2 flush, with the library's own
    timing off (its event records would sit between a call's kernels); then the same calls
    again with it on for the per-kernel times.  Returns (median ms, kernel stats)."""
    import torch
    import block_scaled_precision_tcgen05_gb300 as qk
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)

    def flushed_calls():
        times = []
        for _ in range(iters):
            # read (not write) twice the L2's size: the timed call starts cold, with no
            # dirty lines of the flush left in L2 for its own loads to write back
            flush.sum(dtype=torch.int32)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        return statistics.median(times)

    ms = flushed_calls()
    qk.profile_read(reset=True)
    qk.profile_enable(True)
    flushed_calls()
    qk.profile_enable(False)
    kstats = qk.profile_read(reset=True)
    return ms, kstats


# Every configuration's shapes beside the headline: INT8 256x256x512 (the
# latency configuration) and 30000x21504x5376 with bias, MXFP8 and MXFP4 at
# their configuration shapes, the 15-point FP8 per-token sweep, one shape
# each of the NEXT rows (NVFP4, FP8 blockscale), and MXFP4 / NVFP4 with 64
# rows (the few-row kernels' FP4 modes).
FP8_SWEEP = [(M, N, K) for (N, K) in ((2112, 7168), (7168, 1792), (21504, 5376)) for M in (64, 1024, 4096, 16384, 30000)]
FORMAT_CASES = ([("int8", (256, 256, 512)), ("int8_bias", (30000, 21504, 5376)),
                 ("mxfp8", (16384, 7168, 2048)), ("mxfp8", (32768, 7168, 1792)), ("mxfp8_b32", (16384, 7168, 2048)),
                 ("mxfp4", (8192, 8192, 8192)), ("mxfp4", (8192, 8192, 16384)), ("mxfp4", (16384, 16384, 8192)),
                 ("mxfp4", (16384, 16384, 16384))]
                + [("fp8_ptpc", s) for s in FP8_SWEEP]
                + [("nvfp4", (8192, 8192, 16384)), ("fp8_blockscale", (16384, 7168, 2048)),
                   ("mxfp4", (64, 7168, 2048)), ("nvfp4", (64, 7168, 2048))])


def _device_bf16(gen, rows, K, std, dev, spike=False):
    """bf16 N(0, std^2) [rows, K] drawn on the device (seeded); with `spike`, 1% of the
    entries (a uniform mask) are multiplied by 20, the MXFP8 activation recipe."""
    import torch
    x = torch.randn((rows, K), generator=gen, device=dev, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if spike:
        x[torch.rand((rows, K), generator=gen, device=dev) < 0.01] *= 20.0
    return x.to(torch.bfloat16)


def _b2b_call_ms(call, weights, dev, min_calls=40):
    """Per-call time of back-to-back calls that rotate through `weights`, copies of the
    weight operands whose total is over twice the L2: each call finds its weight evicted
    and streams it from HBM, as successive layers' GEMMs do.  The calls are captured once
    in a CUDA graph and replayed, so the host's per-call work (argument checks, tensor-map
    encoding) is not what is timed; CUDA events around one replay.  If capture fails the
    calls are timed as a plain loop.  Returns (ms per call, whether a graph was used)."""
    import torch
    n = len(weights)
    calls = max(min_calls, 2 * n)
    for i in range(n):
        call(weights[i])
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    graph = None
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
            for i in range(calls):
                call(weights[i % n])
        g.replay()
        torch.cuda.synchronize(dev)
        graph = g
    except Exception:
        torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(calls):
            call(weights[i % n])
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / calls, graph is not None


def _weight_copies(weight_bytes, dev):
    """How many copies of a weight exceed twice the device's L2 (at least 2)."""
    import torch
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 132 * 1024 * 1024
    return max(2, -(-2 * l2 // weight_bytes) + 1)


def secondary_formats(qk, dev, peaks, which):
    """Every configuration shape, one line each: the median of 10 calls, each after an L2
    flush (reading 256 MB), kernel times from the library's own events; the few-row shapes
    (M <= 128) also the per-call time of back-to-back calls over rotating weight copies
    larger than twice the L2 (b2b_ms, b2b_frac_of_hbm).  Operands are drawn on the device with the configurations' distributions
    and quantized by the library's quantizers (INT8, NVFP4 and blockscale use the host
    recipe); the parity tests check the same kernels on the host recipe."""
    import numpy as np
    import torch
    import qk_inputs as qi
    if which == "none":
        return []
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    weights = {}
    results = []
    for kind, (M, N, K) in FORMAT_CASES:
        t_gen = time.time()
        kname2 = None
        weight = call_w = None  # few-row kinds: the weight operands and a call on a copy of them
        if kind in ("mxfp8", "mxfp4", "mxfp8_b32"):
            fp8 = kind != "mxfp4"
            fmt = qi.FMT_MXFP8_E4M3 if fp8 else qi.FMT_MXFP4_E2M1
            A, sA = qk.quantize_mx(fmt, _device_bf16(gen, M, K, 1.0, dev, spike=fp8))
            B, sB = qk.quantize_mx(fmt, _device_bf16(gen, N, K, 0.02 if fp8 else 1.0, dev))
            out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            if kind == "mxfp8_b32":
                # B's scales per 32x32 block: the first row's scales of each 32-row group
                sB = sB[::32].contiguous()
                fn = lambda: qk.gemm_mx_b32(fmt, A, sA, B, sB, None, out)
            else:
                fn = lambda: qk.gemm_mx(fmt, A, sA, B, sB, None, out)
                weight = (B, sB)
                call_w = lambda wt: qk.gemm_mx(fmt, A, sA, wt[0], wt[1], None, out)
            dtype = "fp8" if fp8 else "fp4"
            kname = "gemm_mxfp8" if fp8 else "gemm_mxfp4"
            in_bytes = A.numel() + B.numel() + sA.numel() + sB.numel()
        elif kind == "fp8_ptpc":
            A, sa = qk.quantize_ptpc(_device_bf16(gen, M, K, 1.0, dev))
            if (N, K) not in weights:
                weights[(N, K)] = qk.quantize_ptpc(_device_bf16(gen, N, K, 0.02, dev))
            B, sb = weights[(N, K)]
            out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            fn = lambda: qk.gemm_fp8_rowwise(A, B, sa, sb, None, out)
            weight = (B, sb)
            call_w = lambda wt: qk.gemm_fp8_rowwise(A, wt[0], sa, wt[1], None, out)
            dtype, kname = "fp8", "gemm_fp8"
            in_bytes = A.numel() + B.numel() + 4 * (M + N)
        elif kind == "nvfp4":
            p = qi.nvfp4_problem(M, N, K, seed=0)
            A, sA, B, sB = (_to_dev(x, dev) for x in (p.A, p.sA, p.B, p.sB))
            ga = _to_dev(np.array([p.global_a], np.float32), dev)
            gb = _to_dev(np.array([p.global_b], np.float32), dev)
            out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            fn = lambda: qk.gemm_nvfp4(A, sA, B, sB, ga, gb, None, out)
            weight = (B, sB)
            call_w = lambda wt: qk.gemm_nvfp4(A, sA, wt[0], wt[1], ga, gb, None, out)
            dtype, kname = "fp4", "gemm_nvfp4"
            in_bytes = A.numel() + B.numel() + sA.numel() + sB.numel() + 8
        elif kind == "fp8_blockscale":
            p = qi.blockscale_problem(M, N, K, seed=0)
            A, B, sa, sb = (_to_dev(x, dev) for x in (p.A, p.B, p.sa, p.sb))
            out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            fn = lambda: qk.gemm_fp8_blockscale(A, B, sa, sb, None, out)
            dtype, kname = "fp8", "gemm_fp8_blockscale"
            in_bytes = A.numel() + B.numel() + 4 * (sa.numel() + sb.numel())
        else:
            p = qi.int8_problem(M, N, K, seed=0, bias=True)
            A, B, sa, sb = (_to_dev(x, dev) for x in (p.A, p.B, p.sa, p.sb))
            bias = _bias_dev(p.bias, dev)
            out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            fn = lambda: qk.gemm_int8_rowwise(A, B, sa, sb, bias, out)
            dtype, kname, kname2 = "f16", "gemm_int8_f16", "int8_to_f16"
            in_bytes = A.numel() + B.numel() + 4 * (M + N) + 2 * N
        torch.cuda.synchronize(dev)
        gen_s = time.time() - t_gen
        ms, kstats = time_calls(fn, 10, 3, dev, flush)
        flops = 2.0 * M * N * K
        klaunch, kms = kstats.get(kname, (1, ms))
        kavg = kms / max(klaunch, 1)
        peak = peaks["bf16_tflops"] * RATIO[dtype]
        alg_bytes = in_bytes + 2 * M * N
        tfl = flops / kavg / 1e9
        gbs = alg_bytes / kavg / 1e6
        few = M <= 128
        line = {
            "format": kind, "M": M, "N": N, "K": K,
            "ms": round(ms, 4), "tflops": round(flops / ms / 1e9, 1),
            "kernel_ms": round(kavg, 4), "kernel_tflops": round(tfl, 1),
            "peak_tflops": round(peak, 1), "frac_of_peak": round(tfl / peak, 4),
            "kernel_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "bound": "hbm" if few else "tensor",
            "frac": round(gbs / peaks["hbm_gbs"] if few else tfl / peak, 4),
            "gen_s": round(gen_s, 1),
        }
        if kname2:
            l2, ms2 = kstats.get(kname2, (0, 0.0))
            if l2:
                line["widen_ms"] = round(ms2 / l2, 4)
        if "sf_atoms" in kstats:   # the block-scaled kinds' scale-atom pre-pass
            l3, ms3 = kstats["sf_atoms"]
            line["sf_atoms_ms"] = round(ms3 / max(l3, 1), 4)
        if few and weight is not None:
            # back to back over rotating weight copies larger than twice the L2
            ncopy = _weight_copies(sum(x.numel() * x.element_size() for x in weight), dev)
            wcopies = [tuple(x.clone() for x in weight) for _ in range(ncopy)]
            b2b, graphed = _b2b_call_ms(call_w, wcopies, dev)
            b2b_gbs = alg_bytes / b2b / 1e6
            line.update({"b2b_ms": round(b2b, 4), "b2b_weight_copies": ncopy, "b2b_graph": graphed,
                         "b2b_gbs": round(b2b_gbs, 1), "b2b_frac_of_hbm": round(b2b_gbs / peaks["hbm_gbs"], 4)})
            del wcopies
        results.append(line)
        weight = call_w = None
        del A, B, out
        torch.cuda.empty_cache()
    weights.clear()
    # the quantizers that feed the GEMMs (bandwidth-bound: bf16 in, codes + scales out)
    rows, K = 16384, 7168
    xb = _device_bf16(gen, rows, K, 1.0, dev)
    for name, fn, out_bytes in (
            ("quantize_mxfp8", lambda: qk.quantize_mx(qi.FMT_MXFP8_E4M3, xb), rows * K + rows * K // 32),
            ("quantize_mxfp4", lambda: qk.quantize_mx(qi.FMT_MXFP4_E2M1, xb), rows * K // 2 + rows * K // 32),
            ("quantize_ptpc", lambda: qk.quantize_ptpc(xb), rows * K + 4 * rows)):
        ms, kstats = time_calls(fn, 10, 3, dev, flush)
        klaunch, kms = kstats.get("quantize", (1, ms))
        kavg = kms / max(klaunch, 1)
        alg = 2 * rows * K + out_bytes
        results.append({"format": name, "M": rows, "K": K, "ms": round(ms, 4), "kernel_ms": round(kavg, 4),
                        "kernel_gbs": round(alg / kavg / 1e6, 1), "frac_of_hbm": round(alg / kavg / 1e6 / peaks["hbm_gbs"], 4),
                        "bound": "hbm", "frac": round(alg / kavg / 1e6 / peaks["hbm_gbs"], 4)})
    del xb
    torch.cuda.empty_cache()
    return results


# ----------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ----------------------------------------------------------------------------

def oracle_tiles(p, target_s: float, max_tiles: int = 10000):
    """Runs the oracle on 128x128 output tiles of the problem for about target_s seconds."""
    import oracle
    import qk_inputs as qi
    tiles = qi.sample_tiles(p.M, p.N, max_tiles, seed=17)
    done, macs = 0, 0
    t0 = time.time()
    for (m0, m1, n0, n1) in tiles:
        oracle.gemm_int8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias, m0=m0, m1=m1, n0=n0, n1=n1)
        done += 1
        macs += (m1 - m0) * (n1 - n0) * p.K
        if time.time() - t0 >= target_s:
            break
    return time.time() - t0, done, macs, oracle.num_threads()


def run_reference(args, rank, world):
    import qk_inputs as qi
    if rank != 0:
        return 0
    p = qi.int8_problem(HEADLINE["M"], HEADLINE["N"], HEADLINE["K"], seed=0, bias=False)
    import oracle
    tiles = qi.sample_tiles(p.M, p.N, args.warmup + args.steps + 8, seed=17)
    for (m0, m1, n0, n1) in tiles[:args.warmup]:
        oracle.gemm_int8_rowwise(p.A, p.B, p.sa, p.sb, m0=m0, m1=m1, n0=n0, n1=n1)
    timed = tiles[args.warmup:args.warmup + args.steps]
    macs = 0
    t0 = time.time()
    for (m0, m1, n0, n1) in timed:
        oracle.gemm_int8_rowwise(p.A, p.B, p.sa, p.sb, m0=m0, m1=m1, n0=n0, n1=n1)
        macs += (m1 - m0) * (n1 - n0) * p.K
    secs = time.time() - t0
    tops = 2.0 * macs / secs / 1e12
    sample = f"{len(timed)} output tiles of up to 128x128 (full K={p.K}) of the {p.M}x{p.N}x{p.K} INT8 GEMM, one tile per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(tops, 6), "unit": "TOPS", "n_gpus": world,
        "steps": len(timed), "warmup": args.warmup, "ms_per_step": round(secs * 1000 / max(len(timed), 1), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": f"INT8 row/column-scaled GEMM {p.M}x{p.N}x{p.K}, bf16 out, no bias",
                   "M": p.M, "N": p.N, "K": p.K, "bias": False, "seed": 0},
        "cpu_baseline": {"value": round(tops, 6), "unit": "TOPS", "cores": __import__("oracle").num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(tops, 6), "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_kernel_case(args):
    """A few calls of one kernel kind on one shape (for profiler captures); prints ms per call."""
    import torch
    import block_scaled_precision_tcgen05_gb300 as qk
    import qk_inputs as qi
    M, N, K = (int(v) for v in args.shape.split(","))
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    out_dtype = torch.bfloat16
    if args.kernel_case in ("int8", "int8_fp16", "int8_fp32"):
        p = qi.int8_problem(M, N, K, seed=0, bias=False)
        A, B, sa, sb = (_to_dev(x, dev) for x in (p.A, p.B, p.sa, p.sb))
        out_dtype = {"int8": torch.bfloat16, "int8_fp16": torch.float16, "int8_fp32": torch.float32}[args.kernel_case]
        fn = lambda out: qk.gemm_int8_rowwise(A, B, sa, sb, None, out)
    elif args.kernel_case == "fp8":
        p = qi.fp8_problem(M, N, K, seed=0)
        A, B, sa, sb = (_to_dev(x, dev) for x in (p.A, p.B, p.sa, p.sb))
        fn = lambda out: qk.gemm_fp8_rowwise(A, B, sa, sb, None, out)
    elif args.kernel_case == "blockscale":
        p = qi.blockscale_problem(M, N, K, seed=0)
        A, B, sa, sb = (_to_dev(x, dev) for x in (p.A, p.B, p.sa, p.sb))
        fn = lambda out: qk.gemm_fp8_blockscale(A, B, sa, sb, None, out)
    elif args.kernel_case == "nvfp4":
        import numpy as np
        p = qi.nvfp4_problem(M, N, K, seed=0)
        A, sA, B, sB = (_to_dev(x, dev) for x in (p.A, p.sA, p.B, p.sB))
        ga = _to_dev(np.array([p.global_a], np.float32), dev)
        gb = _to_dev(np.array([p.global_b], np.float32), dev)
        fn = lambda out: qk.gemm_nvfp4(A, sA, B, sB, ga, gb, None, out)
    elif args.kernel_case in ("quantize_ptpc", "quantize_mxfp8"):
        # bf16 [M, K] input (N is not used), the recipe of the benchmark's quantizer lines
        import numpy as np
        rng = np.random.default_rng(0)
        xb = torch.from_numpy(qi.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32)).view(np.int16))
        xb = xb.to(dev).view(torch.bfloat16)
        if args.kernel_case == "quantize_ptpc":
            fn = lambda out: qk.quantize_ptpc(xb)
        else:
            fn = lambda out: qk.quantize_mx(qi.FMT_MXFP8_E4M3, xb)
        N = 1
    elif args.kernel_case == "mxfp8_b32":
        p = qi.mx_problem(qi.FMT_MXFP8_E4M3, M, N, K, seed=0)
        A, sA, B = (_to_dev(x, dev) for x in (p.A, p.sA, p.B))
        sB32 = _to_dev(p.sB[::32], dev)   # the first row's scales of each 32-row group of B
        fn = lambda out: qk.gemm_mx_b32(qi.FMT_MXFP8_E4M3, A, sA, B, sB32, None, out)
    else:
        fmt = qi.FMT_MXFP8_E4M3 if args.kernel_case == "mxfp8" else qi.FMT_MXFP4_E2M1
        p = qi.mx_problem(fmt, M, N, K, seed=0)
        A, sA, B, sB = (_to_dev(x, dev) for x in (p.A, p.sA, p.B, p.sB))
        fn = lambda out: qk.gemm_mx(fmt, A, sA, B, sB, None, out)
    out = torch.empty((M, N), dtype=out_dtype, device=dev)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for _ in range(args.iters):
        fn(out)
    torch.cuda.synchronize(dev)
    ms = (time.time() - t0) * 1000 / args.iters
    print(json.dumps({"kernel_case": args.kernel_case, "M": M, "N": N, "K": K, "iters": args.iters,
                      "wall_ms_per_call": round(ms, 3), "status_word": qk.device_status()}), flush=True)
    return 0


# ----------------------------------------------------------------------------

def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["qk", "reference"], default="qk")
    ap.add_argument("--formats", choices=["default", "none"], default="default",
                    help="none: the headline only (no per-configuration lines)")
    # steps of the end-to-end leg: enough that the pipeline's fill (the first input copy and GEMM,
    # ~5 ms) stays a small part of a region bound by the output's read-back (~6.7 ms per step)
    ap.add_argument("--e2e-steps", type=int, default=24)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--kernel-case", choices=["int8", "int8_fp16", "int8_fp32", "fp8", "mxfp8", "mxfp8_b32", "mxfp4",
                                              "nvfp4", "blockscale", "quantize_ptpc", "quantize_mxfp8"], default=None,
                    help="only run --iters calls of one kernel kind on --shape (profiler captures)")
    ap.add_argument("--shape", default="8192,8192,8192")
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args(argv)
    if args.kernel_case:
        return run_kernel_case(args)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_env()

    if args.impl == "reference":
        return run_reference(args, rank, world)

    import numpy as np  # noqa: F401
    import torch

    import block_scaled_precision_tcgen05_gb300 as qk
    import qk_inputs as qi

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = init_dist(world, "nccl")
    peaks, peak_src = load_peaks()
    M, N, K = HEADLINE["M"], HEADLINE["N"], HEADLINE["K"]
    p = qi.int8_problem(M, N, K, seed=rank, bias=False)
    qk.load_library()

    sampler = ClockSampler(gpu_index_for(local))
    ms, launches, kstats, clocks, wall = time_headline(qk, p, args.steps, args.warmup, dev, dist, sampler)
    max_ms = max_over_ranks(ms, dist, dev)
    flops = 2.0 * M * N * K
    value = whole_job_rate(flops * args.steps, world, max_ms / 1000.0) / 1e12

    e2e_ms, h2d, d2h = time_e2e(qk, p, args.e2e_steps, dev)
    e2e_max = max_over_ranks(e2e_ms, dist, dev)
    e2e_value = whole_job_rate(flops * args.e2e_steps, world, e2e_max / 1000.0) / 1e12

    # roofline of the dominant kernel (the GEMM); the f16 widening pass is reported beside it
    glaunch, gms = kstats.get("gemm_int8_f16", (0, 0.0))
    gavg = gms / max(glaunch, 1)
    sustained = wall >= 2.0
    peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    achieved = flops / (gavg / 1000.0) / 1e12 if gavg > 0 else 0.0
    wl, wms = kstats.get("int8_to_f16", (0, 0.0))
    wavg = wms / max(wl, 1)
    widen_bytes = (M + N) * K * 3
    traffic = profiled_traffic("gemm_int8_f16", f"{M}x{N}x{K}")

    fmt_results = []
    fmt_clocks = None
    cpu = None
    if rank == 0 and world == 1:
        fsampler = ClockSampler(gpu_index_for(local))
        fsampler.start()
        t_f0 = time.time()
        fmt_results = secondary_formats(qk, dev, peaks, args.formats)
        fmt_clocks = fsampler.stop(t_f0, time.time())
        secs, ntiles, macs, cores = oracle_tiles(p, args.cpu_seconds)
        cpu = {"value": round(2.0 * macs / secs / 1e12, 6), "unit": "TOPS", "cores": cores, "kind": "oracle",
               "sample": f"{ntiles} output tiles of up to 128x128 (full K={K}) of this GEMM, seeded positions, "
                         f"{secs:.1f} s on the host cores"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": round(value / (PAGES_INT8_TOPS * world), 3), "dtype": "int8",
            "data": "synthetic",
            "config": {"workload": f"INT8 row/column-scaled GEMM {M}x{N}x{K}, bf16 out, no bias (one replica per GPU)",
                       "M": M, "N": N, "K": K, "bias": False, "seed": "rank",
                       "l2": "inputs larger than L2 (277 MB int8 operands and their 553 MB f16 copies per step)",
                       "parallelism": f"replicas x{world}"},
            "e2e": {"value": round(e2e_value, 2), "unit": "TOPS", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "steps": args.e2e_steps},
            "gpu_launches": int(launches),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4) if peak else None, "traffic": traffic,
                         "kernel": "qk_gemm_kernel, exact INT8 on the f16 pipe: 256x256 tiles on 2-SM CTA pairs, "
                                   "two TMEM accumulators, int32 sums in registers, bulk-store epilogue",
                         "peak_source": f"{peak_src} {'sustained' if sustained else 'burst'} bf16 (f16 rate)",
                         "kernel_ms": round(gavg, 4)},
            "secondary_kernel": {"name": "int8_to_f16", "ms": round(wavg, 4),
                                 "achieved_gbs": round(widen_bytes / (wavg / 1000.0) / 1e9, 1) if wavg else None,
                                 "peak_gbs": peaks["hbm_gbs"],
                                 "frac": round(widen_bytes / (wavg / 1000.0) / 1e9 / peaks["hbm_gbs"], 4) if wavg else None},
            "clocks": clocks,
            "cpu_baseline": cpu,
            "formats": fmt_results,
            "formats_clocks": fmt_clocks,
            "kernel_source_sha1": kernel_source_hash(),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
