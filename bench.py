"""Benchmark of the tensor-core GEMM D = A·B + C on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one D = A·B + C over the workload's synthetic inputs (default: bf16
8192^3, C ~ N(0,1) fp32, D bf16).  ``value`` is TFLOP/s (2*M*N*K per step)
over K back-to-back steps with the inputs resident in HBM, timed with CUDA
events between a barrier + synchronize on both sides (max over ranks).  The
inputs (A+B+C = 512 MiB at the default size) are larger than L2, so no L2
flush runs between steps.  ``e2e`` times the same product through the C ABI
with host buffers (gemm_run_host: H2D of A, B, C, the kernel, D2H of D).

With N > 1 (launched by torch.distributed.run) every rank runs its own
replica of the workload on its own GPU: the GEMM has no exchange step, so
there is no collective on the data path (weak scaling).

``--impl reference`` times the CPU oracle instead (rank 0 only), on bounded
samples of the same workload; it is the deliberately slow fp64 definition,
not a competing GPU implementation.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) of one launch of the dominant kernel, from the ncu capture
# summarised in profiles/; valid only for the kernel sources the capture ran on
MEASURED_TRAFFIC = {
    "bf16_8192x8192x8192_bf16out": {"bytes": 1139664128 + 124062720, "src": "074331377af61419",
                                    "ncu": "profiles/gemm_tc_kernel_bf16_8192x8192x8192_bf16out_launches.md"},
    "mxf8e4m3_8192x8192x8192_c0_f32out": {"bytes": 609121280 + 235741952, "src": "3a8d4b60a298d33a",
                                          "ncu": "profiles/gemm_tc_kernel_mxf8_8192x8192x8192_launches.md"},
    "mxf4e2m1_8192x8192x8192_c0_f32out": {"bytes": 483959040 + 218009856, "src": "7a56a78b84b639d1",
                                          "ncu": "profiles/gemm_tc_kernel_fp4_8192x8192x8192_launches.md"},
    "nvf4e2m1_8192x8192x8192_c0_f32out": {"bytes": 495177472 + 219982848, "src": "6f369e190bf36c4c",
                                          "ncu": "profiles/gemm_tc_kernel_fp4_8192x8192x8192_launches.md"},
    "chain_bf16_32768x4096_256x256_bf16out": {"bytes": 312649216 + 11200512, "src": "fcd2357da88d26b3",
                                              "ncu": "profiles/chain_kernel_bf16_32768x4096_256x256_launches.md"},
}


# the kernel's sources and the host code that encodes its tensor maps (box shapes, swizzle and
# L2 fill granularity change the DRAM traffic as much as the kernel does)
KERNEL_SOURCES = {
    "f16": ["gemm_kernel.cuh", "ptx.cuh", "gemm_internal.h", "gemm_f16.cu", "gemm_api.cu"],
    "mxf8": ["gemm_kernel.cuh", "ptx.cuh", "gemm_internal.h", "gemm_mxf8.cu", "gemm_api.cu"],
    "mxf4": ["gemm_kernel.cuh", "ptx.cuh", "gemm_internal.h", "gemm_mxf4.cu", "gemm_api.cu"],
    "nvf4": ["gemm_kernel.cuh", "ptx.cuh", "gemm_internal.h", "gemm_nvf4.cu", "gemm_api.cu"],
    "chain": ["gemm_kernel.cuh", "ptx.cuh", "gemm_internal.h", "gemm_chain.cu", "gemm_api.cu"],
}


def kernel_family(workload_name: str) -> str:
    for fam in ("mxf8", "mxf4", "nvf4", "chain"):
        if workload_name.startswith(fam):
            return fam
    return "f16"


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and with runs of whitespace collapsed, so that a
    change to comments alone leaves the kernel's hash (and its recorded traffic) valid."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"' or c == "'":                 # a literal: copied up to its closing quote
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(family: str = "f16") -> str:
    """Hash of the CUDA sources (comments stripped) a family's kernel is built and launched from."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family]:
        h.update(f.encode())
        with open(os.path.join(ROOT, "blackwell_tensor_core_tma_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(workload_name: str):
    t = MEASURED_TRAFFIC.get(workload_name)
    if t is None or t["src"] != kernel_source_hash(kernel_family(workload_name)):
        return None, None
    return t["bytes"], t["ncu"]
# dense tensor-core rate of each operand type relative to bf16 (nominal GB300 figures:
# bf16/fp16 2.25, fp8 4.5, fp4 13.5 PFLOP/s)
OVER_BF16 = {"bf16": 1.0, "f16": 1.0, "e4m3": 2.0, "e2m1": 6.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------ distributed

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def aggregate(local_ms: float, units_per_rank: float, world: int, group=None):
    """Whole-job throughput: all ranks' units over the slowest rank's time.

    Returns (max_ms, total units / max seconds).  With world > 1 the max is an
    all-reduce over the default process group (or ``group``).
    """
    max_ms = local_ms
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([local_ms], dtype=torch.float64)
        if dist.get_backend(group) == "nccl":
            t = t.cuda()
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
        max_ms = float(t.item())
    return max_ms, units_per_rank * world / (max_ms / 1e3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu, self.period, self.proc, self.lines = gpu_index, period_ms, None, []
        self._t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(self.period), "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._t:
                self._t.join(timeout=5)

    def summary(self):
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


def smi_index(local_rank: int) -> int:
    """nvidia-smi index of CUDA device local_rank (through CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v.strip() for v in vis.split(",") if v.strip()]
    if local_rank < len(ids) and ids[local_rank].isdigit():
        return int(ids[local_rank])
    return local_rank


def workload(args):
    from blackwell_tensor_core_tma_gb300 import synth
    if args.workload in synth.CHAIN_WORKLOADS:
        w = synth.CHAIN_WORKLOADS[args.workload]
        if args.shape:
            M, N1, N2, K = (int(v) for v in args.shape.lower().split("x"))
            w = synth.scaled_chain(w, M, N1, N2, K)
        return w
    w = synth.WORKLOADS[args.workload]
    if args.shape:
        M, N, K = (int(v) for v in args.shape.lower().split("x"))
        w = synth.scaled(w, M, N, K)
    if args.a_col_major or args.b_row_major:
        w = synth.dataclasses.replace(w, name=w.name + ("+Acol" if args.a_col_major else "") +
                                      ("+Brow" if args.b_row_major else ""),
                                      a_row_major=not args.a_col_major, b_row_major=args.b_row_major)
    return w


# --------------------------------------------------------------- our arm

def gemm_config(w) -> dict:
    """The workload part of the JSON line's config, shared by both arms."""
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "ab": w.ab, "c": "fp32",
            "a_row_major": w.a_row_major, "b_row_major": w.b_row_major, "d": w.d}


def chain_config(w) -> dict:
    return {"workload": w.name, "M": w.M, "K": w.K, "N1": w.N1, "N2": w.N2, "ab": w.ab, "c": "fp32", "d": w.d}


def timed_e2e(step, flops, world, dev, stream, steps, blocks=3):
    """End-to-end rate through the host-buffer entry point: `blocks` separately timed blocks of
    `steps` calls (each copying its inputs up and its result down), after two untimed calls.
    The host link of this machine is shared with its other GPUs' jobs, and a block that meets
    their traffic runs at half speed; the value is the median block, and every block is
    reported beside it."""
    import torch
    for _ in range(2):
        step()
    vals = []
    for _ in range(blocks):
        barrier(world)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        _, rate = aggregate(e0.elapsed_time(e1) / steps, flops, world)
        vals.append(round(rate / 1e12, 3))
    return statistics.median(vals), vals


def tensor_rate(w, info, achieved, clock_summary, kernel_mhz=None):
    """Per-clock view of the roofline: the tensor-pipe rate probe (after the timed region)
    gives the FLOP per SM clock of the plan's MMA shape; the kernel's TFLOP/s is then set
    against that rate at the maximum SM clock and at the SM clock the kernel itself ran at
    (the plan's clock meter: every CTA's clock64 cycles over its globaltimer nanoseconds,
    summed over the timed launches; nvidia-smi's median is the fallback).  The probe's
    operands are hashed values of ordinary magnitude; the per-clock rate does not depend
    on the clock."""
    from blackwell_tensor_core_tma_gb300 import gemm
    r = gemm.gemm_measure_tensor_rate(w.ab, w.block_scaled, info["cta_group"], 8192)
    per_clk, sms = r["flop_per_clk_per_sm"], info["sm_count"]
    max_mhz = clock_summary.get("sm_max_mhz") or 2070.0
    at_max = sms * per_clk * max_mhz * 1e6 / 1e12
    run_mhz = kernel_mhz or clock_summary.get("sm_mhz")
    at_run = sms * per_clk * run_mhz * 1e6 / 1e12 if run_mhz else None
    return {"flop_per_clk_per_sm": round(per_clk, 1), "probe_sm_mhz": round(r["sm_mhz"], 1),
            "probe_tflops": round(r["tflops"], 1), "peak_at_max_clock": round(at_max, 1),
            "max_mhz": max_mhz, "frac_at_max_clock": round(achieved / at_max, 4),
            "run_mhz": round(run_mhz, 1) if run_mhz else None,
            "frac_at_run_clock": round(achieved / at_run, 4) if at_run else None,
            "run_clock_source": ("the kernel's own SM clock over the timed launches (clock meter: clock64 / "
                                 "globaltimer per CTA)") if kernel_mhz else "nvidia-smi median over the timed region"}


def trace_summary(tr, info, steps, w):
    """Per-role clock accounting of a trace build, per launch: where the MMA issuer's
    cycles go per k-block, and the epilogue's per piece."""
    import numpy as np

    from blackwell_tensor_core_tma_gb300 import gemm
    F = {n: i for i, n in enumerate(gemm.TRACE_FIELDS)}
    t = tr.reshape(info["grid"], -1).astype(np.float64) / steps
    lead = t[:, F["mma_kblocks"]] > 0
    kb = t[lead, F["mma_kblocks"]].sum()
    col = lambda n: t[:, F[n]]
    per_kb = lambda n: round(float(col(n)[lead].sum() / kb), 1)
    epi = col("epi_pieces").sum()
    out = {
        "launches": steps, "leader_ctas": int(lead.sum()), "kblocks_per_leader": round(float(kb / lead.sum()), 2),
        "kernel_mhz": round(float(col("kernel_clk").sum() / col("kernel_ns").sum() * 1e3), 1),
        "clk_per_kblock": round(float((col("kernel_clk")[lead] / col("mma_kblocks")[lead]).mean()), 1),
        "mma_per_kblock": {n: per_kb("mma_" + n) for n in ("wait_ab", "wait_sf", "wait_acc", "issue")},
        "mma_first_clk": round(float(col("mma_first")[lead].mean()), 0),
        "mma_tail_clk": round(float((col("kernel_clk") - col("mma_end"))[lead].mean()), 0),
        "prod_per_stage": {n: round(float(col("prod_" + n).sum() / col("prod_stages").sum()), 1)
                           for n in ("wait", "issue")},
        "epi_per_piece_per_warp": {n: round(float(col("epi_" + n).sum() / max(epi, 1)), 1)
                                   for n in ("wait_acc", "tmem_ld", "wait_c", "store")},
        "epi_end_clk": round(float(col("epi_end").max()), 0),
    }
    if w.block_scaled:
        out["copier_per_kblock"] = {n: per_kb("cp_" + n) for n in ("wait", "issue")}
    return out


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    from blackwell_tensor_core_tma_gb300 import gemm, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = workload(args)
    x = synth.make_inputs(w)

    def dev_tensor(a):
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    A, B, C = dev_tensor(x["A"]), dev_tensor(x["B"]), dev_tensor(x["C"])
    SFA = dev_tensor(x["SFA"]) if w.block_scaled else None
    SFB = dev_tensor(x["SFB"]) if w.block_scaled else None
    d_t = torch.bfloat16 if w.d == "bf16" else torch.float32
    D = torch.empty((w.M, w.N), dtype=d_t, device=dev)
    flags = {0: 0, 1: gemm.GEMM_FLAG_FORCE_1CTA, 2: gemm.GEMM_FLAG_FORCE_2CTA}[args.cta_group]
    plan = gemm.Plan(w.M, w.N, w.K, w.ab, w.d, w.block_scaled, flags, a_row_major=w.a_row_major,
                     b_row_major=w.b_row_major)
    if args.stream_k is not None:
        plan.set_stream_k(args.stream_k)
    info = plan.info
    stream = torch.cuda.Stream(device=dev)

    def step():
        plan.run(A, B, C, D, SFA, SFB, stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)
    if plan.last_status() != gemm.GEMM_OK:
        raise RuntimeError("kernel reported a timeout during warm-up")

    # per-launch events on the launching stream give the kernel's duration
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    trace_buf = None
    if args.trace:
        slots = gemm.gemm_testing_trace_slots()
        trace_buf = torch.zeros(info["grid"] * slots, dtype=torch.int64, device=dev)
        gemm.gemm_testing_set_trace(plan.handle, trace_buf, trace_buf.numel() * 8)
    plan.set_clock_meter(True)               # the kernel's own SM clock over the timed launches
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(smi_index(local_rank)) as clocks:
        t0.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    if plan.last_status() != gemm.GEMM_OK:
        raise RuntimeError("kernel reported a timeout in the timed region")
    meter = plan.read_clock_meter()
    plan.set_clock_meter(False)
    trace = None
    if trace_buf is not None:
        gemm.gemm_testing_set_trace(plan.handle, None, 0)
        trace = trace_summary(trace_buf.cpu().numpy(), info, args.steps, w)
    local_ms = t0.elapsed_time(t1) / args.steps
    kernel_ms = statistics.fmean(a.elapsed_time(b) for a, b in ev)
    max_ms, flops_per_s = aggregate(local_ms, w.flops, world)
    value = flops_per_s / 1e12

    # end to end through the C ABI with pinned host buffers
    e2e = None
    if not args.no_e2e:
        hA = torch.from_numpy(x["A"].view(np.int16) if x["A"].dtype == np.uint16 else x["A"]).pin_memory()
        hB = torch.from_numpy(x["B"].view(np.int16) if x["B"].dtype == np.uint16 else x["B"]).pin_memory()
        hC = torch.from_numpy(x["C"]).pin_memory()
        hSFA = torch.from_numpy(x["SFA"]).pin_memory() if w.block_scaled else None
        hSFB = torch.from_numpy(x["SFB"]).pin_memory() if w.block_scaled else None
        hD = torch.empty((w.M, w.N), dtype=d_t).pin_memory()
        e_steps = max(3, min(args.steps, args.e2e_steps))
        e2e_value, blocks = timed_e2e(lambda: plan.run_host(hA, hB, hC, hD, hSFA, hSFB, stream), w.flops, world, dev,
                                  stream, e_steps)
        h2d = x["A"].nbytes + x["B"].nbytes + x["C"].nbytes + \
            (x["SFA"].nbytes + x["SFB"].nbytes if w.block_scaled else 0)
        e2e = {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(hD.numel() * hD.element_size()), "steps": e_steps, "blocks": blocks}

    peaks, source = load_peaks()
    traffic, traffic_src = (args.traffic, "--traffic") if args.traffic is not None else measured_traffic(w.name)
    ratio = OVER_BF16[w.ab]
    peak = peaks["bf16_tflops"] * ratio
    achieved = w.flops / (kernel_ms / 1e3) / 1e12
    sf_bytes = x["SFA"].nbytes + x["SFB"].nbytes if w.block_scaled else 0
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": traffic, "traffic_source": traffic_src,
                "algorithmic_bytes": int(x["A"].nbytes + x["B"].nbytes + x["C"].nbytes + sf_bytes +
                                         w.M * w.N * (2 if w.d == "bf16" else 4)),
                "peak_source": f"{source} bf16 burst (cuBLAS bf16 8192^3)" +
                               (f" x{ratio:g} nominal {w.ab}/bf16" if ratio != 1.0 else ""),
                "frac_of_sustained": round(achieved / (peaks.get("bf16_tflops_sustained", peak) * ratio), 4),
                "kernel": "gemm_tc_kernel",
                "kernel_ms": round(kernel_ms, 5)}
    clock_summary = clocks.summary()
    clock_summary["kernel_sm_mhz"] = round(meter["sm_mhz"], 1) if meter["sm_mhz"] else None
    if not args.no_probe:
        roofline["tensor_rate"] = tensor_rate(w, info, achieved, clock_summary, meter["sm_mhz"] or None)

    out = {
        "metric": "GEMM TFLOP/s and % of GB300 dense tensor peak (bf16 8192^3), vs CPU oracle",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(max_ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.ab == "bf16" else w.ab,
        "data": "synthetic (seeded splitmix64; recipe of the workload)",
        "config": dict(gemm_config(w), cta_group=info["cta_group"],
                       tile=[info["tile_m"], info["tile_n"], info["tile_k"]], stages=info["stages"],
                       grid=info["grid"], replicas=world, l2="no flush: inputs (A+B+C) larger than the 129 MB L2"),
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": args.steps * info["launches_per_run"],
        "clocks": clock_summary,
    }
    if trace is not None:
        out["trace"] = trace
        out["library"] = "trace build (GB300_TRACE=1): timings include the counters' cost"
    plan.close()
    if rank == 0 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline(w, x, args.cpu_seconds)
    return out


def run_ours_chain(args, rank, world, local_rank):
    """The two-product chain D = C + round(A·B)·E through gemm_chain_run."""
    import numpy as np
    import torch

    from blackwell_tensor_core_tma_gb300 import gemm, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = workload(args)
    x = synth.make_chain_inputs(w)

    def dev_tensor(a):
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    A, B, E, C = (dev_tensor(x[k]) for k in ("A", "B", "E", "C"))
    d_t = torch.bfloat16 if w.d == "bf16" else torch.float32
    D = torch.empty((w.M, w.N2), dtype=d_t, device=dev)
    plan = gemm.ChainPlan(w.M, w.N1, w.N2, w.K, w.ab, w.d)
    if args.stream_k is not None:
        plan.set_stream_k(args.stream_k)
    info = plan.info
    stream = torch.cuda.Stream(device=dev)

    def step():
        plan.run(A, B, E, C, D, stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)
    if plan.last_status() != gemm.GEMM_OK:
        raise RuntimeError("kernel reported a timeout during warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(smi_index(local_rank)) as clocks:
        t0.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    if plan.last_status() != gemm.GEMM_OK:
        raise RuntimeError("kernel reported a timeout in the timed region")
    local_ms = t0.elapsed_time(t1) / args.steps
    kernel_ms = statistics.fmean(a.elapsed_time(b) for a, b in ev)
    max_ms, flops_per_s = aggregate(local_ms, w.flops, world)

    e2e = None
    if not args.no_e2e:
        h = {k: torch.from_numpy(x[k].view(np.int16) if x[k].dtype == np.uint16 else x[k]).pin_memory()
             for k in ("A", "B", "E", "C")}
        hD = torch.empty((w.M, w.N2), dtype=d_t).pin_memory()
        e_steps = max(3, min(args.steps, args.e2e_steps))
        e2e_value, blocks = timed_e2e(lambda: plan.run_host(h["A"], h["B"], h["E"], h["C"], hD, stream), w.flops, world,
                                  dev, stream, e_steps)
        h2d = sum(x[k].nbytes for k in ("A", "B", "E", "C"))
        e2e = {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(hD.numel() * hD.element_size()), "steps": e_steps, "blocks": blocks}

    # roofline: the bound is whichever of HBM bytes and tensor FLOPs takes longer at the measured peaks
    peaks, source = load_peaks()
    alg_bytes = int(sum(x[k].nbytes for k in ("A", "B", "E", "C")) + w.M * w.N2 * (2 if w.d == "bf16" else 4))
    t_hbm = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = w.flops / (peaks["bf16_tflops"] * 1e12)
    traffic, traffic_src = (args.traffic, "--traffic") if args.traffic is not None else measured_traffic(w.name)
    if t_hbm >= t_tc:
        achieved = alg_bytes / (kernel_ms / 1e3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "peak_source": f"{source} HBM copy bandwidth"}
    else:
        achieved = w.flops / (kernel_ms / 1e3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                    "peak_source": f"{source} bf16 burst (cuBLAS bf16 8192^3)"}
    roofline.update({"traffic": traffic, "traffic_source": traffic_src, "algorithmic_bytes": alg_bytes,
                     "tensor_tflops": round(w.flops / (kernel_ms / 1e3) / 1e12, 2),
                     "frac_of_tensor_peak": round(w.flops / (kernel_ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
                     "kernel": "chain_kernel", "kernel_ms": round(kernel_ms, 5)})
    out = {
        "metric": "GEMM TFLOP/s and % of GB300 dense tensor peak (bf16 8192^3), vs CPU oracle",
        "value": round(flops_per_s / 1e12, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(max_ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.ab,
        "data": "synthetic (seeded splitmix64; recipe of the workload)",
        "config": dict(chain_config(w), cta_group=info["cta_group"],
                       tile=[info["tile_m"], info["tile_n"], info["tile_k"]], stages=info["stages"],
                       grid=info["grid"], replicas=world, l2="no flush: inputs (A alone) larger than the 129 MB L2"),
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": args.steps * info["launches_per_run"],
        "clocks": clocks.summary(),
    }
    plan.close()
    if rank == 0 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline_chain(w, x, args.cpu_seconds)
    return out


def cpu_baseline_chain(w, x, seconds: float):
    """The oracle's chain on a bounded number of rows of the same workload."""
    import numpy as np

    import oracle
    probe = 64
    t = time.perf_counter()
    oracle.chain(x["A"], x["B"], x["E"], x["C"], w.M, w.N1, w.N2, w.K, w.ab, rows=np.arange(probe))
    per_row = max((time.perf_counter() - t) / probe, 1e-6)
    R = int(max(1, min(w.M, seconds / per_row)))
    t = time.perf_counter()
    oracle.chain(x["A"], x["B"], x["E"], x["C"], w.M, w.N1, w.N2, w.K, w.ab, rows=np.arange(R))
    dt = time.perf_counter() - t
    return {"value": round(2.0 * R * w.N1 * (w.K + w.N2) / dt / 1e12, 6), "unit": "TFLOP/s",
            "cores": oracle.threads(), "kind": "oracle",
            "sample": f"rows 0..{R - 1} of {w.name} (both products, fp64, incl. operand decode), {dt:.1f} s"}


def cpu_baseline(w, x, seconds: float):
    """The oracle's triple loop on a row slab of the same workload (bounded CPU time)."""
    import oracle
    t = time.perf_counter()
    oracle.gemm(x["A"], x["B"], x["C"], w.M, w.N, w.K, w.ab, SFA=x.get("SFA"), SFB=x.get("SFB"),
                block_scaled=w.block_scaled, rows=(0, 1))
    one = time.perf_counter() - t                    # includes decoding all of B once
    rows = 33                                        # enough rows for every core to take some
    t = time.perf_counter()
    oracle.gemm(x["A"], x["B"], x["C"], w.M, w.N, w.K, w.ab, SFA=x.get("SFA"), SFB=x.get("SFB"),
                block_scaled=w.block_scaled, rows=(0, rows))
    two = time.perf_counter() - t
    per_row = max((two - one) / (rows - 1), 1e-6)
    fixed = max(one - per_row, 0.0)
    R = int(max(1, min(w.M, (seconds - fixed) / per_row)))
    t = time.perf_counter()
    oracle.gemm(x["A"], x["B"], x["C"], w.M, w.N, w.K, w.ab, SFA=x.get("SFA"), SFB=x.get("SFB"),
                block_scaled=w.block_scaled, rows=(0, R))
    dt = time.perf_counter() - t
    return {"value": round(2.0 * R * w.N * w.K / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.threads(),
            "kind": "oracle",
            "sample": f"rows 0..{R - 1} of {w.name} (all N and K, fp64 triple loop incl. operand decode), "
                      f"{dt:.1f} s"}


# --------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    import numpy as np

    import oracle
    from blackwell_tensor_core_tma_gb300 import synth

    w = workload(args)
    if isinstance(w, synth.ChainWorkload):
        return run_reference_chain(args, w, world)
    x = synth.make_inputs(w)
    rng = np.random.default_rng(0)
    total_budget = args.reference_seconds
    per_step = total_budget / (args.steps + args.warmup)

    def sample(n):
        r = rng.integers(0, w.M, n)
        c = rng.integers(0, w.N, n)
        t = time.perf_counter()
        oracle.gemm_entries(x["A"], x["B"], x["C"], w.M, w.N, w.K, w.ab, r, c, SFA=x.get("SFA"),
                            SFB=x.get("SFB"), block_scaled=w.block_scaled)
        return time.perf_counter() - t

    probe = 256
    rate = probe / max(sample(probe), 1e-6)          # entries per second
    n = int(max(16, rate * per_step))
    for _ in range(args.warmup):
        sample(n)
    t = time.perf_counter()
    for _ in range(args.steps):
        sample(n)
    dt = (time.perf_counter() - t) / args.steps
    flops = 2.0 * n * w.K
    value = flops / dt / 1e12
    desc = f"{n} random entries of {w.name} per step (each a fp64 sum over K = {w.K})"
    return {
        "impl": "reference",
        "metric": "GEMM TFLOP/s and % of GB300 dense tensor peak (bf16 8192^3), vs CPU oracle",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded splitmix64)",
        "config": gemm_config(w),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def run_reference_chain(args, w, world):
    """The oracle's chain on random rows of the workload (each row: both products, fp64)."""
    import numpy as np

    import oracle
    from blackwell_tensor_core_tma_gb300 import synth
    x = synth.make_chain_inputs(w)
    rng = np.random.default_rng(0)
    per_step = args.reference_seconds / (args.steps + args.warmup)

    def sample(n):
        t = time.perf_counter()
        oracle.chain(x["A"], x["B"], x["E"], x["C"], w.M, w.N1, w.N2, w.K, w.ab, rows=rng.integers(0, w.M, n))
        return time.perf_counter() - t

    rate = 8 / max(sample(8), 1e-6)                  # rows per second
    n = int(max(1, rate * per_step))
    for _ in range(args.warmup):
        sample(n)
    t = time.perf_counter()
    for _ in range(args.steps):
        sample(n)
    dt = (time.perf_counter() - t) / args.steps
    value = 2.0 * n * w.N1 * (w.K + w.N2) / dt / 1e12
    desc = f"{n} random rows of {w.name} per step (both products in fp64)"
    return {
        "impl": "reference",
        "metric": "GEMM TFLOP/s and % of GB300 dense tensor peak (bf16 8192^3), vs CPU oracle",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded splitmix64)",
        "config": chain_config(w),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    from blackwell_tensor_core_tma_gb300 import synth
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=synth.HEADLINE, choices=sorted(synth.WORKLOADS) + sorted(synth.CHAIN_WORKLOADS))
    ap.add_argument("--shape", default=None, help="MxNxK (chain workloads: MxN1xN2xK): the workload's recipe at "
                                                  "other sizes (profiling)")
    ap.add_argument("--cta-group", type=int, choices=[0, 1, 2], default=0,
                    help="force single CTAs (1) or CTA pairs (2); 0 = the plan's choice")
    ap.add_argument("--stream-k", type=int, choices=[0, 1], default=None,
                    help="gemm_plan_set_stream_k: 0 = never, 1 = where the plan's rule takes it (the default)")
    ap.add_argument("--a-col-major", action="store_true", help="store A column-major (M contiguous)")
    ap.add_argument("--b-row-major", action="store_true", help="store B row-major (N contiguous)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-probe", action="store_true", help="skip the tensor-pipe rate probe")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--reference-seconds", type=float, default=120.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the dominant kernel from an ncu capture")
    ap.add_argument("--trace", action="store_true",
                    help="load the trace build of the library (GB300_TRACE=1, built if needed) and add the "
                         "kernels' per-role clock accounting to the line (GEMM workloads; a diagnostic run)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.trace:
        if args.workload in synth.CHAIN_WORKLOADS:
            ap.error("--trace covers the GEMM kernels, not the chain")
        from blackwell_tensor_core_tma_gb300 import build as _libbuild
        _libbuild.build(variant="trace")
        os.environ["GB300GEMM_VARIANT"] = "trace"
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        runner = run_ours_chain if args.workload in synth.CHAIN_WORKLOADS else run_ours
        out = runner(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(out), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
