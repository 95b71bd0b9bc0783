#!/usr/bin/env python3
"""Benchmark: throughput of the half-precision GEMM hot path on GB300.

One step = one C = A . B through the C ABI (hgemm_run) on the workload's full
shape.  Default workload: M = N = K = 4096, bf16 inputs, fp32 accumulate, bf16
output, TN layout; metric TFLOPS = 2MNK / t.  The skinny workload reports GB/s
of compulsory traffic instead.

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and torch.cuda.synchronize on both sides, timed with CUDA events on the
launching stream.  Inputs rotate through enough copies that the bytes touched
between two uses of the same copy exceed twice the L2, so every step reads its
operands from HBM.  SM clocks and throttle reasons are sampled with
nvidia-smi during the timed region.  The end-to-end figure (e2e) is the same
metric with the host->device copy of A and B from pinned memory and the
device->host copy of C inside the timed region; consecutive steps alternate
between two caller streams (--e2e-streams), so that one step's uploads overlap
the previous step's GEMM and download.

After the K timed steps (one GPU only; --no-secondary skips them): a
sustained loop of the same launches lasting >= 1 s, whose clocks the sampler
does see, against the sustained peak; the other target workloads (8192^3 bf16,
the skinny 16x16384x8192 product against HBM) and the two weakest shapes
(1000x3000x4104, 2048^3 fp16), each with its own roofline; and the CPU oracle
on the 256^3 workload and on 2048^3, one thread and all host cores.

N > 1 (torchrun): independent replicas, one per GPU, each running the full
workload (weak scaling); the time is the maximum over ranks.

--impl reference: the CPU oracle timed on the host cores on a bounded sample
(a block of rows of C) of the same workload; that is the reference arm.

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import atexit
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC_TFLOPS = "TFLOPS (2MNK/t) at M=N=K=4096 bf16, fp32 acc; % of dense BF16 tensor peak"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
THROTTLE_BITS = {  # nvidia-smi clocks_event_reasons bit masks
    0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
    0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
    0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}
_SHARED_SOURCES = ["ptx.cuh", "desc.cuh", "sched.cuh", "kernels.h", "clc.cuh"]
KERNEL_SOURCES = {  # the files each kernel is compiled from
    "dense": ["gemm_dense.cu"] + _SHARED_SOURCES,
    "splitk": ["gemm_splitk.cu"] + _SHARED_SOURCES,
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of one kernel's sources: stored ncu traffic is valid only while it matches."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "tensor_core_half_gb300", "csrc", rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(workload: str, variant: int, plan=None):
    """DRAM bytes per launch from a committed ncu summary, if it matches these
    kernels and this launch plan (the stream-K split and the rasterisation
    height change the traffic)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get("%s/%d" % (workload, variant))
    kernel = "splitk" if variant == 4 else "dense"
    if not e or e.get("kernel_hash") != kernel_source_hash(kernel):
        return None
    want = e.get("plan")
    if plan is not None and want is not None:
        have = {"grid": plan.grid, "dp_tiles": plan.dp_tiles, "sk_units": plan.sk_units,
                "sk_ranges": plan.sk_ranges, "group_m": getattr(plan, "group_m", None)}
        if any(have[k] != v for k, v in want.items()):
            return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- clocks ----
class ClockSampler:
    """nvidia-smi sampling in the background; marks let us keep only samples
    taken inside the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.samples = []  # (host time, sm_mhz, max_mhz, power_w, active_mask)
        self.proc = None
        self.thread = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", str(period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # A run that raises before stop() must not leave nvidia-smi looping.
        atexit.register(self.stop)
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()

    def _reader(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 5:
                continue
            try:
                sm = float(parts[1])
                mx = float(parts[2])
                pw = float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else float("nan")
                act = int(parts[4], 16) if parts[4].startswith("0x") else int(parts[4])
            except ValueError:
                continue
            self.samples.append((time.time(), sm, mx, pw, act))

    def stop(self):
        """Ends the sampling process; safe to call more than once."""
        if self.proc is not None and self.proc.poll() is None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed"
        if not inside:  # timed region shorter than the sampling period: nearest samples
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            window = "nearest"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "none"}
        sms = sorted(s[1] for s in inside)
        mask = 0
        for s in inside:
            mask |= s[4]
        reasons = [name for bit, name in THROTTLE_BITS.items() if mask & bit]
        pw = [s[3] for s in inside if not math.isnan(s[3])]
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(inside), "window": window}


def in_kernel_clocks(rows, recorded, expected):
    """SM clock of every CTA of the timed launches from their kernel begin/end
    stamps (cycles over global-timer ns), as median / min / max MHz."""
    from tensor_core_half_gb300 import trace

    mhz = sorted(trace.launch_clocks(rows))
    out = {"source": "SM cycle counter / global timer between each CTA's kernel begin and end, every CTA of "
                     "the K timed launches",
           "stamps": int(recorded), "stamps_expected": int(expected), "cta_launches": len(mhz)}
    if mhz:
        out.update({"sm_mhz_median": round(mhz[len(mhz) // 2], 1), "sm_mhz_min": round(mhz[0], 1),
                    "sm_mhz_max": round(mhz[-1], 1)})
    return out


# --------------------------------------------------------------- helpers ----
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_metric(w):
    """(metric name, unit, per-step amount of the unit's numerator, roofline bound)."""
    if w.name.startswith("skinny"):
        return ("GB/s of compulsory traffic (A + B + C bytes / t) at M=%d N=%d K=%d %s" % (w.M, w.N, w.K, w.in_dtype),
                "GB/s", float(w.compulsory_bytes) / 1e9, "hbm")
    if w.name == "square4096_bf16":
        return METRIC_TFLOPS, "TFLOPS", float(w.flops) / 1e12, "tensor"
    return ("TFLOPS (2MNK/t) at M=%d N=%d K=%d %s, %s acc" % (w.M, w.N, w.K, w.in_dtype, w.acc_dtype), "TFLOPS",
            float(w.flops) / 1e12, "tensor")


def cpu_oracle_sample(w, a_bits, b_bits, target_s: float):
    """Times the oracle (as it stands, all host cores) on a block of rows of C."""
    import numpy as np

    import oracle
    cores = os.cpu_count() or 1
    rows = 8
    while True:
        t0 = time.perf_counter()
        oracle.gemm_entries(a_bits, b_bits, w.M, w.N, w.K, w.layout, w.in_dtype,
                            np.repeat(np.arange(rows, dtype=np.int64), w.N),
                            np.tile(np.arange(w.N, dtype=np.int64), rows), nthreads=cores)
        dt = time.perf_counter() - t0
        if dt >= target_s or rows >= w.M:
            return rows, dt, cores
        rows = min(w.M, max(rows * 2, int(rows * target_s / max(dt, 1e-3) * 1.1)))


def host_cpu_model() -> str:
    """The host CPU: lscpu's model name, else /proc/cpuinfo's (or the Arm part number)."""
    try:
        import subprocess
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read().splitlines()
    except OSError:
        return "unknown"
    for key in ("model name", "Model name", "Hardware"):
        for line in info:
            if line.startswith(key) and ":" in line:
                return line.split(":", 1)[1].strip()
    impl = [l.split(":", 1)[1].strip() for l in info if l.startswith("CPU implementer")]
    part = [l.split(":", 1)[1].strip() for l in info if l.startswith("CPU part")]
    return "CPU implementer %s, part %s" % (impl[0] if impl else "?", part[0] if part else "?")


def oracle_timing(names=("square256_f16", "sweep2048_f16_accf32"), emit=True):
    """The CPU oracle on the small workloads, one thread and all host cores:
    each a median of 3 full products (one run where a single-threaded product
    takes over 30 s), GFLOP/s = 2MNK / t.  Returns one record per run (and
    prints each as a JSON line when emit is set)."""
    import numpy as np

    import oracle
    from tensor_core_half_gb300 import workloads
    cores = os.cpu_count() or 1
    nproc = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else cores
    model = host_cpu_model()
    out = []
    for name in names:
        w = workloads.WORKLOADS[name]
        a, b = workloads.generate_workload(w)
        ab, bb = workloads.bits(a), workloads.bits(b)
        for threads in (1, nproc):
            times = []
            for _ in range(3):
                t0 = time.perf_counter()
                oracle.gemm(ab, bb, w.M, w.N, w.K, w.layout, w.in_dtype, w.out_dtype, nthreads=threads)
                times.append(time.perf_counter() - t0)
                if times[-1] > 30.0:
                    break
            t = float(np.median(times))
            rec = {"oracle_timing": name, "M": w.M, "N": w.N, "K": w.K, "in": w.in_dtype, "threads": threads,
                   "runs": len(times), "seconds": round(t, 4), "gflops": round(2.0 * w.M * w.N * w.K / t / 1e9, 3),
                   "hardware_concurrency": cores, "nproc": nproc, "cpu": model}
            out.append(rec)
            if emit:
                print(json.dumps(rec), flush=True)
    return out


def wake_then_rest(step, dev, load_seconds, rest_seconds):
    """Brings a GPU that has been idle out of its low-clock state: launches
    back to back for load_seconds, then lets it rest for rest_seconds so that
    the power limiter, which engages within tens of milliseconds of full load,
    has recovered when the timed burst starts.  (Measured on GB300 at 4096^3:
    the first bursts of a process on an idle GPU ran ~81 us per launch, bursts
    during or right after 50 ms-3 s of load ~88 us, bursts after such load
    and >= 0.5 s of rest ~77 us.  As the first process on a fresh box, 1 s of
    load and 1 s of rest gave 77.6 us where 0.3 s and 0.6 s had given
    79-80 us on other boxes.)  Returns what it did."""
    import torch
    t0 = time.time()
    n = 0
    while time.time() - t0 < load_seconds:
        for _ in range(32):
            step(n)
            n += 1
        torch.cuda.synchronize(dev)
    loaded = time.time() - t0
    time.sleep(rest_seconds)
    return {"load_launches": n, "load_seconds": round(loaded, 3), "rest_seconds": rest_seconds}


def problem_config(w, world):
    """The workload as both arms name it (the same dict in our line and in the
    reference arm's line)."""
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "layout": w.layout, "in": w.in_dtype,
            "acc": w.acc_dtype, "out": w.out_dtype, "parallelism": "replicas" if world > 1 else "single",
            "l2": "GPU arm: inputs rotate over copies that together exceed 2x L2, so every launch reads its "
                  "operands from HBM; CPU oracle arm: host memory"}


def roofline_for(w, bound, kernel_ms, peaks, peak_src, sustained):
    """The roofline object of one kernel: algorithmic work of one launch over
    its average launch time, against the measured peak of its bound."""
    if bound == "tensor":
        peak = peaks.get("bf16_tflops_sustained" if sustained else "bf16_tflops")
        achieved = (w.flops / 1e12) / (kernel_ms / 1e3)
        return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4),
                "peak_source": "%s %s" % (peak_src, "sustained" if sustained else "burst")}
    peak = peaks.get("hbm_gbs")
    achieved = (w.compulsory_bytes / 1e9) / (kernel_ms / 1e3)
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": peak_src}


def time_workload(w, dev, steps, warmup, n_single, stamps=True):
    """Device-timed launches of one workload through hgemm_run: `steps`
    back-to-back launches between two events (inputs rotating over copies
    larger than 2x L2), then the median of `n_single` launches each between
    its own events.  Before the warm-up, the same load-then-rest as the
    headline.  With `stamps`, every CTA records its kernel begin and end
    (HGEMM_OPT_TRACE_ITEMS = 0) from the first launch on, and those of the
    timed launches give the SM clock inside them.  Returns (ms per launch,
    median single ms, plan, what the load-then-rest did, in-kernel clocks or
    None)."""
    import torch

    from tensor_core_half_gb300 import hgemm, workloads
    a_cpu, b_cpu = workloads.generate_workload(w)
    in_bytes = (a_cpu.numel() + b_cpu.numel()) * 2
    c_bytes = w.M * w.N * 2
    copies = max(1, math.ceil(2 * L2_BYTES / max(1, in_bytes + c_bytes)))
    A = [a_cpu.to(dev) for _ in range(copies)]
    B = [b_cpu.to(dev) for _ in range(copies)]
    C = [torch.empty((w.M, w.N), dtype=workloads.DTYPES[w.out_dtype], device=dev) for _ in range(copies)]
    lay, fin, facc, fout = (hgemm.LAYOUTS[w.layout], hgemm.DTYPES[w.in_dtype], hgemm.DTYPES[w.acc_dtype],
                            hgemm.DTYPES[w.out_dtype])
    st, plan = hgemm.hgemm_plan(w.M, w.N, w.K, lay, fin, facc, fout,
                                torch.cuda.get_device_properties(dev).multi_processor_count)
    stream = torch.cuda.current_stream(dev)
    capacity = 2 * plan.grid * (steps + 2)
    clocks = None
    with hgemm.Handle() as h:
        if stamps:
            h.set_option(hgemm.HGEMM_OPT_TRACE, capacity)
            h.set_option(hgemm.HGEMM_OPT_TRACE_ITEMS, 0)

        def step(i):
            s = hgemm.hgemm_run(h.h, A[i % copies].data_ptr(), B[i % copies].data_ptr(), C[i % copies].data_ptr(),
                                w.M, w.N, w.K, lay, fin, facc, fout, stream.cuda_stream)
            if s != hgemm.HGEMM_OK:
                raise hgemm.HgemmError(s, "hgemm_run (%s)" % w.name)

        protocol = wake_then_rest(step, dev, 0.05, 0.6)
        for i in range(warmup):
            step(i)
        if stamps:  # drop the warm-up's stamps
            st = hgemm.hgemm_trace_read(h.h, 0)[0]
            if st != hgemm.HGEMM_OK:
                raise hgemm.HgemmError(st, "hgemm_trace_read (reset, %s)" % w.name)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
        if stamps:
            st, recorded, rows = hgemm.hgemm_trace_read(h.h, capacity)
            if st != hgemm.HGEMM_OK:
                raise hgemm.HgemmError(st, "hgemm_trace_read (%s)" % w.name)
            h.set_option(hgemm.HGEMM_OPT_TRACE, 0)
            clocks = in_kernel_clocks(rows, recorded, 2 * plan.grid * steps)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_single)]
        for i, (x, y) in enumerate(ev):
            x.record(stream)
            step(i)
            y.record(stream)
        torch.cuda.synchronize(dev)
        single = sorted(x.elapsed_time(y) for x, y in ev)
        st, detail = h.sync_status()
        if st != hgemm.HGEMM_OK:
            raise hgemm.HgemmError(st, "%s (detail %s)" % (w.name, hex(detail)))
    del A, B, C
    torch.cuda.empty_cache()
    return ms, single[len(single) // 2], plan, protocol, clocks


SECONDARY = ("square8192_bf16", "skinny16x16384x8192_bf16", "ragged1000x3000x4104_bf16", "sweep2048_f16_accf32")


# ------------------------------------------------------------------ main ----
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None)
    ap.add_argument("--variant", default="auto")
    ap.add_argument("--stream-k", type=int, default=1, choices=[0, 1, 2])
    ap.add_argument("--schedule", default="static", choices=["static", "dynamic"])
    ap.add_argument("--epilogue", default="tma", choices=["tma", "direct"])
    ap.add_argument("--group-m", type=int, default=0, help="rasterisation group height in tiles (0: default)")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--e2e-streams", type=int, default=2,
                    help="caller streams the end-to-end steps alternate between (1: every step on one stream)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--oracle-timing", action="store_true",
                    help="only time the CPU oracle on the 256^3 and 2048^3 workloads, one thread and all cores")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the other workloads, the oracle timing and the sustained loop after the headline")
    ap.add_argument("--wake-seconds", type=float, default=1.0,
                    help="untimed back-to-back launches that bring an idle GPU to its full clock before the rest")
    ap.add_argument("--rest-seconds", type=float, default=1.0,
                    help="idle time after the wake-up load, before the W warm-up steps and the timed region")
    ap.add_argument("--sustained-seconds", type=float, default=1.2,
                    help="length of the sustained headline loop reported beside the K timed steps")
    ap.add_argument("--no-launch-clocks", action="store_true",
                    help="do not record each CTA's kernel begin/end stamps (SM cycle counter and global timer) "
                         "during the headline, which give the SM clock inside the K timed launches")
    ap.add_argument("--sweep", default=None, metavar="JSONL",
                    help="measure every workload of the table (and --sweep-variants, --sweep-schedules), one JSON "
                         "record per line appended to JSONL; records already there are skipped, so an "
                         "interrupted sweep resumes")
    ap.add_argument("--sweep-variants", default="auto")
    ap.add_argument("--sweep-schedules", default="static")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.oracle_timing:
        oracle_timing()
        return
    if args.sweep:
        sweep(args)
        return

    world, rank, local = dist_setup()
    from tensor_core_half_gb300 import workloads
    w = workloads.WORKLOADS[args.workload or workloads.HEADLINE]
    metric, unit, per_step, bound = workload_metric(w)

    if args.impl == "reference":
        run_reference(args, w, metric, unit, per_step, world, rank)
        return

    import numpy as np
    import torch

    from tensor_core_half_gb300 import hgemm

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    a_cpu, b_cpu = workloads.generate_workload(w)
    dt = workloads.DTYPES[w.out_dtype]
    in_bytes = (a_cpu.numel() + b_cpu.numel()) * 2
    c_bytes = w.M * w.N * 2
    copies = max(1, math.ceil(2 * L2_BYTES / max(1, in_bytes + c_bytes)))
    A = [a_cpu.to(dev) for _ in range(copies)]
    B = [b_cpu.to(dev) for _ in range(copies)]
    C = [torch.empty((w.M, w.N), dtype=dt, device=dev) for _ in range(copies)]
    handle = hgemm.Handle()
    handle.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.VARIANTS[args.variant])
    handle.set_option(hgemm.HGEMM_OPT_STREAM_K, args.stream_k)
    handle.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.SCHEDULES[args.schedule])
    handle.set_option(hgemm.HGEMM_OPT_EPILOGUE, hgemm.EPILOGUES[args.epilogue])
    if args.group_m > 0:
        handle.set_option(hgemm.HGEMM_OPT_GROUP_M, args.group_m)
    st, plan = hgemm.hgemm_plan(w.M, w.N, w.K, hgemm.LAYOUTS[w.layout], hgemm.DTYPES[w.in_dtype],
                                hgemm.DTYPES[w.acc_dtype], hgemm.DTYPES[w.out_dtype],
                                torch.cuda.get_device_properties(dev).multi_processor_count,
                                hgemm.VARIANTS[args.variant], args.group_m, args.stream_k)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    lay, fin, facc, fout = (hgemm.LAYOUTS[w.layout], hgemm.DTYPES[w.in_dtype], hgemm.DTYPES[w.acc_dtype],
                            hgemm.DTYPES[w.out_dtype])
    ptrs = [(A[i].data_ptr(), B[i].data_ptr(), C[i].data_ptr()) for i in range(copies)]

    def step(i):
        a, b, c = ptrs[i % copies]
        s = hgemm.hgemm_run(handle.h, a, b, c, w.M, w.N, w.K, lay, fin, facc, fout, sp)
        if s != hgemm.HGEMM_OK:
            raise hgemm.HgemmError(s, "hgemm_run")

    # The SM clock inside the timed region: nvidia-smi samples every 20 ms,
    # far apart for K launches of well under a millisecond, so every CTA of
    # every launch also records its kernel begin and end (the SM cycle
    # counter against the global timer; two appends per CTA, from the first
    # launch on, so the warm-up runs the same code as the timed launches).
    launch_clocks = world == 1 and not args.no_launch_clocks
    stamp_capacity = 2 * plan.grid * (args.steps + 2)
    if launch_clocks:
        handle.set_option(hgemm.HGEMM_OPT_TRACE, stamp_capacity)
        handle.set_option(hgemm.HGEMM_OPT_TRACE_ITEMS, 0)

    # One checked launch (allocates the workspace, reports any device-side
    # error), then the clock sampler gets going; the W warm-up steps run last,
    # right before the timed region, so that the GPU is not idle in between.
    step(0)
    st, detail = handle.sync_status()
    if st != hgemm.HGEMM_OK:
        raise hgemm.HgemmError(st, "first launch (detail %s)" % hex(detail))
    sampler = ClockSampler(local)
    # Load, then rest (see wake_then_rest), then the W warm-up steps right
    # before the timed region.
    clock_warm = wake_then_rest(step, dev, args.wake_seconds, max(0.3, args.rest_seconds))
    for i in range(args.warmup):
        step(i)

    # ------------------------------------------------ device-timed region ----
    # Two events bracket the K launches: events between launches would break the
    # overlap of consecutive kernels (programmatic dependent launch).
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if launch_clocks:  # drop the warm-up's stamps (this read synchronises the device)
        st = hgemm.hgemm_trace_read(handle.h, 0)[0]
        if st != hgemm.HGEMM_OK:
            raise hgemm.HgemmError(st, "hgemm_trace_read (reset)")
    barrier(world)
    torch.cuda.synchronize(dev)
    h0 = time.time()
    t_start.record(stream)
    for i in range(args.steps):
        step(i)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    h1 = time.time()
    barrier(world)
    st, detail = handle.sync_status()
    if st != hgemm.HGEMM_OK:
        raise hgemm.HgemmError(st, "timed region (detail %s)" % hex(detail))
    total_ms = t_start.elapsed_time(t_end)
    kernel_ms_avg = total_ms / args.steps  # average launch duration in the timed stream
    total_ms_max = max_over_ranks(total_ms, world)
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(h0, h1)
    if launch_clocks:
        st, n_stamps, rows = hgemm.hgemm_trace_read(handle.h, stamp_capacity)
        if st != hgemm.HGEMM_OK:
            raise hgemm.HgemmError(st, "hgemm_trace_read")
        handle.set_option(hgemm.HGEMM_OPT_TRACE, 0)
        clocks["in_kernel"] = in_kernel_clocks(rows, n_stamps, 2 * plan.grid * args.steps)

    # Median of single launches, each bracketed by its own events (outside the
    # timed region; includes the launch overhead the overlap otherwise hides).
    n_med = max(20, min(args.steps, 50))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_med)]
    for i in range(n_med):
        ev[i][0].record(stream)
        step(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    per_launch = sorted(e[0].elapsed_time(e[1]) for e in ev)
    median_ms = per_launch[len(per_launch) // 2]

    # A sustained loop of the same launches, long enough (>= 1 s) for the
    # clock sampler to see the SM clock and the power cap during it; the K
    # timed steps above are far shorter than one sampling period.
    sustained_rec = None
    if world == 1 and not args.no_secondary and args.sustained_seconds > 0:
        n_long = max(args.steps, int(math.ceil(args.sustained_seconds / (kernel_ms_avg / 1e3))))
        s_sampler = ClockSampler(local)
        time.sleep(0.3)
        for i in range(args.warmup):
            step(i)
        l0 = torch.cuda.Event(enable_timing=True)
        l1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        g0 = time.time()
        l0.record(stream)
        for i in range(n_long):
            step(i)
        l1.record(stream)
        torch.cuda.synchronize(dev)
        g1 = time.time()
        time.sleep(0.1)
        s_sampler.stop()
        st, detail = handle.sync_status()
        if st != hgemm.HGEMM_OK:
            raise hgemm.HgemmError(st, "sustained loop (detail %s)" % hex(detail))
        long_ms = l0.elapsed_time(l1) / n_long
        sustained_rec = {"steps": n_long, "seconds": round(n_long * long_ms / 1e3, 3), "ms_per_step": round(long_ms, 5),
                         "value": round(per_step / (long_ms / 1e3), 3), "unit": unit,
                         "clocks": s_sampler.summary(g0, g1)}

    # ------------------------------------------------------ end to end ------
    e2e_steps = args.e2e_steps if args.e2e_steps is not None else max(3, min(args.steps, 50))
    # End to end: the C-ABI call on HOST buffers (hgemm_run_host), which uploads
    # A and B from page-locked memory and downloads C inside every step.
    # Consecutive steps alternate between e2e_streams caller streams, the
    # pipelined use the call is built for: a step's uploads then wait only for
    # the staging set it reuses, not for the previous step's download.
    a_pin = a_cpu.pin_memory()
    b_pin = b_cpu.pin_memory()
    n_es = max(1, args.e2e_streams)
    c_pins = [torch.empty((w.M, w.N), dtype=dt).pin_memory() for _ in range(n_es)]
    e_streams = [stream] + [torch.cuda.Stream(device=dev) for _ in range(n_es - 1)]

    def e2e_step(i):
        j = i % n_es
        s = hgemm.hgemm_run_host(handle.h, a_pin.data_ptr(), b_pin.data_ptr(), c_pins[j].data_ptr(), w.M, w.N, w.K,
                                 lay, fin, facc, fout, e_streams[j].cuda_stream)
        if s != hgemm.HGEMM_OK:
            raise hgemm.HgemmError(s, "hgemm_run_host (e2e)")

    for i in range(2 * n_es):
        e2e_step(i)
    barrier(world)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for es in e_streams[1:]:
        es.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    for es in e_streams[1:]:  # the closing event follows every step's download
        stream.wait_stream(es)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    st, detail = handle.sync_status()
    if st != hgemm.HGEMM_OK:
        raise hgemm.HgemmError(st, "e2e (detail %s)" % hex(detail))

    if rank != 0:
        handle.close()
        return

    value = world * args.steps * per_step / (total_ms_max / 1e3)
    e2e_value = world * e2e_steps * per_step / (e2e_ms / 1e3)
    peaks, peak_src = load_peaks()
    timed_seconds = total_ms / 1e3
    # The sustained (power-capped) peak applies once the loop runs long enough
    # for the power cap to engage, which the clock record shows.
    sustained = timed_seconds > 1.0 or "sw_power_cap" in (clocks.get("reasons") or [])
    roof = roofline_for(w, bound, kernel_ms_avg, peaks, peak_src, sustained)
    roof["traffic"] = load_traffic(w.name, plan.variant, plan)
    roof["kernel_ms_avg"] = round(kernel_ms_avg, 5)
    if sustained_rec is not None and bound == "tensor":
        sustained_rec["roofline"] = roofline_for(w, bound, sustained_rec["ms_per_step"], peaks, peak_src, True)

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        rows, secs, cores = cpu_oracle_sample(w, workloads.bits(a_cpu), workloads.bits(b_cpu), args.cpu_seconds)
        frac = rows / w.M
        cpu_val = (per_step * frac) / secs
        cpu = {"value": round(cpu_val, 6), "unit": unit, "cores": cores, "kind": "oracle",
               "sample": "first %d of %d rows of C (%.3g s, fp64 oracle, %d threads)" % (rows, w.M, secs, cores)}
    handle.close()

    # The other workloads the targets name (8192^3 bf16 and the skinny product
    # against HBM) and the two weakest shapes, timed the same way, each with its
    # own roofline; then the oracle on the 256^3 workload and 2048^3, one
    # thread and all cores, on this host.
    secondary, oracle_recs = None, None
    if world == 1 and not args.no_secondary:
        secondary = []
        for name in SECONDARY:
            sw = workloads.WORKLOADS[name]
            s_metric, s_unit, s_per_step, s_bound = workload_metric(sw)
            n_steps = max(args.steps, 20)
            ms, single_ms, s_plan, s_protocol, s_clocks = time_workload(sw, dev, n_steps, max(args.warmup, 5), 20,
                                                                        not args.no_launch_clocks)
            # a timed region over 1 s runs under the power cap: the sustained peak applies
            r = roofline_for(sw, s_bound, ms, peaks, peak_src, n_steps * ms > 1000.0)
            r["traffic"] = load_traffic(sw.name, s_plan.variant, s_plan)
            secondary.append({"workload": name, "metric": s_metric, "value": round(s_per_step / (ms / 1e3), 3),
                              "unit": s_unit, "steps": n_steps, "ms_per_step": round(ms, 5),
                              "median_single_launch_ms": round(single_ms, 5),
                              "value_at_median_single_launch": round(s_per_step / (single_ms / 1e3), 3),
                              "variant": list(hgemm.VARIANTS)[s_plan.variant], "warmup_protocol": s_protocol,
                              "clocks": {"in_kernel": s_clocks}, "roofline": r})
        oracle_recs = oracle_timing(emit=False)

    config = problem_config(w, world)
    out = {
        "metric": metric, "value": round(value, 3), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms_max / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.in_dtype, "data": "synthetic",
        "config": config,
        "plan": {"variant": list(hgemm.VARIANTS)[plan.variant],
                 "grid": plan.grid if args.schedule == "static" else plan.work_ids * plan.cta_group,
                 "schedule": args.schedule, "epilogue": args.epilogue, "group_m": plan.group_m,
                 "tile": [plan.tile_m, plan.tile_n], "stages": plan.stages,
                 "stream_k": {"dp_tiles": plan.dp_tiles, "sk_units": plan.sk_units, "sk_ranges": plan.sk_ranges,
                              "sk_pieces": plan.sk_pieces} if plan.stream_k else None,
                 "input_copies": copies, "input_bytes": int(copies * (in_bytes + c_bytes))},
        "warmup_protocol": clock_warm,
        "single_launch": {"median_ms": round(median_ms, 5), "launches": n_med,
                          "value_at_median": round(per_step / (median_ms / 1e3), 3)},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 3), "unit": unit, "h2d_bytes_per_step": int(in_bytes),
                "d2h_bytes_per_step": int(c_bytes), "steps": e2e_steps, "api": "hgemm_run_host",
                "streams": n_es},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if sustained_rec is not None:
        out["sustained"] = sustained_rec
    if secondary is not None:
        out["secondary"] = secondary
    if oracle_recs is not None:
        out["oracle_timing"] = oracle_recs
    print(json.dumps(out), flush=True)


def sweep(args):
    """Device-timed rate of every workload (one GPU), appended as JSON lines."""
    import torch

    from tensor_core_half_gb300 import hgemm, workloads

    done = set()
    if os.path.exists(args.sweep):
        with open(args.sweep) as f:
            for line in f:
                if line.strip():
                    r = json.loads(line)
                    done.add((r["workload"], r["variant"], r["schedule"]))
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    peaks, peak_src = load_peaks()
    names = sorted(workloads.WORKLOADS, key=lambda n: workloads.WORKLOADS[n].flops)
    steps = args.steps if args.steps != 3000 else 200  # shorter default than the headline loop
    n_new = 0
    for name in names:
        w = workloads.WORKLOADS[name]
        metric, unit, per_step, bound = workload_metric(w)
        a_cpu, b_cpu = None, None
        for variant in args.sweep_variants.split(","):
            for schedule in args.sweep_schedules.split(","):
                if (name, variant, schedule) in done:
                    continue
                if a_cpu is None:
                    a_cpu, b_cpu = workloads.generate_workload(w)
                in_bytes = (a_cpu.numel() + b_cpu.numel()) * 2
                c_bytes = w.M * w.N * 2
                copies = max(1, math.ceil(2 * L2_BYTES / max(1, in_bytes + c_bytes)))
                A = [a_cpu.to(dev) for _ in range(copies)]
                B = [b_cpu.to(dev) for _ in range(copies)]
                C = [torch.empty((w.M, w.N), dtype=workloads.DTYPES[w.out_dtype], device=dev) for _ in range(copies)]
                h = hgemm.Handle()
                h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.VARIANTS[variant])
                h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.SCHEDULES[schedule])
                lay, fin, facc, fout = (hgemm.LAYOUTS[w.layout], hgemm.DTYPES[w.in_dtype], hgemm.DTYPES[w.acc_dtype],
                                        hgemm.DTYPES[w.out_dtype])
                st, plan = hgemm.hgemm_plan(w.M, w.N, w.K, lay, fin, facc, fout, props.multi_processor_count,
                                            hgemm.VARIANTS[variant], 0, 1, schedule=hgemm.SCHEDULES[schedule])
                if st != hgemm.HGEMM_OK:  # e.g. a forced variant that does not take this layout
                    rec = {"workload": name, "variant": variant, "schedule": schedule,
                           "status": hgemm.hgemm_status_string(st)}
                else:
                    sp = torch.cuda.current_stream(dev).cuda_stream

                    def step(i):
                        s = hgemm.hgemm_run(h.h, A[i % copies].data_ptr(), B[i % copies].data_ptr(),
                                            C[i % copies].data_ptr(), w.M, w.N, w.K, lay, fin, facc, fout, sp)
                        if s != hgemm.HGEMM_OK:
                            raise hgemm.HgemmError(s, "hgemm_run")

                    for i in range(args.warmup):
                        step(i)
                    torch.cuda.synchronize(dev)
                    sampler = ClockSampler(0)
                    time.sleep(0.2)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    h0 = time.time()
                    e0.record()
                    for i in range(steps):
                        step(i)
                    e1.record()
                    torch.cuda.synchronize(dev)
                    h1 = time.time()
                    sampler.stop()
                    ms = e0.elapsed_time(e1) / steps
                    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                          for _ in range(50)]
                    for i, (x, y) in enumerate(ev):
                        x.record()
                        step(i)
                        y.record()
                    torch.cuda.synchronize(dev)
                    single = sorted(x.elapsed_time(y) for x, y in ev)
                    st, detail = h.sync_status()
                    if st != hgemm.HGEMM_OK:
                        raise hgemm.HgemmError(st, "sweep %s (detail %s)" % (name, hex(detail)))
                    value = per_step / (ms / 1e3)
                    peak = peaks.get("bf16_tflops") if bound == "tensor" else peaks.get("hbm_gbs")
                    rec = {"workload": name, "variant": variant, "schedule": schedule, "metric": metric,
                           "value": round(value, 3), "unit": unit, "steps": steps, "ms_per_step": round(ms, 5),
                           "single_launch_ms": {"p10": round(single[5], 5), "median": round(single[25], 5),
                                                "p90": round(single[45], 5)},
                           "roofline": {"bound": bound, "peak": peak, "frac": round(value / peak, 4),
                                        "peak_source": "%s%s" % (peak_src, " burst" if bound == "tensor" else "")},
                           "plan": {"variant": list(hgemm.VARIANTS)[plan.variant], "grid": plan.grid,
                                    "tile": [plan.tile_m, plan.tile_n], "stages": plan.stages,
                                    "group_m": plan.group_m,
                                    "stream_k": bool(plan.stream_k), "sk_pieces": plan.sk_pieces,
                                    "sk_ranges": plan.sk_ranges, "work_ids": plan.work_ids,
                                    "splitk_chunks": plan.splitk_chunks,
                                    "splitk_whole_tiles": plan.splitk_align > 1},
                           "gpu": props.name, "sms": props.multi_processor_count,
                           "clocks": sampler.summary(h0, h1)}
                h.close()
                del A, B, C
                torch.cuda.empty_cache()
                with open(args.sweep, "a") as f:
                    f.write(json.dumps(rec) + "\n")
                n_new += 1
    print(json.dumps({"sweep": args.sweep, "records_added": n_new, "records_skipped": len(done)}), flush=True)


def run_reference(args, w, metric, unit, per_step, world, rank):
    """The CPU oracle on the same workload: each step computes a bounded block of rows."""
    if world > 1 and rank != 0:
        return
    import numpy as np

    import oracle
    from tensor_core_half_gb300 import workloads
    a, b = workloads.generate_workload(w)
    ab, bb = workloads.bits(a), workloads.bits(b)
    cores = os.cpu_count() or 1
    # rows per step: sized so that warm-up plus K steps take about 90 s of oracle work
    per_step_s = max(0.02, min(0.5, 90.0 / (args.steps + min(args.warmup, 3))))
    rows, secs, _ = cpu_oracle_sample(w, ab, bb, per_step_s)
    ri = np.repeat(np.arange(rows, dtype=np.int64), w.N)
    ci = np.tile(np.arange(w.N, dtype=np.int64), rows)
    for _ in range(min(args.warmup, 3)):
        oracle.gemm_entries(ab, bb, w.M, w.N, w.K, w.layout, w.in_dtype, ri, ci, nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm_entries(ab, bb, w.M, w.N, w.K, w.layout, w.in_dtype, ri, ci, nthreads=cores)
    total = time.perf_counter() - t0
    frac = rows / w.M
    value = args.steps * per_step * frac / total
    sample = "first %d of %d rows of C per step (fp64 oracle, %d threads)" % (rows, w.M, cores)
    out = {"impl": "reference", "metric": metric, "value": round(value, 6), "unit": unit, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": problem_config(w, world),
           "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": cores, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "gpu_launches": 0}
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
