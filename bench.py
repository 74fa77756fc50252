"""SGEMM benchmark on GB300: TFLOPS and fraction of the roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--path auto|ffma|tf32x3]

A step is one C = alpha*A*B + beta*C call through the C ABI on the
8192 x 8192 x 8192 workload (row-major FP32, alpha = 1, beta = 0, A and B
i.i.d. N(0,1) from seed 3) by default, inputs resident in HBM.  Rank 0
prints one JSON line.  Under torchrun every rank runs its own independent
replica of the step (a GEMM has no exchange step), so ``value`` is the
FLOPs of all ranks over the slowest rank's time ("weak" scaling).

``--impl reference`` times the FP64 CPU oracle on the same workload instead
(a bounded slab of output rows per step, on the host cores), the only arm
this library has to compare against.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SGEMM TFLOPS on 1 GB300 at 2048³/8192³; % of FP32 FFMA peak (roofline)"
DEFAULT_WORKLOAD = "8192^3"
SECONDARY = "2048^3"
L2_BYTES = 129 * 2 ** 20
FP32_LANES_PER_SM = 128
# nominal dense tensor rates (PFLOP/s) used only to scale a measured bf16 peak to tf32
NOMINAL_TF32_OVER_BF16 = 1.1 / 2.25

WORKLOAD_TEXT = {
    "256^3": "sgemm 256x256x256 row-major fp32, alpha=1 beta=0, A,B U[-1,1] seed 0",
    "2048^3": "sgemm 2048x2048x2048 row-major fp32, alpha=1 beta=0, A,B U[-1,1] seed 1",
    "1000x1500x777": "sgemm 1000x1500x777 row-major fp32, lda=777 ldb=ldc=1500, alpha=1.5 beta=0.5, "
                     "A,B U[-1,1], C0 N(0,1) seed 2",
    "8192^3": "sgemm 8192x8192x8192 row-major fp32, alpha=1 beta=0, A,B N(0,1) seed 3",
    "16384x128x8192": "sgemm 16384x128x8192 row-major fp32, alpha=1 beta=1, A,B,C0 U[-1,1] seed 4",
}


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--path", choices=("auto", "ffma", "tf32x3"), default="auto")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_TEXT), default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--shape", default=None,
                    help="m,n,k of a smaller stand-in of the 8192^3 workload (profiling captures)")
    ap.add_argument("--reduce", type=int, default=0, metavar="N",
                    help="time reduce_sum_f32 on N floats instead of the GEMM (its own JSON line)")
    return ap.parse_args(argv)


def flops(p):
    return 2.0 * p.m * p.n * p.k


def tflops(p, ms, count=1):
    """TFLOPS of `count` problems `p` done in `ms` milliseconds (2mnk per
    problem, the FLOP count the pages' figures use)."""
    return flops(p) * count / (ms * 1e-3) / 1e12


def max_over_ranks(value, world):
    """The largest `value` over all ranks (the slowest rank's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_problem(args):
    from dense_fp32_gemm_06_gb300 import inputs
    if args.shape:
        m, n, k = (int(x) for x in args.shape.split(","))
        return inputs.workload(DEFAULT_WORKLOAD, m=m, n=n, k=k), f"sgemm {m}x{n}x{k} stand-in of 8192^3"
    return inputs.workload(args.workload), WORKLOAD_TEXT[args.workload]


# ----------------------------------------------------------------------------- clocks

class NvmlClockSampler:
    """SM clock, power and clock-event reasons read through NVML (the
    driver's libnvidia-ml, by ctypes) every `period_s` seconds on a
    background thread, so that even a timed region of a few tens of
    milliseconds gets many samples.  Reads only; changes no setting."""

    # nvmlClocksEventReasons bits
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, device_index, period_s=0.005):
        import ctypes
        import threading
        self.ok = False
        self.rows = []
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint(0)
            nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))   # NVML_CLOCK_SM
            get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
        except Exception:
            return
        self.nv, self.h, self.max_mhz = nv, h, float(mx.value)
        self.ok = True
        self.stop_flag = threading.Event()

        def loop():
            clk, pw, rs = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
            while not self.stop_flag.is_set():
                t = time.time()
                if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                    nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
                    get_reasons(h, ctypes.byref(rs))
                    self.rows.append((t, float(clk.value), pw.value / 1000.0, int(rs.value)))
                time.sleep(period_s)

        self.thread = threading.Thread(target=loop, daemon=True)
        self.thread.start()

    def stop(self):
        if self.ok:
            self.stop_flag.set()
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        inside = [r for r in self.rows if t0 <= r[0] <= t1]
        if not inside:
            return None
        reasons = sorted({name for r in inside for bit, name in self.REASONS.items() if r[3] & bit})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(r[1] for r in inside), "reasons": reasons, "samples": len(inside),
                "power_w_median": statistics.median(r[2] for r in inside),
                "source": "NVML every 5 ms during the timed region"}


class SmiClockSampler:
    """nvidia-smi sampled every 100 ms in the background (used when NVML
    cannot be opened directly)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        fd, self.path = tempfile.mkstemp(prefix="sgemm_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[3], parts[5:9]))
                except (ValueError, IndexError):
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05] or rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in inside for i in range(4) if r[4][i].lower() == "active"})
        power = [float(r[3]) for r in inside if r[3].replace(".", "", 1).isdigit()]
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons,
                "samples": len(inside),
                "power_w_median": statistics.median(power) if power else None,
                "source": "nvidia-smi every 100 ms"}


class ClockSampler:
    """Clocks during a timed region: NVML every 5 ms, falling back to
    nvidia-smi every 100 ms when NVML cannot be opened."""

    def __init__(self, device_index):
        self.nvml = NvmlClockSampler(device_index)
        self.smi = None if self.nvml.ok else SmiClockSampler(device_index)

    def stop(self):
        self.nvml.stop()
        if self.smi is not None:
            self.smi.stop()

    def summary(self, t0, t1):
        if self.smi is None:
            got = self.nvml.summary(t0, t1)
            if got is not None:
                return got
            return {"sm_mhz": None, "sm_max_mhz": self.nvml.max_mhz, "reasons": [], "samples": 0,
                    "note": "no NVML sample inside the timed region"}
        return self.smi.summary(t0, t1)


# ----------------------------------------------------------------------------- helpers

# sources that define each kernel family (a traffic figure is void once any
# changes), the planner (sgemm_api.cu) among them: the plan -- tiles, raster
# groups, schedule -- sets the launch whose traffic a record holds.  The
# tensor-core families differ in which operands the GEMM reads as stored
# (raw) and which come split by the split pass.
_TC_SOURCES = ["tf32x3_sgemm.cuh", "tcgen05.cuh", "ptx.cuh", "raster.cuh", "sgemm_api.cu"]
KERNEL_SOURCES = {
    "ffma": ["ffma_sgemm.cuh", "ptx.cuh", "raster.cuh", "sgemm_api.cu"],
    "tf32x3_raw_ab": _TC_SOURCES,
    "tf32x3_raw_a": _TC_SOURCES,
    "tf32x3_raw_b": _TC_SOURCES,
    "tf32x3_presplit": _TC_SOURCES,
}


def tc_family(a_raw, b_raw):
    return {(True, True): "tf32x3_raw_ab", (True, False): "tf32x3_raw_a", (False, True): "tf32x3_raw_b",
            (False, False): "tf32x3_presplit"}[(bool(a_raw), bool(b_raw))]


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and blank lines, so that a kernel's
    hash changes with its code only (string literals in these sources hold
    no comment markers)."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_source_hash(family):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_fp32_gemm_06_gb300", "csrc")
    for name in KERNEL_SOURCES[family]:
        try:
            with open(os.path.join(csrc, name), encoding="utf-8") as fh:
                h.update(name.encode() + strip_comments(fh.read()).encode())
        except OSError:
            h.update(name.encode() + b"<missing>")
    return h.hexdigest()[:16]


def traffic_record(kernel_family, units):
    """DRAM bytes per launch (read + write) of the kernel from the committed
    ncu summaries (`profiles/traffic.json`: per kernel family, one record per
    captured size) when one was captured on this size (`units` = m*n*k),
    else None; None too when the kernel sources changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            recs = json.load(fh).get(kernel_family)
    except (OSError, ValueError):
        return None
    if isinstance(recs, dict):
        recs = [recs]
    for rec in recs or ():
        if rec.get("source_hash") == kernel_source_hash(kernel_family) and rec.get("units") == units:
            return rec.get("dram_bytes_per_launch")
    return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh)
    except (OSError, ValueError):
        return None


def oracle_sample(p, seconds):
    """Times the FP64 oracle on a slab of output rows sized to ~`seconds`;
    returns (tflops, rows, seconds, threads)."""
    import oracle
    oracle.build()
    threads = oracle.max_threads()
    rows = max(1, min(p.m, threads))
    t = time.perf_counter()
    oracle.problem_f64(p, rows=(0, rows))
    dt = time.perf_counter() - t
    rows = int(max(1, min(p.m, rows * max(1.0, seconds / max(dt, 1e-6)))))
    t = time.perf_counter()
    oracle.problem_f64(p, rows=(0, rows))
    dt = time.perf_counter() - t
    return 2.0 * rows * p.n * p.k / dt / 1e12, rows, dt, threads


def oracle_full_small():
    """The whole FP64 oracle (every output) on the three configurations it
    finishes in about a second, on all host cores: the CPU baseline of those
    workloads, timed once each."""
    import oracle
    from dense_fp32_gemm_06_gb300 import inputs
    oracle.build()
    out = []
    for name in ("256^3", "2048^3", "1000x1500x777"):
        q = inputs.workload(name)
        oracle.problem_f64(q, rows=(0, min(q.m, 8)))   # warm (threads, pages)
        t = time.perf_counter()
        oracle.problem_f64(q)
        dt = time.perf_counter() - t
        out.append({"workload": WORKLOAD_TEXT[name], "seconds": dt, "value": flops(q) / dt / 1e12,
                    "unit": "TFLOPS", "cores": oracle.max_threads(), "kind": "oracle",
                    "sample": "every output (full run)"})
    return out


def cublas_side_reference(p, A, B, C, stream, flush, sms):
    """cuBLAS FP32 SGEMM (torch.matmul, TF32 off, so FP32 FFMA) on the same
    operands and stream, CUDA events per launch: context for the library's
    numbers, not a path the library takes."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        Av = A[:, :p.k]
        Bv = B[:, :p.n]
        out = torch.empty(p.m, p.n, device="cuda")
        with torch.cuda.stream(stream):
            for _ in range(3):
                torch.matmul(Av, Bv, out=out)
            count = max(10, int(1.0 / max(1e-6, flops(p) / 60e12)))
            ms = time_launches(lambda: torch.matmul(Av, Bv, out=out), stream, count, flush=flush)
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    med = statistics.median(ms)
    return {"value": tflops(p, med), "unit": "TFLOPS", "median_ms": med, "launches": len(ms),
            "what": "cuBLAS FP32 SGEMM via torch.matmul (allow_tf32 = False), same operands and stream; "
                    "side reference only, not on the library's path"}


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    p, text = load_problem(args)
    oracle.build()
    threads = oracle.max_threads()
    # size one step to ~ (budget / steps) seconds of CPU work
    budget = 150.0
    per_step = max(0.5, min(10.0, budget / max(1, args.steps + args.warmup)))
    probe = min(p.m, threads)
    t = time.perf_counter()
    oracle.problem_f64(p, rows=(0, probe))
    dt = time.perf_counter() - t
    rows = int(max(1, min(p.m, probe * per_step / max(dt, 1e-6))))
    for _ in range(args.warmup):
        oracle.problem_f64(p, rows=(0, rows))
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.problem_f64(p, rows=(0, rows))
        times.append(time.perf_counter() - t)
    total = sum(times)
    value = 2.0 * rows * p.n * p.k * len(times) / total / 1e12
    sample = (f"output rows 0..{rows - 1} of the {args.workload} workload ({rows} x {p.n} outputs, "
              f"k = {p.k}) per step, FP64")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded splitmix64)",
        "config": {"workload": text, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- our arm

def time_launches(fn, stream, steps, flush=None):
    """Per-launch CUDA-event durations (ms) on `stream`."""
    import torch
    evs = []
    for _ in range(steps):
        if flush is not None:
            flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def device_time_ms(fn, stream, reps, flush=None):
    """Device time of one fn() launch sequence (ms): reps x (flush, fn)
    enqueued back to back minus reps x flush alone, each bracketed by CUDA
    events on `stream`.  For kernels shorter than the host's cost of a call,
    where per-launch events would also count the GPU waiting for the host:
    a device-side sleep (a few ms) runs first, so that every launch is
    queued before the first event and the launches then run back to back."""
    import torch

    def run(with_fn):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(4_000_000 + 200_000 * reps)   # clock cycles
        a.record(stream)
        for _ in range(reps):
            if flush is not None:
                flush()
            if with_fn:
                fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    run(True)   # warm
    with_fn = min(run(True) for _ in range(3))
    without = min(run(False) for _ in range(3))
    return max(0.0, (with_fn - without) / reps)


def time_e2e(p, world, host, step_on, steps):
    """End-to-end steps through the C ABI from pinned host memory: each step
    copies its A and B (and C0 when beta != 0) host -> device, runs the
    GEMM and copies C device -> host.  Steps are pipelined the way a
    streaming caller would run them: three device buffer sets, one stream
    for host -> device copies, one for the GEMM, one for device -> host
    copies, so step i+1's inputs and step i-1's result move while step i
    computes (with two sets, step i+1's upload would also wait for step
    i-1's download, which puts both copies of a step on one chain).
    Each of three windows is timed from its first copy in to its last copy
    out; the metric is that of the median window."""
    import torch
    A_h, B_h, C_h, out_h = host
    up, comp, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    nsets = 3
    sets = [(torch.empty_like(A_h, device="cuda"), torch.empty_like(B_h, device="cuda"),
             torch.empty_like(C_h, device="cuda")) for _ in range(nsets)]
    outs = [torch.empty_like(C_h).pin_memory() for _ in range(nsets)]
    done_compute = [None] * nsets
    done_down = [None] * nsets

    def run(n):
        for i in range(n):
            A, B, C = sets[i % nsets]
            with torch.cuda.stream(up):
                if done_compute[i % nsets] is not None:
                    up.wait_event(done_compute[i % nsets])      # the GEMM of step i-3 has read A, B
                if done_down[i % nsets] is not None:
                    up.wait_event(done_down[i % nsets])         # and its result has left C
                A.copy_(A_h, non_blocking=True)
                B.copy_(B_h, non_blocking=True)
                if p.beta != 0:
                    C.copy_(C_h, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(up)
            with torch.cuda.stream(comp):
                comp.wait_event(ready)
                step_on(A, B, C, comp.cuda_stream)
                done_compute[i % nsets] = torch.cuda.Event()
                done_compute[i % nsets].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(done_compute[i % nsets])
                outs[i % nsets].copy_(C, non_blocking=True)
                done_down[i % nsets] = torch.cuda.Event()
                done_down[i % nsets].record(down)

    run(nsets)
    torch.cuda.synchronize()
    # three timed windows of `steps` steps each; the median window is the
    # value (host-copy bandwidth varies between runs on a shared host)
    windows = []
    for _ in range(3):
        done_compute[:] = [None] * nsets
        done_down[:] = [None] * nsets
        t = time.perf_counter()
        run(steps)
        torch.cuda.synchronize()
        windows.append((time.perf_counter() - t) * 1e3 / steps)
    ms = statistics.median(windows)
    h2d = A_h.numel() * 4 + B_h.numel() * 4 + (C_h.numel() * 4 if p.beta != 0 else 0)
    return {"value": tflops(p, ms, world), "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": C_h.numel() * 4, "ms_per_step": ms, "steps": steps,
            "windows_ms_per_step": windows,
            "pipelining": f"{nsets} device buffer sets; copies in, GEMM, copies out on three streams; "
                          f"median of 3 windows of {steps} steps"}


def run_ours(args, rank, world):
    import torch
    import torch.distributed as dist
    from dense_fp32_gemm_06_gb300 import binding, inputs
    import oracle

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    path = {"auto": binding.PATH_AUTO, "ffma": binding.PATH_FFMA, "tf32x3": binding.PATH_TF32X3}[args.path]
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    p, workload_text = load_problem(args)
    A_h = torch.from_numpy(p.A).pin_memory()
    B_h = torch.from_numpy(p.B).pin_memory()
    C_h = torch.from_numpy(p.C0).pin_memory()
    A = A_h.cuda()
    B = B_h.cuda()
    C = C_h.cuda()
    torch.cuda.synchronize()
    operand_bytes = 4 * (A.numel() + B.numel() + C.numel())
    # inputs smaller than twice L2 are flushed (a 2 x L2 write) before every timed launch
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda") \
        if operand_bytes < 2 * L2_BYTES else None
    flush = (lambda: flush_buf.fill_(1.0)) if flush_buf is not None else None

    # the plan of the call below on this device (its measured cluster capacity)
    st, plan = binding.plan(p.m, p.n, p.k, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                            C.data_ptr(), p.ldc, path=path, num_sms=0)
    if st:
        raise SystemExit(f"plan failed: {binding.status_string(st)}")

    def step():
        s = binding.sgemm_raw(p.m, p.n, p.k, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                              C.data_ptr(), p.ldc, sptr, path)
        if s:
            raise SystemExit(f"sgemm failed: {binding.status_string(s)}")

    # quick self-check on sampled outputs before timing
    step()
    torch.cuda.synchronize()
    rows, cols = inputs.sample_indices(p.m, p.n, 256, seed=p.seed + 2000)
    R, E = oracle.problem_f64_sampled(p, rows, cols)
    got = C.cpu().numpy()[rows, cols]
    ok, worst, _ = oracle.within_tolerance(got, R, E, p.beta, p.C0[rows, cols] if p.beta != 0 else None)
    # beta != 0 accumulates into C: restore C0 before timing
    C.copy_(C_h)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    sampler = ClockSampler(dev)
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    per = []
    ev0.record(stream)
    for _ in range(args.steps):
        if flush is not None:
            flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        per.append((a, b))
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    launch_ms = [a.elapsed_time(b) for a, b in per]
    # with L2 flushes between launches the bracket includes the flushes, so
    # the timed region is the sum of the launches' own event intervals
    total_ms = sum(launch_ms) if flush is not None else ev0.elapsed_time(ev1)
    total_ms = max_over_ranks(total_ms, world)
    value = tflops(p, total_ms / args.steps, world)
    med_ms = statistics.median(launch_ms)
    mean_ms = sum(launch_ms) / len(launch_ms)

    # ---- roofline of the dominant kernel
    mhz = clocks.get("sm_mhz") or 2070.0
    ffma_peak = sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
    ffma_basis = (f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 FLOP x {mhz:.0f} MHz "
                  f"(median SM clock sampled during the timed region)")
    if plan["path"] == binding.PATH_FFMA:
        # the step is the one FFMA kernel (or the C = beta*C kernel)
        launches_per_step = 1
        achieved = tflops(p, mean_ms)
        roof = {"bound": "alu", "kernel": "ffma_sgemm_kernel", "achieved": achieved, "peak": ffma_peak,
                "unit": "TFLOP/s", "frac": achieved / ffma_peak, "peak_basis": ffma_basis,
                "traffic": traffic_record("ffma", p.m * p.n * p.k)}
    else:
        ka = binding.ka_of(p.k)
        a_raw, b_raw = bool(plan["a_in_kernel"]), bool(plan["b_in_kernel"])
        # the GEMM, plus one split launch when an operand cannot be read as stored
        launches_per_step = 1 if (a_raw and b_raw) else 2
        if a_raw and b_raw:
            # the call is the GEMM kernel alone (no split pass, no scratch)
            gemm_ms = mean_ms
            gemm_timing = "the whole call: one launch of the GEMM kernel (CUDA events per launch)"
        else:
            # the GEMM's time is the call's minus the split passes it runs,
            # timed alone through the public split entry points
            a_hi = a_lo = b_hi = b_lo = None
            if not a_raw:
                a_hi = torch.empty(p.m * ka, device="cuda")
                a_lo = torch.empty_like(a_hi)
            if not b_raw:
                b_hi = torch.empty(p.n * ka, device="cuda")
                b_lo = torch.empty_like(b_hi)

            def splits_only():
                if not a_raw:
                    binding.tf32x3_split_a(A[:, :p.k], a_hi, a_lo)
                if not b_raw:
                    binding.tf32x3_split_b(B[:, :p.n], b_hi, b_lo)

            for _ in range(3):
                splits_only()
            split_ms = device_time_ms(splits_only, stream, 20, flush=flush)
            gemm_ms = mean_ms - split_ms
            gemm_timing = ("whole call minus the split pass over " +
                           " and ".join(x for x, raw in (("A", a_raw), ("B", b_raw)) if not raw) +
                           " timed alone (device time of 20 back-to-back launches, CUDA events)")
            del a_hi, a_lo, b_hi, b_lo
        achieved = tflops(p, gemm_ms)
        mp = measured_peaks()
        bf16 = (mp or {}).get("bf16_tflops", 1900.0)
        tf32 = bf16 * NOMINAL_TF32_OVER_BF16
        family = tc_family(a_raw, b_raw)
        # an A that TMA cannot read as one tensor is read in four row phases
        a_phased = a_raw and not plan["trans"] and (p.lda % 4 != 0 or A.data_ptr() % 16 != 0)
        traits = [t for t, on in (("A read raw" + (" in row phases" if a_phased else ""), a_raw), ("B read raw", b_raw),
                                  ("CTA pairs", plan["pair"]), ("transposed tiles", plan["trans"]),
                                  ("stream-K", plan["stream_k"] > 0), (f"split-K {plan['split_k']}",
                                                                       plan["split_k"] > 1)) if on]
        roof = {"bound": "tensor", "kernel": "tf32x3_gemm_kernel" + (f"<{', '.join(traits)}>" if traits else ""),
                "achieved": achieved, "peak": tf32 / 3,
                "unit": "TFLOP/s", "frac": achieved / (tf32 / 3),
                "peak_basis": f"TF32 dense peak / 3 (three TF32 products per FP32 product); TF32 peak = "
                              f"measured bf16 {bf16} TFLOP/s ({'of measured' if mp else 'of fallback'}) x "
                              f"nominal tf32/bf16 ratio 1.1/2.25 = {tf32:.1f} TFLOP/s",
                "gemm_kernel_ms": gemm_ms, "gemm_kernel_timing": gemm_timing,
                "split_kernels_ms": mean_ms - gemm_ms, "tensor_pipe_tflops": 3 * achieved,
                "traffic": traffic_record(family, p.m * p.n * p.k)}
    roof["ffma_peak_tflops"] = ffma_peak
    roof["value_over_ffma_peak"] = value / world / ffma_peak

    # ---- end to end through the same C call, host buffers, copies timed
    out_h = torch.empty_like(C_h).pin_memory()

    def step_on(A_, B_, C_, stream_ptr):
        s_ = binding.sgemm_raw(p.m, p.n, p.k, p.alpha, A_.data_ptr(), p.lda, B_.data_ptr(), p.ldb, p.beta,
                               C_.data_ptr(), p.ldc, stream_ptr, path)
        if s_:
            raise SystemExit(f"sgemm failed: {binding.status_string(s_)}")

    e2e = None
    if args.e2e_steps > 0:
        e2e = time_e2e(p, world, (A_h, B_h, C_h, out_h), step_on, args.e2e_steps)

    # ---- secondary size (2048^3 fits in L2: flushed before every launch)
    secondary = None
    if not args.no_secondary and args.workload != SECONDARY and not args.shape:
        q = inputs.workload(SECONDARY)
        qA = torch.from_numpy(q.A).cuda()
        qB = torch.from_numpy(q.B).cuda()
        qC = torch.from_numpy(q.C0).cuda()
        scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")

        def qstep():
            s = binding.sgemm_raw(q.m, q.n, q.k, q.alpha, qA.data_ptr(), q.lda, qB.data_ptr(), q.ldb, q.beta,
                                  qC.data_ptr(), q.ldc, sptr, path)
            if s:
                raise SystemExit(f"sgemm failed: {binding.status_string(s)}")

        for _ in range(5):
            qstep()
        ms = time_launches(qstep, stream, 30, flush=lambda: scratch.fill_(1.0))
        qmed = statistics.median(ms)
        secondary = {"workload": WORKLOAD_TEXT[SECONDARY], "value": tflops(q, qmed), "unit": "TFLOPS",
                     "median_ms": qmed, "launches": len(ms), "l2": "flushed (2 x L2 write) before every launch"}
        del scratch

    # ---- the CUDA-core FFMA path on the same workload, for comparison
    ffma = None
    if plan["path"] != binding.PATH_FFMA and not args.no_secondary:
        def ffma_step():
            s = binding.sgemm_raw(p.m, p.n, p.k, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                                  C.data_ptr(), p.ldc, sptr, binding.PATH_FFMA)
            if s:
                raise SystemExit(f"sgemm failed: {binding.status_string(s)}")
        for _ in range(2):
            ffma_step()
        torch.cuda.synchronize()
        fs = ClockSampler(dev)
        time.sleep(0.3)
        f0 = time.time()
        # about 1.5 s of FFMA work, at least 10 launches
        count = max(10, int(1.5 / max(1e-6, flops(p) / 60e12)))
        fm = time_launches(ffma_step, stream, count, flush=flush)
        f1 = time.time()
        time.sleep(0.25)
        fs.stop()
        fclk = fs.summary(f0, f1)
        f_ms = sum(fm) / len(fm)
        fmhz = fclk.get("sm_mhz") or 2070.0
        fpeak = sms * FP32_LANES_PER_SM * 2 * fmhz * 1e6 / 1e12
        ffma = {"value": tflops(p, f_ms), "unit": "TFLOPS", "ms": f_ms, "launches": len(fm),
                "frac_of_ffma_peak": tflops(p, f_ms) / fpeak, "ffma_peak_tflops": fpeak, "clocks": fclk}

    # ---- side reference: cuBLAS FP32 SGEMM (torch.matmul with TF32 off) on
    # the same operands; never on the library's path, reported for context
    cublas = None
    if not args.no_secondary and not args.shape:
        cublas = cublas_side_reference(p, A, B, C, stream, flush, sms)

    # ---- CPU baseline: the oracle on a bounded slab of the same workload
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tf, nrows, secs, threads = oracle_sample(p, args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
               "sample": f"output rows 0..{nrows - 1} of the workload ({nrows} x {p.n} outputs, "
                         f"k = {p.k}, FP64), {secs:.1f} s"}

    # ---- CPU baseline on the small configurations: the whole oracle, timed
    cpu_configs = None
    if rank == 0 and not args.no_cpu_baseline and not args.shape:
        cpu_configs = oracle_full_small()

    if rank == 0:
        path_name = {binding.PATH_FFMA: "ffma", binding.PATH_TF32X3: "tf32x3"}.get(plan["path"], "?")
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "median_ms": med_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "tf32x3" if plan["path"] == binding.PATH_TF32X3 else "f32",
            "data": "synthetic (seeded splitmix64)",
            "config": {"workload": workload_text, "path": path_name, "kernel_plan": plan,
                       "l2": ("flushed (2 x L2 write) before every timed launch; value from the launches' "
                              "own event intervals") if flush is not None else
                             f"inputs larger than L2 ({operand_bytes / 2**20:.0f} MB of A, B, C vs 129 MB)",
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "check": {"sampled_outputs": int(len(rows)), "within_tolerance": ok,
                                 "worst_ratio": worst}},
            "roofline": roof,
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": args.steps * launches_per_step,
            "cpu_baseline": cpu,
            "cpu_baseline_full": cpu_configs,
            "secondary": secondary,
            "ffma_path": ffma,
            "cublas_side_reference": cublas,
        }
        print(json.dumps(line), flush=True)
    return 0


def run_reduce(args, rank, world):
    """reduce_sum_f32 on N uniform[-1, 1) floats resident in HBM: CUDA events
    over `steps` launches on the launching stream after `warmup`; HBM-bound
    (4N bytes read per call), against the measured copy bandwidth."""
    import torch
    from dense_fp32_gemm_06_gb300 import binding
    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    n = args.reduce
    stream = torch.cuda.current_stream()
    x = torch.empty(n, device="cuda").uniform_(-1, 1)
    out = torch.empty(1, device="cuda")

    def step():
        st = binding.reduce_sum_raw(x.data_ptr(), n, out.data_ptr(), stream.cuda_stream)
        if st:
            raise SystemExit(f"reduce failed: {binding.status_string(st)}")

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev)
    time.sleep(0.1)
    t0 = time.time()
    ms = time_launches(step, stream, args.steps)
    t1 = time.time()
    time.sleep(0.05)
    sampler.stop()
    mean = sum(ms) / len(ms)
    s64 = x.double().sum().item()
    gbs = 4.0 * n / (mean * 1e-3) / 1e9
    world_gbs = gbs * world
    mp = measured_peaks()
    peak = (mp or {}).get("hbm_gbs", 6800.0)
    line = {"metric": "reduce_sum_f32 GB/s (HBM read of x)", "value": world_gbs, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean, "median_ms": statistics.median(ms),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (torch uniform[-1,1))",
            "config": {"workload": f"reduce_sum_f32 of {n} floats ({4 * n / 2**20:.0f} MiB, larger than L2)",
                       "relative_difference_to_fp64_sum": abs(out.item() - s64) / max(1e-30, x.abs().double().sum().item())},
            "roofline": {"bound": "hbm", "kernel": "reduce_sum_kernel", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "peak_basis": ("measured copy bandwidth (MEASURED_PEAKS.json), of measured"
                                                             if mp else "fallback 6800 GB/s, of fallback"),
                         "traffic": None},
            "clocks": sampler.summary(t0, t1), "gpu_launches": args.steps}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.reduce:
        return run_reduce(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    try:
        return run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
