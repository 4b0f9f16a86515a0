"""Throughput benchmark: MXFP8 rowwise+colwise cast of a 16384x16384 bf16
matrix on GB300, in GB/s of algorithmic traffic (bf16 input read + E4M3 codes
and E8M0 scales written), the byte accounting of torchao's cast_bench.py
(torchao PR #12 "Multiply with inverse scale in loop instead of dividing",
section "Performance").

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

One step = one mx_quantize_rowcol call over the whole 16384x16384 input
(already resident in HBM; the input is 512 MiB, larger than L2, so no flush
is needed between steps).  Under torchrun (N > 1) every rank quantizes its
own matrix (row panels of a larger one need no exchange), the steps are
bracketed by barriers and the slowest rank's time counts.  Rank 0 prints one
JSON line.  --impl reference times the scalar CPU oracle on the host cores
instead, on a bounded sample of the same workload per step.
"""
import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "MXFP8 cast GB/s (in+out bytes) and % of GB300 HBM peak at 16384x16384 bf16"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20

# --------------------------------------------------------------------------
# Byte accounting (algorithmic bytes per call)
# --------------------------------------------------------------------------


def mx_bytes(M, K, rowwise=True, colwise=True, dbias=False, gated=False):
    """bf16 input read + E4M3 codes + E8M0 scales written (+ fp32 dbias)."""
    read = M * K * 2 * (2 if gated else 1)
    per_dir = M * K + M * K // 32
    written = per_dir * (int(rowwise) + int(colwise)) + (K * 4 if dbias else 0)
    return read + written


def dgated_bytes(M, N, rowwise=True, colwise=True):
    """Gated backward: grad [M, N] and x [M, 2N] bf16 read, codes and scales
    of the [M, 2N] output written."""
    per_dir = 2 * M * N + 2 * M * N // 32
    return M * N * 2 + M * 2 * N * 2 + per_dir * (int(rowwise) + int(colwise))


def nvfp4_bytes(M, K, rowwise=True, colwise=True):
    """bf16 input + packed E2M1 codes + E4M3 scales, plus the fp32 tensor
    amax read and the fp32 global scale written."""
    per_dir = M * K // 2 + M * K // 16
    return M * K * 2 + per_dir * (int(rowwise) + int(colwise)) + 8


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The sources each timed kernel is built from; a recorded DRAM traffic figure
# counts only while these files are unchanged.
KERNEL_SOURCES = {
    "mx": ("mx_kernels.cu", "mxq_ptx.cuh", "mxq_internal.h"),
    "nvfp4": ("nvfp4_kernels.cu", "mxq_ptx.cuh", "mxq_internal.h"),
}


def kernel_source_sha(family="mx"):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, "fp4_quantization_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key, family="mx"):
    """DRAM bytes per launch from the committed ncu summary
    (profiles/traffic.json), if it was taken on the current kernel sources;
    else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(kernel_key)
    if not entry or entry.get("source_sha") != kernel_source_sha(family):
        return None
    return entry.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------
# Clock sampling (NVML through ctypes; read-only queries)
# --------------------------------------------------------------------------

_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
            0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
            0x100: "display_clock_setting"}


class ClockSampler:
    """Samples the SM clock and the clock-event reasons of one GPU every
    `period` seconds on a background thread (NVML queries only)."""

    def __init__(self, device_index, period=0.002):
        self.period = period
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        try:
            nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if nvml.nvmlInit_v2() != 0:
                return
            handle = ctypes.c_void_p()
            if nvml.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device_index), ctypes.byref(handle)) != 0:
                return
            self._reasons_fn = None
            for fn in ("nvmlDeviceGetCurrentClocksEventReasons",
                       "nvmlDeviceGetCurrentClocksThrottleReasons"):
                try:
                    self._reasons_fn = getattr(nvml, fn)
                    break
                except AttributeError:
                    continue
            self._nvml, self._handle = nvml, handle
            mx = ctypes.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
        except OSError:
            self._nvml = None

    def _run(self):
        clk = ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self._nvml.nvmlDeviceGetClockInfo(self._handle, 1, ctypes.byref(clk)) == 0:
                r = 0
                if self._reasons_fn is not None and self._reasons_fn(self._handle, ctypes.byref(reasons)) == 0:
                    r = int(reasons.value)
                self.samples.append((int(clk.value), r))
            time.sleep(self.period)

    def __enter__(self):
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._thread is not None:
            self._thread.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml unavailable" if self._nvml is None else "nvml"}
        mhz = [s for s, _ in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        names = [n for b, n in _REASONS.items() if bits & b and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": names,
                "samples": len(self.samples), "source": "nvml"}


# --------------------------------------------------------------------------
# Distributed plumbing (barrier + max over ranks only; no data exchange)
# --------------------------------------------------------------------------


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
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


def max_over_ranks(value, world):
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------


def to_device(bits, device):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(device)


def time_device(fn, steps, warmup, world, stream):
    """Run fn() warmup times, then time `steps` calls with CUDA events on
    `stream`, bracketed by barrier + synchronize.  Returns (total ms,
    per-call ms list, slowest-rank total ms)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    per_call = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total = starts[0].elapsed_time(ends[-1])
    return total, per_call, max_over_ranks(total, world)


# The pages' own cold-L2 kernel times for the same workload on GB200 (another
# GPU: context for the cold figure beside them, not a target).  TE PR #3291
# results tables: "specialized plain both 8192x28672", "generic dbias both
# 8192x8192", "NVFP4 2D quantize-transpose both 8192x8192".
PAGES_GB200_COLD_US = {
    "rowcol_8192x28672": 149.4,
    "dbias_rowcol_8192x8192": 52.5,
    "nvfp4_2d_rowtrans_given_amax_8192x8192": 50.1,
}


# Kernel launches per call of each row (the rest launch one kernel).
ROW_LAUNCHES = {"dbias_rowcol_8192x8192": 2, "dbias_dgelu_rowcol_8192x14336": 2,
                "nvfp4_rowtrans_16384x8192": 2}


def rows_measurements(mxq, device, steps, warmup, world, stream, peak, only=None, clock_index=0):
    """The other hot-path variants, each on its own workload (only the one
    named `only` when given), `steps` timed calls each."""
    out = {}
    cases = [
        # The headline workload itself, timed here only when named in `only`
        # (the default run times it as the headline).
        ("rowcol_16384x16384", lambda: synth.rowcol(),
         lambda x, o: mxq.mx_quantize_rowcol(x, mxq.ROWWISE | mxq.COLWISE, **o),
         mx_bytes(16384, 16384), {}),
        ("rowcol_8192x8192", lambda: synth.rowcol(M=8192, K=8192),
         lambda x, o: mxq.mx_quantize_rowcol(x, mxq.ROWWISE | mxq.COLWISE, **o),
         mx_bytes(8192, 8192), {}),
        ("rowcol_8192x28672", lambda: synth.rowcol(M=8192, K=28672),
         lambda x, o: mxq.mx_quantize_rowcol(x, mxq.ROWWISE | mxq.COLWISE, **o),
         mx_bytes(8192, 28672), {}),
        ("gemm_ready_rowcol_16384x16384", lambda: synth.rowcol(),
         lambda x, o: mxq.mx_quantize_rowcol(
             x, mxq.ROWWISE | mxq.COLWISE | mxq.SCALE_RCEIL | mxq.SCALE_SWIZZLED, **o),
         mx_bytes(16384, 16384), {}),
        ("dim1_colwise_16384x16384", lambda: synth.dim1(),
         lambda x, o: mxq.mx_quantize_rowcol(x, mxq.COLWISE, **o), mx_bytes(16384, 16384, rowwise=False),
         dict(q_col=None, s_col=None)),
        ("dbias_rowcol_8192x8192", lambda: synth.dbias(),
         lambda x, o: mxq.mx_quantize_rowcol(x, mxq.ROWWISE | mxq.COLWISE | mxq.DBIAS, **o),
         mx_bytes(8192, 8192, dbias=True), {}),
        ("swiglu_rowcol_8192x2x14336", lambda: synth.swiglu(),
         lambda x, o: mxq.mx_quantize_gated(x, mxq.ROWWISE | mxq.COLWISE, **o),
         mx_bytes(8192, 14336, gated=True), {}),
        ("gelu_rowcol_8192x14336", lambda: synth.gelu(),
         lambda x, o: mxq.mx_quantize_rowcol(x, mxq.ROWWISE | mxq.COLWISE | mxq.ACT_GELU_TANH, **o),
         mx_bytes(8192, 14336), {}),
        ("geglu_rowcol_8192x2x14336", lambda: synth.swiglu(),
         lambda x, o: mxq.mx_quantize_gated(x, mxq.ROWWISE | mxq.COLWISE | mxq.ACT_GELU_TANH, **o),
         mx_bytes(8192, 14336, gated=True), {}),
        ("dbias_dgelu_rowcol_8192x14336",
         lambda: (synth.gelu(seed=8), synth.gelu()),
         lambda x, o: mxq.mx_quantize_dact(x[0], x[1], mxq.ROWWISE | mxq.COLWISE | mxq.DBIAS
                                           | mxq.ACT_GELU_TANH, **o),
         mx_bytes(8192, 14336, gated=True, dbias=True), {}),
        ("dswiglu_rowcol_8192x14336",
         lambda: (synth.gelu(seed=9), synth.swiglu()),
         lambda x, o: mxq.mx_quantize_dgated(x[0], x[1], mxq.ROWWISE | mxq.COLWISE, **o),
         dgated_bytes(8192, 14336), {}),
        ("nvfp4_rowtrans_16384x8192", lambda: synth.nvfp4(),
         lambda x, o: mxq.nvfp4_quantize_transpose(x, mxq.ROWWISE | mxq.COLWISE, **o),
         nvfp4_bytes(16384, 8192), {}),
        ("nvfp4_rowtrans_given_amax_16384x8192", lambda: synth.nvfp4(),
         lambda x, o: mxq.nvfp4_quantize_transpose(x, mxq.ROWWISE | mxq.COLWISE, **o),
         nvfp4_bytes(16384, 8192), {}),
        ("nvfp4_2d_rowtrans_given_amax_16384x8192", lambda: synth.nvfp4(),
         lambda x, o: mxq.nvfp4_quantize_transpose(x, mxq.ROWWISE | mxq.COLWISE | mxq.NVFP4_2D,
                                                   **o),
         nvfp4_bytes(16384, 8192), {}),
        ("nvfp4_2d_rowtrans_given_amax_8192x8192", lambda: synth.nvfp4(M=8192, K=8192),
         lambda x, o: mxq.nvfp4_quantize_transpose(x, mxq.ROWWISE | mxq.COLWISE | mxq.NVFP4_2D,
                                                   **o),
         nvfp4_bytes(8192, 8192), {}),
        ("bf16_amax_16384x8192", lambda: synth.nvfp4(),
         lambda x, o: mxq.bf16_amax(x, **o), 16384 * 8192 * 2 + 4, {}),
    ]
    for name, gen, call, nbytes, _ in cases:
        if only is not None and name not in only.split(","):
            continue
        if only is None and name == "rowcol_16384x16384":
            continue
        data = gen()
        x = (tuple(to_device(d, device) for d in data) if isinstance(data, tuple)
             else to_device(data, device))
        first = call(x, {})                       # allocates the outputs once
        if name.startswith("bf16_amax"):
            keep = {"out": first}
        else:
            keep = dict(first)
        if "given_amax" in name:
            keep["amax"] = mxq.bf16_amax(x)
        elif name.startswith("nvfp4"):
            keep["workspace"] = torch.empty(16, dtype=torch.uint8, device=device)
        if name.startswith("dbias_rowcol"):
            keep["workspace"] = torch.empty(
                max(16, mxq.mxq_workspace_bytes(mxq.OP_ROWCOL, 8192, 8192, 7)), dtype=torch.uint8,
                device=device)
        if name.startswith("dbias_dgelu"):
            keep["workspace"] = torch.empty(
                max(16, mxq.mxq_workspace_bytes(mxq.OP_DACT, 8192, 14336, 7)), dtype=torch.uint8,
                device=device)
        with ClockSampler(clock_index) as clocks:
            total, per_call, _ = time_device(lambda: call(x, keep), steps, warmup, world, stream)
        # Device time per call (events around each call); the loop time per
        # call beside it also holds the host's time between calls, which
        # the shortest calls do not cover.  GB/s and the fraction of peak
        # use the median call.
        med_ms = statistics.median(per_call)
        gbs = nbytes / (med_ms * 1e-3) / 1e9
        launches = ROW_LAUNCHES.get(name, 1)
        out[name] = {"GB_per_s": round(gbs, 1), "us_per_call": round(med_ms * 1e3, 2),
                     "us_min": round(min(per_call) * 1e3, 2),
                     "us_mean": round(statistics.mean(per_call) * 1e3, 2),
                     "calls": steps,
                     "loop_us_per_call": round(total / steps * 1e3, 2),
                     "bytes_per_call": nbytes, "frac_of_hbm_peak": round(gbs / peak, 4),
                     "launches_per_call": launches, "clocks": clocks.summary()}
        if name.startswith("nvfp4_rowtrans_16"):
            out[name]["note"] = ("bytes exclude the tensor-amax pass (a second 256 MiB read), "
                                 "time includes it")
        if name in PAGES_GB200_COLD_US:
            cold_ms = cold_l2_measure(lambda: call(x, keep), 20, stream, device)
            out[name]["cold_us_per_call"] = round(cold_ms * 1e3, 2)
            out[name]["pages_gb200_cold_us"] = PAGES_GB200_COLD_US[name]
        if "given_amax" in name:
            out[name]["note"] = "tensor amax supplied by the caller: the quantize kernel alone"
            if name == "nvfp4_rowtrans_given_amax_16384x8192":
                out[name]["traffic"] = recorded_traffic("nvfp4_rowtrans_16384x8192", "nvfp4")
        del x, first, keep
        torch.cuda.empty_cache()
    return out


def copy_ceiling(device, steps, stream, elems=256 * 2 ** 20):
    """What plain copies of `elems` bf16 values (512 MiB in, 512 MiB out, close
    to the headline cast's 1.09 GB) reach on this GPU, timed with events
    (median and best over `steps` calls): torch's device-to-device copy (a
    memcpy, which ncu cannot capture) and torch's elementwise kernel on the
    same buffers (negation: one read and one write per element, a kernel ncu
    captures in the same units as the cast)."""
    a = torch.empty(elems, dtype=torch.bfloat16, device=device).normal_()
    b = torch.empty_like(a)
    nbytes = 2 * a.numel() * a.element_size()
    out = {"bytes_per_call": nbytes}
    for name, fn in (("memcpy", lambda: b.copy_(a)), ("elementwise_neg", lambda: torch.neg(a, out=b))):
        _, per_call, _ = time_device(fn, max(3, steps), 3, 1, stream)
        med = statistics.median(per_call)
        out[name] = {"us_per_call": round(med * 1e3, 2),
                     "GB_per_s": round(nbytes / (med * 1e-3) / 1e9, 1),
                     "best_GB_per_s": round(nbytes / (min(per_call) * 1e-3) / 1e9, 1)}
    return out


def cold_l2_measure(fn, steps, stream, device, flush_bytes=512 * 2 ** 20):
    """Median per-call time with L2 flushed before every call (a 512 MiB
    scratch buffer zeroed between calls, outside the timed events)."""
    scratch = torch.empty(flush_bytes, dtype=torch.uint8, device=device)
    times = []
    for _ in range(steps):
        scratch.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e))
    del scratch
    return statistics.median(times)


def e2e_measure(mxq, bits, device, steps, warmup, stream):
    """Same metric through the public API with host buffers: every step is
    one mx_quantize_rowcol_host call, which copies the input from pinned
    host memory to the device, quantizes it and copies every output back to
    pinned host memory (panels pipelined inside the call)."""
    M, K = bits.shape
    x_host = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    outs = mxq.mx_quantize_rowcol_host(x_host, mxq.ROWWISE | mxq.COLWISE)
    ws = torch.empty(max(256, mxq.mxq_workspace_bytes(mxq.OP_ROWCOL_HOST, M, K, 3)),
                     dtype=torch.uint8, device=device)

    def step():
        mxq.mx_quantize_rowcol_host(x_host, mxq.ROWWISE | mxq.COLWISE, workspace=ws, **outs)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    h2d = M * K * 2
    d2h = sum(v.numel() * v.element_size() for v in outs.values())
    return ms, h2d, d2h


def host_threads():
    """Host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def oracle_on_threads(bits, flags, threads):
    """The oracle as it stands, on `threads` host threads: row panels (multiples
    of 32 rows, so no block straddles two panels), one oracle call per
    panel (the ctypes call releases the GIL).  Returns seconds."""
    import concurrent.futures
    import oracle
    M = bits.shape[0]
    per = max(32, (M // threads) // 32 * 32)
    panels = [bits[r:r + per] for r in range(0, M, per)]
    oracle.mx_quantize(bits[:32], flags)    # load/build outside the timing
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as pool:
        t0 = time.perf_counter()
        list(pool.map(lambda p: oracle.mx_quantize(p, flags), panels))
        return time.perf_counter() - t0


def cpu_baseline(bits):
    """The oracle as it stands on the whole workload (the bench's own input),
    on every host core (row panels, one thread each) -- the same definition
    as the reference arm's step -- and, for context, on one thread over the
    first 1024 rows."""
    rows, K = bits.shape
    threads = host_threads()
    dt = oracle_on_threads(bits, 3, threads)
    dt1 = oracle_on_threads(bits[:1024], 3, 1) * (rows / 1024)
    gbs = mx_bytes(rows, K) / dt / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"all {rows} rows ({rows}x{K} bf16, the bench's input), rowwise+colwise, "
                      f"{dt:.2f} s on {threads} host threads (row panels)",
            "one_thread": {"value": round(mx_bytes(rows, K) / dt1 / 1e9, 4), "unit": "GB/s",
                           "sample": f"first 1024 rows on 1 thread, scaled x{rows / 1024:g}"}}


def gpu_arm(args):
    import fp4_quantization_gb300 as mxq

    world, rank, local = dist_setup()
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream()
    peak, peak_kind = measured_peaks()
    clock_index = local if world > 1 else int(os.environ.get("MXQ_NVML_INDEX", "0"))
    if args.only == "copy_ceiling":
        # The denominator's own kind of kernel (torch's device copy) on a
        # 512 MiB bf16 buffer: for profiling it beside the cast in the same
        # units.  Not part of the hot path.
        print(json.dumps({"only": args.only, "copy": copy_ceiling(device, args.steps, stream)}),
              flush=True)
        return
    if args.only:
        # One hot-path variant alone (profiling runs); no headline line.
        rows = rows_measurements(mxq, device, args.steps, args.warmup, world, stream, peak,
                                 only=args.only, clock_index=clock_index)
        if rank == 0:
            print(json.dumps({"only": args.only, "rows": rows}), flush=True)
        return
    M, K = args.M, args.K
    bits = synth.rowcol(M=M, K=K)
    x = to_device(bits, device)
    outs = mxq.mx_quantize_rowcol(x, mxq.ROWWISE | mxq.COLWISE)
    nbytes = mx_bytes(M, K)

    def step():
        mxq.mx_quantize_rowcol(x, mxq.ROWWISE | mxq.COLWISE, **outs)

    with ClockSampler(clock_index) as clocks:
        total_ms, per_call, total_max = time_device(step, args.steps, args.warmup, world, stream)
    avg_call_ms = statistics.mean(per_call)
    value = nbytes * world / (total_max * 1e-3 / args.steps) / 1e9
    achieved = nbytes / (avg_call_ms * 1e-3) / 1e9

    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_max / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16->e4m3+e8m0",
        "data": "synthetic: N(0,1) bf16, Philox seed 5",
        "config": {"workload": f"mxfp8_rowwise_colwise_{M}x{K}", "M": M, "K": K, "block": 32,
                   "directions": "rowwise+colwise", "parallelism": f"replicas x{world}",
                   "l2": f"input {M * K * 2 // 2**20} MiB > 129 MiB L2: no flush between steps"},
        "clocks": clocks.summary(),
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} hbm_gbs (copy, burst)", "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic(f"mx_rowcol_{M}x{K}"),
                     "kernel": "mx_cast_tile_kernel<rowwise|colwise>",
                     "bytes_per_launch": nbytes},
    }
    cold_ms = cold_l2_measure(step, max(10, min(args.steps, 50)), stream, device)
    result["cold_l2"] = {"us_per_call": round(cold_ms * 1e3, 2),
                         "GB_per_s": round(nbytes / (cold_ms * 1e-3) / 1e9, 1),
                         "how": "median over calls, 512 MiB zeroed before each (untimed)"}
    if args.rows:
        result["rows"] = rows_measurements(mxq, device, max(50, args.steps), max(3, args.warmup),
                                           world, stream, peak, clock_index=clock_index)
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 20))
        ms, h2d, d2h = e2e_measure(mxq, bits, device, e2e_steps, 3, stream)
        result["e2e"] = {"value": round(nbytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "ms_per_step": round(ms, 4), "steps": e2e_steps}
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(bits)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# --------------------------------------------------------------------------
# Reference arm: the oracle on the host cores
# --------------------------------------------------------------------------


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    K = 16384
    budget_s = 90.0
    threads = host_threads()
    per_row_s = 16384 * 2 / 12e6 / threads  # about 12 M elements/s per thread and direction pair
    rows = int(budget_s / (args.steps + args.warmup) / per_row_s) // 32 * 32
    rows = max(32, min(rows, 16384))
    bits = synth.rowcol(M=rows, K=K)
    for _ in range(args.warmup):
        oracle_on_threads(bits, 3, threads)
    dt = sum(oracle_on_threads(bits, 3, threads) for _ in range(args.steps))
    nbytes = mx_bytes(rows, K)
    gbs = nbytes * args.steps / dt / 1e9
    sample = (f"first {rows} of 16384 rows ({rows}x{K} bf16) per step, rowwise+colwise, "
              f"{threads} host threads (row panels)")
    print(json.dumps({
        "impl": "reference",
        "metric": METRIC,
        "value": round(gbs, 5),
        "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16->e4m3+e8m0",
        "data": "synthetic: N(0,1) bf16, Philox seed 5",
        "config": {"workload": "mxfp8_rowwise_colwise_16384x16384", "M": 16384, "K": K,
                   "block": 32, "directions": "rowwise+colwise"},
        "cpu_baseline": {"value": round(gbs, 5), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--rows", dest="rows", action="store_true", default=True,
                   help="also time the other hot-path variants (default)")
    p.add_argument("--no-rows", dest="rows", action="store_false")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--only", default=None,
                   help="time just these variants of the 'rows' object, comma-separated "
                        "(profiling runs)")
    p.add_argument("--M", type=int, default=16384,
                   help="rows of the timed cast (16384 for the headline number)")
    p.add_argument("--K", type=int, default=16384, help="columns of the timed cast")
    args = p.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
