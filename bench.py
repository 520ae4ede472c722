"""Benchmark of the tiled GEMM (+ReLU) on one GB300 per process.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl tl|reference] [--no-cpu-baseline] [--no-e2e]

One step is one call of the C ABI (tl_gemm) on one seeded synthetic input set of
the workload: the whole hot path (TMA producer, tcgen05 MMA, ReLU/cast epilogue,
TMA store) in one persistent kernel launch.  Inputs are resident in HBM before the
timed region.  Between timed steps the inputs rotate over enough independent sets
that the working set exceeds twice the L2 cache, so every step reads its operands
from HBM (or the operands alone are larger than L2).

Prints ONE JSON line (rank 0): the metric (TFLOP/s), the roofline of the GEMM
kernel against the measured peaks, the CPU oracle's rate on the host cores, the
end-to-end rate from pinned host buffers, and the SM clocks seen during the run.

With N > 1 (torchrun), every rank runs the same workload on its own GPU: the path
has no exchange step, so the ranks are replicas (weak scaling) and only the timing
barrier and the max-over-ranks reduction use torch.distributed.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

L2_BYTES = 126 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["tiled_gemm_gb300/csrc/gemm_kernel.cuh", "tiled_gemm_gb300/csrc/sm103_ptx.cuh",
                  "tiled_gemm_gb300/csrc/attn_kernel.cuh", "tiled_gemm_gb300/csrc/mx_kernel.cuh",
                  "tiled_gemm_gb300/csrc/tl_gemm.cu"]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on these sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    entry = table.get(workload)
    if not entry or entry.get("kernel_source_hash") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


def rotation_sets(bytes_per_set: int) -> int:
    """Input sets the timed steps rotate over, so that the working set exceeds twice the
    L2 cache (1 when one set alone does)."""
    return 1 if bytes_per_set >= 2 * L2_BYTES else int(math.ceil(2 * L2_BYTES / bytes_per_set))


def l2_note(bytes_per_set: int) -> str:
    rot = rotation_sets(bytes_per_set)
    if rot == 1:
        return "operands larger than 2x L2"
    return f"inputs rotate over {rot} sets ({rot * bytes_per_set / 2**20:.0f} MiB > 2x L2)"


def max_over_ranks(x: float, dist, device) -> float:
    """The largest value of x over all ranks (x itself without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sig4(x: float) -> float:
    """x to 4 significant figures (the oracle's rates are far below 1 TFLOP/s, where a
    fixed number of decimals would keep too few digits)."""
    return float(f"{x:.4g}")


def whole_job_tflops(flops_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Throughput of the whole job: every rank ran `steps` steps; the slowest rank's time."""
    return flops_per_step * steps * world / (max_ms * 1e-3) / 1e12


# Dense 8-bit tensor throughput over 16-bit on this part (nominal 4.5 vs 2.25 PFLOP/s):
# the 8-bit peak is the measured bf16 peak times this ratio.
FP8_OVER_BF16 = 2.0


def tensor_peak_scale(w) -> float:
    return FP8_OVER_BF16 if getattr(w, "fp8", False) else 1.0


def is_hbm_bound(w: workloads.Workload, peaks: dict) -> bool:
    ridge = tensor_peak_scale(w) * peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    return w.flops / w.bytes_moved < ridge


def roofline(w, avg_launch_ms: float, peaks: dict, peaks_src: str, clocks, attn: bool) -> dict:
    """The dominant kernel against its roofline: algorithmic flops (or bytes, for a
    product under the ridge point) per launch over the average launch time, and the
    fraction of the measured peak.  fp16 and bf16 share the dense tensor rate; 8-bit
    operands take it times FP8_OVER_BF16.  The sustained figure (cuBLAS looping under
    the power cap) applies when the timed region ran under the power cap (sw_power_cap
    seen in the clock samples); otherwise the burst one."""
    hbm = False if attn else is_hbm_bound(w, peaks)
    capped = "sw_power_cap" in ((clocks or {}).get("reasons") or [])
    if hbm:
        achieved = w.bytes_moved / (avg_launch_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s"}
    else:
        achieved = w.flops / (avg_launch_ms * 1e-3) / 1e12
        peak = tensor_peak_scale(w) * peaks["bf16_tflops_sustained" if capped else "bf16_tflops"]
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                "unit": "TFLOP/s"}
    roof["frac"] = round(achieved / peak, 4)
    roof["peak_source"] = (f"{peaks_src} ({'copy' if hbm else 'sustained, power cap seen' if capped else 'burst'})"
                           + (" bf16 x 2 for 8-bit operands" if tensor_peak_scale(w) > 1 and not hbm
                              else ""))
    if not hbm:
        roof["frac_of_burst"] = round(achieved / (tensor_peak_scale(w) * peaks["bf16_tflops"]), 4)
    return roof


class ClockSampler:
    """nvidia-smi clock/throttle samples every 50 ms while the timed region runs (the
    fallback when NVML cannot be loaded in-process)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="tl_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which: str) -> None:
        """Start of the pre-heat, start or end of the timed region (the nvidia-smi record
        keeps every sample)."""

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return dict(summarise_clocks(lines), source="nvidia-smi every 50 ms")


# NVML clock-event reason bits (nvmlClocksEventReason*) that the record names
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


def nvml_reason_names(mask: int) -> set:
    return {name for bit, name in NVML_REASONS.items() if mask & bit}


class NvmlClockSampler:
    """SM clock, power and clock-event reasons read in-process through NVML every
    `period_s` (read-only queries: nothing on the GPU is changed).  Samples are kept
    between mark("start") and mark("end"); a timed region too short for `min_samples`
    samples takes, in addition, the last samples of the pre-heat replays that run back to
    back before it (from mark("preheat") on: the same graphs, the GPU never idle)."""

    def __init__(self, uuid: str | None, pci_bus_id: str | None, index: int,
                 period_s: float = 0.001, min_samples: int = 5):
        import ctypes
        import threading
        self._ct = ctypes
        self._threading = threading
        self.period_s = period_s
        self.min_samples = min_samples
        self.samples = []            # (host time, sm MHz, power W, reason mask)
        self.window = [None, None]
        self.preheat = None
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.handle = ctypes.c_void_p()
        found = False
        for key in ([f"GPU-{uuid}", uuid] if uuid else []):
            if key and self.lib.nvmlDeviceGetHandleByUUID(
                    ctypes.c_char_p(key.encode()), ctypes.byref(self.handle)) == 0:
                found = True
                break
        if not found and pci_bus_id:
            found = self.lib.nvmlDeviceGetHandleByPciBusId_v2(
                ctypes.c_char_p(pci_bus_id.encode()), ctypes.byref(self.handle)) == 0
        if not found:
            if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index),
                                                      ctypes.byref(self.handle)) != 0:
                raise OSError("no NVML handle for the device")
        self.matched = "uuid" if found and uuid else ("pci" if found else "index")
        self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_mhz = (float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(
            self.handle, ctypes.c_int(1), ctypes.byref(mx)) == 0 else None)
        self._stop = threading.Event()
        self._thread = None

    def _read(self):
        ct = self._ct
        clk, mw, reasons = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        ok = self.lib.nvmlDeviceGetClockInfo(self.handle, ct.c_int(1), ct.byref(clk)) == 0
        pw = self.lib.nvmlDeviceGetPowerUsage(self.handle, ct.byref(mw)) == 0
        rs = self._reasons(self.handle, ct.byref(reasons)) == 0
        if ok:
            self.samples.append((time.perf_counter(), float(clk.value),
                                 mw.value / 1000.0 if pw else None,
                                 int(reasons.value) if rs else 0))

    def _run(self):
        while not self._stop.is_set():
            self._read()
            time.sleep(self.period_s)

    def start(self):
        self._thread = self._threading.Thread(target=self._run, daemon=True)
        self._thread.start()

    def mark(self, which: str) -> None:
        now = time.perf_counter()
        if which == "preheat":
            self.preheat = now
        else:
            self.window[0 if which == "start" else 1] = now

    def stop(self) -> dict:
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=5)
        self.lib.nvmlShutdown()
        picked, n_timed, lead_ms = clock_window([s[0] for s in self.samples], self.preheat,
                                                self.window[0], self.window[1],
                                                self.min_samples)
        rec = summarise_samples([(self.samples[i][1], self.max_mhz, self.samples[i][2],
                                  nvml_reason_names(self.samples[i][3])) for i in picked])
        rec["timed_samples"] = n_timed
        rec["source"] = f"NVML every {self.period_s * 1e3:.0f} ms ({self.matched})"
        if lead_ms > 0:
            rec["source"] += (f"; timed region plus the last {lead_ms:.1f} ms of the "
                              "pre-heat replays right before it")
        return rec


def clock_window(times, t_pre, t0, t1, min_samples: int):
    """Indices of the clock samples that describe the timed region [t0, t1]: the samples
    inside it, and, if they are fewer than min_samples, as many of the latest samples
    taken since t_pre (the start of the back-to-back pre-heat) as make up the count.
    Returns (indices, samples inside the region, ms of pre-heat taken before t0)."""
    inside = [i for i, t in enumerate(times)
              if (t0 is None or t >= t0) and (t1 is None or t <= t1)]
    lead = []
    if len(inside) < min_samples and t0 is not None and t_pre is not None:
        before = [i for i, t in enumerate(times) if t_pre <= t < t0]
        lead = before[max(0, len(before) - (min_samples - len(inside))):]
    lead_ms = (t0 - times[lead[0]]) * 1e3 if lead else 0.0
    return lead + inside, len(inside), lead_ms


def clock_sampler(dev_index: int):
    """An NVML sampler for the CUDA device, or the nvidia-smi one if NVML is missing."""
    uuid = pci = None
    try:
        import torch
        props = torch.cuda.get_device_properties(dev_index)
        u = getattr(props, "uuid", None)
        uuid = str(u) if u is not None else None
        if hasattr(props, "pci_bus_id"):
            pci = (f"{getattr(props, 'pci_domain_id', 0):08x}:{props.pci_bus_id:02x}:"
                   f"{getattr(props, 'pci_device_id', 0):02x}.0")
    except Exception:
        pass
    try:
        return NvmlClockSampler(uuid, pci, dev_index)
    except (OSError, AttributeError):
        return ClockSampler(f"GPU-{uuid}" if uuid else str(dev_index))


def summarise_samples(samples) -> dict:
    """Median SM clock over the busy samples (above half the highest), the highest clock
    limit and power seen, and every throttle reason active in any sample.  Each sample
    is (SM MHz, max SM MHz or None, power W or None, set of reason names)."""
    if not samples:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    sm = [s[0] for s in samples]
    smax = [s[1] for s in samples if s[1] is not None]
    power = [s[2] for s in samples if s[2] is not None]
    reasons = set().union(*[s[3] for s in samples])
    busy = [s for s in sm if s > 0.5 * max(sm)] or sm
    return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax) if smax else None,
            "power_w_max": max(power) if power else None, "samples": len(sm),
            "reasons": sorted(reasons)}


def summarise_clocks(lines) -> dict:
    """summarise_samples over `nvidia-smi --format=csv,noheader,nounits` rows of
    ClockSampler.QUERY (unparsable rows are skipped)."""
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    samples = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm, smax, power = float(parts[1]), float(parts[2]), float(parts[3])
        except ValueError:
            continue
        samples.append((sm, smax, power,
                        {n for n, v in zip(names, parts[5:9]) if v.lower() == "active"}))
    return summarise_samples(samples)


# ------------------------------------------------------------------ CPU oracle ----

def oracle_rate(w: workloads.Workload, a_cpu, b_cpu, budget_s: float, threads: int):
    """Oracle TFLOP/s on whole-row slices of the workload, repeated for ~budget_s."""
    import oracle
    oracle.build()
    rows = max(1, min(w.M, threads))            # one output row per thread to start
    done_flops, elapsed, reps = 0, 0.0, 0
    a_rows = a_cpu if w.trans_a else None
    while elapsed < budget_s:
        if w.trans_a:
            sl_a, M_s = a_rows[:, :rows].contiguous(), rows
            lda = rows
        else:
            sl_a, M_s = a_cpu[:rows].contiguous(), rows
            lda = w.K
        t0 = time.perf_counter()
        if w.fp8:
            oracle.gemm_fp8(sl_a, b_cpu, M_s, w.N, w.K, lda=lda, a_fmt=w.dtype, b_fmt=w.b_fmt,
                            out_dtype=w.c_dtype, alpha=w.alpha, trans_a=w.trans_a,
                            trans_b=w.trans_b, relu=w.relu, threads=threads)
        else:
            oracle.gemm(sl_a, b_cpu, M_s, w.N, w.K, lda=lda, dtype=w.dtype,
                        trans_a=w.trans_a, trans_b=w.trans_b, relu=w.relu, threads=threads)
        dt = time.perf_counter() - t0
        elapsed += dt
        done_flops += 2 * M_s * w.N * w.K
        reps += 1
        if dt < budget_s / 20 and rows < w.M:
            rows = min(w.M, rows * 2)
    return done_flops / elapsed / 1e12, elapsed, done_flops, rows, reps


def oracle_rate_mx(w: workloads.MxWorkload, a_cpu, b_cpu, sa_cpu, budget_s: float, sb_cpu,
                   threads: int):
    """Oracle TFLOP/s of the block-scaled product on whole-row slices, for ~budget_s."""
    import oracle
    oracle.build()
    rows = max(1, min(w.M, threads))
    done_flops, elapsed, reps = 0, 0.0, 0
    while elapsed < budget_s:
        t0 = time.perf_counter()
        oracle.gemm_mx(a_cpu[:rows].contiguous(), b_cpu, sa_cpu[:rows].contiguous(), sb_cpu,
                       rows, w.N, w.K, a_fmt=w.a_fmt, b_fmt=w.b_fmt, out_dtype=w.out_dtype,
                       sfa_ld=w.sf_ld, sfb_ld=w.sf_ld, relu=w.relu, threads=threads)
        dt = time.perf_counter() - t0
        elapsed += dt
        done_flops += 2 * rows * w.N * w.K
        reps += 1
        if dt < budget_s / 20 and rows < w.M:
            rows = min(w.M, rows * 2)
    return done_flops / elapsed / 1e12, elapsed, done_flops, rows, reps


# ------------------------------------------------------------------ GPU arm ----

def graph_chunks(steps: int, rot: int, max_calls: int = 64, one_graph_max: int = 4096):
    """Split `steps` consecutive calls into the CUDA graphs of the timed region.

    Returns [(first step, calls, reuse)].  Up to one_graph_max steps: one graph of all of
    them (no graph boundary between calls).  More steps: one graph of G calls (G a
    multiple of the rotation, so every replay walks the same input sets in order)
    replayed steps // G times (reuse = True marks replays of that first graph), then the
    remainder."""
    if steps <= 0:
        return []
    if steps <= one_graph_max:
        return [(0, steps, False)]
    G = rot * max(1, math.ceil(max_calls / rot))
    n_full, rem = divmod(steps, G)
    chunks = [(i * G, G, i > 0) for i in range(n_full)]
    if rem:
        chunks.append((n_full * G, rem, False))
    return chunks


def percentile(xs, q: float) -> float:
    """Linear-interpolation percentile (q in [0, 100]) of a non-empty list."""
    s = sorted(xs)
    pos = (len(s) - 1) * q / 100.0
    lo = int(math.floor(pos))
    hi = min(lo + 1, len(s) - 1)
    return s[lo] + (s[hi] - s[lo]) * (pos - lo)


def spread_of(chunk_ms, chunks) -> dict:
    """Per-call time of each timed sequence (its events' interval over its calls): min,
    p10, p50, p90 and max over the sequences of the largest size (a shorter remainder is
    left out, so that every figure averages the same number of calls)."""
    size = max(c[1] for c in chunks)
    per_call = [ms / c[1] for ms, c in zip(chunk_ms, chunks) if c[1] == size]
    return {"chunks": len(per_call), "calls_per_chunk": size,
            "ms_per_call": {"min": round(min(per_call), 6),
                            "p10": round(percentile(per_call, 10), 6),
                            "p50": round(percentile(per_call, 50), 6),
                            "p90": round(percentile(per_call, 90), 6),
                            "max": round(max(per_call), 6)}}


def spread_line(spread, flops: int):
    """The spread record with the throughput at each per-call time (TFLOP/s; the
    slowest chunk gives the lowest rate)."""
    if not spread:
        return None
    ms = spread["ms_per_call"]
    return dict(spread, tflops={k: round(flops / (v * 1e-3) / 1e12, 1) for k, v in ms.items()})


def timed_graph_steps(args, step, rot: int, stream, dist, dev, tl, preheat_s: float = 2.0):
    """Warm-up, then exactly args.steps calls of step(i) replayed as CUDA graphs, timed
    with events on `stream` between barriers; returns (max-over-ranks ms, clocks,
    spread).

    Before the timed region the graphs are replayed, untimed, for about preheat_s, so
    that the timed steps run at the clock the GPU settles at under this load (for the
    large products, the power cap) rather than at the first milliseconds' boost."""
    import torch

    w0 = torch.cuda.Event(enable_timing=True)
    w1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            if i == args.warmup - 2:
                w0.record(stream)
            step(i)
        w1.record(stream)
    torch.cuda.synchronize()
    status, word = tl.tl_device_status(reset=True)
    if status != tl.TL_OK:
        raise RuntimeError(f"device-side wait gave up during warm-up: {word:#x}")
    step_ms = max(w0.elapsed_time(w1) / 2.0, 1e-3)
    if args.steps <= 0:
        # default: a timed region of ~1.5 s
        args.steps = int(min(200000, max(50, math.ceil(1500.0 / step_ms))))
        args.steps = int(max_over_ranks(float(args.steps), dist, dev))

    # The timed steps run as CUDA-graph replays of consecutive library calls (one call
    # per step, inputs rotating as in eager mode), so host-side launch cost does not
    # hide the device time of small problems.  Exactly args.steps calls are timed.
    chunks = graph_chunks(args.steps, rot)

    def capture(first, n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(first, first + n):
                step(i)
        return g

    graphs = []
    for first, n, reuse in chunks:
        graphs.append(graphs[0] if reuse else capture(first, n))
    # The pre-heat graph walks every input set once, in order, so that the first timed
    # call finds its set as cold as every later one.
    G = rot * max(1, math.ceil(64 / rot))
    pre = graphs[0] if chunks[0][1] == G else capture(0, G)
    distinct = list({id(g): g for g in graphs + [pre]}.values())
    with torch.cuda.stream(stream):
        for g in distinct:                     # one untimed replay of each graph
            g.replay()
    torch.cuda.synchronize()
    # pre-heat: untimed replays, back to back with the timed ones
    reps = int(min(100000, max(1, math.ceil(preheat_s * 1e3 / (step_ms * G)))))
    if preheat_s <= 0:
        reps = 1

    clocks = clock_sampler(torch.cuda.current_device())
    clocks.start()
    events = [torch.cuda.Event(enable_timing=True) for _ in range(len(chunks) + 1)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    pre_ev = torch.cuda.Event()
    with torch.cuda.stream(stream):
        pre_ev.record(stream)
        for _ in range(reps):
            pre.replay()
        events[0].record(stream)
        for j, g in enumerate(graphs):
            g.replay()
            events[j + 1].record(stream)
    # the clock record covers the device's timed region: from when the first event
    # completes (polled) to the end of the last replay (and, for a short region, the end
    # of the pre-heat that runs back to back before it)
    while not pre_ev.query():
        time.sleep(0.0002)
    clocks.mark("preheat")
    while not events[0].query():
        time.sleep(0.0002)
    clocks.mark("start")
    torch.cuda.synchronize()
    clocks.mark("end")
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    total_ms = events[0].elapsed_time(events[-1])
    chunk_ms = [events[j].elapsed_time(events[j + 1]) for j in range(len(chunks))]
    status, word = tl.tl_device_status(reset=True)
    if status != tl.TL_OK:
        raise RuntimeError(f"device-side wait gave up in the timed region: {word:#x}")
    if len(chunks) == 1:
        # one graph: the spread comes from five more replays of the timed sequence, each
        # between its own events, after the timed region (nothing is added inside it)
        # (behind one untimed replay, so that the GPU is busy while the first timed
        # replay is submitted, as in the timed region, which follows the pre-heat)
        rep_ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        with torch.cuda.stream(stream):
            pre.replay()
            rep_ev[0].record(stream)
            for j in range(5):
                graphs[0].replay()
                rep_ev[j + 1].record(stream)
        torch.cuda.synchronize()
        chunk_ms = [rep_ev[j].elapsed_time(rep_ev[j + 1]) for j in range(5)]
        chunks = chunks * 5
    spread = spread_of(chunk_ms, chunks)
    spread["preheat_ms"] = round(reps * step_ms * G, 1)
    return max_over_ranks(total_ms, dist, dev), clk, spread


def library_context(name: str, step, rot: int, stream, steps: int, flops: int,
                    preheat_s: float = 2.0) -> dict:
    """The same workload through a vendor library (a library run, never inspected), timed
    as the kernel is: CUDA-graph replays of consecutive calls on the rotating inputs.
    Context for the reader only; any failure is reported, never raised."""
    import torch
    try:
        with torch.cuda.stream(stream):
            for i in range(3):
                step(i)
        torch.cuda.synchronize()
        G = rot * max(1, math.ceil(64 / rot))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(G):
                step(i)
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        # the same pre-heat as the library's own timed steps, so both run at the clock
        # the load sustains
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < preheat_s:
            with torch.cuda.stream(stream):
                g.replay()
            torch.cuda.synchronize()
        reps = max(2, steps // (4 * G))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / (reps * G)
        return {"library": name, "tflops": round(flops / (ms * 1e-3) / 1e12, 3),
                "ms_per_step": round(ms, 5), "steps": reps * G}
    except Exception as e:          # context only: never fail the measurement for it
        return {"library": name, "error": str(e).splitlines()[0][:200]}


def e2e_pipeline(args, inputs_cpu, out_shape, out_dtype, compute, flops: int, world: int,
                 stream, dist, dev, tl) -> dict:
    """The same metric end to end through the public call from pinned host buffers.

    Every step uploads its inputs, runs compute(device inputs, device output) and
    downloads the output, all inside the timed region.  As a serving loop would, the
    steps are pipelined: copies in, the computation and the copy out run on three
    streams over two device buffer sets, so step i's computation overlaps step i+1's
    upload and step i-1's download; a set is reused only after its download finished.
    Like the device-resident number, the timed steps replay CUDA graphs of that
    pipeline (host launch cost excluded); the same steps enqueued eagerly from Python
    are timed too and reported as eager_ms_per_step.  (Uploads split over two streams
    were measured no faster: ~210 GB/s either way.)"""
    import torch

    hosts = [x.pin_memory() for x in inputs_cpu]
    e_sets = []
    for _ in range(2):
        ins = [torch.empty_like(x, device=dev) for x in inputs_cpu]
        out_d = torch.empty(out_shape, dtype=out_dtype, device=dev)
        out_h = torch.empty(out_shape, dtype=out_dtype).pin_memory()
        e_sets.append((ins, out_d, out_h))
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    e_graph = 50                              # pipelined steps per graph
    e_steps = e_graph * max(1, min(args.steps, 200) // e_graph)

    def run(n):
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        freed = [None, None]           # download of the set's previous step done
        for i in range(n):
            k = i % 2
            ins, out_d, out_h = e_sets[k]
            if freed[k] is not None:
                s_in.wait_event(freed[k])
            with torch.cuda.stream(s_in):
                for d, h in zip(ins, hosts):
                    d.copy_(h, non_blocking=True)
                uploaded = torch.cuda.Event()
                uploaded.record(s_in)
            stream.wait_event(uploaded)
            compute(ins, out_d)
            computed = torch.cuda.Event()
            computed.record(stream)
            s_out.wait_event(computed)
            with torch.cuda.stream(s_out):
                out_h.copy_(out_d, non_blocking=True)
                freed[k] = torch.cuda.Event()
                freed[k].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    def timed(fn):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):        # graph replays go to the current stream
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    run(4)                                     # warm-up, eager
    torch.cuda.synchronize()
    eager_ms = timed(lambda: run(e_graph))
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        run(e_graph)
    with torch.cuda.stream(stream):
        g_e2e.replay()                         # one untimed replay
    torch.cuda.synchronize()

    def replays():
        for _ in range(e_steps // e_graph):
            g_e2e.replay()

    e_ms = max_over_ranks(timed(replays), dist, dev)
    status, word = tl.tl_device_status(reset=True)
    if status != tl.TL_OK:
        raise RuntimeError(f"device-side wait gave up in the end-to-end run: {word:#x}")
    return {"value": round(whole_job_tflops(flops, e_steps, world, e_ms), 3),
            "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(sum(x.numel() * x.element_size() for x in inputs_cpu)),
            "d2h_bytes_per_step": int(math.prod(out_shape) *
                                      torch.empty((), dtype=out_dtype).element_size()),
            "steps": e_steps, "ms_per_step": round(e_ms / e_steps, 4),
            "eager_ms_per_step": round(eager_ms / e_graph, 4),
            "pipelined": "upload, compute and download on three streams, two buffer sets; "
                         "graphs of 50 steps"}


def run_tl(args, w: workloads.Workload, rank: int, world: int, dist) -> dict:
    import torch

    import tiled_gemm_gb300 as tl

    dev = torch.device("cuda", torch.cuda.current_device())
    a_cpu, b_cpu = workloads.make_inputs(w)
    per_set = w.bytes_moved
    rot = rotation_sets(per_set)
    sets = []
    a0, b0 = a_cpu.to(dev), b_cpu.to(dev)
    for i in range(rot):
        a = a0 if i == 0 else a0.clone()
        b = b0 if i == 0 else b0.clone()
        c = torch.empty((w.M, w.N), dtype=w.torch_dtype, device=dev)
        sets.append((a, b, c))
    plan = None
    if w.plan is not None:
        bm, bn, bk, st = w.plan
        plan = tl.plan_for(0, 0, 0, bm, bn, bk, st)
    stream = torch.cuda.Stream(device=dev)
    lda = w.M if w.trans_a else w.K
    eb = w.elem_bytes
    launches_per_step = 1 + int((lda * eb) % 16 != 0) + int(
        ((w.K if w.trans_b else w.N) * eb) % 16 != 0)

    def gemm_call(a, b, c):
        if w.fp8:
            tl.gemm_fp8(a, b, trans_a=w.trans_a, trans_b=w.trans_b, relu=w.relu, alpha=w.alpha,
                        out=c, plan=plan, stream=stream)
        else:
            tl.gemm(a, b, trans_a=w.trans_a, trans_b=w.trans_b, relu=w.relu, out=c, plan=plan,
                    stream=stream)

    def step(i):
        a, b, c = sets[i % rot]
        gemm_call(a, b, c)

    max_ms, clk, spread = timed_graph_steps(args, step, rot, stream, dist, dev, tl,
                                            preheat_s=args.preheat_s)
    e2e = None
    if not args.no_e2e:
        e2e = e2e_pipeline(args, [a_cpu, b_cpu], (w.M, w.N), w.torch_dtype,
                           lambda ins, out: gemm_call(ins[0], ins[1], out), w.flops, world,
                           stream, dist, dev, tl)
    context = None
    if not w.fp8:
        def lib_step(i):
            a, b, c = sets[i % rot]
            torch.matmul(a.t() if w.trans_a else a, b.t() if w.trans_b else b, out=c)
            if w.relu:
                c.relu_()
        context = library_context("torch.matmul (cuBLAS)" + (" + relu_" if w.relu else ""),
                                  lib_step, rot, stream, args.steps, w.flops, args.preheat_s)
    return {"total_ms": max_ms, "clocks": clk, "spread": spread, "e2e": e2e, "context": context,
            "rotation_sets": rot, "launches_per_step": launches_per_step,
            "plan": tl.tl_gemm_plan(w.M, w.N, w.K, w.dtype, int(w.trans_a), int(w.trans_b),
                                    torch.cuda.get_device_properties(dev).multi_processor_count)
            .as_dict() if plan is None else
            tl.tl_plan_complete(w.M, w.N, w.K, *w.plan, dtype=w.dtype).as_dict()}


def run_mx(args, w: workloads.MxWorkload, rank: int, world: int, dist) -> dict:
    import torch

    import tiled_gemm_gb300 as tl

    dev = torch.device("cuda", torch.cuda.current_device())
    ins_cpu = workloads.make_mx_inputs(w)
    rot = rotation_sets(w.bytes_moved)
    first = [x.to(dev) for x in ins_cpu]
    sets = [(first if i == 0 else [x.clone() for x in first]) +
            [torch.empty((w.M, w.N), dtype=w.c_torch_dtype, device=dev)] for i in range(rot)]
    stream = torch.cuda.Stream(device=dev)

    def call(ins, out):
        tl.gemm_mx(ins[0], ins[1], ins[2], ins[3], relu=w.relu, out=out, stream=stream)

    def step(i):
        st = sets[i % rot]
        call(st[:4], st[4])

    max_ms, clk, spread = timed_graph_steps(args, step, rot, stream, dist, dev, tl,
                                            preheat_s=args.preheat_s)
    e2e = None
    if not args.no_e2e:
        e2e = e2e_pipeline(args, list(ins_cpu), (w.M, w.N), w.c_torch_dtype, call, w.flops,
                           world, stream, dist, dev, tl)
    return {"total_ms": max_ms, "clocks": clk, "spread": spread, "e2e": e2e,
            "rotation_sets": rot, "launches_per_step": 1,
            "plan": {"tile": [128, 128, 128], "stages": 4, "cta_group": 1,
                     "grid": [math.ceil(w.N / 128), math.ceil(w.M / 128)]}}


def run_attn(args, w: workloads.AttnWorkload, rank: int, world: int, dist) -> dict:
    import torch

    import tiled_gemm_gb300 as tl

    dev = torch.device("cuda", torch.cuda.current_device())
    q_cpu, k_cpu, v_cpu = workloads.make_attn_inputs(w)
    rot = rotation_sets(w.bytes_moved)
    q0, k0, v0 = (x.to(dev) for x in (q_cpu, k_cpu, v_cpu))
    sets = [(q0, k0, v0, torch.empty_like(q0)) if i == 0 else
            (q0.clone(), k0.clone(), v0.clone(), torch.empty_like(q0)) for i in range(rot)]
    stream = torch.cuda.Stream(device=dev)

    def step(i):
        q, k, v, o = sets[i % rot]
        tl.attention(q, k, v, causal=w.causal, out=o, stream=stream)

    max_ms, clk, spread = timed_graph_steps(args, step, rot, stream, dist, dev, tl,
                                            preheat_s=args.preheat_s)

    def lib_step(i):
        q, k, v, _ = sets[i % rot]
        torch.nn.functional.scaled_dot_product_attention(
            q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2), is_causal=w.causal)

    context = library_context("torch scaled_dot_product_attention", lib_step, rot, stream,
                              args.steps, w.flops, args.preheat_s)
    e2e = None
    if not args.no_e2e:
        e2e = e2e_pipeline(args, [q_cpu, k_cpu, v_cpu], tuple(q_cpu.shape), w.torch_dtype,
                           lambda ins, out: tl.attention(ins[0], ins[1], ins[2], causal=w.causal,
                                                         out=out, stream=stream),
                           w.flops, world, stream, dist, dev, tl)
    return {"total_ms": max_ms, "clocks": clk, "spread": spread, "e2e": e2e,
            "context": context, "rotation_sets": rot, "launches_per_step": 1,
            "plan": {"q_tile": 128, "kv_tile": 128, "kv_stages": 2, "s_buffers": 3,
                     "grid": "persistent, at most one CTA per SM"}}


def oracle_rate_attn(w: workloads.AttnWorkload, q, k, v, budget_s: float, threads: int):
    """Oracle TFLOP/s on output rows spread over the sequence, repeated for ~budget_s."""
    import numpy as np

    import oracle
    oracle.build()
    rng = np.random.default_rng(0)
    n, done_flops, elapsed, reps = 16, 0, 0.0, 0
    code = oracle.F16 if w.dtype == workloads.F16 else oracle.BF16
    while elapsed < budget_s:
        bs = rng.integers(0, w.B, n)
        is_ = rng.integers(0, w.S, n)
        hs = rng.integers(0, w.H, n)
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, bs, is_, hs, dtype=code, causal=w.causal, threads=threads)
        dt = time.perf_counter() - t0
        elapsed += dt
        keys = (is_ + 1) if w.causal else np.full(n, w.S)
        done_flops += int(4 * w.D * keys.sum())
        reps += 1
        if dt < budget_s / 20:
            n *= 2
    return done_flops / elapsed / 1e12, elapsed, done_flops, n, reps


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps; 0 (default) sizes the timed region to ~1.5 s")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=workloads.HEADLINE,
                    choices=sorted(workloads.WORKLOADS) + sorted(workloads.ATTN_WORKLOADS)
                    + sorted(workloads.MX_WORKLOADS))
    ap.add_argument("--impl", default="tl", choices=["tl", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--preheat-s", type=float, default=2.0,
                    help="untimed replays before the timed region, in seconds (0: one round)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    attn = args.workload in workloads.ATTN_WORKLOADS
    mx = args.workload in workloads.MX_WORKLOADS
    w = (workloads.ATTN_WORKLOADS[args.workload] if attn else
         workloads.MX_WORKLOADS[args.workload] if mx else workloads.WORKLOADS[args.workload])
    metric = ("attention forward TFLOP/s and % of GB300 dense fp16/bf16 peak, 1 GPU" if attn
              else "block-scaled 8-bit GEMM TFLOP/s and % of GB300 dense fp8 peak, 1 GPU" if mx
              else "GEMM+ReLU TFLOP/s and % of GB300 dense fp16/bf16 peak, 1 GPU")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    peaks, peaks_src = load_peaks()
    threads = os.cpu_count() or 1

    if attn:
        config = {"workload": w.name, "B": w.B, "S": w.S, "H": w.H, "D": w.D,
                  "dtype": w.dtype_name, "causal": w.causal, "inputs": w.description,
                  "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                  "l2": l2_note(w.bytes_moved)}
    elif mx:
        config = {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dtype": w.dtype_name,
                  "layout": "A [M,K], B [N,K], both K-major", "scales": "E8M0 per 32 K",
                  "out": "bf16" if w.out_dtype == workloads.BF16 else "f16",
                  "epilogue": "relu" if w.relu else "none", "inputs": w.description,
                  "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                  "l2": l2_note(w.bytes_moved)}
    else:
        config = {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dtype": w.dtype_name,
                  "trans_a": w.trans_a, "trans_b": w.trans_b,
                  "epilogue": "relu" if w.relu else "none", "inputs": w.description,
                  "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                  "l2": l2_note(w.bytes_moved)}

    cpu_inputs = []              # drawn once, on first use

    def cpu_rate(budget, nthreads=threads):
        if not cpu_inputs:
            cpu_inputs.extend(workloads.make_attn_inputs(w) if attn else
                              workloads.make_mx_inputs(w) if mx else workloads.make_inputs(w))
        if attn:
            q, k, v = cpu_inputs
            r, el, fl, n, reps = oracle_rate_attn(w, q, k, v, budget, nthreads)
            return r, el, fl, f"{reps} oracle runs of up to {n} output rows of {w.B * w.S * w.H}"
        if mx:
            a_cpu, b_cpu, sa_cpu, sb_cpu = cpu_inputs
            r, el, fl, rows, reps = oracle_rate_mx(w, a_cpu, b_cpu, sa_cpu, budget, sb_cpu,
                                                   nthreads)
            return r, el, fl, f"{reps} oracle runs on row slices (up to {rows} of {w.M} rows)"
        a_cpu, b_cpu = cpu_inputs
        r, el, fl, rows, reps = oracle_rate(w, a_cpu, b_cpu, budget, nthreads)
        return r, el, fl, f"{reps} oracle runs on row slices (up to {rows} of {w.M} rows)"

    if args.impl == "reference":
        # The oracle on the host cores, rank 0 only: each step a bounded row slice.
        if rank != 0:
            return
        if args.steps <= 0:
            args.steps = 10
        budget = max(0.5, 150.0 / (args.steps + args.warmup))
        for _ in range(args.warmup):
            cpu_rate(min(budget, 1.0))
        rates, times = [], []
        for _ in range(args.steps):
            r, el, fl, what = cpu_rate(budget)
            rates.append(r)
            times.append(el)
        value = statistics.mean(rates)
        line = {"metric": metric,
                "value": sig4(value), "unit": "TFLOP/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(1e3 * statistics.mean(times), 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic", "impl": "reference", "config": config,
                "cpu_baseline": {"value": sig4(value), "unit": "TFLOP/s", "cores": threads,
                                 "kind": "oracle",
                                 "sample": f"{what} per step, ~{budget:.1f} s of CPU work "
                                           "per step"},
                "e2e": {"value": sig4(value), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    dist = None
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl")
        dist = tdist
    else:
        torch.cuda.set_device(0)

    # The oracle's CPU baseline runs before any CUDA work of this process touches the
    # GPU's clocks (rank 0, N = 1 only).
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r, el, fl, what = cpu_rate(args.cpu_budget_s)
        # one thread for a short sample: the per-core rate, and the single-core time that
        # the whole workload would take
        r1, el1, fl1, what1 = cpu_rate(min(args.cpu_budget_s, 2.0), 1)
        cpu = {"value": sig4(r), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{what}, {fl / 1e9:.2f} GFLOP in {el:.1f} s",
               "single_core": {"value": sig4(r1), "unit": "TFLOP/s",
                               "sample": f"{what1}, {fl1 / 1e9:.3f} GFLOP in {el1:.1f} s",
                               "workload_s": round(w.flops / (r1 * 1e12), 1)}}

    res = (run_attn if attn else run_mx if mx else run_tl)(args, w, rank, world, dist)
    total_ms = res["total_ms"]
    value = whole_job_tflops(w.flops, args.steps, world, total_ms)
    avg_launch_ms = total_ms / args.steps        # back-to-back launches in the graph
    roof = roofline(w, avg_launch_ms, peaks, peaks_src, res.get("clocks"), attn)
    roof["traffic"] = load_traffic(w.name)
    roof["kernel_ms"] = round(avg_launch_ms, 6)
    roof["algorithmic"] = {"flops_per_launch": w.flops, "bytes_per_launch": w.bytes_moved}
    if rank != 0:
        return
    line = {"metric": metric,
            "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype_name, "data": "synthetic (seeded CPU generator)",
            "config": config,
            "roofline": roof, "cpu_baseline": cpu, "e2e": res["e2e"],
            "gpu_launches": res["launches_per_step"] * args.steps,
            "clocks": res["clocks"], "spread": spread_line(res.get("spread"), w.flops),
            "plan": res["plan"],
            "context": res.get("context"),
            "pct_of_nominal": round(100 * value / world / (2250.0 * tensor_peak_scale(w)), 2),
            "nominal_tflops": 2250.0 * tensor_peak_scale(w)}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
