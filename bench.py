#!/usr/bin/env python3
"""Benchmark of the GEMV library on one GB300 (or N replicas, one per GPU).

Headline: achieved HBM GB/s of the FP16 4096x14336 GEMV (the decode
down-projection shape), and its memory-bandwidth utilisation against the
pure-read ceiling measured in the same run ("membound", sections "Results" and
"Why GEMV, and why MBU").

One step = one GEMV launch over the whole workload: choose the kernel, stage
x, stream A, accumulate, reduce, write y.  Weights rotate through enough
copies (at least max(256 MiB, 4 x L2)) that every launch reads A cold from
HBM ("membound", gotcha 1); x stays resident.  The K timed steps are one CUDA
graph of exactly K back-to-back launches (or replays of a graph of B launches
plus one graph of the remainder), each graph replayed during warm-up; right
before the timed region a short spin kernel (so that the host's submission of
the graph is not timed) and an untimed replay of one rotation of the weights
(so that the first timed launch follows a launch of the same kernel, as in a
decode loop).  Time comes from CUDA events on the launching stream.  Algorithmic bytes per step = A +
scales + x read once, y written once ("Making GEMV Fast", section "Memory
Access").

Besides the headline the line carries, unless --no-configs: every workload of
the five families (FP32 1024^2, FP16 4096^2, the FP16 decode shapes, the
square sweep in FP32 and FP16, INT8/INT4 at both decode shapes) with its
automatic kernel, time per launch in a chain of plain launches and in an
overlapped chain, GB/s, MBU against the probe and the 8 TB/s spec, and the
parity error over every row against the CPU oracle; plus FP16, INT8 and INT4
at each decode shape timed in interleaved rounds (best round per kernel) with
their speed-up over FP16 ("membound", "dequant GEMV").

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead (the reference arm: there is no runnable upstream
code).
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

DEFAULT_WORKLOAD = "f16_down_4096x14336"
METRIC = "achieved HBM GB/s and MBU% (vs measured pure-read) for FP16 4096x14336 GEMV"
SPEC_HBM_GBS = 8000.0           # HBM3e nominal
FALLBACK_HBM_GBS = 6800.0       # used only if MEASURED_PEAKS.json is absent
PUBLISHED = {"f16_down_4096x14336": (417.0, "membound page, RTX 4080 Laptop (Ada sm_89): context only")}
ROTATE_MIN_BYTES = 256 << 20
GATE_CYCLES = 100_000           # spin kernel ahead of a timed region (~50 us)
GRAPH_MAX = 1000                # launches per captured graph

KERNEL_NAMES = {"vec": "mbg_warprow_kernel", "tile": "mbg_rowtile_kernel", "bulk": "mbg_bulkpipe_kernel",
                "band": "mbg_rowband_kernel", "sband": "mbg_stageband_kernel", "elem": "mbg_elem_kernel",
                "mma": "mbg_mmaband_kernel", "smma": "mbg_mmastage_kernel"}

# the five workload families, in the order they are reported
CONFIG_WORKLOADS = ["f32_1024", "f16_4096", "f16_up_14336x4096", "f16_down_4096x14336",
                    "sweep_f32_2048", "sweep_f32_4096", "sweep_f32_8192", "sweep_f32_16384",
                    "sweep_f16_2048", "sweep_f16_4096", "sweep_f16_8192", "sweep_f16_16384",
                    "q8_4096x14336", "q8_14336x4096", "q4_4096x14336", "q4_14336x4096",
                    # format options: binary16 weights with an FP32 x, INT8 with one scale per row
                    "f16x32_down_4096x14336", "q8row_4096x14336"]
# FP16 / INT8 / INT4 at one shape, timed in interleaved rounds
INTERLEAVED = {"4096x14336": ("f16_down_4096x14336", "q8_4096x14336", "q4_4096x14336"),
               "14336x4096": ("f16_up_14336x4096", "q8_14336x4096", "q4_14336x4096")}


# ---------------------------------------------------------------------------
# byte model and rotation (pure host arithmetic, tested in test_bench_math)
# ---------------------------------------------------------------------------

def a_bytes(dtype: str, M: int, N: int) -> int:
    per = {"f32": 4 * N, "f16": 2 * N, "q8": N, "q4": N // 2, "f16x32": 2 * N, "q8row": N}[dtype]
    return M * per


def scale_bytes(dtype: str, M: int, N: int) -> int:
    if dtype == "q8row":
        return 2 * M
    return 2 * M * synth.n_groups(N) if dtype in ("q8", "q4") else 0


def x_bytes(dtype: str, N: int) -> int:
    return (4 if dtype in ("f32", "f16x32") else 2) * N


def f16_weights(dtype: str) -> bool:
    return dtype in ("f16", "f16x32")


def f32_x(dtype: str) -> bool:
    return dtype in ("f32", "f16x32")


def algorithmic_bytes(dtype: str, M: int, N: int) -> int:
    """A + scales + x read once, y (FP32) written once."""
    return a_bytes(dtype, M, N) + scale_bytes(dtype, M, N) + x_bytes(dtype, N) + 4 * M


def rotation_copies(weight_bytes: int, l2_bytes: int) -> int:
    target = max(ROTATE_MIN_BYTES, 4 * l2_bytes)
    return max(2, math.ceil(target / max(1, weight_bytes)))


def gbs(nbytes: float, seconds: float) -> float:
    return nbytes / seconds / 1e9 if seconds > 0 else float("nan")


def split_steps(steps: int, batch: int):
    """(full graph replays, tail launches) for exactly `steps` launches."""
    batch = max(1, batch)
    return steps // batch, steps % batch


def graph_plan(steps: int, copies: int, graph_max: int = GRAPH_MAX):
    """Graphs that make up exactly `steps` launches: [(launches, replays), ...].

    Up to graph_max steps: one graph of exactly `steps` launches, replayed
    once.  Beyond: a graph of B launches (a multiple of the rotation count, so
    replays continue the rotation) replayed steps // B times, plus one graph of
    the remainder."""
    if steps <= graph_max:
        return [(steps, 1)]
    batch = max(copies, graph_max // copies * copies)
    full, tail = split_steps(steps, batch)
    plan = [(batch, full)]
    if tail:
        plan.append((tail, 1))
    return plan


# sources of the kernels whose DRAM traffic is recorded (GEMV variants and
# their dispatch, the row softmax); the probes, the host-buffer copy, the
# quantiser and the dequantisation helpers do not change those kernels
TRAFFIC_SOURCES = ("gemv_api.cu", "gemv_device.cuh", "gemv_internal.h", "gemv_kernels.cuh", "gemv_f32.cu",
                   "gemv_f16.cu", "gemv_f16x32.cu", "gemv_q8.cu", "gemv_q4.cu", "gemv_softmax.cu")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "memory_bound_gemv_gb300", "csrc")
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "of measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "of fallback"


def recorded_traffic(workload: str, variant: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernels are unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    entry = rec.get("entries", {}).get(f"{workload}:{variant}")
    return None if entry is None else entry.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------

def rank_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def max_over_ranks(value: float, device=None) -> float:
    """Max of a scalar over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
REASON_NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def parse_clock_line(line: str):
    parts = [p.strip() for p in line.split(",")]
    if len(parts) != len(CLOCK_FIELDS):
        return None
    try:
        sm = float(parts[1])
        smax = float(parts[2])
    except ValueError:
        return None
    reasons = [n for n, v in zip(REASON_NAMES, parts[5:]) if v.lower() == "active"]
    return {"sm": sm, "sm_max": smax, "reasons": reasons}


def summarise_clocks(samples, t0, t1):
    inside = [s for s in samples if t0 is not None and t1 is not None and t0 <= s["t"] <= t1]
    if not inside:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    return {"sm_mhz": statistics.median(s["sm"] for s in inside),
            "sm_max_mhz": max(s["sm_max"] for s in inside),
            "reasons": sorted({r for s in inside for r in s["reasons"]}), "samples": len(inside)}


class ClockSampler:
    """nvidia-smi sampled every 50 ms; windows are host-time intervals."""

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        self.error = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={','.join(CLOCK_FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "50", "-i", gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError as e:
            self.error = str(e)

    def _read(self):
        for line in self.proc.stdout:
            s = parse_clock_line(line)
            if s is not None:
                s["t"] = time.monotonic()
                self.samples.append(s)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def window(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": f"nvidia-smi unavailable: {self.error}"}
        return summarise_clocks(self.samples, t0, t1)


def gpu_id_for(dev: int) -> str:
    import torch
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if uuid:
            return uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
    except (AttributeError, RuntimeError):
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[dev]
    return str(dev)


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def sample_bytes(w, nrows: int) -> int:
    """Algorithmic bytes of GEMV over `nrows` rows of workload w (x read once)."""
    per_row = (a_bytes(w.dtype, 1, w.N) + scale_bytes(w.dtype, 1, w.N) + 4)
    return nrows * per_row + x_bytes(w.dtype, w.N)


def oracle_rows(w, rows):
    """Inputs for the given rows only (the generator is counter-based)."""
    import numpy as np
    r0, r1 = min(rows), max(rows) + 1
    A = synth.weight_rows(w, r0, r1 - r0)
    s = synth.scale_rows(w, r0, r1 - r0) if w.quantised else None
    idx = np.asarray(rows, dtype=np.int64) - r0
    return A, synth.x_vector(w), s, idx


def time_oracle(w, seconds: float, threads: int, rows_per_call: int):
    """Repeat the oracle over a block of rows until `seconds` of CPU work."""
    import oracle
    orc = oracle.load()
    rows = list(range(min(rows_per_call, w.M)))
    A, x, s, idx = oracle_rows(w, rows)
    n = len(rows)
    orc.gemv(w.dtype, A, x, n, w.N, scales=s, rows=idx, threads=threads)  # warm
    calls, t0 = 0, time.perf_counter()
    while True:
        orc.gemv(w.dtype, A, x, n, w.N, scales=s, rows=idx, threads=threads)
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return gbs(calls * sample_bytes(w, n), el), calls, n, el


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    rank, _, world = rank_env()
    if rank != 0:
        return 0
    w = synth.WORKLOADS[args.workload]
    import oracle
    orc = oracle.load()
    threads = cpu_threads()
    # calibrate rows per step so that warm-up + timed steps stay within budget
    probe_rows = min(w.M, 64)
    A, x, s, idx = oracle_rows(w, list(range(probe_rows)))
    t0 = time.perf_counter()
    orc.gemv(w.dtype, A, x, probe_rows, w.N, scales=s, rows=idx, threads=threads)
    per_row = (time.perf_counter() - t0) / probe_rows
    budget = args.reference_seconds
    steps_total = max(1, args.steps + args.warmup)
    rows = int(max(1, min(w.M, budget / steps_total / max(per_row, 1e-9))))
    A, x, s, idx = oracle_rows(w, list(range(rows)))
    for _ in range(args.warmup):
        orc.gemv(w.dtype, A, x, rows, w.N, scales=s, rows=idx, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.gemv(w.dtype, A, x, rows, w.N, scales=s, rows=idx, threads=threads)
    el = time.perf_counter() - t0
    value = gbs(args.steps * sample_bytes(w, rows), el)
    sample = (f"each step: oracle (double precision, all {threads} host threads) over rows "
              f"0..{rows - 1} of the {w.M}x{w.N} {w.dtype} workload")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / max(1, args.steps) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64)",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "weights": w.dtype},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU helpers
# ---------------------------------------------------------------------------

class Resident:
    """One workload in device memory: weight copies for the rotation, x, y."""

    def __init__(self, w, dev, l2, inp=None):
        import numpy as np
        import torch
        self.w = w
        self.inp = inp if inp is not None else synth.make(w)

        def to_dev(arr, f16bits):
            a = np.ascontiguousarray(arr)
            return torch.from_numpy(a.view(np.float16) if f16bits else a).to(dev)

        A0 = to_dev(self.inp["A"], f16_weights(w.dtype))
        self.x = to_dev(self.inp["x"], not f32_x(w.dtype))
        S0 = to_dev(self.inp["scales"], True) if w.quantised else None
        if w.dtype == "q8row":
            S0 = S0.reshape(-1)  # one scale per row: [M]
        self.wbytes = a_bytes(w.dtype, w.M, w.N) + scale_bytes(w.dtype, w.M, w.N)
        self.copies = rotation_copies(self.wbytes, l2)
        self.As = [A0] + [A0.clone() for _ in range(self.copies - 1)]
        self.Ss = [S0] + [S0.clone() for _ in range(self.copies - 1)] if w.quantised else [None] * self.copies
        self.y = torch.empty(w.M, dtype=torch.float32, device=dev)
        self.step_bytes = algorithmic_bytes(w.dtype, w.M, w.N)

    def launch(self, i, overlap=False):
        import memory_bound_gemv_gb300 as mbg
        k = i % self.copies
        mbg.gemv(self.w.dtype, self.As[k], self.x, self.Ss[k], y=self.y, overlap=overlap)

    def free(self):
        self.As = self.Ss = self.x = self.y = None


class Timer:
    """Graphs of back-to-back launches timed with CUDA events on one stream.

    Every timed pass is preceded by an untimed replay of one full rotation
    (launches on copies 0 .. copies-1): the first timed launch then follows a
    launch of the same kernel, as every later one does, and reads copy 0,
    which was last touched `copies` launches (at least 4 x L2 of weights)
    earlier.  Measured on the headline: one launch alone takes ~22 us, the
    first of a short chain ~7-10 us more than the steady 15.9 us, because
    consecutive launches hide each other's ramp; without the pre-roll a
    20-launch region carries that once."""

    def __init__(self, dev, stream, l2):
        self.dev = dev
        self.stream = stream

    def capture(self, launch, plan, overlap=False, copies=None):
        """Graphs for the plan, plus (first) the pre-roll graph of one rotation."""
        import torch
        graphs = []
        with torch.cuda.stream(self.stream):
            sizes = ([copies] if copies else []) + [n for n, _ in plan]
            for n in sizes:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream):
                    for i in range(n):
                        launch(i, overlap)
                graphs.append(g)
        self.stream.synchronize()
        return graphs

    def replay(self, graphs, plan):
        for g, (_, reps) in zip(graphs[1:], plan):
            for _ in range(reps):
                g.replay()

    def warm(self, graphs, plan, launches):
        """Replays every graph at least once and at least `launches` launches in all."""
        import torch
        done = 0
        with torch.cuda.stream(self.stream):
            graphs[0].replay()
            while True:
                for g, (n, _) in zip(graphs[1:], plan):
                    g.replay()
                    done += n
                if done >= launches:
                    break
        self.stream.synchronize()

    def timed(self, graphs, plan):
        """Seconds for one pass of the plan: a spin kernel first (the host's
        submissions are not timed), then the untimed pre-roll, then the plan
        between two events."""
        import torch
        with torch.cuda.stream(self.stream):
            torch.cuda._sleep(GATE_CYCLES)
            graphs[0].replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            self.replay(graphs, plan)
            e1.record(self.stream)
        e1.synchronize()
        return e0.elapsed_time(e1) * 1e-3

    def hold(self, graphs, plan, seconds):
        """Replays the plan back to back for about `seconds` (clock sampling)."""
        import torch
        t_end = time.monotonic() + seconds
        with torch.cuda.stream(self.stream):
            while time.monotonic() < t_end:
                self.replay(graphs, plan)
                self.stream.synchronize()


def probe_ceiling(mbg, stream, probe_buf, sink, reps):
    import torch
    probe_bytes = probe_buf.numel() * probe_buf.element_size()
    res = {}
    with torch.cuda.stream(stream):
        for v, name in enumerate(mbg.probe_variants()):
            for _ in range(2):
                mbg.gemv_probe_read(probe_buf, sink, v)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                mbg.gemv_probe_read(probe_buf, sink, v)
            e1.record(stream)
            e1.synchronize()
            res[name] = gbs(reps * probe_bytes, e0.elapsed_time(e1) * 1e-3)
    # bit 63 of the sink: a bulk-copy probe gave up waiting (its time means nothing)
    if (int(sink.item()) >> 63) & 1:
        raise SystemExit("a bulk-copy probe timed out; no MBU denominator")
    return res


def parity_all_rows(w, inp, y_gpu):
    """Max normalised error of y_gpu against the oracle over every row."""
    import oracle
    orc = oracle.load()
    y_ref, den = orc.gemv(w.dtype, inp["A"], inp["x"], w.M, w.N, scales=inp.get("scales"),
                          threads=cpu_threads())
    return oracle.max_normalised_error(y_gpu, y_ref, den)


TOL = {"f32": 1e-5, "f16": 2e-3, "q8": 2e-3, "q4": 2e-3, "f16x32": 1e-5, "q8row": 2e-3}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import torch

    import memory_bound_gemv_gb300 as mbg

    rank, local_rank, world = rank_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    w = synth.WORKLOADS[args.workload]
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 << 20))
    stream = torch.cuda.Stream(dev)
    timer = Timer(dev, stream, l2)
    R = Resident(w, dev, l2)
    step_bytes = R.step_bytes

    vid = mbg.select_variant(w.dtype, R.As[0], R.x)
    vinfo = mbg.variants(w.dtype)[vid]

    # first launch: kept for the parity check (every row against the oracle)
    with torch.cuda.stream(stream):
        R.launch(0)
    stream.synchronize()
    y_first = R.y.cpu().numpy().copy()
    if mbg.gemv_get_device_error(stream) != mbg.OK:
        raise SystemExit("device status word set on the first launch")

    # ---- pure-read probe (before) ----
    probe_bytes = int(args.probe_gib * (1 << 30)) // 16 * 16
    probe_buf = torch.randint(-2 ** 31, 2 ** 31 - 1, (probe_bytes // 4,), dtype=torch.int32, device=dev)
    sink = torch.zeros(1, dtype=torch.int64, device=dev)
    probe_before = probe_ceiling(mbg, stream, probe_buf, sink, args.probe_reps)

    # ---- the timed region: exactly K launches from warmed graphs ----
    with torch.cuda.stream(stream):
        for i in range(min(3, R.copies)):
            R.launch(i)
    stream.synchronize()
    plan = graph_plan(args.steps, R.copies, args.graph_max)
    graphs = timer.capture(R.launch, plan, copies=R.copies)
    timer.warm(graphs, plan, args.warmup)

    sampler = ClockSampler(gpu_id_for(local_rank)) if not args.no_clocks else None
    if sampler is not None:
        time.sleep(0.3)  # let nvidia-smi start
    barrier()
    torch.cuda.synchronize(dev)
    t_host0 = time.monotonic()
    elapsed = timer.timed(graphs, plan)
    t_host1 = time.monotonic()
    barrier()
    # the same graphs replayed for a while right after, so that the clocks
    # under this load are sampled (a timed region of a few launches is far
    # shorter than the sampling interval)
    clock_t0 = time.monotonic()
    if sampler is not None:
        timer.hold(graphs, plan, args.clock_seconds)
    clock_t1 = time.monotonic()
    t_max = max_over_ranks(elapsed, dev)
    per_launch = elapsed / max(1, args.steps)
    value = gbs(world * args.steps * step_bytes, t_max)
    del graphs

    # ---- the same chain launched with programmatic dependent launch ----
    # (gemv_ex with GEMV_FLAG_OVERLAP_PRECEDING: each launch may start while
    # the previous one finishes; weights are never written by the chain)
    overlap = None
    if not args.no_overlap:
        g_ov = timer.capture(R.launch, plan, overlap=True, copies=R.copies)
        timer.warm(g_ov, plan, args.warmup)
        barrier()
        ov_t = max_over_ranks(timer.timed(g_ov, plan), dev)
        barrier()
        overlap = {"value": gbs(world * args.steps * step_bytes, ov_t), "unit": "GB/s", "steps": args.steps,
                   "ms_per_step": ov_t / args.steps * 1e3,
                   "how": "the same launches in the same graphs, each launched with programmatic dependent "
                          "launch (weights requested before waiting for the previous launch)"}
        del g_ov

    # ---- a long chain for comparison with the short timed region ----
    long_chain = None
    if not args.no_long_chain:
        lplan = graph_plan(args.long_steps, R.copies, args.graph_max)
        lg = timer.capture(R.launch, lplan, copies=R.copies)
        timer.warm(lg, lplan, 1)
        lt = timer.timed(lg, lplan)
        long_chain = {"steps": args.long_steps, "us_per_launch": lt / args.long_steps * 1e6,
                      "value": gbs(args.long_steps * step_bytes, lt), "unit": "GB/s"}
        del lg

    # ---- the same launches without graphs (host-launched stream), for context ----
    eager_steps = min(args.steps, 2000)
    with torch.cuda.stream(stream):
        for i in range(R.copies):
            R.launch(i)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for i in range(eager_steps):
            R.launch(i)
        f1.record(stream)
    f1.synchronize()
    eager_gbs = gbs(eager_steps * step_bytes, f0.elapsed_time(f1) * 1e-3)

    probe_after = probe_ceiling(mbg, stream, probe_buf, sink, args.probe_reps)
    probe_all = {k: max(probe_before[k], probe_after[k]) for k in probe_before}
    best_probe = max(probe_all, key=probe_all.get)
    ceiling = probe_all[best_probe]
    if overlap is not None:
        overlap["mbu_probe_pct"] = 100.0 * overlap["value"] / world / ceiling
    if long_chain is not None:
        long_chain["mbu_probe_pct"] = 100.0 * long_chain["value"] / ceiling

    # ---- end to end through the C ABI: x from pinned host memory, y back ----
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, mbg, R, stream, world, dev)

    # ---- every workload of the five families ----
    configs = None
    if not args.no_configs and world == 1:
        R.free()
        del probe_buf
        torch.cuda.empty_cache()
        configs = measure_configs(args, mbg, dev, l2, stream, timer, ceiling)

    peak, peak_kind = measured_peak()
    achieved = gbs(step_bytes, per_launch)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_kind": peak_kind,
                "traffic": recorded_traffic(w.name, vinfo["name"]),
                "kernel": f"{KERNEL_NAMES[vinfo['kind']]} {vinfo['name']}"}
    clocks = {"sm_mhz": None, "note": "disabled"}
    if sampler is not None:
        held = sampler.window(clock_t0, clock_t1)
        inside = sampler.window(t_host0, t_host1)
        sampler.stop()
        clocks = dict(held)
        clocks["timed_region_samples"] = inside["samples"]
        clocks["window"] = (f"nvidia-smi every 50 ms while the timed graphs were replayed back to back for "
                            f"{clock_t1 - clock_t0:.1f} s right after the timed region "
                            f"({(t_host1 - t_host0) * 1e3:.2f} ms, {inside['samples']} samples inside it)")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = cpu_threads()
        cb, calls, nrows, el = time_oracle(w, args.cpu_seconds, threads, args.cpu_rows)
        cb1, calls1, nrows1, el1 = time_oracle(w, args.cpu_seconds, 1, args.cpu_rows)
        cpu = {"value": cb, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{calls} oracle passes over rows 0..{nrows - 1} of the workload "
                         f"({el:.1f} s, double precision, {threads} threads)",
               "single_thread": {"value": cb1, "unit": "GB/s", "cores": 1,
                                 "sample": f"{calls1} passes over rows 0..{nrows1 - 1} ({el1:.1f} s, 1 thread)"}}

    parity_err = parity_all_rows(w, R.inp, y_first)
    published = PUBLISHED.get(w.name)
    launch_desc = " + ".join(f"{reps} replay{'s' if reps > 1 else ''} of a CUDA graph of {n} back-to-back launches"
                             for n, reps in plan)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max / max(1, args.steps) * 1e3,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (value / world / published[0]) if published else None,
        "vs_baseline_note": published[1] if published else None,
        "dtype": w.dtype, "data": "synthetic (seeded SplitMix64; weights and x normal(0,0.02) "
                                  "rounded to FP16)" if w.dtype == "f16" else "synthetic (seeded SplitMix64)",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "weights": w.dtype,
                   "variant": vinfo["name"], "rotation_copies": R.copies,
                   "rotation_bytes": R.copies * R.wbytes, "l2_bytes": l2,
                   "l2_policy": "inputs larger than L2: the weights rotate through the copies, so each launch "
                                "reads a copy last touched `rotation_copies` launches earlier (cold from HBM)",
                   "launch": f"timed: {launch_desc}; each graph replayed during warm-up; right before the timed "
                             f"region a spin kernel (so no host submission is timed) and an untimed replay of one "
                             f"rotation ({R.copies} launches), so that the first timed launch follows a launch of "
                             f"the same kernel as every later one does",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "mbu": {"probe_gbs": ceiling, "probe_variant": best_probe,
                "mbu_probe_pct": 100.0 * achieved / ceiling,
                "mbu_spec_pct": 100.0 * achieved / SPEC_HBM_GBS,
                "probe_before": probe_before, "probe_after": probe_after},
        "roofline": roofline,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "parity_max_normalised_error_all_rows": parity_err,
        "eager_stream_gbs": eager_gbs,
        "overlap": overlap,
        "long_chain": long_chain,
        "ms_per_launch": per_launch * 1e3,
        "configs": configs,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
        if args.json_out:
            with open(args.json_out, "w") as f:
                json.dump(line, f, indent=1)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def measure_e2e(args, mbg, R, stream, world, dev):
    """One gemv_ex_host call per step through the C ABI, x in and y out through
    page-locked host memory; timed on the host clock (including the final
    synchronisation) and, for comparison, with CUDA events."""
    import torch
    w = R.w
    if w.dtype == "q8row":
        return None
    L = mbg.lib()
    x_host = R.x.cpu().pin_memory()
    y_host = torch.empty(w.M, dtype=torch.float32).pin_memory()
    x_dev = torch.empty_like(R.x)
    steps = min(args.steps, args.e2e_steps) if args.e2e_steps > 0 else args.steps
    steps = max(steps, args.e2e_min_steps)
    dt = mbg.DTYPES[w.dtype]
    a_ptrs = [a.data_ptr() for a in R.As]
    s_ptrs = [s.data_ptr() if s is not None else None for s in R.Ss]
    xh, xd, yh = x_host.data_ptr(), x_dev.data_ptr(), y_host.data_ptr()
    sp = ctypes.c_void_p(stream.cuda_stream)
    fn = L.gemv_ex_host

    def run(flags, n):
        for i in range(n):
            k = i % R.copies
            st = fn(dt, a_ptrs[k], xh, xd, yh, w.M, w.N, s_ptrs[k], flags, sp)
            if st != mbg.OK:
                raise SystemExit(f"gemv_ex_host: {mbg.status_string(st)}")

    out = {}
    for flags, key in ((0, "plain"), (mbg.FLAG_OVERLAP_PRECEDING, "overlap")):
        run(flags, min(args.warmup + 10, 100))
        stream.synchronize()
        barrier()
        h0 = torch.cuda.Event(enable_timing=True)
        h1 = torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        h0.record(stream)
        run(flags, steps)
        h1.record(stream)
        stream.synchronize()
        wall = time.perf_counter() - t0
        barrier()
        out[key] = (max_over_ranks(wall, dev), max_over_ranks(h0.elapsed_time(h1) * 1e-3, dev))
    wall, ev = out["plain"]
    return {"value": gbs(world * steps * R.step_bytes, wall), "unit": "GB/s",
            "h2d_bytes_per_step": int(R.x.numel() * R.x.element_size()),
            "d2h_bytes_per_step": int(w.M * 4), "steps": steps,
            "us_per_step": wall / steps * 1e6,
            "how": "host wall clock (perf_counter) around `steps` gemv_ex_host calls through the C ABI and the "
                   "final stream synchronisation: per step x is read from pinned host memory by a copy kernel "
                   "into a device buffer, the GEMV runs after it with programmatic dependent launch and writes "
                   "y into pinned host memory; weights resident and rotated",
            "device_events_value": gbs(world * steps * R.step_bytes, ev),
            "overlap_value": gbs(world * steps * R.step_bytes, out["overlap"][0]),
            "overlap_how": "the same calls with GEMV_FLAG_OVERLAP_PRECEDING (each copy of x may start before "
                           "the previous GEMV ends), host wall clock"}


def measure_configs(args, mbg, dev, l2, stream, timer, ceiling):
    """Every workload of the five families: time per launch (plain and overlapped
    chains), GB/s, MBU, parity over every row; FP16 / INT8 / INT4 interleaved."""
    import torch
    out = {"how": f"per workload: automatic kernel; a CUDA graph of ~{args.config_launches} back-to-back "
                  f"launches over the rotated weights, replayed once to warm and once timed after an untimed "
                  f"replay of one rotation; "
                  f"MBU against the run's probe ceiling ({ceiling:.0f} GB/s) and the 8 TB/s spec; parity: the "
                  f"first launch against the double-precision oracle over every row",
           "workloads": {}, "interleaved": {}}
    resident = {}
    keep = {name for group in INTERLEAVED.values() for name in group}
    t_start = time.monotonic()

    def chain(R, overlap):
        n = R.copies * max(1, math.ceil(args.config_launches / R.copies))
        plan = [(n, 1)]
        g = timer.capture(R.launch, plan, overlap=overlap, copies=R.copies)
        timer.warm(g, plan, 1)
        t = timer.timed(g, plan)
        return g, plan, t / n

    for name in CONFIG_WORKLOADS:
        w = synth.WORKLOADS[name]
        R = Resident(w, dev, l2)
        with torch.cuda.stream(stream):
            R.launch(0)
        stream.synchronize()
        y0 = R.y.cpu().numpy().copy()
        err = parity_all_rows(w, R.inp, y0)
        vid = mbg.select_variant(w.dtype, R.As[0], R.x)
        vname = mbg.variants(w.dtype)[vid]["name"]
        vkind = mbg.variants(w.dtype)[vid]["kind"]
        g, plan, t = chain(R, False)
        g_ov, _, t_ov = chain(R, True)
        rec = {"M": w.M, "N": w.N, "weights": w.dtype, "variant": vname,
               "kernel": KERNEL_NAMES[vkind], "bytes": R.step_bytes, "rotation_copies": R.copies,
               "us": t * 1e6, "gbs": gbs(R.step_bytes, t),
               "mbu_probe_pct": 100.0 * gbs(R.step_bytes, t) / ceiling,
               "mbu_spec_pct": 100.0 * gbs(R.step_bytes, t) / SPEC_HBM_GBS,
               "overlap_us": t_ov * 1e6, "overlap_gbs": gbs(R.step_bytes, t_ov),
               "overlap_mbu_probe_pct": 100.0 * gbs(R.step_bytes, t_ov) / ceiling,
               "parity_max_normalised_error": err, "parity_rows": w.M, "tolerance": TOL[w.dtype],
               "parity_ok": bool(err <= TOL[w.dtype])}
        if mbg.gemv_get_device_error(stream) != mbg.OK:
            rec["device_status"] = "timeout reported"
        out["workloads"][name] = rec
        if name in keep:
            R.inp = None
            resident[name] = (R, g, plan)
        else:
            R.free()
            del g
        del g_ov
        torch.cuda.empty_cache()

    # the fixed cost of one launch in such a chain: the smallest GEMV (FP16,
    # 2 x 512, 2 KB of weights, L2-resident), timed the same way; a matrix of
    # B bytes cannot take less than about B / probe + this per launch
    import numpy as np
    wf = synth.random_case("f16", 2, 512, 7)
    inf = synth.make(wf)
    A_f = torch.from_numpy(inf["A"].view(np.float16)).to(dev)
    x_f = torch.from_numpy(inf["x"].view(np.float16)).to(dev)
    y_f = torch.empty(2, dtype=torch.float32, device=dev)
    floor = {"shape": "f16 2x512 (2 KB of weights, L2-resident)"}
    for key, ov in (("us", False), ("overlap_us", True)):
        def launch(i, overlap):
            mbg.gemv("f16", A_f, x_f, None, y=y_f, overlap=overlap)
        plan = [(args.config_launches, 1)]
        g = timer.capture(launch, plan, overlap=ov, copies=2)
        timer.warm(g, plan, 1)
        floor[key] = timer.timed(g, plan) / args.config_launches * 1e6
        del g
    out["launch_floor"] = floor

    for shape, names in INTERLEAVED.items():
        best = {n: float("inf") for n in names}
        for _ in range(args.interleave_rounds):
            for n in names:
                R, g, plan = resident[n]
                best[n] = min(best[n], timer.timed(g, plan) / plan[0][0])
        f16_t = best[names[0]]
        entry = {}
        for n in names:
            R = resident[n][0]
            entry[R.w.dtype] = {"workload": n, "us": best[n] * 1e6, "gbs": gbs(R.step_bytes, best[n]),
                                "mbu_probe_pct": 100.0 * gbs(R.step_bytes, best[n]) / ceiling,
                                "x_fp16": f16_t / best[n]}
        out["interleaved"][shape] = entry
    out["interleaved_how"] = (f"FP16, INT8 and INT4 graphs of the same shape timed in turn, "
                              f"{args.interleave_rounds} rounds, best round per kernel; x_fp16 = FP16 time / "
                              f"kernel time (\"membound\", dequant GEMV: INT4 cap 3.87x)")
    for R, g, plan in resident.values():
        R.free()
    resident.clear()
    torch.cuda.empty_cache()
    out["seconds"] = time.monotonic() - t_start
    return out


SOFTMAX_METRIC = "achieved HBM GB/s (one read + one write per element) and MBU% vs measured copy ceiling for FP16 row softmax"


def run_softmax(args):
    """Row softmax ("membound", "Bonus kernel"): bytes = 2 (read) + 2 (write) per element;
    the denominator is the copy probe, because the kernel reads and writes every element."""
    import numpy as np
    import torch

    import memory_bound_gemv_gb300 as mbg

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    w = synth.SOFTMAX_WORKLOADS[args.workload]
    bits = synth.weight_rows(w, 0, w.M)
    x0 = torch.from_numpy(bits.view(np.float16)).to(dev)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20))
    copies = rotation_copies(2 * w.M * w.N, l2)
    xs = [x0] + [x0.clone() for _ in range(copies - 1)]
    y = torch.empty_like(x0)
    step_bytes = 4 * w.M * w.N
    stream = torch.cuda.Stream(dev)
    timer = Timer(dev, stream, l2)
    with torch.cuda.stream(stream):
        mbg.gemv_softmax_f16(x0, y=y)
    stream.synchronize()
    y_first = y.cpu().numpy().view(np.uint16).copy()

    half = (int(args.probe_gib * (1 << 30)) // 2) // 16 * 16
    src = torch.randint(-2 ** 31, 2 ** 31 - 1, (half // 4,), dtype=torch.int32, device=dev)
    dst = torch.empty_like(src)

    def copy_probe():
        res = {}
        with torch.cuda.stream(stream):
            for v, name in enumerate(mbg.copy_probe_variants()):
                for _ in range(2):
                    mbg.gemv_probe_copy(src, dst, v)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(args.probe_reps):
                    mbg.gemv_probe_copy(src, dst, v)
                e1.record(stream)
                e1.synchronize()
                res[name] = gbs(2 * half * args.probe_reps, e0.elapsed_time(e1) * 1e-3)
        return res

    def launch(i, overlap=False):
        mbg.gemv_softmax_f16(xs[i % copies], y=y)

    before = copy_probe()
    plan = graph_plan(args.steps, copies, min(args.graph_max, 50 * copies))
    graphs = timer.capture(launch, plan, copies=copies)
    timer.warm(graphs, plan, args.warmup)
    t = timer.timed(graphs, plan)
    steps = args.steps
    after = copy_probe()
    best = {k: max(before[k], after[k]) for k in before}
    ceiling = max(best.values())
    value = gbs(steps * step_bytes, t)
    rows = sorted({0, w.M // 2, w.M - 1})
    import oracle
    ref = oracle.load().softmax(bits, w.M, w.N, rows=rows, threads=cpu_threads())
    got = y_first[rows].view(np.float16).astype(np.float64)
    err = float(np.max(np.abs(got - ref) / np.maximum(ref, 1e-4)))
    peak, peak_kind = measured_peak()
    line = {"metric": SOFTMAX_METRIC, "value": value, "unit": "GB/s", "n_gpus": 1, "steps": steps,
            "warmup": args.warmup, "ms_per_step": t / steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic (seeded SplitMix64 normal(0, 2) logits rounded to FP16)",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "rotation_copies": copies,
                       "l2_policy": "inputs larger than L2: the logits rotate through the copies",
                       "launch": " + ".join(f"{reps} x graph of {n} launches" for n, reps in plan)},
            "mbu": {"copy_probe_gbs": ceiling, "mbu_copy_pct": 100.0 * value / ceiling, "probes": best},
            "roofline": {"bound": "hbm", "achieved": value, "peak": peak, "unit": "GB/s",
                         "frac": value / peak, "peak_kind": peak_kind,
                         "traffic": recorded_traffic(w.name, "auto")},
            "parity_rows_max_rel_err": err, "gpu_launches": steps}
    print(json.dumps(line), flush=True)
    if args.json_out:
        with open(args.json_out, "w") as f:
            json.dump(line, f, indent=1)
    return 0


def run_profile(args):
    """Each kernel launched once (for an ncu capture of the top kernel)."""
    import numpy as np
    import torch

    import memory_bound_gemv_gb300 as mbg

    torch.cuda.set_device(0)
    w = synth.WORKLOADS[args.workload]
    inp = synth.make(w)
    A = torch.from_numpy(inp["A"].view(np.float16) if f16_weights(w.dtype) else inp["A"]).cuda()
    x = torch.from_numpy(inp["x"] if f32_x(w.dtype) else inp["x"].view(np.float16)).cuda()
    S = torch.from_numpy(inp["scales"].view(np.float16)).cuda() if w.quantised else None
    if w.dtype == "q8row":
        S = S.reshape(-1)
    if args.variant:
        vid = [v["id"] for v in mbg.variants(w.dtype) if v["name"] == args.variant]
        if not vid:
            raise SystemExit(f"no variant {args.variant!r} for {w.dtype}")
        vid = vid[0]
        y = mbg.gemv_run_variant(w.dtype, vid, A, x, S)
    else:
        vid = mbg.select_variant(w.dtype, A, x)
        y = mbg.gemv(w.dtype, A, x, S)
    torch.cuda.synchronize()
    print(json.dumps({"profile": w.name, "variant": mbg.variants(w.dtype)[vid]["name"],
                      "y0": float(y[0].item())}))
    return 0


def run_profile_softmax(args):
    """One launch of the row softmax (for an ncu capture)."""
    import numpy as np
    import torch

    import memory_bound_gemv_gb300 as mbg

    torch.cuda.set_device(0)
    w = synth.SOFTMAX_WORKLOADS[args.workload]
    x = torch.from_numpy(synth.weight_rows(w, 0, w.M).view(np.float16)).cuda()
    y = mbg.gemv_softmax_f16(x)
    torch.cuda.synchronize()
    print(json.dumps({"profile": w.name, "y00": float(y[0, 0].item())}))
    return 0


def run_profile_aux(args):
    """The kernels off the GEMV and softmax paths, each launched once (for one ncu capture):
    every read and copy probe pattern over 256 MiB (twice L2), the quantiser (INT8 per group,
    INT8 per row, INT4) of the FP16 4096x14336 decode matrix and the dequantisation of its output,
    one host-buffer call (x fetched by the copy kernel), the zero fill of an N = 0 call and the
    softmax kernel for any layout (rows of 8191 values)."""
    import numpy as np
    import torch

    import memory_bound_gemv_gb300 as mbg

    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    gen = torch.Generator(device="cpu").manual_seed(7)
    words = (256 << 20) // 4
    buf = torch.randint(-2 ** 31, 2 ** 31 - 1, (words,), dtype=torch.int32, generator=gen).to(dev)
    sink = torch.zeros(1, dtype=torch.int64, device=dev)
    for v in range(len(mbg.probe_variants())):
        mbg.gemv_probe_read(buf, sink, v)
    dst = torch.empty_like(buf)
    for v in range(len(mbg.copy_probe_variants())):
        mbg.gemv_probe_copy(buf, dst, v)
    torch.cuda.synchronize()
    del buf, dst
    w = synth.WORKLOADS[DEFAULT_WORKLOAD]
    inp = synth.make(w)
    W = torch.from_numpy(inp["A"].view(np.float16)).to(dev)
    A8, S8 = mbg.quantize(W, "q8")
    mbg.quantize(W, "q8row")
    A4, S4 = mbg.quantize(W, "q4")
    mbg.gemv_dequant_q8(A8, S8)
    mbg.gemv_dequant_q4(A4, S4)
    x_host = torch.from_numpy(inp["x"].view(np.float16)).pin_memory()
    x_dev = torch.empty(w.N, dtype=torch.float16, device=dev)
    y_host = mbg.gemv_host("f16", W, x_host, x_dev)
    y0 = torch.full((w.M,), 7.0, device=dev)
    _ = mbg.lib().gemv_f32(0, 0, y0.data_ptr(), w.M, 0, None)
    xs = torch.randn(8192, 8191, generator=gen).to(torch.float16).to(dev)
    ys = mbg.gemv_softmax_f16(xs)  # 8191 is no multiple of 8: the any-layout kernel
    torch.cuda.synchronize()
    print(json.dumps({"profile": "aux", "y0": float(y_host[0].item()), "zero_fill": float(y0.abs().max().item()),
                      "softmax_row_sum": float(ys[0].float().sum().item())}))
    return 0


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--op", choices=("gemv", "softmax", "aux"), default="gemv",
                   help="aux (with --profile): the probes, quantiser, host copy and edge kernels once each")
    p.add_argument("--workload", default=None,
                   choices=sorted(synth.WORKLOADS) + sorted(synth.SOFTMAX_WORKLOADS))
    p.add_argument("--graph-max", type=int, default=GRAPH_MAX, help="launches per captured graph")
    p.add_argument("--probe-gib", type=float, default=1.0)
    p.add_argument("--probe-reps", type=int, default=10)
    p.add_argument("--e2e-steps", type=int, default=5000, help="e2e steps (at most --steps)")
    p.add_argument("--e2e-min-steps", type=int, default=200, help="e2e steps at least")
    p.add_argument("--long-steps", type=int, default=2000, help="launches of the comparison long chain")
    p.add_argument("--clock-seconds", type=float, default=1.0)
    p.add_argument("--config-launches", type=int, default=200)
    p.add_argument("--interleave-rounds", type=int, default=5)
    p.add_argument("--cpu-seconds", type=float, default=5.0)
    p.add_argument("--cpu-rows", type=int, default=512)
    p.add_argument("--reference-seconds", type=float, default=60.0)
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-overlap", action="store_true")
    p.add_argument("--no-long-chain", action="store_true")
    p.add_argument("--no-configs", action="store_true", help="skip the per-workload block")
    p.add_argument("--profile", action="store_true", help="one launch of the GEMV, for ncu")
    p.add_argument("--variant", default=None, help="kernel variant name for --profile")
    p.add_argument("--json-out", default=None)
    args = p.parse_args(argv)
    if args.steps < 1 or args.warmup < 0:
        p.error("--steps must be >= 1 and --warmup >= 0")
    if args.op == "aux":
        if not args.profile:
            p.error("--op aux runs only with --profile")
        return run_profile_aux(args)
    if args.workload is None:
        args.workload = "softmax_8192x8192" if args.op == "softmax" else DEFAULT_WORKLOAD
    if args.op == "softmax":
        if args.workload not in synth.SOFTMAX_WORKLOADS:
            p.error("--op softmax needs a softmax_* workload")
        if args.profile:
            return run_profile_softmax(args)
        return run_softmax(args)
    if args.workload not in synth.WORKLOADS:
        p.error("GEMV workloads: " + ", ".join(sorted(synth.WORKLOADS)))
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
