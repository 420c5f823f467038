#!/usr/bin/env python3
"""Benchmark of the GEMV library on one GB300 (or N replicas, one per GPU).

Headline: achieved HBM GB/s of the FP16 4096x14336 GEMV (the decode
down-projection shape), and its memory-bandwidth utilisation against the
pure-read ceiling measured in the same run ("membound", sections "Results" and
"Why GEMV, and why MBU").

One step = one GEMV launch over the whole workload: choose the kernel, stage
x, stream A, accumulate, reduce, write y.  Weights rotate through enough
copies (at least max(256 MiB, 4 x L2)) that every launch reads A cold from
HBM ("membound", gotcha 1); x stays resident.  Steps are replayed from CUDA
graphs of back-to-back launches and timed with CUDA events on the launching
stream.  Algorithmic bytes per step = A + scales + x read once, y written
once ("Making GEMV Fast", section "Memory Access").

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead (the reference arm: there is no runnable upstream
code).
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


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "memory_bound_gemv_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        # the probe kernels (their own file) do not touch the recorded kernels
        if f.endswith((".cu", ".cuh", ".h")) and f != "gemv_probe.cu":
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


class ClockSampler:
    """nvidia-smi sampled every 50 ms; keeps the samples inside [mark_start, mark_end]."""

    def __init__(self, gpu_id: str):
        self.samples = []
        self.window = [None, None]
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

    def mark_start(self):
        self.window[0] = time.monotonic()

    def mark_end(self):
        self.window[1] = time.monotonic()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": f"nvidia-smi unavailable: {self.error}"}
        t0, t1 = self.window
        inside = [s for s in self.samples if t0 is not None and t1 is not None and t0 <= s["t"] <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "timed region shorter than the sampling interval"}
        reasons = sorted({r for s in inside for r in s["reasons"]})
        return {"sm_mhz": statistics.median(s["sm"] for s in inside),
                "sm_max_mhz": max(s["sm_max"] for s in inside), "reasons": reasons,
                "samples": len(inside)}


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
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import numpy as np
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
    inp = synth.make(w)

    def to_dev(arr, kind):
        if kind == "f16bits":
            return torch.from_numpy(np.ascontiguousarray(arr).view(np.float16)).to(dev)
        return torch.from_numpy(np.ascontiguousarray(arr)).to(dev)

    A0 = to_dev(inp["A"], "f16bits" if f16_weights(w.dtype) else "raw")
    x = to_dev(inp["x"], "raw" if f32_x(w.dtype) else "f16bits")
    S0 = to_dev(inp["scales"], "f16bits") if w.quantised else None
    if w.dtype == "q8row":
        S0 = S0.reshape(-1)  # one scale per row: [M]
    wbytes = a_bytes(w.dtype, w.M, w.N) + scale_bytes(w.dtype, w.M, w.N)
    copies = rotation_copies(wbytes, l2)
    As = [A0] + [A0.clone() for _ in range(copies - 1)]
    Ss = [S0] + [S0.clone() for _ in range(copies - 1)] if w.quantised else [None] * copies
    y = torch.empty(w.M, dtype=torch.float32, device=dev)
    step_bytes = algorithmic_bytes(w.dtype, w.M, w.N)
    stream = torch.cuda.Stream(dev)

    vid = mbg.select_variant(w.dtype, A0, x)
    vinfo = mbg.variants(w.dtype)[vid]

    def launch(i, overlap=False):
        mbg.gemv(w.dtype, As[i % copies], x, Ss[i % copies], y=y, overlap=overlap)

    # first launch: keep the result for the parity sample of the cpu_baseline leg
    with torch.cuda.stream(stream):
        launch(0)
    stream.synchronize()
    y_first = y.cpu().numpy().copy()
    if mbg.gemv_get_device_error(stream) != mbg.OK:
        raise SystemExit("device status word set on the first launch")

    # ---- pure-read probe (before) ----
    probe_bytes = int(args.probe_gib * (1 << 30)) // 16 * 16
    probe_buf = torch.randint(-2 ** 31, 2 ** 31 - 1, (probe_bytes // 4,), dtype=torch.int32, device=dev)
    sink = torch.zeros(1, dtype=torch.int64, device=dev)
    probe_names = mbg.probe_variants()

    def run_probes(reps=args.probe_reps):
        res = {}
        with torch.cuda.stream(stream):
            for v, name in enumerate(probe_names):
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

    probe_before = run_probes()

    # ---- graphs of back-to-back launches ----
    batch = copies * max(1, math.ceil(args.graph_batch / copies))
    n_full, n_tail = split_steps(args.steps, batch)
    stream.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(stream):
        for i in range(3):
            launch(i)
    stream.synchronize()
    g_main = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_main, stream=stream):
        for i in range(batch):
            launch(i)
    g_tail = None
    if n_tail:
        g_tail = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_tail, stream=stream):
            for i in range(n_tail):
                launch(i)

    # warm-up: W launches
    w_full, w_tail = split_steps(args.warmup, batch)
    with torch.cuda.stream(stream):
        for _ in range(w_full):
            g_main.replay()
        for i in range(w_tail):
            launch(i)
    stream.synchronize()

    sampler = ClockSampler(gpu_id_for(local_rank)) if not args.no_clocks else None
    if sampler is not None:
        time.sleep(0.3)  # let nvidia-smi start
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    if sampler is not None:
        sampler.mark_start()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n_full):
            g_main.replay()
        if g_tail is not None:
            g_tail.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    if sampler is not None:
        sampler.mark_end()
    barrier()
    elapsed = e0.elapsed_time(e1) * 1e-3
    if sampler is not None:
        sampler.stop()
    t_max = max_over_ranks(elapsed, dev)
    per_launch = elapsed / max(1, args.steps)
    value = gbs(world * args.steps * step_bytes, t_max)

    # ---- the same chain launched with programmatic dependent launch ----
    # (gemv_ex with GEMV_FLAG_OVERLAP_PRECEDING: each launch may start while
    # the previous one finishes; weights are never written by the chain)
    overlap = None
    if not args.no_overlap and n_full > 0:
        g_ov = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for i in range(copies):
                launch(i, overlap=True)
        stream.synchronize()
        with torch.cuda.graph(g_ov, stream=stream):
            for i in range(batch):
                launch(i, overlap=True)
        with torch.cuda.stream(stream):
            for _ in range(max(1, w_full)):
                g_ov.replay()
        stream.synchronize()
        barrier()
        with torch.cuda.stream(stream):
            o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            o0.record(stream)
            for _ in range(n_full):
                g_ov.replay()
            o1.record(stream)
        o1.synchronize()
        barrier()
        ov_t = max_over_ranks(o0.elapsed_time(o1) * 1e-3, dev)
        ov_steps = n_full * batch
        overlap = {"value": gbs(world * ov_steps * step_bytes, ov_t), "unit": "GB/s", "steps": ov_steps,
                   "ms_per_step": ov_t / ov_steps * 1e3,
                   "how": "same graph of back-to-back launches, each launched with programmatic "
                          "dependent launch (weights requested before waiting for the previous launch)"}
        del g_ov

    # ---- the same launches without graphs (host-launched stream), for context ----
    eager_steps = min(args.steps, 2000)
    with torch.cuda.stream(stream):
        for i in range(copies):
            launch(i)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for i in range(eager_steps):
            launch(i)
        f1.record(stream)
    f1.synchronize()
    eager_gbs = gbs(eager_steps * step_bytes, f0.elapsed_time(f1) * 1e-3)

    probe_after = run_probes()
    probe_all = {k: max(probe_before[k], probe_after[k]) for k in probe_before}
    best_probe = max(probe_all, key=probe_all.get)
    ceiling = probe_all[best_probe]
    if overlap is not None:
        overlap["mbu_probe_pct"] = 100.0 * overlap["value"] / world / ceiling

    # ---- end to end: x from pinned host memory, y back to pinned host memory ----
    e2e = None
    if not args.no_e2e:
        x_host = x.cpu().pin_memory()
        y_host = torch.empty(w.M, dtype=torch.float32).pin_memory()
        x_dev = torch.empty_like(x)
        e2e_steps = min(args.steps, args.e2e_steps)

        def e2e_run(overlap_flag):
            # one public call per step: x_host -> device, the GEMV, y written to y_host
            def e2e_step(i):
                if w.dtype == "q8row":
                    x_dev.copy_(x_host, non_blocking=True)
                    mbg.gemv(w.dtype, As[i % copies], x_dev, Ss[i % copies], y=y_dev_rowscale)
                    y_host.copy_(y_dev_rowscale, non_blocking=True)
                else:
                    mbg.gemv_host(w.dtype, As[i % copies], x_host, x_dev, Ss[i % copies], y_host=y_host,
                                  overlap=overlap_flag)

            with torch.cuda.stream(stream):
                for i in range(min(args.warmup, 50)):
                    e2e_step(i)
                stream.synchronize()
                barrier()
                h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                h0.record(stream)
                for i in range(e2e_steps):
                    e2e_step(i)
                h1.record(stream)
            h1.synchronize()
            barrier()
            return max_over_ranks(h0.elapsed_time(h1) * 1e-3, dev)

        y_dev_rowscale = torch.empty_like(y)
        e2e_t = e2e_run(False)
        e2e_ov = e2e_run(True) if w.dtype != "q8row" else None
        e2e = {"value": gbs(world * e2e_steps * step_bytes, e2e_t), "unit": "GB/s",
               "h2d_bytes_per_step": int(x.numel() * x.element_size()),
               "d2h_bytes_per_step": int(y.numel() * y.element_size()),
               "steps": e2e_steps,
               "how": "per step one gemv_ex_host call through the C ABI: x read from pinned host memory "
                      "by a copy kernel into a device buffer, the GEMV launched after it with programmatic "
                      "dependent launch, y written by the GEMV into pinned host memory; weights resident "
                      "and rotated" if w.dtype != "q8row" else
                      "per step: pinned x -> device, gemv through the C ABI, y -> pinned host",
               "overlap_value": gbs(world * e2e_steps * step_bytes, e2e_ov) if e2e_ov else None,
               "overlap_how": "the same calls with GEMV_FLAG_OVERLAP_PRECEDING (each copy of x may "
                              "start before the previous GEMV ends)"}

    peak, peak_kind = measured_peak()
    achieved = gbs(step_bytes, per_launch)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_kind": peak_kind,
                "traffic": recorded_traffic(w.name, vinfo["name"]),
                "kernel": f"gemv_{vinfo['kind']}_kernel {vinfo['name']}"}
    clocks = sampler.summary() if sampler is not None else {"sm_mhz": None, "note": "disabled"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        threads = cpu_threads()
        cb, calls, nrows, el = time_oracle(w, args.cpu_seconds, threads, args.cpu_rows)
        rows = list(range(nrows))
        A_s, x_s, s_s, idx = oracle_rows(w, rows)
        y_ref, den = oracle.load().gemv(w.dtype, A_s, x_s, nrows, w.N, scales=s_s, rows=idx,
                                        threads=threads)
        cpu = {"value": cb, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{calls} oracle passes over rows 0..{nrows - 1} of the workload "
                         f"({el:.1f} s, double precision, {threads} threads)",
               "parity_max_normalised_error": oracle.max_normalised_error(y_first[:nrows], y_ref, den)}

    published = PUBLISHED.get(w.name)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max / max(1, args.steps) * 1e3,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (value / world / published[0]) if published else None,
        "vs_baseline_note": published[1] if published else None,
        "dtype": w.dtype, "data": "synthetic (seeded SplitMix64; weights and x normal(0,0.02) "
                                  "rounded to FP16)" if w.dtype == "f16" else "synthetic (seeded SplitMix64)",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "weights": w.dtype,
                   "variant": vinfo["name"], "rotation_copies": copies,
                   "rotation_bytes": copies * wbytes, "l2_bytes": l2,
                   "l2_policy": "inputs larger than L2: weights rotate through the copies, each "
                                "launch reads A cold from HBM",
                   "launch": f"CUDA graph of {batch} back-to-back launches",
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
        "eager_stream_gbs": eager_gbs,
        "overlap": overlap,
        "ms_per_launch": per_launch * 1e3,
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

    before = copy_probe()
    batch = copies * max(1, math.ceil(min(args.graph_batch, 50) / copies))
    n_full, n_tail = split_steps(args.steps, batch)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(batch):
            mbg.gemv_softmax_f16(xs[i % copies], y=y)
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup // batch)):
            g.replay()
    stream.synchronize()
    with torch.cuda.stream(stream):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(max(1, n_full)):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    steps = max(1, n_full) * batch
    t = e0.elapsed_time(e1) * 1e-3
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
                       "launch": f"CUDA graph of {batch} back-to-back launches"},
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


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30000)
    p.add_argument("--warmup", type=int, default=300)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--op", choices=("gemv", "softmax"), default="gemv")
    p.add_argument("--workload", default=None,
                   choices=sorted(synth.WORKLOADS) + sorted(synth.SOFTMAX_WORKLOADS))
    p.add_argument("--graph-batch", type=int, default=100)
    p.add_argument("--probe-gib", type=float, default=1.0)
    p.add_argument("--probe-reps", type=int, default=10)
    p.add_argument("--e2e-steps", type=int, default=5000)
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--cpu-rows", type=int, default=512)
    p.add_argument("--reference-seconds", type=float, default=60.0)
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-overlap", action="store_true")
    p.add_argument("--profile", action="store_true", help="one launch of the GEMV, for ncu")
    p.add_argument("--variant", default=None, help="kernel variant name for --profile")
    p.add_argument("--json-out", default=None)
    args = p.parse_args(argv)
    if args.steps < 1 or args.warmup < 0:
        p.error("--steps must be >= 1 and --warmup >= 0")
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
