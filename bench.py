"""Benchmark of the streaming-reduction hot path on GB300.

One step runs every kernel of the path once over its full synthetic workload:

  gemv      packed-int8 dequant GEMV, W 8192 x 16384, one vector
  segments  ragged row sums of 65,536 segments of 63 x 32 f32
  batched   packed-int8 dequant-dot, its own W (same shape and values as the
            GEMV's, a separate array) against 16 vectors
  wide      ragged row sums of a 16,384 x 16,384 f32 matrix

The four workloads are independent, so a step runs them as two lanes (CUDA
streams) that overlap: segments then batched on one, wide then gemv on the
other; an event forks both lanes off the launching stream and the step ends
when both have joined it again.  Each kernel reads its own arrays and every
array exceeds the 129 MB L2, so no kernel finds another's data in L2.

The metric is HBM GB/s over algorithmic bytes (only the bytes the method
must move: active rows, metadata, outputs).  Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --profile {gemv,segments,batched,batched_dp4a,wide,...} [--launches N]
      (no timing: runs one kernel's workload for an ncu capture)
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "HBM GB/s and % of GB300 peak: ragged f32 row-sum, packed-int8 dequant-dot"
WORKLOAD = ("gemv 8192x16384 int8 + 65536 ragged 63x32 f32 segments + batched dot 8192x16384x16 "
            "int8 + 16384x16384 f32 ragged wide rows")
ORDER = ("gemv", "segments", "batched", "wide")
#: the step's concurrent lanes: each lane is a CUDA stream running its kernels in
#: order; measured best of the two- and three-lane splits (segments is bound by
#: instruction issue and leaves HBM time that the wide rows use)
STEP_LANES = (("segments", "batched"), ("wide", "gemv"))
#: the same step on one stream (`--lanes 1`), for comparison
ONE_LANE = (ORDER,)
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------------------
# workload
# ----------------------------------------------------------------------------

def make_inputs():
    import synth
    seg = synth.batched_segments()
    wide = synth.wide_rows()
    gemv = synth.dequant_gemv()
    bat = synth.dequant_batched()
    return {"segments": seg, "wide": wide, "gemv": gemv, "batched": bat}


def leading(n: int, frac: float) -> int:
    """The number of leading units a sample of fraction `frac` takes (all when frac >= 1)."""
    return n if frac >= 1.0 else max(1, min(n, int(np.ceil(frac * n))))


def algorithmic_bytes(inp, frac: float = 1.0) -> dict:
    """Bytes each kernel must move once: active data, metadata and outputs; with
    frac < 1, those of the leading segments / rows of each workload only."""
    seg, wide = inp["segments"], inp["wide"]
    out = {}
    m = leading(seg["num_segments"], frac)
    c = seg["counts"][:m].astype(np.int64)
    out["segments"] = int(128 * c.sum() + m * (4 + 4 + 16))
    m = leading(wide["num_segments"], frac)
    L = wide["counts"][:m].astype(np.int64)
    out["wide"] = int(4 * L.sum() + m * (4 + 16))
    for name in ("gemv", "batched"):
        d = inp[name]
        n, k = d["w"].shape
        n = leading(n, frac)
        b = d["x"].shape[0]
        out[name] = int(n * k + 4 * n + b * k + 4 * b + 4 * n * b)
    return out


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic():
    """Per-kernel DRAM bytes per launch from the committed ncu summary, each valid
    only while the sources of that workload's kernels hash to the value recorded
    with it."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return {}
    out = {}
    for name, rec in d.get("workloads", {}).items():
        if rec.get("source_hash") == source_hash(name):
            out[name] = rec.get("bytes_per_launch")
    return out


#: the source files each workload's kernels are built from
KERNEL_SOURCES = {
    "segments": ("row_sum.cu",), "wide": ("row_sum.cu",),
    "gemv": ("dequant_dot.cu",), "batched": ("dot_tc.cu", "dot_tc_rows.cu", "tc_ptx.cuh"),
    "packed": ("packed_dot.cu",),
    "sum_rows": ("lane_sum.cu",), "sum_vector_rows": ("lane_sum.cu",), "guarded_rows": ("lane_sum.cu",),
    "routed": ("routed.cu",),
}
SHARED_SOURCES = ("common.cuh", "internal.h", "loom_api.cu")


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and blank lines (string and character
    literals kept whole), so that editing a comment leaves the hash unchanged."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
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
    lines = (line.rstrip() for line in "".join(out).split("\n"))
    return "\n".join(line for line in lines if line)


def source_hash(workload: str) -> str:
    """Hash of the code (comments and blank lines left out) that a workload's
    kernels are built from."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "int8_dequant_dot_gb300", "csrc")
    for f in sorted(KERNEL_SOURCES[workload] + SHARED_SOURCES):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + b"\0" + strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


class DeviceWorkload:
    """Device copies of the inputs and outputs, and one launch per kernel."""

    def __init__(self, inp, torch, loom, stream, depth=0):
        self.torch, self.loom, self.stream = torch, loom, stream
        self.inp = inp
        dev = torch.device("cuda")
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        seg, wide, gemv, bat = inp["segments"], inp["wide"], inp["gemv"], inp["batched"]
        self.d = {
            "seg_values": t(seg["values"]), "seg_counts": t(seg["counts"]), "seg_init": t(seg["initial"]),
            "wide_values": t(wide["values"]), "wide_counts": t(wide["counts"]),
            "w": t(gemv["w"].view("<i4")), "sw": t(gemv["scale_w"]),
            "x1": t(gemv["x"].view("<i4")), "sx1": t(gemv["scale_x"]),
            "wb": t(bat["w"].view("<i4")), "swb": t(bat["scale_w"]),
            "x16": t(bat["x"].view("<i4")), "sx16": t(bat["scale_x"]),
        }
        i32, f32 = torch.int32, torch.float32
        S, R = seg["num_segments"], wide["num_segments"]
        self.o = {
            "seg": tuple(torch.empty(S, dtype=dt, device=dev) for dt in (i32, i32, f32, f32)),
            "wide": tuple(torch.empty(R, dtype=dt, device=dev) for dt in (i32, i32, f32, f32)),
            "y1": torch.empty((8192, 1), dtype=f32, device=dev),
            "y16": torch.empty((8192, 16), dtype=f32, device=dev),
        }
        self.tuning = loom.make_tuning(depth=depth) if depth else None
        # one kernel each for segments, wide and gemv; the batched dot is one tensor-core
        # launch, or two when its schedule splits bands between CTAs (streaming + finishing)
        L = loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT, [8192, 16384, 16, 1, 0, 0, 0, 0, 1])
        self.launches_per_step = 3 + (2 if L["kernel"] == loom.LOOM_KERNEL_DOT_TENSOR_SPLIT else 1)

    def launch(self, name, stream=None):
        L, d, o = self.loom, self.d, self.o
        s = self.stream if stream is None else stream
        if name == "segments":
            L.loom_row_sum_batched_ex(d["seg_values"], 65536, 2016, 63, 32, d["seg_counts"], d["seg_init"],
                                      8, out=o["seg"], tuning=self.tuning, stream=s)
        elif name == "wide":
            L.loom_row_sum_batched_ex(d["wide_values"], 16384, 16384, 16384, 1, d["wide_counts"], None,
                                      8, out=o["wide"], tuning=self.tuning, stream=s)
        elif name == "gemv":
            L.loom_i8_dequant_dot_ex(d["w"], d["sw"], 8192, 16384, d["x1"], d["sx1"], 1, y=o["y1"],
                                     tuning=self.tuning, stream=s)
        elif name == "batched":
            L.loom_i8_dequant_dot_ex(d["wb"], d["swb"], 8192, 16384, d["x16"], d["sx16"], 16, y=o["y16"],
                                     tuning=self.tuning, stream=s)
        else:
            raise ValueError(name)


class Step:
    """One step: the lanes (STEP_LANES by default) forked off the launching stream by an
    event, each on a stream of its own, and joined back by one event per lane."""

    def __init__(self, torch, work, lanes=STEP_LANES):
        self.work, self.lanes = work, lanes
        self.streams = [torch.cuda.Stream() for _ in lanes]
        self.fork = torch.cuda.Event()
        self.joins = [torch.cuda.Event() for _ in lanes]

    def run(self, main):
        self.fork.record(main)
        for lane, s, j in zip(self.lanes, self.streams, self.joins):
            s.wait_event(self.fork)
            for name in lane:
                self.work.launch(name, stream=s)
            j.record(s)
        for j in self.joins:
            main.wait_event(j)


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons every 20 ms; each
    sample carries nvidia-smi's own timestamp, so that only the samples taken
    inside the timed region are reported."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.index = index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    @staticmethod
    def parse(out: str):
        """(wall-clock seconds, sm MHz, max MHz, set of active reasons) per sample line."""
        import datetime
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = {nm for nm, v in zip(ClockSampler.NAMES, parts[5:9]) if v.lower() == "active"}
            rows.append((t, sm, mx, reasons))
        return rows

    def stop(self, window=None):
        """Summary of the samples inside `window` (wall-clock start, end); when no
        sample falls inside it, of all samples, marked as such."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return self.summarise(self.parse(out), window)

    @staticmethod
    def summarise(rows, window=None):
        if not rows:
            return None
        inside = [r for r in rows if window and window[0] <= r[0] <= window[1]]
        use = inside or rows
        reasons = set()
        for r in use:
            reasons |= r[3]
        out = {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
               "reasons": sorted(reasons), "samples": len(use), "in_timed_region": bool(inside)}
        if window:
            out["timed_region_ms"] = round((window[1] - window[0]) * 1e3, 1)
        return out


# ----------------------------------------------------------------------------
# CPU oracle baseline (and the reference arm)
# ----------------------------------------------------------------------------

def oracle_step(inp, threads, frac: float = 1.0):
    """One oracle pass over every workload (frac < 1: their leading segments / rows)."""
    import oracle
    seg, wide, gemv, bat = inp["segments"], inp["wide"], inp["gemv"], inp["batched"]
    n = leading(gemv["w"].shape[0], frac)
    oracle.i8_dequant_dot(gemv["w"][:n], gemv["scale_w"][:n], gemv["x"], gemv["scale_x"], threads=threads)
    m = leading(seg["num_segments"], frac)
    oracle.row_sum_batched(seg["values"][:m], 2016, 63, 32, seg["counts"][:m], seg["initial"][:m], 8,
                           threads=threads)
    n = leading(bat["w"].shape[0], frac)
    oracle.i8_dequant_dot(bat["w"][:n], bat["scale_w"][:n], bat["x"], bat["scale_x"], threads=threads)
    m = leading(wide["num_segments"], frac)
    oracle.row_sum_batched(wide["values"][:m], 16384, 16384, 1, wide["counts"][:m], None, 8, threads=threads)


def oracle_workload(inp, name, threads, frac: float = 1.0):
    """One oracle pass over one workload (frac < 1: its leading segments / rows)."""
    import oracle
    if name in ("gemv", "batched"):
        d = inp[name]
        n = leading(d["w"].shape[0], frac)
        oracle.i8_dequant_dot(d["w"][:n], d["scale_w"][:n], d["x"], d["scale_x"], threads=threads)
    elif name == "segments":
        d = inp["segments"]
        m = leading(d["num_segments"], frac)
        oracle.row_sum_batched(d["values"][:m], 2016, 63, 32, d["counts"][:m], d["initial"][:m], 8,
                               threads=threads)
    else:
        d = inp["wide"]
        m = leading(d["num_segments"], frac)
        oracle.row_sum_batched(d["values"][:m], 16384, 16384, 1, d["counts"][:m], None, 8, threads=threads)


def cpu_per_workload(inp, threads, budget_s: float = 1.5) -> dict:
    """The oracle on each workload alone, single-threaded and on `threads` host
    threads: GB/s over the algorithmic bytes of a leading sample of the workload
    sized so that the single-threaded pass takes about `budget_s` seconds."""
    out = {}
    for name in ORDER:
        probe = 1.0 / 64
        t0 = time.perf_counter()
        oracle_workload(inp, name, 1, probe)
        t_probe = max(time.perf_counter() - t0, 1e-6)
        frac = min(1.0, probe * budget_s / t_probe)
        nbytes = algorithmic_bytes(inp, frac)[name]
        t0 = time.perf_counter()
        oracle_workload(inp, name, 1, frac)
        t1 = time.perf_counter() - t0
        reps, t0 = 0, time.perf_counter()
        while True:
            oracle_workload(inp, name, threads, frac)
            reps += 1
            tn = (time.perf_counter() - t0) / reps
            if time.perf_counter() - t0 >= budget_s / 2 or reps >= 50:
                break
        out[name] = {"gbs_1_thread": nbytes / t1 / 1e9, f"gbs_{threads}_threads": nbytes / tn / 1e9,
                     "sample_fraction": frac, "sample_bytes": nbytes}
    return out


def cpu_baseline(inp, total_bytes, threads, budget_s: float = 10.0):
    """The oracle as it stands on the host cores: whole steps (all four
    workloads) repeated until about `budget_s` seconds of work have run."""
    oracle_step(inp, threads)   # warm caches and the thread pool
    steps, t0 = 0, time.perf_counter()
    while True:
        oracle_step(inp, threads)
        steps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or steps >= 1000:
            break
    per = dt / steps
    return {"value": total_bytes / per / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{steps} full steps (all four workloads, {total_bytes / 1e9:.2f} GB of algorithmic bytes "
                      f"each), fp64/int64 C oracle, {threads} threads over independent segments/rows; "
                      f"{dt:.1f} s",
            "per_workload": cpu_per_workload(inp, threads),
            "per_workload_sample": "each workload alone: a leading sample of its segments / rows sized so that "
                                   "one single-threaded pass takes about 1.5 s, timed on 1 thread and on all "
                                   "host threads"}


#: wall-clock budget of the reference arm's K timed steps
REFERENCE_BUDGET_S = 120.0


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle timed as it stands on the host cores.  Each
    timed step is one oracle pass over the leading fraction of every workload's
    segments / rows, the fraction chosen so that the K steps take about two minutes
    at most (the whole workload when that fits)."""
    if rank != 0:
        return
    inp = make_inputs()
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle_step(inp, threads)   # first warm-up step: the full workload, timed for the sample size
    t_full = time.perf_counter() - t0
    for _ in range(max(args.warmup - 1, 0)):
        oracle_step(inp, threads)
    frac = min(1.0, REFERENCE_BUDGET_S / (max(args.steps, 1) * t_full))
    for _ in range(2):   # a pass has a fixed cost too: size the sample on its own timing
        if frac >= 1.0:
            break
        t0 = time.perf_counter()
        oracle_step(inp, threads, frac)
        frac = min(1.0, frac * REFERENCE_BUDGET_S / (max(args.steps, 1) * (time.perf_counter() - t0)))
    total = sum(algorithmic_bytes(inp, frac).values())
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(inp, threads, frac)
    dt = (time.perf_counter() - t0) / args.steps
    value = total / dt / 1e9
    sample = ("each step: one oracle pass over " +
              ("every workload in full" if frac >= 1.0 else
               f"the leading {100 * frac:.1f}% of every workload's segments / rows") +
              f" ({total / 1e9:.3f} GB of algorithmic bytes), fp64/int64 C oracle, {threads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64+i64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": "host threads", "sample_fraction": frac},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def slowest_rank_ms(elapsed_ms: float, dist, device) -> float:
    """The timed region's length on the slowest rank (every rank gets it)."""
    if dist is None:
        return elapsed_ms
    import torch
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, bytes_per_rank_step: int, ms_per_step: float) -> float:
    """Replicas: every rank moves the whole workload each step, so the job moves
    world times the bytes in the slowest rank's step time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def run_ours(args, rank, world, dist):
    import torch
    import int8_dequant_dot_gb300 as loom

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    stream = torch.cuda.Stream()
    inp = make_inputs()
    alg = algorithmic_bytes(inp)
    total = sum(alg.values())
    work = DeviceWorkload(inp, torch, loom, stream, depth=args.depth)
    lanes = STEP_LANES if args.lanes == 2 else ONE_LANE
    step = Step(torch, work, lanes)

    def barrier():
        if dist is not None:
            dist.barrier()

    # warm-up
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step.run(stream)
    stream.synchronize()

    # timed region: K whole steps between two events on the launching stream.
    # Within a lane nothing is recorded between the kernels: an event between two
    # launches costs about 2 us and stops the next kernel from being scheduled
    # while the previous one drains (programmatic dependent launch).
    step_start = torch.cuda.Event(enable_timing=True)
    step_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)   # let the sampler attach before the timed work
    t_region = time.time()
    with torch.cuda.stream(stream):
        # keep the device busy for ~1 ms while the host queues the first steps, so
        # that the events below never time host-side launch work on an idle device
        torch.cuda._sleep(2_000_000)
        step_start.record(stream)
        for _ in range(args.steps):
            step.run(stream)
        step_end.record(stream)
    stream.synchronize()
    region = (t_region, time.time())
    torch.cuda.synchronize()
    barrier()

    # per-kernel durations for the roofline: the same K steps again, the kernels
    # one after another on one stream, each launch between two events of its own
    # (so each kernel runs alone, as ncu sees it)
    ev = {name: [] for name in ORDER}
    with torch.cuda.stream(stream):
        torch.cuda._sleep(2_000_000)
        for _ in range(args.steps):
            for name in ORDER:
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                work.launch(name)
                b.record(stream)
                ev[name].append((a, b))
    stream.synchronize()
    clk = clocks.stop(region)
    elapsed_ms = slowest_rank_ms(step_start.elapsed_time(step_end), dist, "cuda")
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_gbs(world, total, ms_per_step)

    peak, peak_kind = measured_peak()
    traffic = recorded_traffic()
    kernels = {}
    alone = {name: [a.elapsed_time(b) for a, b in ev[name]] for name in ORDER}
    sum_alone = sum(sum(t) / len(t) for t in alone.values())
    for name in ORDER:
        times = alone[name]
        avg = sum(times) / len(times)
        gbs = alg[name] / (avg * 1e-3) / 1e9
        kernels[name] = {"alg_bytes": alg[name], "avg_ms": avg, "min_ms": min(times), "GB/s": gbs,
                         "frac_of_" + peak_kind: gbs / peak,
                         "frac_of_nominal_8TBs": gbs / 8000.0,
                         "share": avg / sum_alone}
    dominant = max(ORDER, key=lambda n: kernels[n]["avg_ms"])
    dk = kernels[dominant]
    tr = traffic.get(dominant)
    roofline = {"bound": "hbm", "kernel": dominant, "achieved": dk["GB/s"], "peak": peak,
                "unit": "GB/s", "frac": dk["GB/s"] / peak, "peak_source": peak_kind,
                "traffic": tr, "alg_bytes": dk["alg_bytes"]}

    # end to end through the public API: pinned host inputs -> device -> kernels -> host results
    e2e = run_e2e(args, inp, total, torch, loom, stream, work)
    # the pages' other examples (packed dot, per-lane sums), each timed on its own (not part of the step)
    extras = measure_extras(args, torch, loom, stream, peak, peak_kind)
    extras["read_ahead"] = read_ahead_study(torch, loom, stream, work, alg)
    extras["stream_floor"] = stream_floor(torch, loom, stream, work, alg, extras)
    work2 = DeviceWorkload(inp, torch, loom, stream, depth=args.depth)
    extras["stream_floor"]["trains"] = floor_trains(torch, loom, stream, work, work2, alg)
    del work2
    extras["stream_floor"]["step"] = step_floor(torch, loom, stream, total, ms_per_step)
    extras["batched_engines"] = engine_study(torch, loom, stream, work, alg)

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32+i32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "alg_bytes_per_step": total,
                   "l2": "inputs larger than L2 (each >= 134 MB vs 129 MB); consecutive kernels read "
                         "different arrays", "parallelism": f"replicas x{world}" if world > 1 else "1 gpu",
                   "depth": args.depth or "default",
                   "step_lanes": [list(lane) for lane in lanes],
                   "timing": "value: K steps between two events; each step forks its lanes (CUDA streams, "
                             "step_lanes) off the launching stream and joins them; no event between the "
                             "kernels of a lane (each may be scheduled while the previous drains); kernels: the "
                             "same K steps again, serially on one stream, with an event pair around every launch"},
        "roofline": roofline,
        "kernels": kernels,
        "e2e": e2e,
        "gpu_launches": work.launches_per_step * args.steps,
        "clocks": clk,
        "extras": extras,
    }
    if rank == 0:
        threads = os.cpu_count() or 1
        line["cpu_baseline"] = cpu_baseline(inp, total, threads)
        print(json.dumps(line), flush=True)


PACKED_WORKLOAD = "packed dot: 128 instances x 128 records x 2048 lanes, 64 activation streams"


def packed_alg_bytes(d) -> int:
    """Per instance: the active records' words and scales, their activation rows,
    the initial sums, the count and the outputs."""
    c = d["counts"].astype(np.int64)
    L, S = d["lanes"], d["streams"]
    return int((c * L * 6).sum() + (c * S * 16).sum() + d["problems"] * (L * 8 + 4))


def lane_alg_bytes(d) -> int:
    """Per segment: the active rows, the count and the outputs."""
    c = d["counts"].astype(np.int64)
    row = d["lanes"] * d["width"] * 4
    return int((c * row).sum() + d["num_segments"] * (4 + d["lanes"] * 4))


ROUTED_WORKLOAD = ("routed row combine: 4096 tokens x 8 routes (1 in 16 missing), payload rows of 2048 f32 "
                   "each read once")


def routed_alg_bytes(d) -> int:
    """The ids, the present routes' weights and payload rows, and the outputs."""
    valid = int((d["ids"] >= 0).sum())
    return int(d["ids"].size * 4 + valid * 4 + valid * d["width"] * 4 + d["tokens"] * d["width"] * 4)


def _time_single(args, torch, stream, call, flush, sink):
    """Single launches, each after a 512 MB read that leaves nothing of the inputs
    in L2; CUDA events on the launching stream.  Returns the times in ms."""
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            call()
    stream.synchronize()
    times = []
    for _ in range(min(max(args.steps, 5), 200)):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            sink.copy_(flush.view(torch.int32).sum())
            torch.cuda._sleep(200_000)
            a.record(stream)
            call()
            b.record(stream)
        stream.synchronize()
        times.append(a.elapsed_time(b))
    return times


def _extra_line(workload, alg, times, peak, peak_kind, traffic, launch):
    avg = sum(times) / len(times)
    gbs = alg / (avg * 1e-3) / 1e9
    return {"workload": workload, "alg_bytes": alg, "avg_ms": avg, "median_ms": statistics.median(times),
            "min_ms": min(times), "launches": len(times),
            "l2": "512 MB read before each launch",
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "peak_source": peak_kind, "traffic": traffic},
            "grid": launch["grid"], "block": launch["block"][0]}


def measure_extras(args, torch, loom, stream, peak, peak_kind):
    import synth
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    flush = torch.ones(512 << 20, dtype=torch.uint8, device="cuda")
    sink = torch.zeros((), dtype=torch.int64, device="cuda")
    traffic = recorded_traffic()
    out = {}

    d = synth.packed_dot_case()
    f, sc, rhs = t(d["fields"]), t(d["scales"].view(np.int16)), t(d["rhs"])
    counts, init = t(d["counts"]), t(d["initial"])
    y = torch.empty((d["problems"], d["lanes"]), dtype=torch.float32, device="cuda")
    times = _time_single(args, torch, stream,
                         lambda: loom.loom_packed_dot(f, sc, rhs, counts, 0, init, out=y, stream=stream), flush, sink)
    L = loom.loom_launch_config(loom.LOOM_OP_PACKED_DOT, [d["problems"], d["records"], d["lanes"], d["streams"]])
    out["packed_dot"] = _extra_line(PACKED_WORKLOAD, packed_alg_bytes(d), times, peak, peak_kind,
                                    traffic.get("packed"), L)
    # trains over two copies of the inputs, beside the read-only probe's trains
    copies = [(f, sc, rhs), (f.clone(), sc.clone(), rhs.clone())]
    srcs, word = floor_srcs(torch, packed_alg_bytes(d))
    tr = train_vs_floor(torch, loom, stream,
                        lambda i: loom.loom_packed_dot(*copies[i], counts, 0, init, out=y, stream=stream),
                        packed_alg_bytes(d), srcs, word)
    out["packed_dot"]["trains"] = tr | {"note": TRAIN_NOTE}
    del f, sc, rhs, counts, init, y, d, copies, srcs

    d = synth.routed_case()
    ids, wts, pay = t(d["ids"]), t(d["weights"]), t(d["payload"])
    o = torch.empty((d["tokens"], d["width"]), dtype=torch.float32, device="cuda")
    times = _time_single(args, torch, stream, lambda: loom.loom_routed_combine(ids, wts, pay, out=o, stream=stream),
                         flush, sink)
    L = loom.loom_launch_config(loom.LOOM_OP_ROUTED_COMBINE, [d["tokens"], d["routes"], d["rows"], d["width"]])
    out["routed_combine"] = _extra_line(ROUTED_WORKLOAD, routed_alg_bytes(d), times, peak, peak_kind,
                                        traffic.get("routed"), L)
    del ids, wts, pay, o, d

    for name, S, R, W, guarded in (("sum_rows", 65536, 64, 1, False), ("sum_vector_rows", 16384, 64, 4, False),
                                   ("guarded_rows", 16384, 63, 4, True)):
        d = synth.lane_segments(num_segments=S, rows=R, lanes=32, width=W)
        v, c = t(d["values"]), t(d["counts"])
        o = torch.empty((S, 32), dtype=torch.float32, device="cuda")
        if guarded:
            call = lambda: loom.loom_sum_guarded_rows(v, S, R * 32 * 4, R, 32, c, 0, 4, 32, out=o, stream=stream)
            what = f"guarded ragged rows: {S} segments x {R} rows x 32 lanes x 4, counts U[0,{R}], 4 columns, 32 lanes"
        else:
            call = lambda: loom.loom_sum_rows(v, S, R * 32 * W, R, 32, W, c, 0, out=o, stream=stream)
            what = f"per-lane sums (width {W}): {S} segments x {R} rows x 32 lanes, counts U[0,{R}]"
        times = _time_single(args, torch, stream, call, flush, sink)
        L = loom.loom_launch_config(loom.LOOM_OP_LANE_SUMS, [S, R, 32, W])
        out[name] = _extra_line(what, lane_alg_bytes(d), times, peak, peak_kind, traffic.get(name), L)
        del v, c, o, d
    del flush
    return out


#: read-only probe schedules (kind, depth, CTAs per SM) tried for every byte count
FLOOR_SCHEDULES = ((0, 4, 4), (0, 8, 4), (0, 8, 2), (1, 4, 4), (1, 8, 4), (1, 8, 8), (2, 2, 12), (2, 4, 6))
FLOOR_KINDS = ("grid_stride", "warp_range", "bulk_ring")


def _after_flush(torch, stream, flush, sink, call):
    """One launch after a 512 MB read, timed by events on the stream; ms."""
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        sink.copy_(flush.view(torch.int32).sum())
        torch.cuda._sleep(200_000)
        a.record(stream)
        call()
        b.record(stream)
    stream.synchronize()
    return a.elapsed_time(b)


def stream_floor(torch, loom, stream, work, alg, extras, reps: int = 21):
    """The single-launch streaming floor: for the algorithmic byte count of every
    workload, the best median over FLOOR_SCHEDULES of a launch that only reads
    that many bytes (loom_stream_floor), beside the kernel's own single-launch
    median; both after a 512 MB read, all launches interleaved."""
    flush = torch.ones(512 << 20, dtype=torch.uint8, device="cuda")
    sink = torch.zeros((), dtype=torch.int64, device="cuda")
    word = torch.zeros(1, dtype=torch.int64, device="cuda")
    sizes = dict(alg)
    for name, line in extras.items():
        if isinstance(line, dict) and "alg_bytes" in line:
            sizes[name] = line["alg_bytes"]
    src = torch.empty(max(sizes.values()) + 16, dtype=torch.uint8, device="cuda")
    floor_t = {(n, sc): [] for n in sizes for sc in FLOOR_SCHEDULES}
    kern_t = {n: [] for n in alg}
    for rep in range(reps + 1):
        for n, nbytes in sizes.items():
            nb = nbytes // 16 * 16
            for sc in FLOOR_SCHEDULES:
                t = _after_flush(torch, stream, flush, sink,
                                 lambda: loom.loom_stream_floor(src, nb, sc[0], sc[1], sc[2], word, stream=stream))
                if rep:
                    floor_t[(n, sc)].append(t)
        for n in alg:
            t = _after_flush(torch, stream, flush, sink, lambda: work.launch(n))
            if rep:
                kern_t[n].append(t)
    out = {}
    for n, nbytes in sizes.items():
        meds = {sc: statistics.median(floor_t[(n, sc)]) for sc in FLOOR_SCHEDULES}
        best = min(meds, key=meds.get)
        k_ms = statistics.median(kern_t[n]) if n in kern_t else extras[n]["median_ms"]
        out[n] = {"bytes": nbytes, "floor_us": meds[best] * 1e3,
                  "floor_schedule": {"kind": FLOOR_KINDS[best[0]], "depth": best[1], "ctas_per_sm": best[2]},
                  "floor_GB/s": nbytes / (meds[best] * 1e-3) / 1e9, "kernel_us": k_ms * 1e3,
                  "kernel_over_floor": k_ms / meds[best]}
    del flush, src
    return {"note": "single launches after a 512 MB read, medians of %d; floor = best schedule of a read-only "
                    "launch over the same byte count (loom_stream_floor)" % reps, "workloads": out}


def _run_train(torch, stream, call, train: int):
    """`train` launches back to back between two events, call(i) alternating i = 0, 1
    between two copies of the inputs; the mean per launch in ms."""
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(200_000)
        a.record(stream)
        for i in range(train):
            call(i & 1)
        b.record(stream)
    stream.synchronize()
    return a.elapsed_time(b) / train


def train_vs_floor(torch, loom, stream, call, nbytes: int, srcs, word, reps: int = 7, train: int = 20):
    """A kernel's trains (call(i) alternating two input copies) beside the read-only
    probe's trains over the same byte count (every FLOOR_SCHEDULES entry, alternating
    two source buffers); medians over `reps` trains, the probe's best schedule."""
    nb = nbytes // 16 * 16
    floor_t = {sc: [] for sc in FLOOR_SCHEDULES}
    kern_t = []
    for rep in range(reps + 1):
        for sc in FLOOR_SCHEDULES:
            t = _run_train(torch, stream,
                           lambda i: loom.loom_stream_floor(srcs[i], nb, sc[0], sc[1], sc[2], word, stream=stream), train)
            if rep:
                floor_t[sc].append(t)
        t = _run_train(torch, stream, call, train)
        if rep:
            kern_t.append(t)
    meds = {sc: statistics.median(v) for sc, v in floor_t.items()}
    best = min(meds, key=meds.get)
    k_ms = statistics.median(kern_t)
    return {"floor_us": meds[best] * 1e3,
            "floor_schedule": {"kind": FLOOR_KINDS[best[0]], "depth": best[1], "ctas_per_sm": best[2]},
            "floor_GB/s": nbytes / (meds[best] * 1e-3) / 1e9, "kernel_us": k_ms * 1e3,
            "kernel_GB/s": nbytes / (k_ms * 1e-3) / 1e9, "kernel_over_floor": k_ms / meds[best]}


def floor_srcs(torch, nbytes: int):
    """Two source buffers for the read-only probe's trains, and its sink word."""
    n = nbytes // 16 * 16 + 16
    return ([torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(2)],
            torch.zeros(1, dtype=torch.int64, device="cuda"))


TRAIN_NOTE = ("trains of 20 launches between two events, alternating two copies of the inputs; mean per "
              "launch, median of 7 trains; floor = best schedule of the read-only probe")


def floor_trains(torch, loom, stream, work, work2, alg, reps: int = 7, train: int = 20):
    """The streaming floor measured on trains of launches rather than single
    launches: `train` launches back to back between two events, alternating
    between two copies of the inputs (so no launch finds its bytes in L2), the
    mean per launch; the median over `reps` trains.  The same for the read-only
    probe over the same byte count, alternating between two source buffers.  The
    event timer ticks in ~1 us steps, so the trains resolve what single launches
    cannot; consecutive launches may overlap their ramp and tail (each kernel may
    be scheduled while the previous drains), as in the step."""
    srcs, word = floor_srcs(torch, max(alg.values()))
    works = (work, work2)
    out = {n: train_vs_floor(torch, loom, stream, lambda i, n=n: works[i].launch(n), nbytes, srcs, word, reps, train)
           for n, nbytes in alg.items()}
    del srcs
    return {"note": TRAIN_NOTE, "workloads": out}


def step_floor(torch, loom, stream, total: int, ms_per_step: float, reps: int = 7, train: int = 20):
    """The read-only probe over the whole step's algorithmic bytes in one launch,
    timed in trains (best of FLOOR_SCHEDULES, median of `reps` trains, alternating
    two source buffers), beside the step's own time per step (K back-to-back steps):
    how far the four kernels together are from reading their bytes once."""
    srcs, word = floor_srcs(torch, total)
    nb = total // 16 * 16
    times = {sc: [] for sc in FLOOR_SCHEDULES}
    for rep in range(reps + 1):
        for sc in FLOOR_SCHEDULES:
            t = _run_train(torch, stream,
                           lambda i: loom.loom_stream_floor(srcs[i], nb, sc[0], sc[1], sc[2], word, stream=stream), train)
            if rep:
                times[sc].append(t)
    del srcs
    meds = {sc: statistics.median(v) for sc, v in times.items()}
    best = min(meds, key=meds.get)
    return {"bytes": total, "floor_us": meds[best] * 1e3,
            "floor_schedule": {"kind": FLOOR_KINDS[best[0]], "depth": best[1], "ctas_per_sm": best[2]},
            "floor_GB/s": total / (meds[best] * 1e-3) / 1e9, "step_us": ms_per_step * 1e3,
            "step_over_floor": ms_per_step / meds[best],
            "note": "one read-only launch over the step's bytes, trains of 20; the step: K back-to-back steps"}


def engine_study(torch, loom, stream, work, alg, reps: int = 21):
    """The batched dot (8192 x 16384 x 16) on both engines, alternated: the
    tensor-core kernel against the dp4a kernel with lanes across the batch."""
    flush = torch.ones(512 << 20, dtype=torch.uint8, device="cuda")
    sink = torch.zeros((), dtype=torch.int64, device="cuda")
    d, o = work.d, work.o
    ys = {}
    tunings = {"tensor": loom.make_tuning(path=loom.LOOM_PATH_TENSOR),
               "dp4a": loom.make_tuning(path=loom.LOOM_PATH_STAGED)}
    times = {k: [] for k in tunings}
    for rep in range(reps + 1):
        for k, tu in tunings.items():
            y = torch.empty((8192, 16), dtype=torch.float32, device="cuda")
            t = _after_flush(torch, stream, flush, sink, lambda: loom.loom_i8_dequant_dot_ex(
                d["wb"], d["swb"], 8192, 16384, d["x16"], d["sx16"], 16, y=y, tuning=tu, stream=stream))
            if rep:
                times[k].append(t)
            ys[k] = y
    same = bool(torch.equal(ys["tensor"].view(torch.int32), ys["dp4a"].view(torch.int32)))
    del flush
    return {k: {"median_us": statistics.median(v) * 1e3, "GB/s": alg["batched"] / (statistics.median(v) * 1e-3) / 1e9}
            for k, v in times.items()} | {"same_bits": same, "auto_picks": "tensor"}


def read_ahead_study(torch, loom, stream, work, alg):
    """The pages' own comparison: the serial control (read-ahead depth 1) against
    a deeper ring, same kernels and workloads, alternated ABAB; single launches
    after a 512 MB read, CUDA events.  Not part of the step.  The row sums'
    deeper arm is their default depth; the GEMV's default is already depth 1
    (its read-ahead comes from sixteen one-stage rings per SM), so its deeper arm
    is two stages per warp with half the warps: the same ring bytes per CTA."""
    flush = torch.ones(512 << 20, dtype=torch.uint8, device="cuda")
    sink = torch.zeros((), dtype=torch.int64, device="cuda")
    serial = loom.make_tuning(depth=1)
    deeper = {"segments": (None, "default (4)"), "wide": (None, "default (2)"),
              "gemv": (loom.make_tuning(depth=2, warps_per_cta=4), "2 (4 warps per CTA)")}
    out = {}
    for name in ("segments", "wide", "gemv"):
        times = {"depth1": [], "deeper": []}
        for rep in range(6):
            for label, tu in (("depth1", serial), ("deeper", deeper[name][0])):
                saved = work.tuning
                work.tuning = tu
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    sink.copy_(flush.view(torch.int32).sum())
                    torch.cuda._sleep(200_000)
                    a.record(stream)
                    work.launch(name)
                    b.record(stream)
                stream.synchronize()
                work.tuning = saved
                if rep > 0:
                    times[label].append(a.elapsed_time(b))
        out[name] = {k: {"avg_ms": sum(v) / len(v), "GB/s": alg[name] / (sum(v) / len(v) * 1e-3) / 1e9}
                     for k, v in times.items()}
        out[name]["deeper"]["depth"] = deeper[name][1]
    del flush
    return out


#: the inputs and outputs of each workload on the end-to-end path
E2E_INPUTS = {"segments": ("seg_counts", "seg_init"), "wide": ("wide_counts",),
              "gemv": ("w", "sw", "x1", "sx1"), "batched": ("wb", "swb", "x16", "sx16")}
E2E_OUTPUTS = {"segments": "seg", "wide": "wide", "gemv": "y1", "batched": "y16"}


class E2EStep:
    """One end-to-end step through the binding with host buffers.  The step moves
    its inputs from pinned host memory to the device -- the dense ones (weights,
    vectors, scales, counts, initial sums) with copies, the two ragged f32 arrays
    with loom_stage_rows, which moves only the rows the row sums read -- runs the
    four kernels and reads the results back into pinned host buffers.  Each lane
    of the step uploads, runs and reads back its own workloads in
    order, so one lane's kernels overlap the other's uploads."""

    def __init__(self, inp, torch, loom, work, lanes=STEP_LANES):
        self.loom, self.work, self.lanes = loom, work, lanes
        self.dense = {}
        for key, arr in (("seg_counts", inp["segments"]["counts"]), ("seg_init", inp["segments"]["initial"]),
                         ("wide_counts", inp["wide"]["counts"]), ("w", inp["gemv"]["w"].view("<i4")),
                         ("sw", inp["gemv"]["scale_w"]), ("x1", inp["gemv"]["x"].view("<i4")),
                         ("sx1", inp["gemv"]["scale_x"]), ("wb", inp["batched"]["w"].view("<i4")),
                         ("swb", inp["batched"]["scale_w"]), ("x16", inp["batched"]["x"].view("<i4")),
                         ("sx16", inp["batched"]["scale_x"])):
            self.dense[key] = torch.from_numpy(np.ascontiguousarray(arr)).pin_memory()
        seg, wide = inp["segments"], inp["wide"]
        self.ragged = {
            "segments": (torch.from_numpy(np.ascontiguousarray(seg["values"]).reshape(-1)).pin_memory(),
                         "seg_values", "seg_counts", seg),
            "wide": (torch.from_numpy(np.ascontiguousarray(wide["values"]).reshape(-1)).pin_memory(),
                     "wide_values", "wide_counts", wide)}
        self.outs = {"seg": work.o["seg"], "wide": work.o["wide"], "y1": (work.o["y1"],), "y16": (work.o["y16"],)}
        self.host_out = {k: tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in grp)
                         for k, grp in self.outs.items()}
        staged = 4 * (int(seg["counts"].astype(np.int64).sum()) * seg["lanes"] +
                      int(wide["counts"].astype(np.int64).sum()))
        self.h2d = sum(t.numel() * t.element_size() for t in self.dense.values()) + staged
        self.d2h = sum(t.numel() * t.element_size() for grp in self.host_out.values() for t in grp)
        self.torch = torch
        self.streams = [torch.cuda.Stream() for _ in lanes]
        self.fork = torch.cuda.Event()
        self.joins = [torch.cuda.Event() for _ in lanes]

    def run(self, main):
        torch, d = self.torch, self.work.d
        self.fork.record(main)
        for lane, s, j in zip(self.lanes, self.streams, self.joins):
            s.wait_event(self.fork)
            with torch.cuda.stream(s):
                for name in lane:
                    for key in E2E_INPUTS[name]:
                        d[key].copy_(self.dense[key], non_blocking=True)
                    if name in self.ragged:
                        h, dv, dc, g = self.ragged[name]
                        self.loom.loom_stage_rows(h, d[dv], g["num_segments"], g["seg_stride"], g["rows"],
                                                  g["lanes"], d[dc], stream=s)
                    self.work.launch(name, stream=s)
                    key = E2E_OUTPUTS[name]
                    for hb, db in zip(self.host_out[key], self.outs[key]):
                        hb.copy_(db, non_blocking=True)
            j.record(s)
        for j in self.joins:
            main.wait_event(j)


def run_e2e(args, inp, total, torch, loom, stream, work):
    """The metric end to end (E2EStep), every step inside the timed region."""
    e2e = E2EStep(inp, torch, loom, work, STEP_LANES if args.lanes == 2 else ONE_LANE)
    steps = max(1, min(args.steps, 5))
    e2e.run(stream)
    stream.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(steps):
            e2e.run(stream)
        b.record(stream)
    stream.synchronize()
    ms = a.elapsed_time(b) / steps
    return {"value": total / (ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": e2e.h2d,
            "d2h_bytes_per_step": e2e.d2h, "ms_per_step": ms, "steps": steps,
            "h2d": "dense inputs by copy; the ragged f32 arrays by loom_stage_rows (active rows only); "
                   "each lane of the step uploads, runs and reads back its own workloads"}


#: algorithmic bytes of the step's workloads (the seeded inputs fix them), for --profile floor_<workload>
FLOOR_PROFILE_BYTES = {"gemv": 134_299_652, "segments": 265_410_432, "batched": 135_036_992, "wide": 535_147_296}


def run_profile(args):
    """One kernel's workload, `--launches` times, for an ncu capture (not timed)."""
    import torch
    import int8_dequant_dot_gb300 as loom
    import synth
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    if args.profile.startswith("floor_"):
        # the read-only probe over a workload's algorithmic byte count, in the
        # schedule that measured best for the step's workloads (bulk-copy ring,
        # depth 2, 12 CTAs per SM)
        nb = FLOOR_PROFILE_BYTES[args.profile[len("floor_"):]] * args.scale // 16 * 16
        src = torch.empty(nb + 16, dtype=torch.uint8, device="cuda")
        word = torch.zeros(1, dtype=torch.int64, device="cuda")
        with torch.cuda.stream(stream):
            for _ in range(args.launches):
                loom.loom_stream_floor(src, nb, 2, 2, 12, word, stream=stream)
        stream.synchronize()
        print(json.dumps({"profile": args.profile, "launches": args.launches, "bytes": nb}))
        return
    if args.profile == "packed":
        d = synth.packed_dot_case()
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        f, sc, rhs, counts, init = (t(d["fields"]), t(d["scales"].view(np.int16)), t(d["rhs"]), t(d["counts"]),
                                    t(d["initial"]))
        with torch.cuda.stream(stream):
            for _ in range(args.launches):
                loom.loom_packed_dot(f, sc, rhs, counts, 0, init, stream=stream)
        stream.synchronize()
        print(json.dumps({"profile": args.profile, "launches": args.launches}))
        return
    if args.profile == "routed":
        d = synth.routed_case()
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        ids, wts, pay = t(d["ids"]), t(d["weights"]), t(d["payload"])
        with torch.cuda.stream(stream):
            for _ in range(args.launches):
                loom.loom_routed_combine(ids, wts, pay, stream=stream)
        stream.synchronize()
        print(json.dumps({"profile": args.profile, "launches": args.launches}))
        return
    if args.profile in ("sum_rows", "sum_vector_rows", "guarded_rows"):
        S, R, W = {"sum_rows": (65536, 64, 1), "sum_vector_rows": (16384, 64, 4),
                   "guarded_rows": (16384, 63, 4)}[args.profile]
        d = synth.lane_segments(num_segments=S, rows=R, lanes=32, width=W)
        v = torch.from_numpy(d["values"]).cuda()
        c = torch.from_numpy(d["counts"]).cuda()
        with torch.cuda.stream(stream):
            for _ in range(args.launches):
                if args.profile == "guarded_rows":
                    loom.loom_sum_guarded_rows(v, S, R * 128, R, 32, c, 0, 4, 32, stream=stream)
                else:
                    loom.loom_sum_rows(v, S, R * 32 * W, R, 32, W, c, 0, stream=stream)
        stream.synchronize()
        print(json.dumps({"profile": args.profile, "launches": args.launches}))
        return
    sc = args.scale
    if args.profile in ("segments", "wide"):
        inp = {"segments": synth.batched_segments(num_segments=65536 * sc) if args.profile == "segments" else None,
               "wide": synth.wide_rows() if args.profile == "wide" else None}
    else:
        inp = {"gemv": synth.dequant_gemv(n_rows=8192 * sc) if args.profile == "gemv" else None,
               "batched": (synth.dequant_batched(n_rows=8192 * sc)
                           if args.profile in ("batched", "batched_dp4a") else None)}
    work = _SingleWorkload(args.profile, inp, torch, loom, stream, args.depth)
    with torch.cuda.stream(stream):
        for _ in range(args.launches):
            work.launch()
    stream.synchronize()
    print(json.dumps({"profile": args.profile, "launches": args.launches}))


class _SingleWorkload:
    def __init__(self, name, inp, torch, loom, stream, depth):
        self.name, self.loom, self.stream = name, loom, stream
        dev = torch.device("cuda")
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        self.tuning = loom.make_tuning(depth=depth) if depth else None
        if name == "batched_dp4a":   # the batched workload on the dp4a engine (the engine comparison)
            name = "batched"
            self.tuning = loom.make_tuning(depth=depth, path=loom.LOOM_PATH_STAGED)
        self.name = name
        if name == "segments":
            s = inp["segments"]
            self.args = (t(s["values"]), s["num_segments"], 2016, 63, 32, t(s["counts"]), t(s["initial"]), 8)
        elif name == "wide":
            s = inp["wide"]
            self.args = (t(s["values"]), 16384, 16384, 16384, 1, t(s["counts"]), None, 8)
        else:
            s = inp[name]
            b = s["x"].shape[0]
            self.args = (t(s["w"].view("<i4")), t(s["scale_w"]), s["n_rows"], 16384, t(s["x"].view("<i4")),
                         t(s["scale_x"]), b)

    def launch(self):
        if self.name in ("segments", "wide"):
            self.loom.loom_row_sum_batched_ex(*self.args, tuning=self.tuning, stream=self.stream)
        else:
            self.loom.loom_i8_dequant_dot_ex(*self.args, tuning=self.tuning, stream=self.stream)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)   # ~0.35 s timed: 16+ clock samples inside it
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--depth", type=int, default=0, help="read-ahead depth (0 = library default)")
    ap.add_argument("--profile", choices=ORDER + ("batched_dp4a", "packed", "sum_rows", "sum_vector_rows",
                                                  "guarded_rows", "routed")
                    + tuple("floor_" + n for n in ORDER), default=None)
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--scale", type=int, default=1,
                    help="with --profile segments/gemv/batched/floor_*: that many times the rows (segments) "
                         "of the workload, for captures of the same kernel over a longer launch")
    ap.add_argument("--lanes", type=int, choices=(1, 2), default=2,
                    help="2: the step's two concurrent stream lanes; 1: every kernel on one stream")
    args = ap.parse_args()
    if args.warmup < 3 and args.profile is None:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.profile:
        run_profile(args)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as dist_mod
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    try:
        run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
