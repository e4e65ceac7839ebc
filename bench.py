#!/usr/bin/env python3
"""Benchmark of the entropy-bounded softmax (constrained_softmax) on GB300.

One step = one constrained_softmax launch over the whole workload (every row:
max, T = 1 pass, bisection, output), inputs resident in HBM.  The default
workload is batch 32 x 50000 classes, the latency case quoted by "BURT-IMMA
CUDA Kernel API Reference" (section 2.1 Performance Notes, section 7.1:
0.8 ms on an RTX 3080).  Prints one JSON line:
  value       rows/s over all GPUs (device-timed, CUDA events);
  e2e         rows/s through the public API with pinned-host inputs, H2D
              and D2H copies of every step inside the timed region
              (consecutive steps on two streams, so that copies overlap the
              neighbouring steps; the serial figure is reported beside it);
  roofline    the kernel against the slower of HBM (8 bytes per class) and
              the ex2 unit ((1 + bisection steps) ex2 per class per row),
              both peaks measured on this GPU (HBM: the copy bandwidth
              recorded for the machine, ex2: a probe kernel run here);
  cpu_baseline  the CPU oracle on this host's cores on a bounded sample.

--impl reference times the CPU oracle instead (the reference arm); under
torchrun every rank runs an independent replica (rows are independent; no
collective is on the data path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from entropy_bounded_softmax_gb300 import workloads as wl  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
METRIC = "rows/s and effective HBM GB/s (% of roofline); latency at 32x50000"
# The page's figure for this workload: 0.8 ms for batch 32 x 50000 classes
# on an RTX 3080 (another machine: context, not a target).
PAGE_LATENCY_MS = {"latency_32x50000": 0.8}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=wl.LATENCY.name,
                    help="one of: " + ", ".join(
                        list(wl.WORKLOADS) + [w.name for w in wl.sweep_workloads()]
                        + list(wl.ATTENTION_WORKLOADS)
                        + list(wl.BIENCODER_WORKLOADS)))
    ap.add_argument("--variant", choices=["auto", "rowgroup", "cluster"],
                    default="auto")
    ap.add_argument("--param", type=int, default=0,
                    help="lanes per row (rowgroup) or CTAs per row (cluster)")
    ap.add_argument("--threads", type=int, default=0,
                    help="cluster variant: threads per CTA (0 = automatic)")
    ap.add_argument("--strict", action="store_true",
                    help="cluster variant: halve the bracket one "
                         "evaluation per round (the bisection itself)")
    ap.add_argument("--batch", type=int, default=0,
                    help="use only the first BATCH rows of the workload "
                         "(profiling captures); 0 = the whole workload")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--soak-s", type=float, default=1.5,
                    help="untimed load before the timed region, for the "
                         "clock samples")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-configuration timings that follow "
                         "the headline")
    ap.add_argument("--no-graph", action="store_true",
                    help="time plain stream launches instead of one CUDA "
                         "graph of the K launches")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--op", choices=["forward", "backward", "attention",
                                     "biencoder"],
                    default="forward",
                    help="backward: time the gradient kernel, (1/T) p "
                         "(g - <g, p>), on the workload's shape; attention: "
                         "time attention_softmax on an attention workload "
                         "(default attention_32x8x512); biencoder: the fused "
                         "biencoder_attention (default "
                         "biencoder_32x8x512x64x64)")
    return ap.parse_args(argv)


def find_workload(name: str) -> wl.Workload:
    if name in wl.WORKLOADS:
        return wl.WORKLOADS[name]
    for w in wl.sweep_workloads():
        if w.name == name:
            return w
    raise SystemExit(f"unknown workload {name!r}")


# ------------------------------------------------------------ distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def reduce_max(dist, value: float, device=None) -> float:
    """Max of a float over ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rows_per_s(rows_per_rank: int, world: int,
                         max_seconds: float) -> float:
    """Whole-job throughput: all ranks' rows over the slowest rank's time."""
    return rows_per_rank * world / max_seconds


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons (200 ms)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        rows = [p for (t, p) in self.samples if t0 <= t <= t1]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------------ peaks
def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


def measured_bf16_tflops() -> float:
    """The measured dense bf16 GEMM rate (TFLOP/s) of this machine, else
    the recorded fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return 1900.0


def probe_ex2_peak(torch, cs, stream_ptr) -> float:
    """ex2/s of the whole GPU from the probe kernel (best of 5)."""
    n = cs.cs_probe_ex2_sink_floats()
    sink = torch.empty(n, dtype=torch.float32, device="cuda")
    iters = 256
    best = 0.0
    for _ in range(8):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        st, count = cs.cs_probe_ex2(sink.data_ptr(), iters, stream_ptr)
        b.record()
        b.synchronize()
        if st != 0:
            raise RuntimeError(f"probe failed: {st}")
        ms = a.elapsed_time(b)
        if ms < 20.0:
            iters = int(iters * max(2.0, 40.0 / max(ms, 1e-3)))
            continue
        best = max(best, count / (ms * 1e-3))
    return best


# --------------------------------------------------------- algorithmic work
def entropy_at_one(x: np.ndarray) -> np.ndarray:
    """H(1) of every row in fp64 (scipy), the workload property that decides
    which rows run the bisection."""
    import scipy.special
    out = np.empty(x.shape[0])
    step = 256
    for r0 in range(0, x.shape[0], step):
        blk = x[r0:r0 + step].astype(np.float64)
        p = scipy.special.softmax(blk, axis=1)
        out[r0:r0 + step] = scipy.special.entr(p).sum(axis=1)
    return out


def searched_rows(w: wl.Workload, x: np.ndarray, h1=None) -> int:
    """Rows whose entropy at T = 1 exceeds the bound (they run the full
    bisection)."""
    h1 = entropy_at_one(x) if h1 is None else h1
    return int(np.sum(h1 > np.float32(w.entropy_bound)))


def formula_ex2(w: wl.Workload, n_search: int) -> int:
    """The roofline's exponentials: (1 + max_iter) per class of a searched
    row, 1 per class of the others (the T = 1 pass; the output pass is not
    counted)."""
    return (w.batch + n_search * w.max_iter) * w.num_classes


def ex2_issued(evals, C: int, plan: dict) -> int:
    """Exponentials the kernel issued, from its per-row evaluation counts
    (T = 1, every point of the search, the output): each counted temperature
    costs one exponential per class, except the fan's (plans with
    fan_points), whose three temperatures share one exponential and two
    squarings."""
    e = evals.long()
    total = int(e.sum().item())
    nf = int(plan.get("fan_points", 0) or 0)
    if nf > 1:
        fan_rows = int((e >= nf + 2).sum().item())
        total -= (nf - 1) * fan_rows
    return total * C


def ex2_roofline(ex2_formula: int, ex2_executed: int | None, io_bytes: int,
                 t_kernel: float, ex2_peak: float, hbm_gbs: float) -> dict:
    """The kernel against the slower of HBM (io_bytes at the measured copy
    bandwidth) and the ex2 unit (the formula's exponentials at the probe's
    rate); frac_executed counts instead the exponentials the kernel issued
    (every temperature each row was evaluated at, from the kernel's own
    per-row counts, output pass included)."""
    ex2_rate = ex2_formula / t_kernel
    hbm_rate = io_bytes / t_kernel / 1e9
    t_hbm = io_bytes / (hbm_gbs * 1e9)
    t_ex2 = ex2_formula / ex2_peak
    if t_ex2 >= t_hbm:
        roof = {"bound": "alu", "unit": "Gex2/s", "achieved": ex2_rate / 1e9,
                "peak": ex2_peak / 1e9, "frac": ex2_rate / ex2_peak,
                "peak_source": "measured ex2 probe (burst)"}
    else:
        roof = {"bound": "hbm", "unit": "GB/s", "achieved": hbm_rate,
                "peak": hbm_gbs, "frac": hbm_rate / hbm_gbs,
                "peak_source": "measured copy bandwidth"}
    roof.update({
        "algorithmic_bytes": io_bytes,
        "algorithmic_ex2": ex2_formula,
        "executed_ex2": ex2_executed,
        "frac_executed": (ex2_executed / t_kernel / ex2_peak
                          if ex2_executed is not None else None),
        "hbm_gbs": hbm_rate,
        "hbm_frac": hbm_rate / hbm_gbs,
        "hbm_peak": hbm_gbs,
        "roofline_us": max(t_hbm, t_ex2) * 1e6,
        "frac_of_roofline": max(t_hbm, t_ex2) / t_kernel,
    })
    return roof


# ------------------------------------------------------------ reference arm
def run_oracle_sample(w: wl.Workload, x: np.ndarray, seconds: float,
                      threads: int) -> dict:
    """The CPU oracle, as it stands, on whole rows of the workload until
    `seconds` have passed (at least one batch of `threads` rows; threads =
    1 gives the single-core figure)."""
    import oracle
    oracle.load()
    done = 0
    t0 = time.perf_counter()
    r = 0
    while True:
        rows = [(r + i) % x.shape[0] for i in range(threads)]
        oracle.constrained_softmax(x[rows], w.entropy_bound, w.t_min,
                                   w.t_max, w.max_iter, threads=threads)
        done += len(rows)
        r += threads
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"rows": done, "seconds": dt, "rows_per_s": done / dt}


def reference_arm(args, w: wl.Workload) -> int:
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    threads = oracle.default_threads()
    x = wl.generate(w)
    oracle.load()
    # Each step: the oracle on `threads` whole rows, one per core, so the
    # whole --steps/--warmup run stays within a few minutes.
    rows_per_step = threads
    for i in range(args.warmup):
        rows = [(i * rows_per_step + j) % w.batch for j in range(rows_per_step)]
        oracle.constrained_softmax(x[rows], w.entropy_bound, w.t_min,
                                   w.t_max, w.max_iter, threads=threads)
    t0 = time.perf_counter()
    for i in range(args.steps):
        rows = [(i * rows_per_step + j) % w.batch for j in range(rows_per_step)]
        oracle.constrained_softmax(x[rows], w.entropy_bound, w.t_min,
                                   w.t_max, w.max_iter, threads=threads)
    dt = time.perf_counter() - t0
    value = rows_per_step * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "rows/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, "cpu"),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{rows_per_step} whole rows per step "
                                   f"({args.steps} steps)"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w: wl.Workload, l2: str) -> dict:
    return {"workload": w.name, "batch": w.batch,
            "num_classes": w.num_classes, "logits": w.note,
            "entropy_bound": w.entropy_bound, "t_min": w.t_min,
            "t_max": w.t_max, "max_iter": w.max_iter, "seed": w.seed,
            "l2": l2}


# ----------------------------------------------------------------- timing
def time_launches(args, torch, launch, stream, dist, local) -> dict:
    """Soak (clock samples start), then the K timed launches: once as plain
    stream launches and once as one CUDA graph of the same K launches (host
    launch overhead out of the device timing), each bracketed by a barrier
    and a synchronize; CUDA events on the launching stream."""
    sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else 0)
    sampler.start()
    t_soak = time.time()
    i = 0
    while time.time() - t_soak < args.soak_s:
        for _ in range(50):
            launch(i)
            i += 1
        torch.cuda.synchronize()

    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cap = torch.cuda.current_stream().cuda_stream
            for j in range(args.steps):
                launch(j, cap)
        graph.replay()
        torch.cuda.synchronize()

    def timed(use_graph: bool) -> float:
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        e_a = torch.cuda.Event(enable_timing=True)
        e_b = torch.cuda.Event(enable_timing=True)
        e_a.record(stream)
        if use_graph:
            graph.replay()
        else:
            for j in range(args.steps):
                launch(j)
        e_b.record(stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        return e_a.elapsed_time(e_b)

    stream_ms = timed(False)
    ms = timed(True) if graph is not None else stream_ms
    t_end = time.time()
    sampler.stop()
    return {"stream_ms": stream_ms, "ms": ms, "graph": graph, "t0": t_soak,
            "t1": t_end, "sampler": sampler}


# -------------------------------------------------------------------- e2e
E2E_SLOTS = 3


def time_e2e(torch, make_slot, step, stream, e_steps: int) -> dict:
    """End-to-end steps through the public API.  make_slot() returns one
    set of device and pinned-host buffers; step(slot) enqueues one whole
    step on the current stream: the host-to-device copy of its inputs, the
    call, the device-to-host copy of its result.  Timed twice with CUDA
    events on `stream`: pipelined (consecutive steps alternate between
    E2E_SLOTS streams and buffer sets, so one step's copies overlap the
    neighbouring steps' call and copies, as a serving loop would run them)
    and serial (every step on one stream).  Returns ms per step of each."""
    slots = [make_slot() for _ in range(E2E_SLOTS)]
    streams = [torch.cuda.Stream(device=stream.device)
               for _ in range(E2E_SLOTS)]

    def run(n: int, pipelined: bool) -> float:
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for st in streams:
            st.wait_event(e0)
        # The current stream is switched with set_stream (a fraction of the
        # host time of the stream context manager, on the step's path).
        prev = torch.cuda.current_stream(stream.device)
        for i in range(n):
            k = i % E2E_SLOTS if pipelined else 0
            torch.cuda.set_stream(streams[k])
            step(slots[k])
        torch.cuda.set_stream(prev)
        for st in streams:
            stream.wait_stream(st)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    run(3, True)
    run(3, False)
    return {"pipelined": run(e_steps, True), "serial": run(e_steps, False)}


def pinned_copy_gbs(torch, dev, nbytes: int = 1 << 28) -> dict:
    """Bandwidth of one large cudaMemcpyAsync between pinned host memory and
    the device, each direction alone and both at once on two streams (best
    of 3, CUDA events): the ceiling of the e2e steps' copies."""
    h = torch.empty(nbytes // 4, dtype=torch.float32).pin_memory()
    h2 = torch.empty(nbytes // 4, dtype=torch.float32).pin_memory()
    d = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)
    d2 = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def best(fn) -> float:
        t = []
        for _ in range(3):
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            s1.wait_event(a)
            s2.wait_event(a)
            fn()
            torch.cuda.current_stream().wait_stream(s1)
            torch.cuda.current_stream().wait_stream(s2)
            b.record()
            b.synchronize()
            t.append(a.elapsed_time(b) * 1e-3)
        return min(t)

    def h2d():
        with torch.cuda.stream(s1):
            d.copy_(h, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)

    def both():
        h2d()
        d2h()

    out = {"h2d_gbs": nbytes / best(h2d) / 1e9,
           "d2h_gbs": nbytes / best(d2h) / 1e9,
           "both_gbs": 2 * nbytes / best(both) / 1e9,
           "bytes": nbytes}
    del h, h2, d, d2
    return out


def e2e_entry(value: float, ms: dict, h2d: int, d2h: int,
              copy_bw: dict | None = None) -> dict:
    out = {"value": value, "unit": "rows/s", "ms_per_step": ms["pipelined"],
           "ms_per_step_serial": ms["serial"],
           "pipeline": f"{E2E_SLOTS} streams, one buffer set each; "
                       "every step copies its inputs in and its result out",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    if copy_bw:
        out["pinned_copy"] = copy_bw
        # The step's copies alone at the measured pinned-copy bandwidth.
        out["copy_bound_ms"] = 1e3 * max(
            h2d / (copy_bw["h2d_gbs"] * 1e9), d2h / (copy_bw["d2h_gbs"] * 1e9),
            (h2d + d2h) / (copy_bw["both_gbs"] * 1e9))
    return out


# ---------------------------------------------------------------- our arm
def our_arm(args, w: wl.Workload) -> int:
    import torch
    import entropy_bounded_softmax_gb300 as cs

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")

    x = wl.generate(w)
    B, C = x.shape
    elems = B * C
    io_bytes = 8 * elems
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    opts = cs.options(cs.VARIANTS[args.variant], args.param, args.threads,
                      int(args.strict))

    # Inputs larger than L2 between timed launches: rotate through enough
    # input/output pairs that one pass over them is >= 3x L2.
    nbuf = max(1, math.ceil(3 * L2_BYTES / io_bytes)) if io_bytes < 3 * L2_BYTES else 1
    xs = torch.from_numpy(x).to(dev)
    ins = [xs] + [xs.clone() for _ in range(nbuf - 1)]
    outs = [torch.empty_like(xs) for _ in range(nbuf)]
    t_outs = [torch.empty(B, dtype=torch.float32, device=dev)
              for _ in range(nbuf)]
    l2_note = (f"rotating {nbuf} input/output pairs "
               f"({nbuf * io_bytes / 2**20:.0f} MiB > L2)") if nbuf > 1 else \
        f"inputs larger than L2 ({io_bytes / 2**20:.0f} MiB)"

    def launch(i: int, stream_ptr: int = sptr) -> None:
        k = i % nbuf
        st = cs.cs_constrained_softmax_ex(
            ins[k].data_ptr(), outs[k].data_ptr(), B, C,
            w.entropy_bound, w.t_min, w.t_max, w.max_iter,
            t_outs[k].data_ptr(), opts, stream_ptr)
        if st != 0:
            raise RuntimeError(f"cs_constrained_softmax failed: {st}")

    cs.get_error()
    for i in range(max(3, args.warmup)):
        launch(i)
    torch.cuda.synchronize()
    plan = cs.plan(B, C, args.variant, args.param, args.threads,
                   args.strict)

    tm = time_launches(args, torch, launch, stream, dist, local)
    stream_ms, local_ms, graph = tm["stream_ms"], tm["ms"], tm["graph"]
    t_soak, t_end, sampler = tm["t0"], tm["t1"], tm["sampler"]
    total_ms = reduce_max(dist, local_ms, dev)
    stream_ms_max = reduce_max(dist, stream_ms, dev)
    ms_per_step = total_ms / args.steps
    value = aggregate_rows_per_s(B, world, ms_per_step * 1e-3)
    err = cs.get_error()

    # End to end through the public API: pinned host input, H2D copy, the
    # call, D2H of the probabilities and temperatures, all inside events.
    h_in = torch.from_numpy(x).pin_memory()

    def make_slot():
        return {"d_in": torch.empty((B, C), dtype=torch.float32, device=dev),
                "out": torch.empty((B, C), dtype=torch.float32, device=dev),
                "t": torch.empty(B, dtype=torch.float32, device=dev),
                "h_out": torch.empty((B, C), dtype=torch.float32).pin_memory(),
                "h_t": torch.empty(B, dtype=torch.float32).pin_memory()}

    def e2e_step(sl):
        sl["d_in"].copy_(h_in, non_blocking=True)
        cs.constrained_softmax(sl["d_in"], w.entropy_bound, w.t_min, w.t_max,
                               w.max_iter, out=sl["out"], t_out=sl["t"],
                               variant=args.variant, param=args.param,
                               threads=args.threads, strict=args.strict)
        sl["h_out"].copy_(sl["out"], non_blocking=True)
        sl["h_t"].copy_(sl["t"], non_blocking=True)

    e2e = time_e2e(torch, make_slot, e2e_step, stream, max(1, args.e2e_steps))
    e2e = {k: reduce_max(dist, v, dev) for k, v in e2e.items()}
    e2e_value = aggregate_rows_per_s(B, world, e2e["pipelined"] * 1e-3)
    copy_bw = pinned_copy_gbs(torch, dev)

    # The exponentials the kernel issues: one untimed launch with the
    # per-row evaluation counts (the search is deterministic, so every timed
    # launch issues the same).
    evals = torch.zeros(B, dtype=torch.int32, device=dev)
    cs.constrained_softmax(ins[0], w.entropy_bound, w.t_min, w.t_max,
                           w.max_iter, out=outs[0], variant=args.variant,
                           param=args.param, threads=args.threads,
                           strict=args.strict, evals_out=evals)
    ex2_executed = ex2_issued(evals, C, plan)

    line = None
    if rank == 0:
        peaks = measured_peaks()
        ex2_peak = probe_ex2_peak(torch, cs, sptr)
        n_search = searched_rows(w, x)
        exps = formula_ex2(w, n_search)
        t_kernel = ms_per_step * 1e-3
        hbm_rate = io_bytes / t_kernel / 1e9
        roof = ex2_roofline(exps, ex2_executed, io_bytes, t_kernel, ex2_peak,
                            peaks["hbm_gbs"])
        roof.update({
            "traffic": None,
            "traffic_note": "DRAM bytes need an ncu capture of this build; "
                            "not measured in this run",
            "kernel": "cluster_kernel" if plan["variant"] == 2 else "rowgroup_kernel",
            "searched_rows": n_search,
            "evals_per_row_mean": (
                float(evals.float().mean().item()) if B else None),
        })
        cpu = None
        if not args.no_cpu_baseline:
            import oracle
            threads = oracle.default_threads()
            s = run_oracle_sample(w, x, args.cpu_seconds, threads)
            s1 = run_oracle_sample(w, x, args.cpu_seconds / 2, 1)
            cpu = {"value": s["rows_per_s"], "unit": "rows/s",
                   "cores": threads, "kind": "oracle",
                   "sample": f"{s['rows']} whole rows of the workload in "
                             f"{s['seconds']:.1f} s, one row per thread",
                   "single_core": {
                       "value": s1["rows_per_s"], "unit": "rows/s",
                       "cores": 1,
                       "sample": f"{s1['rows']} whole rows in "
                                 f"{s1['seconds']:.1f} s on one thread"}}
        clocks = sampler.summary(t_soak, t_end)
        page_ms = PAGE_LATENCY_MS.get(w.name)
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "latency_ms": ms_per_step,
            "launch": "cuda_graph" if graph is not None else "stream",
            "ms_per_step_stream_launches": stream_ms_max / args.steps,
            "hbm_gbs": hbm_rate, "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": (value / (B / (page_ms * 1e-3))) if page_ms else None,
            "baseline_note": ("page figure 0.8 ms on an RTX 3080 for this "
                              "shape (another machine)") if page_ms else None,
            "dtype": "f32", "data": "synthetic",
            "config": dict(workload_config(w, l2_note),
                           parallelism=f"replicas x{world}",
                           variant=args.variant, strict=args.strict,
                           plan=plan),
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": e2e_entry(e2e_value, e2e, 4 * elems, 4 * elems + 4 * B,
                             copy_bw),
            "gpu_launches": args.steps,
            "clocks": clocks,
            "device_errors": sorted(err),
        }
        if not args.no_per_config and not args.batch:
            line["per_config"] = per_config_runs(
                torch, cs, dev, stream, ex2_peak, peaks["hbm_gbs"],
                skip=w.name, cpu=not args.no_cpu_baseline)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------ per config
def per_config_workloads() -> list[tuple[wl.Workload, str]]:
    """Every configuration of the benchmark besides the headline's, with
    its logit type: 4 x 1000, the 65536 x 64 router, 256 x 131072 long rows
    and the six points of the 4096 x 32000 sweep in fp32; then the long
    rows, the 32 x 50000 rows and one sweep point with bf16 logits (the
    work-reducing input form: 6 bytes per class instead of 8)."""
    out = [(w, "f32") for w in [wl.SMALL, wl.LATENCY, wl.ROUTER, wl.LONG]
           + wl.sweep_workloads()]
    sweep02 = next(w for w in wl.sweep_workloads() if w.name.endswith("b0.2_it20"))
    out += [(wl.LATENCY, "bf16"), (wl.LONG, "bf16"), (sweep02, "bf16")]
    return out


def per_config_runs(torch, cs, dev, stream, ex2_peak: float, hbm_gbs: float,
                    skip: str = "", cpu: bool = True,
                    min_seconds: float = 0.4) -> dict:
    """Each configuration timed in this process after the headline, by the
    headline's rules: automatic plan, a CUDA graph of launches over enough
    rotating input/output pairs to exceed L2 (or one pair larger than L2),
    replayed for at least min_seconds between CUDA events on the launching
    stream, with the SM clocks sampled during that region.  Each entry
    carries the time per launch, rows/s, HBM GB/s, both ex2 fractions, the
    plan and the clocks."""
    sptr = stream.cuda_stream
    sampler = ClockSampler(dev.index if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else 0)
    sampler.start()
    results = {}
    cache = {}
    for w, dt in per_config_workloads():
        if w.name == skip and dt == "f32":
            continue
        base = w.name.split("_b")[0] if w.name.startswith(wl.SWEEP.name) else w.name
        key = (base, dt)
        if key not in cache:
            cache.clear()
            xw = wl.generate(w)
            if dt == "bf16":
                bits = wl.to_bf16_bits(xw)
                xw = wl.bf16_to_f32(bits)
                dev_x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
            else:
                dev_x = torch.from_numpy(xw)
            cache[key] = (xw, entropy_at_one(xw), dev_x)
        x, h1, dev_x = cache[key]
        B, C = x.shape
        in_bytes = 2 if dt == "bf16" else 4
        io_bytes = (in_bytes + 4) * B * C
        nbuf = (max(1, math.ceil(3 * L2_BYTES / io_bytes))
                if io_bytes < 3 * L2_BYTES else 1)
        xs = dev_x.to(dev)
        ins = xs.unsqueeze(0).repeat(nbuf, 1, 1) if nbuf > 1 else xs.unsqueeze(0)
        outs = torch.empty((nbuf, B, C), dtype=torch.float32, device=dev)
        touts = torch.empty((nbuf, B), dtype=torch.float32, device=dev)
        entry_fn = (cs.cs_constrained_softmax_bf16_ex if dt == "bf16"
                    else cs.cs_constrained_softmax_ex)

        def launch(i: int, sp: int = sptr) -> None:
            k = i % nbuf
            st = entry_fn(
                ins[k].data_ptr(), outs[k].data_ptr(), B, C, w.entropy_bound,
                w.t_min, w.t_max, w.max_iter, touts[k].data_ptr(), None, sp)
            if st != 0:
                raise RuntimeError(f"{w.name}: status {st}")

        for i in range(max(3, min(nbuf, 50))):
            launch(i)
        torch.cuda.synchronize()
        K = max(20, nbuf)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cap = torch.cuda.current_stream().cuda_stream
            for j in range(K):
                launch(j, cap)
        graph.replay()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        graph.replay()
        torch.cuda.synchronize()
        one = max(time.perf_counter() - t0, 1e-6)
        reps = max(1, math.ceil(min_seconds / one))
        t_clk0 = time.time()
        e_a = torch.cuda.Event(enable_timing=True)
        e_b = torch.cuda.Event(enable_timing=True)
        e_a.record(stream)
        for _ in range(reps):
            graph.replay()
        e_b.record(stream)
        torch.cuda.synchronize()
        t_clk1 = time.time()
        ms = e_a.elapsed_time(e_b) / (K * reps)
        evals = torch.zeros(B, dtype=torch.int32, device=dev)
        cs.constrained_softmax(ins[0], w.entropy_bound, w.t_min, w.t_max,
                               w.max_iter, out=outs[0], evals_out=evals)
        n_eval = int(evals.sum().item())
        n_search = searched_rows(w, x, h1)
        t_kernel = ms * 1e-3
        roof = ex2_roofline(formula_ex2(w, n_search),
                            ex2_issued(evals, C, cs.plan(B, C)), io_bytes,
                            t_kernel, ex2_peak, hbm_gbs)
        entry = {
            "batch": B, "num_classes": C, "entropy_bound": w.entropy_bound,
            "max_iter": w.max_iter, "logits": dt, "bytes_per_class": in_bytes + 4,
            "launches_timed": K * reps,
            "ms_per_step": ms, "rows_per_s": B / t_kernel,
            "hbm_gbs": roof["hbm_gbs"], "bound": roof["bound"],
            "frac": roof["frac"], "frac_executed": roof["frac_executed"],
            "hbm_frac": roof["hbm_frac"], "roofline_us": roof["roofline_us"],
            "searched_rows": n_search, "evals_per_row_mean": n_eval / B,
            "plan": cs.plan(B, C),
            "l2": (f"rotating {nbuf} input/output pairs" if nbuf > 1
                   else "inputs larger than L2"),
            "clocks": sampler.summary(t_clk0, t_clk1),
        }
        if cpu and w.name == wl.SMALL.name:
            import oracle
            smp = run_oracle_sample(w, x, 1.0, 1)
            entry["cpu_baseline_single_core"] = {
                "value": smp["rows_per_s"], "unit": "rows/s", "cores": 1,
                "kind": "oracle",
                "sample": f"{smp['rows']} whole rows in "
                          f"{smp['seconds']:.1f} s on one thread"}
        results[w.name if dt == "f32" else f"{w.name}_bf16"] = entry
        del graph, ins, outs, touts, xs, evals
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    sampler.stop()
    return results


# --------------------------------------------------------------- backward
BACKWARD_METRIC = ("backward rows/s and effective HBM GB/s (% of roofline) "
                   "of grad = (1/T) p (g - <g, p>)")


def backward_inputs_cpu(w: wl.Workload, rows: np.ndarray):
    """p (by the oracle's softmax at the seeded T), g, T for some rows."""
    import oracle
    x = wl.generate(w, rows)
    g, T = wl.backward_inputs(w, rows)
    p = np.zeros(x.shape, dtype=np.float32)
    for i in range(x.shape[0]):
        if np.isfinite(T[i]):
            p[i] = oracle.softmax(x[i], float(T[i])).astype(np.float32)
    return p, g, T


def run_oracle_backward_sample(w: wl.Workload, seconds: float) -> dict:
    """The oracle's backward, as it stands (one thread), on whole rows of
    the workload (a cycled sample of at most 256 rows, inputs prepared
    outside the timed loop) until `seconds` have passed."""
    import oracle
    oracle.load()
    rows = np.arange(min(w.batch, max(1, (1 << 24) // w.num_classes), 256))
    p, g, T = backward_inputs_cpu(w, rows)
    done = 0
    t0 = time.perf_counter()
    while True:
        oracle.constrained_softmax_backward(p, g, T)
        done += rows.size
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"rows": done, "seconds": dt, "rows_per_s": done / dt,
            "sample_rows": int(rows.size)}


def backward_reference_arm(args, w: wl.Workload) -> int:
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.load()
    n = min(w.batch, max(1, (1 << 22) // w.num_classes))
    rows = np.arange(n)
    p, g, T = backward_inputs_cpu(w, rows)
    for _ in range(args.warmup):
        oracle.constrained_softmax_backward(p, g, T)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.constrained_softmax_backward(p, g, T)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    line = {
        "impl": "reference", "op": "backward", "metric": BACKWARD_METRIC,
        "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, "cpu"),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1,
                         "kind": "oracle",
                         "sample": f"the first {n} rows per step "
                                   f"({args.steps} steps)"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def backward_arm(args, w: wl.Workload) -> int:
    """One step = one backward launch over the whole workload: p (the
    forward kernel's output on the workload's logits), its temperatures and
    a seeded upstream gradient, all resident in HBM."""
    import torch
    import entropy_bounded_softmax_gb300 as cs

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")

    x = wl.generate(w)
    g, _ = wl.backward_inputs(w)
    B, C = x.shape
    elems = B * C
    io_bytes = 12 * elems + 4 * B
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    xs = torch.from_numpy(x).to(dev)
    p0, t0 = cs.constrained_softmax(xs, w.entropy_bound, w.t_min, w.t_max,
                                    w.max_iter, return_t=True)
    del xs
    g0 = torch.from_numpy(g).to(dev)
    nbuf = max(1, math.ceil(3 * L2_BYTES / io_bytes)) if io_bytes < 3 * L2_BYTES else 1
    ps = [p0] + [p0.clone() for _ in range(nbuf - 1)]
    gs = [g0] + [g0.clone() for _ in range(nbuf - 1)]
    outs = [torch.empty_like(p0) for _ in range(nbuf)]
    l2_note = (f"rotating {nbuf} input/output sets "
               f"({nbuf * io_bytes / 2**20:.0f} MiB > L2)") if nbuf > 1 else \
        f"inputs larger than L2 ({io_bytes / 2**20:.0f} MiB)"
    opts = cs.options(cs.VARIANTS[args.variant], args.param, args.threads, 0)

    def launch(i: int, stream_ptr: int = sptr) -> None:
        k = i % nbuf
        st = cs.cs_constrained_softmax_backward_ex(
            ps[k].data_ptr(), gs[k].data_ptr(), t0.data_ptr(),
            outs[k].data_ptr(), B, C, opts, stream_ptr)
        if st != 0:
            raise RuntimeError(f"cs_constrained_softmax_backward failed: {st}")

    for i in range(max(3, args.warmup)):
        launch(i)
    torch.cuda.synchronize()
    plan = cs.plan_backward(B, C, args.variant, args.param, args.threads)
    tm = time_launches(args, torch, launch, stream, dist, local)
    total_ms = reduce_max(dist, tm["ms"], dev)
    stream_ms_max = reduce_max(dist, tm["stream_ms"], dev)
    ms_per_step = total_ms / args.steps
    value = aggregate_rows_per_s(B, world, ms_per_step * 1e-3)

    # End to end through the public API: pinned host p, g and T copied in,
    # the call, the gradient copied out, all inside the events.
    h_p = p0.cpu().pin_memory()
    h_g = torch.from_numpy(g).pin_memory()
    h_t = t0.cpu().pin_memory()

    def make_slot():
        return {"p": torch.empty_like(p0), "g": torch.empty_like(p0),
                "t": torch.empty_like(t0), "out": torch.empty_like(p0),
                "h_out": torch.empty((B, C), dtype=torch.float32).pin_memory()}

    def e2e_step(sl):
        sl["p"].copy_(h_p, non_blocking=True)
        sl["g"].copy_(h_g, non_blocking=True)
        sl["t"].copy_(h_t, non_blocking=True)
        cs.constrained_softmax_backward(sl["p"], sl["g"], sl["t"],
                                        out=sl["out"], variant=args.variant,
                                        param=args.param,
                                        threads=args.threads)
        sl["h_out"].copy_(sl["out"], non_blocking=True)

    e2e = time_e2e(torch, make_slot, e2e_step, stream, max(1, args.e2e_steps))
    e2e = {k: reduce_max(dist, v, dev) for k, v in e2e.items()}
    e2e_value = aggregate_rows_per_s(B, world, e2e["pipelined"] * 1e-3)

    line = None
    if rank == 0:
        peaks = measured_peaks()
        t_kernel = ms_per_step * 1e-3
        hbm_rate = io_bytes / t_kernel / 1e9
        kernel = ("bwd_cluster_kernel" if plan["variant"] == 2
                  else "bwd_rowgroup_kernel")
        roof = {"bound": "hbm", "unit": "GB/s", "achieved": hbm_rate,
                "peak": peaks["hbm_gbs"], "frac": hbm_rate / peaks["hbm_gbs"],
                "traffic": None, "kernel": kernel,
                "algorithmic_bytes": io_bytes,
                "peak_source": f"{peaks['source']} copy bandwidth",
                "roofline_us": io_bytes / (peaks["hbm_gbs"] * 1e9) * 1e6}
        cpu = None
        if not args.no_cpu_baseline:
            s = run_oracle_backward_sample(w, args.cpu_seconds)
            cpu = {"value": s["rows_per_s"], "unit": "rows/s", "cores": 1,
                   "kind": "oracle",
                   "sample": f"{s['rows']} rows ({s['sample_rows']} distinct "
                             f"rows of the workload, cycled) in "
                             f"{s['seconds']:.1f} s on one thread"}
        line = {
            "op": "backward", "metric": BACKWARD_METRIC, "value": value,
            "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step,
            "launch": "cuda_graph" if tm["graph"] is not None else "stream",
            "ms_per_step_stream_launches": stream_ms_max / args.steps,
            "hbm_gbs": hbm_rate, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": dict(workload_config(w, l2_note),
                           parallelism=f"replicas x{world}",
                           variant=args.variant, plan=plan,
                           upstream_gradient="N(0,1) fp32, seeded"),
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": e2e_entry(e2e_value, e2e, 8 * elems + 4 * B, 4 * elems),
            "gpu_launches": args.steps,
            "clocks": tm["sampler"].summary(tm["t0"], tm["t1"]),
        }
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------- attention
ATTENTION_METRIC = ("attention_softmax rows/s and effective HBM GB/s "
                    "(% of roofline)")


def attention_bytes(w) -> int:
    """Algorithmic HBM bytes of one launch: every kept score read once,
    every output written once, the mask read once."""
    S = w.seq_len
    kept = w.batch * w.heads * (S * (S + 1) // 2 if w.causal else S * S)
    mask = 4 * w.batch * S if w.mask != "none" else 0
    return 4 * kept + 4 * w.elements + mask


def attention_config(w, l2: str) -> dict:
    return {"workload": w.name, "batch": w.batch, "heads": w.heads,
            "seq_len": w.seq_len, "causal": w.causal, "mask": w.mask,
            "scores": w.note, "seed": w.seed, "l2": l2}


def run_oracle_attention_sample(w, x, mask, seconds: float,
                                threads: int) -> dict:
    """The oracle as it stands on whole (batch, head) blocks of rows of the
    workload, cycled, until `seconds` have passed."""
    import oracle
    oracle.load()
    S = w.seq_len
    blk = x.reshape(w.batch * w.heads, S, S)
    done = 0
    k = 0
    t0 = time.perf_counter()
    while True:
        b = (k // w.heads) % w.batch
        one = blk[k % blk.shape[0]][None, None]
        oracle.attention_softmax(one, None if mask is None else mask[b:b + 1],
                                 w.causal, threads=threads)
        done += S
        k += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"rows": done, "seconds": dt, "rows_per_s": done / dt}


def attention_reference_arm(args, w) -> int:
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    threads = oracle.default_threads()
    S = w.seq_len
    n_blocks = max(1, min(w.batch * w.heads, (1 << 22) // (S * S) or 1))
    x = wl.generate_attention(w, np.arange(n_blocks * S)).reshape(
        n_blocks, 1, S, S)
    mask = wl.attention_mask(w)
    m0 = None if mask is None else mask[:1]
    for _ in range(args.warmup):
        for k in range(n_blocks):
            oracle.attention_softmax(x[k:k + 1], m0, w.causal, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for k in range(n_blocks):
            oracle.attention_softmax(x[k:k + 1], m0, w.causal, threads=threads)
    dt = time.perf_counter() - t0
    value = n_blocks * S * args.steps / dt
    line = {
        "impl": "reference", "op": "attention", "metric": ATTENTION_METRIC,
        "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": attention_config(w, "cpu"),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{n_blocks} (batch, head) blocks of "
                                   f"{S} rows per step ({args.steps} steps)"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def attention_arm(args, w) -> int:
    """One step = one attention_softmax launch over the whole workload,
    scores and mask resident in HBM."""
    import torch
    import entropy_bounded_softmax_gb300 as cs

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")

    B, H, S = w.batch, w.heads, w.seq_len
    x = wl.generate_attention(w).reshape(B, H, S, S)
    mask = wl.attention_mask(w)
    io_bytes = attention_bytes(w)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    xs = torch.from_numpy(x).to(dev)
    md = torch.from_numpy(mask).to(dev) if mask is not None else None
    nbuf = max(1, math.ceil(3 * L2_BYTES / io_bytes)) if io_bytes < 3 * L2_BYTES else 1
    ins = [xs] + [xs.clone() for _ in range(nbuf - 1)]
    outs = [torch.empty_like(xs) for _ in range(nbuf)]
    l2_note = (f"rotating {nbuf} score/output pairs "
               f"({nbuf * io_bytes / 2**20:.0f} MiB > L2)") if nbuf > 1 else \
        f"inputs larger than L2 ({io_bytes / 2**20:.0f} MiB)"
    opts = cs.options(cs.VARIANTS[args.variant], args.param, args.threads, 0)
    m_ptr = md.data_ptr() if md is not None else None

    def launch(i: int, stream_ptr: int = sptr) -> None:
        k = i % nbuf
        st = cs.cs_attention_softmax_ex(ins[k].data_ptr(), outs[k].data_ptr(),
                                        m_ptr, B, H, S, int(w.causal), opts,
                                        stream_ptr)
        if st != 0:
            raise RuntimeError(f"cs_attention_softmax failed: {st}")

    cs.get_error()
    for i in range(max(3, args.warmup)):
        launch(i)
    torch.cuda.synchronize()
    plan = cs.plan_attention(B, H, S, True, args.variant, args.param,
                             args.threads)
    tm = time_launches(args, torch, launch, stream, dist, local)
    total_ms = reduce_max(dist, tm["ms"], dev)
    stream_ms_max = reduce_max(dist, tm["stream_ms"], dev)
    ms_per_step = total_ms / args.steps
    rows = B * H * S
    value = aggregate_rows_per_s(rows, world, ms_per_step * 1e-3)
    err = cs.get_error()

    # End to end: pinned host scores (and mask) in, the public call, the
    # weights out.
    h_x = torch.from_numpy(x).pin_memory()
    h_m = torch.from_numpy(mask).pin_memory() if mask is not None else None

    def make_slot():
        return {"x": torch.empty_like(xs),
                "m": torch.empty_like(md) if md is not None else None,
                "out": torch.empty_like(xs),
                "h_out": torch.empty((B, H, S, S),
                                     dtype=torch.float32).pin_memory()}

    def e2e_step(sl):
        sl["x"].copy_(h_x, non_blocking=True)
        if sl["m"] is not None:
            sl["m"].copy_(h_m, non_blocking=True)
        cs.attention_softmax(sl["x"], sl["m"], w.causal, out=sl["out"],
                             variant=args.variant, param=args.param,
                             threads=args.threads)
        sl["h_out"].copy_(sl["out"], non_blocking=True)

    e2e = time_e2e(torch, make_slot, e2e_step, stream, max(1, args.e2e_steps))
    e2e = {k: reduce_max(dist, v, dev) for k, v in e2e.items()}
    e2e_value = aggregate_rows_per_s(rows, world, e2e["pipelined"] * 1e-3)

    line = None
    if rank == 0:
        peaks = measured_peaks()
        t_kernel = ms_per_step * 1e-3
        hbm_rate = io_bytes / t_kernel / 1e9
        kernel = ("attn_cta_kernel" if plan["variant"] == 2
                  else "attn_rowgroup_kernel")
        roof = {"bound": "hbm", "unit": "GB/s", "achieved": hbm_rate,
                "peak": peaks["hbm_gbs"], "frac": hbm_rate / peaks["hbm_gbs"],
                "traffic": None, "kernel": kernel,
                "algorithmic_bytes": io_bytes,
                "peak_source": f"{peaks['source']} copy bandwidth",
                "roofline_us": io_bytes / (peaks["hbm_gbs"] * 1e9) * 1e6}
        cpu = None
        if not args.no_cpu_baseline:
            import oracle
            threads = oracle.default_threads()
            s = run_oracle_attention_sample(w, x, mask, args.cpu_seconds,
                                            threads)
            cpu = {"value": s["rows_per_s"], "unit": "rows/s",
                   "cores": threads, "kind": "oracle",
                   "sample": f"{s['rows']} rows in whole (batch, head) "
                             f"blocks of the workload, cycled, in "
                             f"{s['seconds']:.1f} s"}
        page_ms = 0.2 if w.name == "attention_32x8x512" else None
        line = {
            "op": "attention", "metric": ATTENTION_METRIC, "value": value,
            "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step,
            "launch": "cuda_graph" if tm["graph"] is not None else "stream",
            "ms_per_step_stream_launches": stream_ms_max / args.steps,
            "hbm_gbs": hbm_rate, "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "baseline_note": ("page figure 0.2 ms on an RTX 3080 for this "
                              "shape (another machine)") if page_ms else None,
            "dtype": "f32", "data": "synthetic",
            "config": dict(attention_config(w, l2_note),
                           parallelism=f"replicas x{world}",
                           variant=args.variant, plan=plan),
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": e2e_entry(e2e_value, e2e,
                             4 * w.elements + (4 * B * S if mask is not None else 0),
                             4 * w.elements),
            "gpu_launches": args.steps,
            "clocks": tm["sampler"].summary(tm["t0"], tm["t1"]),
            "device_errors": sorted(err),
        }
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------- biencoder
BIENC_METRIC = ("biencoder_attention query rows/s, with its ex2, fp32 FMA "
                "and HBM rooflines")
# fp32 FMA peak of the SIMT pipes, from unit counts: 152 SMs x 128 fp32
# lanes x 2 flops per FMA at the 2.07 GHz maximum SM clock.
FP32_SIMT_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def bienc_config(w, l2: str) -> dict:
    return {"workload": w.name, "batch": w.batch, "heads": w.heads,
            "query_len": w.query_len, "context_len": w.context_len,
            "d_head": w.d_head, "entropy_bound": w.entropy_bound,
            "inputs": w.note, "seed": w.seed, "l2": l2}


def bienc_reference_arm(args, w) -> int:
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.load()
    q, k, v = wl.generate_biencoder(w)
    scale = 1.0 / math.sqrt(w.d_head)
    # Each step: the oracle on one (batch, head) pair's queries.
    for i in range(args.warmup):
        b, h = divmod(i % (w.batch * w.heads), w.heads)
        oracle.biencoder_attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                   v[b:b + 1, h:h + 1], scale, w.entropy_bound)
    t0 = time.perf_counter()
    for i in range(args.steps):
        b, h = divmod(i % (w.batch * w.heads), w.heads)
        oracle.biencoder_attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                   v[b:b + 1, h:h + 1], scale, w.entropy_bound)
    dt = time.perf_counter() - t0
    value = w.query_len * args.steps / dt
    threads = oracle.default_threads()
    line = {
        "impl": "reference", "op": "biencoder", "metric": BIENC_METRIC,
        "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": bienc_config(w, "cpu"),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"one (batch, head) pair of {w.query_len} "
                                   f"queries per step ({args.steps} steps)"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def bienc_arm(args, w) -> int:
    """One step = one fused biencoder_attention launch over the workload,
    inputs resident in HBM."""
    import torch
    import entropy_bounded_softmax_gb300 as cs

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    q, k, v = wl.generate_biencoder(w)
    B, H, Q, K, D = w.batch, w.heads, w.query_len, w.context_len, w.d_head
    scale = 1.0 / math.sqrt(D)
    io_bytes = 4 * (2 * B * H * Q * D + 2 * B * H * K * D)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    qs, ks, vs = (torch.from_numpy(a).to(dev) for a in (q, k, v))
    nbuf = max(1, math.ceil(3 * L2_BYTES / io_bytes)) if io_bytes < 3 * L2_BYTES else 1
    sets = [(qs, ks, vs)] + [tuple(a.clone() for a in (qs, ks, vs))
                             for _ in range(nbuf - 1)]
    outs = [torch.empty_like(qs) for _ in range(nbuf)]
    l2_note = (f"rotating {nbuf} input/output sets "
               f"({nbuf * io_bytes / 2**20:.0f} MiB > L2)") if nbuf > 1 else \
        f"inputs larger than L2 ({io_bytes / 2**20:.0f} MiB)"

    def launch(i: int, stream_ptr: int = sptr) -> None:
        j = i % nbuf
        a, b_, c = sets[j]
        st = cs.cs_biencoder_attention(a.data_ptr(), b_.data_ptr(),
                                       c.data_ptr(), outs[j].data_ptr(), B, Q,
                                       K, D, H, scale, w.entropy_bound,
                                       stream_ptr)
        if st != 0:
            raise RuntimeError(f"cs_biencoder_attention failed: {st}")

    cs.get_error()
    for i in range(max(3, args.warmup)):
        launch(i)
    torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(dev)
    optin = int(getattr(props, "shared_memory_per_block_optin", 232448))
    st, plan = cs.cs_plan_biencoder_host(B, Q, K, D, H, None, optin)
    plan = plan.as_dict()
    tm = time_launches(args, torch, launch, stream, dist, local)
    total_ms = reduce_max(dist, tm["ms"], dev)
    stream_ms_max = reduce_max(dist, tm["stream_ms"], dev)
    ms_per_step = total_ms / args.steps
    rows = B * H * Q
    value = aggregate_rows_per_s(rows, world, ms_per_step * 1e-3)
    err = cs.get_error()

    h_q, h_k, h_v = (torch.from_numpy(a).pin_memory() for a in (q, k, v))

    def make_slot():
        return {"q": torch.empty_like(qs), "k": torch.empty_like(ks),
                "v": torch.empty_like(vs), "out": torch.empty_like(qs),
                "h_out": torch.empty(q.shape, dtype=torch.float32).pin_memory()}

    def e2e_step(sl):
        sl["q"].copy_(h_q, non_blocking=True)
        sl["k"].copy_(h_k, non_blocking=True)
        sl["v"].copy_(h_v, non_blocking=True)
        cs.biencoder_attention(sl["q"], sl["k"], sl["v"], scale,
                               w.entropy_bound, out=sl["out"])
        sl["h_out"].copy_(sl["out"], non_blocking=True)

    e2e = time_e2e(torch, make_slot, e2e_step, stream, max(1, args.e2e_steps))
    e2e = {kk: reduce_max(dist, vv, dev) for kk, vv in e2e.items()}
    e2e_value = aggregate_rows_per_s(rows, world, e2e["pipelined"] * 1e-3)

    line = None
    if rank == 0:
        import oracle
        peaks = measured_peaks()
        ex2_peak = probe_ex2_peak(torch, cs, sptr)
        t_kernel = ms_per_step * 1e-3
        # Searched rows from the oracle's step-1 scores on a sample of
        # (batch, head) pairs, scaled to the launch.
        nbh = min(8, B * H)
        sc = oracle.biencoder_scores(q.reshape(B * H, 1, Q, D)[:nbh],
                                     k.reshape(B * H, 1, K, D)[:nbh], scale)
        import scipy.special
        pr = scipy.special.softmax(sc.reshape(-1, K).astype(np.float64), axis=1)
        Hs = scipy.special.entr(pr).sum(axis=1)
        searched = float(np.mean(Hs > np.float32(w.entropy_bound))) * rows
        exps = (rows + searched * 20) * K
        tc = bool(plan.get("tensor_cores"))
        # Step 1 (and, on the fused path, step 3) on the fp32 FMA pipes;
        # with the tensor-core step 3, its three TF32 products per fp32
        # product at the TF32 rate (half the measured bf16 rate, the
        # nominal ratio of the two).
        flops = (2.0 if tc else 4.0) * rows * K * D
        tc_flops = 3 * 2.0 * rows * K * D if tc else 0.0
        tf32_peak = 0.5 * measured_bf16_tflops() * 1e12
        t_hbm = io_bytes / (peaks["hbm_gbs"] * 1e9)
        t_ex2 = exps / ex2_peak
        t_fma = flops / (FP32_SIMT_TFLOPS * 1e12)
        t_tc = tc_flops / tf32_peak if tc else 0.0
        bound = max(("hbm", t_hbm), ("ex2", t_ex2), ("fma", t_fma),
                    key=lambda kv: kv[1])
        roof = {"bound": "hbm" if bound[0] == "hbm" else "alu",
                "limit": bound[0],
                "unit": {"hbm": "GB/s", "ex2": "Gex2/s", "fma": "TFLOP/s"}[bound[0]],
                "achieved": {"hbm": io_bytes / t_kernel / 1e9,
                             "ex2": exps / t_kernel / 1e9,
                             "fma": flops / t_kernel / 1e12}[bound[0]],
                "peak": {"hbm": peaks["hbm_gbs"], "ex2": ex2_peak / 1e9,
                         "fma": FP32_SIMT_TFLOPS}[bound[0]],
                "frac": bound[1] / t_kernel, "traffic": None,
                "kernel": "bienc_kernel", "algorithmic_bytes": io_bytes,
                "algorithmic_ex2": exps, "algorithmic_flops": flops,
                "roofline_us": {"hbm": t_hbm * 1e6, "ex2": t_ex2 * 1e6,
                                "fma": t_fma * 1e6, "tensor_tf32": t_tc * 1e6},
                "tensor_core_step3": tc, "tensor_flops": tc_flops,
                "peak_source": "hbm: measured copy bandwidth; ex2: probe; "
                               "fma: 152 SMs x 128 lanes x 2 flops x 2.07 GHz; "
                               "tf32: half the measured bf16 GEMM rate"}
        cpu = None
        if not args.no_cpu_baseline:
            t0 = time.perf_counter()
            n = 0
            while time.perf_counter() - t0 < args.cpu_seconds:
                b, h = divmod(n % (B * H), H)
                oracle.biencoder_attention(q[b:b + 1, h:h + 1],
                                           k[b:b + 1, h:h + 1],
                                           v[b:b + 1, h:h + 1], scale,
                                           w.entropy_bound)
                n += 1
            dt = time.perf_counter() - t0
            cpu = {"value": n * Q / dt, "unit": "rows/s",
                   "cores": oracle.default_threads(), "kind": "oracle",
                   "sample": f"{n} (batch, head) pairs of {Q} queries in "
                             f"{dt:.1f} s"}
        line = {
            "op": "biencoder", "metric": BIENC_METRIC, "value": value,
            "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step,
            "launch": "cuda_graph" if tm["graph"] is not None else "stream",
            "ms_per_step_stream_launches": stream_ms_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "baseline_note": ("page figure 0.5 ms on an RTX 3080 for this "
                              "shape (another machine)")
            if w.name == "biencoder_32x8x512x64x64" else None,
            "dtype": "f32", "data": "synthetic",
            "config": dict(bienc_config(w, l2_note),
                           parallelism=f"replicas x{world}", plan=plan),
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": e2e_entry(e2e_value, e2e,
                             4 * (B * H * Q * D + 2 * B * H * K * D),
                             4 * B * H * Q * D),
            "gpu_launches": args.steps * (2 if plan.get("tensor_cores") else 1),
            "clocks": tm["sampler"].summary(tm["t0"], tm["t1"]),
            "device_errors": sorted(err),
        }
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None) -> int:
    args = parse_args(argv)
    if args.op == "biencoder":
        name = args.workload if args.workload in wl.BIENCODER_WORKLOADS \
            else wl.BIENC_PAGE.name
        bw = wl.BIENCODER_WORKLOADS[name]
        if args.impl == "reference":
            return bienc_reference_arm(args, bw)
        return bienc_arm(args, bw)
    if args.op == "attention":
        name = args.workload if args.workload in wl.ATTENTION_WORKLOADS \
            else wl.ATTN_PAGE.name
        aw = wl.ATTENTION_WORKLOADS[name]
        if args.impl == "reference":
            return attention_reference_arm(args, aw)
        return attention_arm(args, aw)
    w = find_workload(args.workload)
    if args.batch:
        w = w.with_(batch=min(args.batch, w.batch),
                    name=f"{w.name}[:{min(args.batch, w.batch)}]")
    if args.op == "backward":
        if args.impl == "reference":
            return backward_reference_arm(args, w)
        return backward_arm(args, w)
    if args.impl == "reference":
        return reference_arm(args, w)
    return our_arm(args, w)


if __name__ == "__main__":
    sys.exit(main())
