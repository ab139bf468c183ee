#!/usr/bin/env python
"""Benchmark: AWQ W4A16 awq_gemm on one GB300.

Headline (the JSON line's `value`): decode GB/s on the 70B-shaped linears at M = 1 --
one step is the three linears 8192x8192, 8192x28672, 28672x8192 (group size 128, fp16
bias), one awq_gemm call (one kernel launch) each, through prepared AwqLinear layers.
Weights rotate over R independent sets whose total exceeds 3x the 129 MB L2, so every
step streams its weights from HBM.  Steps are replayed from CUDA graphs and timed with
CUDA events on the replay stream: W warm-up steps, then repetitions of exactly K timed
steps until the repetitions cover at least 0.5 s; the reported step time is the median
repetition.  nvidia-smi clocks are sampled during every timed region.

Extra blocks on the same line: `prefill` -- TFLOP/s of the 70B linears at M = 4096 (the
three linears per step, eager launches, inputs larger than L2) through prepared layers with
the tile-packed weights (awq_gemm_packed; the one-off awq_repack timed separately), beside
awq_gemm on the checkpoint layout and awq_dequant + cuBLAS on the same step; `prefill_7b` --
the same for the 7B linears at M = 2048; `decode_7b` -- the 7B decode step (M = 1: 4096x4096, 4096x11008,
11008x4096, bias); `e2e` -- the headline step end to end through the public call with
pinned host buffers (one host-to-device copy of the step's activations, three calls, one
device-to-host copy of the outputs, a synchronize per step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain restatement of the method the tests
check against) on the host cores on a bounded column sample of the same workload.
Prints one JSON line (rank 0).  Multi-GPU (torchrun): each rank runs an independent
replica; the reported value is the sum over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = ("awq_gemm GB/s (decode, % HBM roofline) and TFLOP/s (prefill, % fp16 peak) "
          "on 1 GB300")
UNIT = "GB/s"
LINEARS = ["70b_m1_8192x8192", "70b_m1_8192x28672", "70b_m1_28672x8192"]
WORKLOAD_NAME = ("70B decode M=1: linears 8192x8192, 8192x28672, 28672x8192; "
                 "group_size 128; fp16 bias")
LINEARS_7B = ["7b_decode_m1_4096x4096_bias", "7b_decode_m1_4096x11008_bias",
              "7b_decode_m1_11008x4096_bias"]
WORKLOAD_7B = ("7B decode M=1: linears 4096x4096, 4096x11008, 11008x4096; group_size 128; "
               "fp16 bias")
PREFILL = ["70b_m4096_8192x8192", "70b_m4096_8192x28672", "70b_m4096_28672x8192"]
WORKLOAD_PREFILL = ("70B prefill M=4096: linears 8192x8192, 8192x28672, 28672x8192; "
                    "group_size 128; fp16 bias")
PREFILL_7B = ["7b_prefill_m2048_4096x11008", "7b_prefill_m2048_11008x4096"]
WORKLOAD_PREFILL_7B = "7B prefill M=2048: linears 4096x11008, 11008x4096; group_size 128; no bias"
L2_BYTES = 129e6
FALLBACK_HBM_GBS = 6800.0
FALLBACK_TFLOPS = 1900.0
MIN_TIMED_S = 0.5  # every timed region repeats its K-step repetitions until it covers this


def algorithmic_bytes(M, K, N, G, bias):
    """Bytes the method must move once: packed weights, zeros, scales, x, y, bias."""
    G = K if G == -1 else G
    ng = K // G
    return K * N // 2 + ng * N // 2 + 2 * ng * N + 2 * M * K + 2 * M * N + (2 * N if bias else 0)


def workload_linears(set_index: int, names=None):
    out = []
    for name in (names or LINEARS):
        cfg, si, _, M, K, N, G, b = synth.workload(name)
        seed = synth.seed_for(cfg, si) + 100000 * set_index
        out.append(synth.awq_linear(seed, M, K, N, group_size=G, bias=b))
    return out


def step_bytes(lins):
    return sum(algorithmic_bytes(d["M"], d["K"], d["N"], d["group_size"], d["bias"] is not None)
               for d in lins)


def step_flop(names):
    tot = 0.0
    for name in names:
        _, _, _, M, K, N, _, _ = synth.workload(name)
        tot += 2.0 * M * N * K
    return tot


# DRAM traffic of the decode kernel per launch (dram__bytes_read.sum + dram__bytes_write.sum),
# averaged over the three linears of one headline step, from the ncu launch list of
# `python bench.py --steps 20 --warmup 3 --no-cpu-baseline --decode-only` (its summary is
# the decode launch-list profile under profiles/); valid only for the kernel source it was
# measured on (SHA-256 of the files below), else reported as null.
TRAFFIC_BYTES_PER_LAUNCH = 93_185_075
TRAFFIC_SOURCES = {
    "w4a16_weight_only_gb300/csrc/awq_decode_tma.cu":
        "3abd9c35b548d6d2a6de5abf5895ead1aa80163b256e434f3e0379e9d03701e0",
    "w4a16_weight_only_gb300/csrc/awq_ptx.cuh":
        "7488ac9d3e1525b7a303d4e435be38b50cdcbf4b04c725918e9c8ee96f8b2e02",
}


def measured_traffic():
    import hashlib
    for rel, digest in TRAFFIC_SOURCES.items():
        try:
            with open(os.path.join(ROOT, rel), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None
        except OSError:
            return None
    return TRAFFIC_BYTES_PER_LAUNCH


def _peaks_file():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except Exception:
        return None


def peaks():
    p = _peaks_file()
    try:
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak(sustained: bool):
    """Dense fp16 tensor peak: the measured bf16 cuBLAS figure (fp16 runs at the same nominal
    rate), sustained for a kernel timed inside a long loop, burst for one timed alone."""
    p = _peaks_file()
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    try:
        return float(p[key]), f"measured ({key}; fp16 nominal rate equal to bf16)"
    except Exception:
        return FALLBACK_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples; keeps those taken inside [start, end]."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(index)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        self.rows = None

    def start(self):
        self.t0 = time.time()

    def end(self):
        self.t1 = time.time()

    def _collect(self):
        if self.rows is not None or self.proc is None:
            return
        time.sleep(0.05)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:], parts[3]))
            except Exception:
                continue
        self.rows = rows

    def window(self, t0, t1):
        """Summary of the samples taken inside [t0, t1] (wall clock, seconds)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        self._collect()
        rows = self.rows
        inside = [r for r in rows if t0 - 0.02 <= r[0] <= t1 + 0.02]
        used = inside
        if not used and rows:
            mid = 0.5 * (t0 + t1)
            used = sorted(rows, key=lambda r: abs(r[0] - mid))[:2]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in used for i, v in enumerate(r[3]) if v == "Active"})
        power = []
        for r in used:
            try:
                power.append(float(r[4]))
            except ValueError:
                pass
        return {"sm_mhz": statistics.median([r[1] for r in used]) if used else None,
                "sm_max_mhz": max(r[2] for r in used) if used else None,
                "power_w_median": statistics.median(power) if power else None,
                "reasons": reasons, "samples": len(inside)}

    def finish(self):
        return self.window(self.t0, self.t1)


def dist_setup(args):
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
    return rank, world, local


def reduce_max(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_step: int, steps: int, world: int, elapsed_max_s: float) -> float:
    """Whole-job throughput: every rank ran `steps` steps of `bytes_per_step` algorithmic
    bytes; the job took the slowest rank's time."""
    return world * bytes_per_step * steps / elapsed_max_s / 1e9


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------- CPU oracle ----

def oracle_sample(width: int):
    """Column sample of the workload: for each linear, its first `width` output columns
    (itself a valid AWQ linear of N = width).  Returns (inputs, algorithmic bytes)."""
    lins = workload_linears(0)
    sub = []
    for d in lins:
        w = min(width, d["N"])
        sub.append({"x": d["x"], "qweight": np.ascontiguousarray(d["qweight"][:, :w // 8]),
                    "qzeros": np.ascontiguousarray(d["qzeros"][:, :w // 8]),
                    "scales": np.ascontiguousarray(d["scales"][:, :w]),
                    "bias": None if d["bias"] is None else d["bias"][:w],
                    "group_size": d["group_size"], "M": d["M"], "K": d["K"], "N": w})
    return sub, step_bytes(sub)


def oracle_step(sub):
    import oracle
    for d in sub:
        oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], d["group_size"])


def cpu_baseline(seconds: float = 12.0):
    width = 512
    sub, nbytes = oracle_sample(width)
    oracle_step(sub)
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_step(sub)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": nbytes * n / el / 1e9, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first {width} output columns of each of the three 70B linears (M=1), "
                      f"{n} passes in {el:.1f} s; numpy fp64 matmul (BLAS threads), "
                      "unpack/dequant single-threaded"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    # size each step so that warm-up + timed steps end within about two minutes
    probe_sub, _ = oracle_sample(256)
    t0 = time.perf_counter()
    oracle_step(probe_sub)
    per256 = max(time.perf_counter() - t0, 1e-4)
    budget = 120.0 / max(1, args.steps + args.warmup)
    width = int(max(8, min(28672, 256 * budget / per256)) // 8 * 8)
    sub, nbytes = oracle_sample(width)
    for _ in range(args.warmup):
        oracle_step(sub)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(sub)
    el = time.perf_counter() - t0
    value = nbytes * args.steps / el / 1e9
    widths = ", ".join(f"{d['K']}x{d['N']}" for d in sub)
    desc = (f"first min({width}, N) output columns of each of the three 70B linears (M=1) per "
            f"step (K x columns: {widths}); numpy fp64 matmul (BLAS threads), unpack/dequant "
            "single-threaded")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD_NAME + " (column sample)", "sample_width": width},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------- GPU path ----

def timed_repetitions(run_k, k, stream, min_s=MIN_TIMED_S, max_reps=100000):
    """Repetitions of exactly k steps (run_k(k) enqueues them on `stream`), each bracketed by
    CUDA events recorded on that stream, until the repetitions cover min_s.  Returns the
    per-repetition times (s) and the wall-clock window of the region."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True)]
    w0 = time.time()
    evs[0].record(stream)
    total, reps = 0.0, 0
    while reps < max_reps:
        # enqueue a batch of repetitions, then measure what they took
        batch = 1 if reps == 0 else max(1, min(256, int(reps * (min_s - total) / max(total, 1e-9)) + 1))
        for _ in range(batch):
            run_k(k)
            e = torch.cuda.Event(enable_timing=True)
            e.record(stream)
            evs.append(e)
            reps += 1
        evs[-1].synchronize()
        total = evs[0].elapsed_time(evs[-1]) / 1e3
        if total >= min_s:
            break
    w1 = time.time()
    times = [evs[i].elapsed_time(evs[i + 1]) / 1e3 for i in range(len(evs) - 1)]
    return times, (w0, w1)


def _device_sets(names, R, torch, awq):
    """R independent weight sets (set 0 from the workload seeds) with their activations,
    outputs and prepared AwqLinear layers (static weights, as at model load)."""
    lins0 = workload_linears(0, names)
    sets = []
    for r in range(R):
        lins = lins0 if r == 0 else workload_linears(r, names)
        dev = []
        for d in lins:
            t = {k: torch.from_numpy(d[k]).cuda() for k in ("x", "qweight", "qzeros", "scales")}
            t["bias"] = torch.from_numpy(d["bias"]).cuda() if d["bias"] is not None else None
            t["y"] = torch.empty((d["M"], d["N"]), dtype=torch.float16, device="cuda")
            t["G"] = d["group_size"]
            t["layer"] = awq.AwqLinear(t["qweight"], t["qzeros"], t["scales"], t["bias"], t["G"])
            dev.append(t)
        sets.append(dev)
    return lins0, sets


def _decode_region(names, args, world, torch, awq, stream, clocks):
    """The decode step over rotating weight sets, replayed from CUDA graphs; returns the
    median step time, the timing details and the sets (for the end-to-end runs)."""
    lins0 = workload_linears(0, names)
    per_set = sum(d["qweight"].nbytes + d["qzeros"].nbytes + d["scales"].nbytes for d in lins0)
    R = max(2, int(np.ceil(3.0 * L2_BYTES / per_set)))
    _, sets = _device_sets(names, R, torch, awq)
    sp = stream.cuda_stream

    def step(r):
        for t in sets[r]:
            t["layer"](t["x"], out=t["y"], stream=sp)

    # one graph of exactly K steps (weight sets in rotation) when K is moderate, so that a timed
    # repetition is one replay; for large K a graph of R steps replayed, plus single steps
    kg = args.steps if args.steps <= 512 else R
    with torch.cuda.stream(stream):
        for r in range(R):  # eager warm-up (first calls set kernel attributes)
            step(r)
        stream.synchronize()
        cycle = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cycle, stream=stream):
            for i in range(kg):
                step(i % R)
        singles = []
        for r in range(R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(r)
            singles.append(g)

    def run_steps(k):
        full, rem = divmod(k, kg)
        for _ in range(full):
            cycle.replay()
        for r in range(rem):
            singles[r % R].replay()

    with torch.cuda.stream(stream):
        run_steps(max(args.warmup, 3))
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        times, (w0, w1) = timed_repetitions(run_steps, args.steps, stream)
        torch.cuda.synchronize()
        barrier(world)
    awq.device_status()
    t_step = statistics.median(times) / args.steps
    return {"t_step": t_step, "reps": len(times), "timed_s": sum(times), "R": R,
            "per_set": per_set, "win": (w0, w1), "sets": sets,
            "nbytes": step_bytes(lins0), "launches": len(names) * args.steps * len(times)}


def _prefill_region(names, args, world, torch, awq, stream):
    """A prefill step (the linears `names`, one call each), eager launches, inputs larger
    than L2, timed three ways: prepared layers with the tile-packed copy (awq_gemm_packed;
    the one-off repack timed separately), prepared layers on the checkpoint layout
    (awq_gemm), and the pages' large-batch strategy (awq_dequant to a dense fp16 weight,
    then a library GEMM) as a comparator."""
    lins = workload_linears(0, names)
    dev = []
    for d in lins:
        t = {k: torch.from_numpy(d[k]).cuda() for k in ("x", "qweight", "qzeros", "scales")}
        t["bias"] = torch.from_numpy(d["bias"]).cuda() if d["bias"] is not None else None
        t["y"] = torch.empty((d["M"], d["N"]), dtype=torch.float16, device="cuda")
        t["G"] = d["group_size"]
        t["plain"] = awq.AwqLinear(t["qweight"], t["qzeros"], t["scales"], t["bias"], t["G"])
        dev.append(t)
    del lins
    sp = stream.cuda_stream
    # the one-off conversion, timed on its own (median of 5 passes over the step's linears)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for t in dev:
            t["layer"] = awq.AwqLinear(t["qweight"], t["qzeros"], t["scales"], t["bias"], t["G"],
                                       packed=True)
        rp = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for t in dev:
                awq.awq_repack(t["qweight"], t["qzeros"], t["scales"], t["G"], out=t["layer"].packed,
                               stream=stream)
            b.record(stream)
            b.synchronize()
            rp.append(a.elapsed_time(b) / 1e3)
    t_repack = statistics.median(rp)

    def timed_step(run_k):
        with torch.cuda.stream(stream):
            run_k(max(args.warmup, 3))
            torch.cuda.synchronize()
            barrier(world)
            times, win = timed_repetitions(run_k, args.steps, stream)
            torch.cuda.synchronize()
            barrier(world)
        return statistics.median(times) / args.steps, len(times), sum(times), win

    def run_packed(k):
        for _ in range(k):
            for t in dev:
                t["layer"](t["x"], out=t["y"], stream=sp)

    def run_plain(k):
        for _ in range(k):
            for t in dev:
                t["plain"](t["x"], out=t["y"], stream=sp)

    for t in dev:
        t["wd"] = torch.empty((t["qweight"].shape[0], t["y"].shape[1]), dtype=torch.float16,
                              device="cuda")

    def run_ref(k):
        for _ in range(k):
            for t in dev:
                awq.awq_dequant(t["qweight"], t["qzeros"], t["scales"], t["G"], out=t["wd"],
                                stream=stream)
                if t["bias"] is not None:
                    torch.addmm(t["bias"], t["x"], t["wd"], out=t["y"])
                else:
                    torch.matmul(t["x"], t["wd"], out=t["y"])

    out = {"packed": timed_step(run_packed), "checkpoint": timed_step(run_plain),
           "ref": timed_step(run_ref), "t_repack": t_repack}
    awq.device_status()
    del dev
    torch.cuda.empty_cache()
    return out


def _prefill_block(names, workload, args, world, torch, awq, stream, windows, key):
    pf = _prefill_region(names, args, world, torch, awq, stream)
    flop = step_flop(names)
    t_p, reps, timed_s, win = pf["packed"]
    tp = reduce_max(t_p, world)
    peak_s, src_s = tensor_peak(sustained=True)
    peak_b, _ = tensor_peak(sustained=False)
    ach = flop / t_p / 1e12
    t_c, reps_c, timed_c, win_c = pf["checkpoint"]
    t_r, reps_r, timed_r, win_r = pf["ref"]
    windows[key] = win
    windows[key + ".checkpoint_layout"] = win_c
    windows[key + ".dequant_plus_cublas"] = win_r
    return {
        "workload": workload, "metric": "TFLOP/s", "value": world * flop / tp / 1e12,
        "unit": "TFLOP/s", "ms_per_step": tp * 1e3, "flop_per_step": flop,
        "path": "awq_gemm_packed (tile-packed weights, AwqLinear(packed=True))",
        "roofline": {"bound": "tensor", "achieved": ach, "peak": peak_s, "unit": "TFLOP/s",
                     "frac": ach / peak_s, "peak_source": src_s + ": the step loop runs for "
                     "seconds under the power cap", "frac_of_burst_peak": ach / peak_b,
                     "kernel": "packed_kernel (tcgen05, A operand in TMEM)", "traffic": None},
        "timing": f"{reps} repetitions of {args.steps} steps ({timed_s:.3f} s); eager launches; "
                  "inputs larger than L2",
        "repack_ms_one_off": pf["t_repack"] * 1e3,
        "checkpoint_layout": {"ms_per_step": t_c * 1e3, "TFLOP_s": flop / t_c / 1e12,
                              "note": "awq_gemm on the checkpoint layout (prefill_kernel, "
                                      "dequantized tile in shared memory)",
                              "timing": f"{reps_c} repetitions ({timed_c:.3f} s)"},
        "dequant_plus_cublas": {"ms_per_step": t_r * 1e3, "TFLOP_s": flop / t_r / 1e12,
                                "timing": f"{reps_r} repetitions ({timed_r:.3f} s)",
                                "note": "awq_dequant to a dense fp16 weight, then torch.addmm "
                                        "(cuBLAS), per linear: comparator, not the product"},
        "gpu_launches": len(names) * args.steps * reps}


def _e2e(reg, args, world, torch, stream):
    """The headline step end to end through the public call: per step one pinned
    host-to-device copy of the step's activations, the three calls, one device-to-host copy
    of the outputs and a synchronize; eagerly and replayed from CUDA graphs.  Each loop
    covers at least MIN_TIMED_S."""
    sets, R = reg["sets"], reg["R"]
    xsz = [t["x"].numel() for t in sets[0]]
    ysz = [t["y"].numel() for t in sets[0]]
    hx_all = torch.cat([t["x"].reshape(-1).cpu() for t in sets[0]]).pin_memory()
    hy_all = torch.empty(sum(ysz), dtype=torch.float16).pin_memory()
    xd_all = torch.empty(sum(xsz), dtype=torch.float16, device="cuda")
    yd_all = torch.empty(sum(ysz), dtype=torch.float16, device="cuda")
    xd = [v.view(t["x"].shape) for v, t in zip(torch.split(xd_all, xsz), sets[0])]
    yd = [v.view(t["y"].shape) for v, t in zip(torch.split(yd_all, ysz), sets[0])]
    h2d, d2h = hx_all.numel() * 2, hy_all.numel() * 2
    sp = stream.cuda_stream

    def e2e_step(r):
        with torch.cuda.stream(stream):
            xd_all.copy_(hx_all, non_blocking=True)
            for t, xv, yv in zip(sets[r], xd, yd):
                t["layer"](xv, out=yv, stream=sp)
            hy_all.copy_(yd_all, non_blocking=True)
        stream.synchronize()

    def loop(fn):
        for i in range(max(args.warmup, 3)):
            fn(i % R)
        barrier(world)
        w0 = time.time()
        n, t0 = 0, time.perf_counter()
        e0 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        while True:
            for _ in range(args.steps):
                fn(n % R)
                n += 1
            if time.perf_counter() - t0 >= MIN_TIMED_S:
                break
        e1 = torch.cuda.Event(enable_timing=True)
        e1.record(stream)
        e1.synchronize()
        wins.append((w0, time.time()))
        return n, reduce_max(e0.elapsed_time(e1) / 1e3, world)

    wins = []
    n_e, el_e = loop(e2e_step)
    graphs = []
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    for r in range(R):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=cap):
            xd_all.copy_(hx_all, non_blocking=True)
            for t, xv, yv in zip(sets[r], xd, yd):
                t["layer"](xv, out=yv, stream=cap.cuda_stream)
            hy_all.copy_(yd_all, non_blocking=True)
        graphs.append(gr)
    stream.wait_stream(cap)

    def graph_step(r):
        with torch.cuda.stream(stream):
            graphs[r].replay()
        stream.synchronize()

    n_g, el_g = loop(graph_step)
    nbytes = reg["nbytes"]
    return ({"value": world * nbytes * n_e / el_e / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
             "d2h_bytes_per_step": d2h, "steps": n_e, "timed_s": el_e, "win": wins[0]},
            {"value": world * nbytes * n_g / el_g / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
             "d2h_bytes_per_step": d2h, "steps": n_g, "timed_s": el_g, "win": wins[1],
             "note": "input copy, three calls, output copy per step, replayed from CUDA graphs; "
                     "a synchronize per step"})


def run_ours(args, rank, world, local):
    import torch
    from w4a16_weight_only_gb300 import build as _build
    _build.build()
    import w4a16_weight_only_gb300 as awq

    torch.cuda.set_device(local)
    if not awq.runtime_available():
        raise RuntimeError("awq runtime unavailable: " + awq.last_error())
    stream = torch.cuda.Stream()
    clocks = ClockSampler(local)
    time.sleep(0.3)
    hbm, hbm_kind = peaks()

    # headline: 70B decode
    reg = _decode_region(LINEARS, args, world, torch, awq, stream, clocks)
    t_max = reduce_max(reg["t_step"], world)
    nbytes = reg["nbytes"]
    value = world * nbytes / t_max / 1e9
    achieved = nbytes / reg["t_step"] / 1e9
    e2e, e2e_graph = _e2e(reg, args, world, torch, stream)
    del reg["sets"]
    torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "M": 1, "group_size": 128, "bias": True,
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {reg['R']} rotating weight sets, "
                         f"{reg['R'] * reg['per_set'] / 1e6:.0f} MB > 3 x 129 MB",
                   "bytes_per_step": nbytes, "launch": "CUDA graph replays of AwqLinear calls",
                   "timing": f"{reg['reps']} repetitions of {args.steps} steps "
                             f"({reg['timed_s']:.3f} s timed); median repetition"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "peak_source": hbm_kind + " (hbm_gbs, STREAM copy)",
                     "kernel": "decode_tma_kernel (awq_gemm decode path)",
                     "traffic": measured_traffic(),
                     "traffic_unit": "bytes per launch (mean of the three linears)",
                     "algorithmic_bytes_per_launch": nbytes / len(LINEARS)},
        "e2e": e2e,
        "e2e_graph": e2e_graph,
        "gpu_launches": reg["launches"],
    }
    windows = {"": reg["win"], "e2e": e2e.pop("win"), "e2e_graph": e2e_graph.pop("win")}
    if not args.decode_only:
        r7 = _decode_region(LINEARS_7B, args, world, torch, awq, stream, clocks)
        del r7["sets"]
        torch.cuda.empty_cache()
        t7 = reduce_max(r7["t_step"], world)
        line["decode_7b"] = {
            "workload": WORKLOAD_7B, "value": world * r7["nbytes"] / t7 / 1e9, "unit": UNIT,
            "ms_per_step": t7 * 1e3, "bytes_per_step": r7["nbytes"],
            "roofline": {"bound": "hbm", "achieved": r7["nbytes"] / r7["t_step"] / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": r7["nbytes"] / r7["t_step"] / 1e9 / hbm,
                         "peak_source": hbm_kind},
            "timing": f"{r7['reps']} repetitions of {args.steps} steps ({r7['timed_s']:.3f} s); "
                      f"{r7['R']} rotating weight sets; CUDA graph replays",
            "gpu_launches": r7["launches"]}
        windows["decode_7b"] = r7["win"]
        line["prefill"] = _prefill_block(PREFILL, WORKLOAD_PREFILL, args, world, torch, awq, stream,
                                         windows, "prefill")
        line["prefill_7b"] = _prefill_block(PREFILL_7B, WORKLOAD_PREFILL_7B, args, world, torch, awq,
                                            stream, windows, "prefill_7b")
    # clock samples of every timed region (the sampler ran throughout)
    for key, (w0, w1) in windows.items():
        clk = clocks.window(w0, w1)
        if key == "":
            line["clocks"] = clk
        elif "." in key:
            a, b = key.split(".")
            line[a][b]["clocks"] = clk
        else:
            line[key]["clocks"] = clk
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    return line if rank == 0 else None


def run_case(args, local):
    """Profiling driver: one workload linear, --steps eager awq_gemm calls after --warmup
    calls, nothing else on the GPU (for ncu launch lists and captures)."""
    import torch
    from w4a16_weight_only_gb300 import build as _build
    _build.build()
    import w4a16_weight_only_gb300 as awq
    torch.cuda.set_device(local)
    import re
    m8 = re.fullmatch(r"w8_m(\d+)_(\d+)x(\d+)", args.case)
    if m8:  # 8-bit codes: w8_m<M>_<K>x<N>, G = 128, bias
        M, K, N = (int(v) for v in m8.groups())
        d = synth.awq8_linear(5000 + M + K + N, M, K, N, group_size=128, bias=True)
        gemm = awq.awq_gemm_w8
    else:
        d = synth.workload_inputs(args.case)
        gemm = awq.awq_gemm
    t = {k: torch.from_numpy(d[k]).cuda() for k in ("x", "qweight", "qzeros", "scales")}
    b = torch.from_numpy(d["bias"]).cuda() if d["bias"] is not None else None
    y = torch.empty((d["M"], d["N"]), dtype=torch.float16, device="cuda")
    if args.packed:  # the tile-packed layout: one repack, then the calls AwqLinear(packed=True) makes
        pk = awq.awq_repack(t["qweight"], t["qzeros"], t["scales"], d["group_size"])
        for i in range(args.warmup + args.steps):
            awq.awq_gemm_packed(t["x"], pk, b, d["K"], d["N"], d["group_size"], out=y, workspace="auto")
    else:
        for i in range(args.warmup + args.steps):
            gemm(t["x"], t["qweight"], t["qzeros"], t["scales"], b, group_size=d["group_size"],
                 out=y, path=args.path)
    torch.cuda.synchronize()
    awq.device_status()
    print(json.dumps({"case": args.case, "path": "packed" if args.packed else args.path,
                      "launches": args.warmup + args.steps}))


def run_sweep(args, local):
    """Per-workload table (one JSON line per synth.WORKLOADS entry): small-M shapes as HBM
    GB/s over CUDA-graph replays of rotating weight copies (together > 3x L2), large-M
    shapes as TFLOP/s over back-to-back launches, beside cuBLAS fp16 on the dense weight
    and awq_dequant + cuBLAS for the large ones.  Not the bench contract line."""
    import torch
    from w4a16_weight_only_gb300 import build as _build
    _build.build()
    import w4a16_weight_only_gb300 as awq
    torch.cuda.set_device(local)
    hbm, hbm_kind = peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tflops = float(json.load(f)["bf16_tflops"])
        tf_kind = "measured bf16 burst (fp16 nominal rate equal)"
    except Exception:
        tflops, tf_kind = 1900.0, "fallback"
    names = [(w[2], "f16") for w in synth.WORKLOADS]
    # bf16 activations / scales on the decode bench linears, a small batch, prefill, 70B
    names += [(n, "bf16") for n in ("7b_decode_m1_4096x4096_bias", "7b_decode_m1_4096x11008_bias",
                                    "7b_decode_m1_11008x4096_bias", "7b_smallbatch_m16_4096x11008",
                                    "7b_prefill_m2048_4096x11008", "70b_m1_8192x28672")]
    if args.case:
        names = [(n, dt) for (n, dt) in names if args.case in (n if dt == "f16" else n + "_bf16")]
    stream = torch.cuda.Stream()

    def timed(fn, reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(reps):
                fn()
            b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / reps * 1e3  # us

    for name, dt in names:
        d = synth.workload_inputs(name, dt)
        M, K, N, G = d["M"], d["K"], d["N"], d["group_size"]
        tdt = torch.bfloat16 if dt == "bf16" else torch.float16
        x = torch.from_numpy(d["x"]).to(tdt).cuda()
        qw = torch.from_numpy(d["qweight"]).cuda()
        qz = torch.from_numpy(d["qzeros"]).cuda()
        sc = torch.from_numpy(d["scales"]).to(tdt).cuda()
        bias = torch.from_numpy(d["bias"]).to(tdt).cuda() if d["bias"] is not None else None
        y = torch.empty((M, N), dtype=tdt, device="cuda")
        if dt == "bf16":
            name = name + "_bf16"
        nbytes = algorithmic_bytes(M, K, N, G, bias is not None)
        flop = 2.0 * M * N * K
        line = {"workload": name, "dtype": dt, "M": M, "K": K, "N": N, "group_size": G,
                "bias": bias is not None,
                "path": awq.select_path(x, qw, qz, sc, bias, G, y)}
        if M <= 32:
            # graph replays of back-to-back calls on rotating weight copies, twice: with
            # AWQ_GEMM_STATIC_WEIGHTS (prepared layers, as the bench's AwqLinear calls; the
            # headline figure) and in the default stream order (weights read after the wait)
            R = max(2, min(16, int(3 * L2_BYTES // nbytes) + 1))
            sets = [(qw.clone(), qz.clone(), sc.clone()) for _ in range(R)]
            calls = max(R, (240 // R) * R)

            def replayed(static):
                torch.cuda.synchronize()
                with torch.cuda.stream(stream):
                    for i in range(3 * R):
                        w = sets[i % R]
                        awq.awq_gemm(x, w[0], w[1], w[2], bias, group_size=G, out=y, stream=stream,
                                     static_weights=static)
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        for i in range(calls):
                            w = sets[i % R]
                            awq.awq_gemm(x, w[0], w[1], w[2], bias, group_size=G, out=y, stream=stream,
                                         static_weights=static)
                times = sorted(timed(g.replay, 1) / calls for _ in range(5))
                del g
                return times[2]

            t = replayed(True)
            t_def = replayed(False)
            line.update({"us": t, "GB_s": nbytes / t / 1e3, "frac_hbm": nbytes / t / 1e3 / hbm,
                         "mode": "static weights (prepared layers)",
                         "default_order_us": t_def, "default_order_GB_s": nbytes / t_def / 1e3,
                         "weight_copies": R, "launches_per_graph": calls})
            if K % 64 == 0 and (G == -1 or G % 64 == 0):
                # the tile-packed copies (what AwqLinear(packed=True) calls), replayed the same
                # way; GB/s of the same algorithmic bytes, so the times compare directly
                pks = [awq.awq_repack(w[0], w[1], w[2], G, stream=stream) for w in sets]
                torch.cuda.synchronize()
                with torch.cuda.stream(stream):
                    for i in range(3 * R):
                        awq.awq_gemm_packed(x, pks[i % R], bias, K, N, G, out=y, stream=stream)
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        for i in range(calls):
                            awq.awq_gemm_packed(x, pks[i % R], bias, K, N, G, out=y, stream=stream)
                t_p = sorted(timed(g.replay, 1) / calls for _ in range(5))[2]
                del g, pks
                line.update({"packed_us": t_p, "packed_GB_s": nbytes / t_p / 1e3,
                             "packed_frac_hbm": nbytes / t_p / 1e3 / hbm})
            del sets
        else:
            fn = lambda: awq.awq_gemm(x, qw, qz, sc, bias, group_size=G, out=y, stream=stream)
            timed(fn, 3)
            t = timed(fn, 10)
            wd = awq.awq_dequant(qw, qz, sc, group_size=G)
            torch.cuda.synchronize()
            mm = lambda: torch.matmul(x, wd, out=y)
            timed(mm, 3)
            t_mm = timed(mm, 10)
            dq = lambda: awq.awq_dequant(qw, qz, sc, group_size=G, out=wd, stream=stream)
            timed(dq, 3)
            t_dq = timed(dq, 10)
            line.update({"us": t, "TFLOP_s": flop / t / 1e6, "frac_tensor": flop / t / 1e6 / tflops,
                         "cublas_fp16_dense_us": t_mm, "cublas_fp16_dense_TFLOP_s": flop / t_mm / 1e6,
                         "dequant_plus_cublas_us": t_dq + t_mm})
            del wd
            if K % 64 == 0 and (G == -1 or G % 64 == 0):
                # the tile-packed layout: the one-off repack, then awq_gemm_packed with the
                # stream's workspace (stream-K where the plan takes it)
                pk = awq.awq_repack(qw, qz, sc, G, stream=stream)
                rp = lambda: awq.awq_repack(qw, qz, sc, G, out=pk, stream=stream)
                timed(rp, 2)
                t_rp = timed(rp, 5)
                ws = torch.zeros((awq.awq_gemm_packed_workspace_size(),), dtype=torch.uint8, device="cuda")
                fp = lambda: awq.awq_gemm_packed(x, pk, bias, K, N, G, out=y, stream=stream, workspace=ws)
                timed(fp, 3)
                t_p = timed(fp, 10)
                line.update({"packed_us": t_p, "packed_TFLOP_s": flop / t_p / 1e6,
                             "packed_frac_tensor": flop / t_p / 1e6 / tflops, "repack_us": t_rp})
                del pk, ws
        awq.device_status()
        line.update({"hbm_peak_GB_s": hbm, "hbm_peak": hbm_kind, "tensor_peak_TFLOP_s": tflops,
                     "tensor_peak": tf_kind})
        print(json.dumps(line), flush=True)
        del x, qw, qz, sc, bias, y
        torch.cuda.empty_cache()
    if not args.case or "quantize" in args.case:
        run_quantize_sweep(awq, timed, hbm, hbm_kind)
    if not args.case or "moe" in args.case:
        run_grouped_sweep(awq, timed, hbm, hbm_kind)
    if not args.case or "w8" in args.case:
        run_w8_sweep(awq, timed, hbm, hbm_kind)


def w8_bytes(M, K, N, G, bias):
    """Bytes an 8-bit linear must move: one byte per code and per zero, fp16 scales, x, y, bias."""
    ng = K // G
    return K * N + ng * N + 2 * ng * N + 2 * M * K + 2 * M * N + (2 * N if bias else 0)


def run_w8_sweep(awq, timed, hbm, hbm_kind):
    """awq_gemm_w8 (8-bit codes) on the 7B decode linears, a 16-row batch and a 70B MLP
    linear: HBM GB/s over CUDA-graph replays of rotating weight copies (together > 3x L2),
    for the automatic path, for the plain generic kernel, and for awq_gemm_packed on the
    8-bit tile-packed copies."""
    import torch
    stream = torch.cuda.Stream()
    for (M, K, N) in ((1, 4096, 4096), (1, 4096, 11008), (1, 11008, 4096), (16, 4096, 11008),
                      (1, 8192, 28672)):
        G = 128
        d = synth.awq8_linear(5000 + M + K + N, M, K, N, group_size=G, bias=True)
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        x, bias = dev(d["x"]), dev(d["bias"])
        w = (dev(d["qweight"]), dev(d["qzeros"]), dev(d["scales"]))
        nbytes = w8_bytes(M, K, N, G, True)
        R = max(2, min(16, int(3 * L2_BYTES // nbytes) + 1))
        sets = [w] + [tuple(t.clone() for t in w) for _ in range(R - 1)]
        y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        line = {"workload": f"w8_m{M}_{K}x{N}", "bits": 8, "M": M, "K": K, "N": N, "group_size": G,
                "bias": True, "weight_copies": R, "hbm_peak_GB_s": hbm, "hbm_peak": hbm_kind}
        for path in ("auto", "generic"):
            calls = max(R, ((240 if path == "auto" else 40) // R) * R)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                for i in range(2 * R):
                    s = sets[i % R]
                    awq.awq_gemm_w8(x, s[0], s[1], s[2], bias, G, out=y, path=path, stream=stream)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(calls):
                        s = sets[i % R]
                        awq.awq_gemm_w8(x, s[0], s[1], s[2], bias, G, out=y, path=path, stream=stream)
            t = sorted(timed(g.replay, 1) / calls for _ in range(5))[2]
            awq.device_status()
            key = "" if path == "auto" else "generic_"
            line.update({key + "us": t, key + "GB_s": nbytes / t / 1e3,
                         key + "frac_hbm": nbytes / t / 1e3 / hbm})
            del g
        # the 8-bit tile-packed copies (the small-batch kernel), replayed the same way
        pks = [awq.awq_repack(s[0], s[1], s[2], G, stream=stream, bits=8) for s in sets]
        calls = max(R, (240 // R) * R)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for i in range(2 * R):
                awq.awq_gemm_packed(x, pks[i % R], bias, K, N, G, out=y, stream=stream, bits=8)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(calls):
                    awq.awq_gemm_packed(x, pks[i % R], bias, K, N, G, out=y, stream=stream, bits=8)
        t = sorted(timed(g.replay, 1) / calls for _ in range(5))[2]
        awq.device_status()
        line.update({"packed_us": t, "packed_GB_s": nbytes / t / 1e3, "packed_frac_hbm": nbytes / t / 1e3 / hbm})
        del g, pks
        print(json.dumps(line), flush=True)
        del sets, w, x, y
        torch.cuda.empty_cache()
    # large M: TFLOP/s of back-to-back launches, beside dequant + cuBLAS fp16
    tflops = 1900.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tflops = float(json.load(f)["bf16_tflops"])
    except Exception:
        pass
    for (M, K, N) in ((512, 4096, 11008), (2048, 4096, 11008), (2048, 11008, 4096), (4096, 8192, 28672)):
        G = 128
        d = synth.awq8_linear(5100 + M + K + N, M, K, N, group_size=G, bias=True)
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        x, bias = dev(d["x"]), dev(d["bias"])
        qw, qz, sc = dev(d["qweight"]), dev(d["qzeros"]), dev(d["scales"])
        y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        flop = 2.0 * M * N * K
        # eager launches on the current stream (the one `timed` records its events on)
        fn = lambda: awq.awq_gemm_w8(x, qw, qz, sc, bias, G, out=y)
        timed(fn, 3)
        t = timed(fn, 10)
        wd = awq.awq_dequant_w8(qw, qz, sc, G)
        torch.cuda.synchronize()
        mm = lambda: torch.matmul(x, wd, out=y)
        timed(mm, 3)
        t_mm = timed(mm, 10)
        dq = lambda: awq.awq_dequant_w8(qw, qz, sc, G)
        timed(dq, 3)
        t_dq = timed(dq, 10)
        # the 8-bit tile-packed layout: one-off repack, then awq_gemm_packed_w8 with a workspace
        pk = awq.awq_repack(qw, qz, sc, G, bits=8)
        rp = lambda: awq.awq_repack(qw, qz, sc, G, out=pk, bits=8)
        timed(rp, 2)
        t_rp = timed(rp, 5)
        ws = torch.zeros((awq.awq_gemm_packed_workspace_size(),), dtype=torch.uint8, device="cuda")
        fp = lambda: awq.awq_gemm_packed(x, pk, bias, K, N, G, out=y, workspace=ws, bits=8)
        timed(fp, 3)
        t_p = timed(fp, 10)
        awq.device_status()
        print(json.dumps({"workload": f"w8_m{M}_{K}x{N}", "bits": 8, "M": M, "K": K, "N": N,
                          "group_size": G, "bias": True, "us": t, "TFLOP_s": flop / t / 1e6,
                          "frac_tensor": flop / t / 1e6 / tflops, "cublas_fp16_dense_us": t_mm,
                          "dequant_plus_cublas_us": t_dq + t_mm, "packed_us": t_p,
                          "packed_TFLOP_s": flop / t_p / 1e6, "packed_frac_tensor": flop / t_p / 1e6 / tflops,
                          "repack_us": t_rp, "tensor_peak_TFLOP_s": tflops}),
              flush=True)
        del x, qw, qz, sc, y, wd, pk, ws
        torch.cuda.empty_cache()


def run_grouped_sweep(awq, timed, hbm, hbm_kind):
    """awq_gemm_grouped on a mixture-of-experts layer shaped like the 7B MLP with E = 8
    experts and top-2 routing (synthetic): HBM GB/s of the bytes the launch must move (the
    experts that received rows, their metadata, x, y) over CUDA-graph replays of rotating
    copies of the stacked weights (together > 3x L2)."""
    import torch
    stream = torch.cuda.Stream()
    for (K, N) in ((4096, 14336), (14336, 4096)):
        for T in (1, 16):
            E, topk, G = 8, 2, 128
            d = synth.moe_inputs(4000 + T + K, T, topk, E, K, N, group_size=G)
            active = int((np.diff(d["offsets"]) > 0).sum())
            R = d["R"]
            nbytes = active * (K * N // 2 + (K // G) * N // 2 + 2 * (K // G) * N) + 2 * R * K + 2 * R * N
            dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
            x, offs = dev(d["x"]), dev(d["offsets"])
            w = (dev(d["qweight"]), dev(d["qzeros"]), dev(d["scales"]))
            copies = max(2, int(3 * L2_BYTES // (active * K * N // 2)) + 1)
            sets = [w] + [tuple(t.clone() for t in w) for _ in range(copies - 1)]
            y = torch.empty((R, N), dtype=torch.float16, device="cuda")
            calls = max(copies, (60 // copies) * copies)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                for i in range(2 * copies):
                    s = sets[i % copies]
                    awq.awq_gemm_grouped(x, s[0], s[1], s[2], offs, None, G, out=y, stream=stream)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(calls):
                        s = sets[i % copies]
                        awq.awq_gemm_grouped(x, s[0], s[1], s[2], offs, None, G, out=y, stream=stream)
            t = sorted(timed(g.replay, 1) / calls for _ in range(5))[2]
            awq.device_status()
            print(json.dumps({"workload": f"moe_e{E}_top{topk}_t{T}_{K}x{N}", "E": E, "topk": topk,
                              "tokens": T, "rows": R, "active_experts": active, "K": K, "N": N,
                              "group_size": G, "us": t, "GB_s": nbytes / t / 1e3,
                              "frac_hbm": nbytes / t / 1e3 / hbm, "weight_copies": copies,
                              "launches_per_graph": calls, "hbm_peak_GB_s": hbm,
                              "hbm_peak": hbm_kind}), flush=True)
            del sets, g, w, x, y
            torch.cuda.empty_cache()
    # prefill-sized routed batches (T = 4096 tokens, top-2 of 8 experts): TFLOP/s of the routed
    # rows, the grouped decode kernel beside the grouped tile-packed kernel (one-off repack of
    # the experts timed separately)
    tflops = 1900.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tflops = float(json.load(f)["bf16_tflops"])
    except Exception:
        pass
    for (K, N) in ((4096, 14336), (14336, 4096)):
        E, topk, G, T = 8, 2, 128, 4096
        d = synth.moe_inputs(4100 + K, T, topk, E, K, N, group_size=G)
        R = d["R"]
        flop = 2.0 * R * K * N
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        x, offs = dev(d["x"]), dev(d["offsets"])
        qw, qz, sc = dev(d["qweight"]), dev(d["qzeros"]), dev(d["scales"])
        y = torch.empty((R, N), dtype=torch.float16, device="cuda")
        # launches on the current stream: the one `timed` makes current and records on
        fd = lambda: awq.awq_gemm_grouped(x, qw, qz, sc, offs, None, G, out=y)
        timed(fd, 1)
        t_dec = timed(fd, 3)
        pk = awq.awq_repack_experts(qw, qz, sc, G)
        t_rp = timed(lambda: awq.awq_repack_experts(qw, qz, sc, G), 2)
        fp = lambda: awq.awq_gemm_packed_grouped(x, pk, offs, K, N, None, G, out=y)
        timed(fp, 3)
        t_p = timed(fp, 10)
        # the same experts and rows in bf16 (scales and x cast on the device, experts repacked)
        xb, yb = x.to(torch.bfloat16), torch.empty((R, N), dtype=torch.bfloat16, device="cuda")
        pkb = awq.awq_repack_experts(qw, qz, sc.to(torch.bfloat16), G)
        fb = lambda: awq.awq_gemm_packed_grouped(xb, pkb, offs, K, N, None, G, out=yb)
        timed(fb, 3)
        t_b = timed(fb, 10)
        awq.device_status()
        print(json.dumps({"workload": f"moe_prefill_e{E}_top{topk}_t{T}_{K}x{N}", "E": E, "topk": topk,
                          "tokens": T, "rows": R, "K": K, "N": N, "group_size": G,
                          "grouped_decode_us": t_dec, "grouped_decode_TFLOP_s": flop / t_dec / 1e6,
                          "packed_us": t_p, "packed_TFLOP_s": flop / t_p / 1e6,
                          "packed_frac_tensor": flop / t_p / 1e6 / tflops, "repack_experts_us": t_rp,
                          "packed_bf16_us": t_b, "packed_bf16_TFLOP_s": flop / t_b / 1e6,
                          "tensor_peak_TFLOP_s": tflops}), flush=True)
        del x, qw, qz, sc, y, pk, xb, yb, pkb
        torch.cuda.empty_cache()


def quantize_bytes(N, K, G):
    """Bytes awq_quantize_rtn must move: the fp16 weight once, the packed outputs once."""
    ng = K // G
    return 2 * N * K + N * K // 2 + ng * N // 2 + 2 * ng * N


def run_quantize_sweep(awq, timed, hbm, hbm_kind):
    """awq_quantize_rtn on the 7B linears' fp16 weights [N, K], G = 128, both modes: HBM
    GB/s over CUDA-graph replays of calls on rotating weight copies (together > 3x L2)."""
    import torch
    stream = torch.cuda.Stream()
    for (N, K) in ((4096, 4096), (11008, 4096), (4096, 11008)):
        G = 128
        nbytes = quantize_bytes(N, K, G)
        R = max(2, int(3 * L2_BYTES // (2 * N * K)) + 1)
        gen = torch.Generator(device="cuda").manual_seed(N + K)
        ws = [(torch.randn((N, K), generator=gen, device="cuda") * 0.02).half() for _ in range(R)]
        outs = [(torch.empty((K, N // 8), dtype=torch.int32, device="cuda"),
                 torch.empty((K // G, N // 8), dtype=torch.int32, device="cuda"),
                 torch.empty((K // G, N), dtype=torch.float16, device="cuda")) for _ in range(R)]
        calls = max(R, (60 // R) * R)
        for sym in (False, True):
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                for i in range(2 * R):
                    awq.awq_quantize_rtn(ws[i % R], G, sym, out=outs[i % R], stream=stream)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(calls):
                        awq.awq_quantize_rtn(ws[i % R], G, sym, out=outs[i % R], stream=stream)
            t = sorted(timed(g.replay, 1) / calls for _ in range(5))[2]
            awq.device_status()
            print(json.dumps({"workload": f"quantize_rtn_{'sym' if sym else 'asym'}_{N}x{K}_g{G}",
                              "N": N, "K": K, "group_size": G, "sym": sym, "us": t,
                              "GB_s": nbytes / t / 1e3, "frac_hbm": nbytes / t / 1e3 / hbm,
                              "weight_copies": R, "launches_per_graph": calls,
                              "hbm_peak_GB_s": hbm, "hbm_peak": hbm_kind}), flush=True)
            del g
        del ws, outs
        torch.cuda.empty_cache()


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def run_cpu_oracle(args):
    """CPU oracle table (no GPU): the C oracle's dequant and fp64 linear on every workload
    shape (synth.WORKLOADS; --configs selects), timed in full, one JSON line per shape.
    Threads: OpenMP's default (all host cores) unless OMP_NUM_THREADS says otherwise; the
    dequant is single-threaded by construction."""
    from oracle import c_oracle
    c_oracle.build()
    cfgs = {int(c) for c in args.configs.split(",")} if args.configs else None
    threads = int(os.environ.get("OMP_NUM_THREADS", "0")) or os.cpu_count()
    model = cpu_model()
    for (cfg, idx, name, M, K, N, G, bias) in synth.WORKLOADS:
        if cfgs is not None and cfg not in cfgs:
            continue
        d = synth.workload_inputs(name)
        args_ = (d["qweight"], d["qzeros"], d["scales"], G)
        t0 = time.perf_counter()
        c_oracle.dequant_f32(*args_)
        t_dq = time.perf_counter() - t0
        t0 = time.perf_counter()
        c_oracle.gemm(d["x"], d["qweight"], d["qzeros"], d["scales"], d["bias"], G)
        t_gemm = time.perf_counter() - t0
        print(json.dumps({"workload": name, "config": cfg, "M": M, "K": K, "N": N, "group_size": G,
                          "kind": "C oracle", "dequant_s": t_dq,
                          "linear_s": t_gemm, "linear_includes_dequant": True,
                          "GB_s": step_bytes([d]) / t_gemm / 1e9,
                          "GFLOP_s": 2.0 * M * N * K / t_gemm / 1e9,
                          "threads": threads, "cores": os.cpu_count(), "cpu": model}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-only", action="store_true",
                    help="headline decode step (and its end-to-end runs) only, no extra blocks")
    ap.add_argument("--case", default=None,
                    help="profiling mode: run only this workload linear (see synth.WORKLOADS, or "
                         "w8_m<M>_<K>x<N> for 8-bit codes)")
    ap.add_argument("--path", default="auto", choices=["auto", "decode", "prefill", "generic"])
    ap.add_argument("--packed", action="store_true",
                    help="profiling mode: repack once, then call awq_gemm_packed with the stream's workspace")
    ap.add_argument("--sweep", action="store_true",
                    help="per-workload table (one JSON line per workload), not the bench line")
    ap.add_argument("--cpu-oracle", action="store_true",
                    help="time the C oracle (dequant, fp64 linear) on every workload shape; no GPU")
    ap.add_argument("--configs", default=None, help="--cpu-oracle: comma-separated config indices")
    args = ap.parse_args(argv)
    if args.cpu_oracle:
        run_cpu_oracle(args)
        return
    rank, world, local = dist_setup(args)
    if args.sweep:
        run_sweep(args, local)
        return
    if args.case:
        run_case(args, local)
        return
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
