#!/usr/bin/env python3
"""NVFP4 block-scaled GEMM benchmark: device-timed TFLOP/s and roofline fraction.

One step = one pass of the hot path over one batch of synthetic input:
``nvfp4_gemm_run_grouped`` on inputs already resident in HBM with scales already
repacked (the repack is a once-per-weight preparation, timed separately in
``step_with_repack``).

Every workload of the problem statement is timed in one run (``per_config``):
the 128x128x256 single tile, the skinny-M 128x7168x16384 problem, the dense
8192^3 problem, the two-group and the eight-group MoE problems.  The headline
``value``, ``roofline``, ``e2e`` and ``cpu_baseline`` belong to the largest
one, the compute-bound 8192^3 problem (``--workload`` picks another).

Timing: W untimed warm-up steps, then exactly K steps replayed from CUDA graphs
right after one untimed warm replay, timed with CUDA events on the launching
stream with a device synchronisation on both sides; the steps cycle through R
independent input sets whose total size is more than three times the L2 cache,
so no step finds its operands in L2.  ``e2e`` is the same metric through the C
ABI with host buffers: every step copies the step's inputs from pinned host
memory, repacks both scale tensors, runs the GEMM and copies C back, all inside
the timed region (two device buffer sets, so one step's host-to-device copies
overlap the previous step's work).

``--impl reference`` times the CPU oracle (the only reference this method has)
on a bounded sample of the same workload.

One GPU only: the library's kernels load shared tiles with cluster multicast,
which stays within one GPU's memory, and nothing here shards.  Launched with
more than one rank or ``--gpus`` > 1, rank 0 prints an ``unavailable`` line and
every rank exits without touching a GPU.
"""
import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from block_scaled_fp4_nvfp4_gb300 import workloads  # noqa: E402

METRIC = "NVFP4 (grouped) GEMM TFLOPS, device-timed, and % of FP4-tensor/HBM roofline"
HEADLINE_WORKLOAD = "dense_8192x8192x8192"
FP4_OVER_BF16 = 13.5 / 2.25   # nominal dense ratio, used to scale the measured bf16 peak
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["gemm_kernel.cu", "gemm_params.h", "ptx.cuh", "descriptors.h", "schedule.h"]


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE_WORKLOAD, choices=list(workloads.WORKLOADS))
    ap.add_argument("--configs", default="all",
                    help="comma-separated workloads timed in per_config ('all', or 'none')")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target oracle sample time")
    ap.add_argument("--check", action="store_true", help="oracle check of set 0 (sampled)")
    ap.add_argument("--no-quantize", action="store_true", help="skip the fused quantize + repack leg")
    ap.add_argument("--no-repack-step", action="store_true", help="skip the step_with_repack leg")
    ap.add_argument("--clock-window-s", type=float, default=1.0,
                    help="seconds of untimed back-to-back steps after each timed region, sampled for the "
                         "clock record (0: sample the timed region only)")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, "block_scaled_fp4_nvfp4_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel sources changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def roofline_terms(wl, peaks):
    """(bound, t_hbm, t_fp4, hbm GB/s, fp4 TFLOP/s) of a workload."""
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    fp4 = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])) * FP4_OVER_BF16
    t_hbm = wl.bytes / (hbm * 1e9)
    t_fp4 = wl.flops / (fp4 * 1e12)
    return ("hbm" if t_hbm >= t_fp4 else "tensor"), t_hbm, t_fp4, hbm, fp4


class ClockSampler:
    """nvidia-smi clocks / throttle reasons every 100 ms, started before the
    timed regions; each region takes the samples that fall inside it, else the
    nearest ones (a region shorter than the sampling period)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.rows = []
        self.path = os.path.join("/tmp", "nvfp4_clocks_%d_%d.csv" % (os.getpid(), index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                self.rows.append((ts, float(parts[2]), float(parts[3]), parts[4], parts[5:]))
            except (ValueError, IndexError):
                continue
        os.unlink(self.path)

    def window(self, t0, t1, margin=0.05, label="timed"):
        """Samples taken within [t0 - margin, t1 + margin] (a negative margin
        trims the ends)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        inside = [r for r in self.rows if t0 - margin <= r[0] <= t1 + margin]
        window = label
        if not inside:
            inside = sorted(self.rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:3]
            window = "adjacent (timed region %.4f s, shorter than the 0.1 s sampling period)" % (t1 - t0)
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        reasons = set()
        for r in inside:
            for n, fl in zip(self.NAMES, r[4][1:5]):
                if fl.lower().startswith("active"):
                    reasons.add(n)

        def watts(s):
            try:
                return float(s)
            except ValueError:
                return 0.0
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": max(r[2] for r in inside),
                "power_w_max": max(watts(r[3]) for r in inside), "reasons": sorted(reasons),
                "samples": len(inside), "window": window}


def one_gpu_only(args):
    """True (after printing the line on rank 0) when asked for more than one GPU."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus <= 1 and world <= 1:
        return False
    if int(os.environ.get("RANK", "0")) == 0:
        print(json.dumps({"impl": args.impl, "metric": METRIC, "n_gpus": max(args.gpus, world),
                          "unavailable": "one GPU only: the GEMM runs on a single GB300 and nothing "
                                         "shards; no multi-GPU path is built"}), flush=True)
    return True


# ------------------------------------------------------------------ CPU oracle timing
def _oracle_columns(p, ncols, threads):
    import oracle
    t0 = time.perf_counter()
    oracle.gemm(p["A"], p["B"][:, :ncols].contiguous(), p["SFA"], p["SFB"][:, :ncols].contiguous(),
                p["M"], ncols, p["K"], 1, nthreads=threads)
    return time.perf_counter() - t0


def _oracle_sample(wl, seed=0):
    import oracle
    probs = workloads.make_inputs(wl, seed=seed)
    p = max(probs, key=lambda q: q["M"] * q["N"] * q["K"])
    p = dict(p, A=p["A"][:1], B=p["B"][:1], SFA=p["SFA"][:1], SFB=p["SFB"][:1])
    return p, oracle.max_threads()


def time_oracle(wl, target_s, seed=0):
    """Time the oracle (as it stands) on whole output columns of the workload's
    largest group, growing the sample until it takes about target_s.  Returns
    (TFLOP/s, seconds, threads, description)."""
    p, threads = _oracle_sample(wl, seed)
    M, N, K = p["M"], p["N"], p["K"]
    ncols = 1
    while True:
        dt = _oracle_columns(p, ncols, threads)
        if dt >= target_s * 0.5 or ncols >= N:
            break
        ncols = min(N, max(ncols * 2, int(ncols * target_s / max(dt, 1e-3) * 0.9)))
    desc = "oracle on %d of %d output columns of the %dx%dx%d problem (all %d rows), %d threads" % (
        ncols, N, M, N, K, M, threads)
    return 2.0 * M * ncols * K / dt / 1e12, dt, threads, desc


def run_reference(args):
    """The reference arm: the CPU oracle timed on the host cores, each step a
    bounded sample (whole output columns) sized so the run ends in minutes."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    wl = workloads.WORKLOADS[args.workload]
    p, threads = _oracle_sample(args.workload)
    M, N, K = p["M"], p["N"], p["K"]
    t1 = _oracle_columns(p, 1, threads)
    t2 = _oracle_columns(p, 2, threads)
    per_col = max(t2 - t1, t1 / 2, 1e-6)
    budget = 120.0 / max(1, args.steps + args.warmup)
    ncols = int(max(1, min(N, budget / per_col)))
    secs = []
    for i in range(args.warmup + args.steps):
        dt = _oracle_columns(p, ncols, threads)
        if i >= args.warmup:
            secs.append(dt)
    step_s = float(np.mean(secs)) if secs else float("nan")
    value = 2.0 * M * ncols * K / step_s / 1e12
    desc = "oracle on %d of %d output columns of the %dx%dx%d problem (all %d rows) per step, %d threads" % (
        ncols, N, M, N, K, M, threads)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "shapes_MNKL": wl.shapes, "seed": 0},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU timing
def size_matched_copy(nbytes, dev, stream, l2, iters=200):
    """HBM rate of the copy that defines the measured peak (torch copy_,
    read + write bytes) at the size of one launch: a buffer of nbytes/2
    copied per launch, rotating over sets that together exceed L2.  A single
    launch of tens of MB spends a visible part of its time ramping up and
    draining, so this is the practical ceiling for a launch of that size."""
    half = max(16, (nbytes // 2) // 16 * 16)
    nsets = max(2, math.ceil(3 * l2 / (2 * half)) + 1)
    src = [torch.full((half,), 1, dtype=torch.uint8, device=dev) for _ in range(nsets)]
    dst = [torch.empty((half,), dtype=torch.uint8, device=dev) for _ in range(nsets)]
    with torch.cuda.stream(stream):
        for i in range(nsets):
            dst[i].copy_(src[i])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(iters):
            dst[i % nsets].copy_(src[i % nsets])
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / iters * 1e3
    del src, dst
    return {"bytes_per_launch": 2 * half, "us": us, "achieved": 2 * half / (us * 1e-6) / 1e9, "unit": "GB/s",
            "how": "torch copy_ of %.1f MB (read + write), %d buffer pairs rotating, CUDA events" % (
                half / 1e6, nsets)}


def device_inputs(binding, wl, sets, dev):
    """R seeded input sets of a workload on the device, scales repacked."""
    host0 = None
    dev_sets = []
    for r in range(sets):
        probs = workloads.make_inputs(wl, seed=r)
        if r == 0:
            host0 = probs
        d = []
        for p in probs:
            M, N, K, L = p["M"], p["N"], p["K"], p["L"]
            q = dict(M=M, N=N, K=K, L=L)
            q["A"] = p["A"].to(dev)
            q["B"] = p["B"].to(dev)
            q["SFA"] = binding.repack_scales(p["SFA"].to(dev), M, K, L)
            q["SFB"] = binding.repack_scales(p["SFB"].to(dev), N, K, L)
            q["C"] = torch.empty((L, M, N), dtype=torch.float16, device=dev)
            d.append(q)
        dev_sets.append(d)
    torch.cuda.synchronize()
    return host0, dev_sets


def launch_grouped(binding, d, stream):
    binding.nvfp4_gemm_run_grouped(
        len(d), [q["A"] for q in d], [q["B"] for q in d], [q["SFA"] for q in d], [q["SFB"] for q in d],
        [q["C"] for q in d], [q["M"] for q in d], [q["N"] for q in d], [q["K"] for q in d],
        [q["L"] for q in d], stream)


def time_launches(binding, dev_sets, steps, warmup, stream, flush=None):
    """W eager warm-up launches (they also size the library's per-stream
    split-K workspace before capture), then K launches replayed from CUDA graphs
    (one graph per pass over the R input sets, one for the remainder), right
    after one untimed warm replay.  With `flush` (a buffer larger than L2, for
    workloads too small to rotate through L2) every step first overwrites the
    buffer and only the launch itself, between two events, is timed.  Returns
    (elapsed ms of the K steps, wall-clock start, end)."""
    sets = len(dev_sets)
    with torch.cuda.stream(stream):
        for i in range(max(warmup, sets)):
            launch_grouped(binding, dev_sets[i % sets], stream)
    torch.cuda.synchronize()
    binding.nvfp4_gemm_check_device_status(stream)
    if flush is not None:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        t_wall0 = time.time()
        with torch.cuda.stream(stream):
            for i in range(steps):
                flush.fill_(i & 0xFF)
                ev[i][0].record(stream)
                launch_grouped(binding, dev_sets[i % sets], stream)
                ev[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall1 = time.time()
        binding.nvfp4_gemm_check_device_status(stream)
        return sum(a.elapsed_time(b) for a, b in ev), t_wall0, t_wall1
    full, rem = divmod(steps, sets)
    graphs = []
    for count, reps in ((sets, full), (rem, 1)):
        if count == 0 or reps == 0:
            continue
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(count):
                launch_grouped(binding, dev_sets[i % sets], stream)
        graphs.append((g, reps))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for g, _ in graphs:          # warm replay, directly followed by the timed one
            g.replay()
        t_wall0 = time.time()
        e0.record(stream)
        for g, reps in graphs:
            for _ in range(reps):
                g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    binding.nvfp4_gemm_check_device_status(stream)
    del graphs
    return e0.elapsed_time(e1), t_wall0, t_wall1


def check_sampled(host0, dev_set):
    import oracle
    out = []
    for gi, p in enumerate(host0):
        C = dev_set[gi]["C"]
        rng = np.random.default_rng(gi)
        n = 2000
        ls, ms, ns = rng.integers(0, p["L"], n), rng.integers(0, p["M"], n), rng.integers(0, p["N"], n)
        ref, absacc = oracle.gemm_points(p["A"], p["B"], p["SFA"], p["SFB"], p["M"], p["N"], p["K"],
                                         ls, ms, ns, L=p["L"])
        g = C[torch.as_tensor(ls), torch.as_tensor(ms), torch.as_tensor(ns)].cpu().numpy()
        ok, worst, _ = oracle.compare(g, ref, absacc)
        out.append({"group": gi, "ok": ok, "worst_ratio": worst})
    return out


def measure_workload(binding, name, args, dev, stream, l2, peaks, peak_src):
    """Device-timed K steps of one workload with its roofline."""
    wl = workloads.WORKLOADS[name]
    sets = max(2, math.ceil(3 * l2 / wl.bytes) + 1)
    flush = None
    if sets > 16:
        # too small to rotate through L2: overwrite a 2 x L2 buffer before every step
        sets = 2
        flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
        l2_note = "L2 flushed before every step (%.0f MB written), each launch timed alone" % (2 * l2 / 1e6)
    else:
        l2_note = "rotating %d input sets, %.0f MB > 3 x L2 (%.0f MB)" % (sets, sets * wl.bytes / 1e6, l2 / 1e6)
    host0, dev_sets = device_inputs(binding, wl, sets, dev)
    elapsed_ms, tw0, tw1 = time_launches(binding, dev_sets, args.steps, args.warmup, stream, flush)
    launch = binding.nvfp4_gemm_last_launch()
    # The timed region is mostly far shorter than nvidia-smi's 100 ms sampling
    # period, so its samples can miss the load.  For the clock record the same
    # steps then run back to back, untimed, for about --clock-window-s seconds
    # while the sampler keeps running.
    # Chunks of about a quarter second of device time (K steps where every
    # step also flushes L2), until the window's wall time is reached.
    load_wall = None
    if args.clock_window_s > 0:
        per_step = max(elapsed_ms / args.steps * 1e-3, 1e-6)
        chunk = args.steps if flush is not None else int(min(100000, max(args.steps, math.ceil(0.25 / per_step))))
        n = 0
        lw0 = time.time()
        while True:
            time_launches(binding, dev_sets, chunk, 0, stream, flush)
            n += chunk
            if time.time() - lw0 >= args.clock_window_s:
                break
        load_wall = (lw0, time.time(), n)
    launch_s = elapsed_ms / args.steps * 1e-3
    bound, t_hbm, t_fp4, hbm, fp4 = roofline_terms(wl, peaks)
    if bound == "hbm":
        achieved, peak, unit = wl.bytes / launch_s / 1e9, hbm, "GB/s"
    else:
        achieved, peak, unit = wl.flops / launch_s / 1e12, fp4, "TFLOP/s"
    # a same-size copy is only meaningful where the inputs rotate through more
    # than L2 (not for the launch-latency-bound single tile)
    copy_ref = size_matched_copy(wl.bytes, dev, stream, l2) if bound == "hbm" and flush is None else None
    res = {
        "workload": wl.name, "shapes_MNKL": wl.shapes, "steps": args.steps, "warmup": args.warmup,
        "us_per_launch": launch_s * 1e6, "tflops": wl.flops / launch_s / 1e12,
        "l2": l2_note,
        "launch": launch,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": ncu_traffic(wl.name),
                     "peak_source": "%s (%s)" % (peak_src, "hbm_gbs" if bound == "hbm" else
                                                 "bf16_tflops x 6 nominal fp4/bf16"),
                     "algorithmic_bytes_per_launch": wl.bytes, "flops_per_launch": wl.flops,
                     "avg_launch_us": launch_s * 1e6,
                     "size_matched_copy": copy_ref,
                     "frac_of_size_matched_copy": None if copy_ref is None else achieved / copy_ref["achieved"]},
        "roofline_fraction_min_time": max(t_hbm, t_fp4) / launch_s,
        "_wall": (tw0, tw1),
        "_load_wall": load_wall,
    }
    del flush
    if args.check:
        res["check"] = check_sampled(host0, dev_sets[0])
    return res, host0, dev_sets


def repack_step(binding, host0, dev_sets, steps, dev, stream, wl):
    """Both scale repacks inside every step, then the GEMM (not the headline)."""
    sets = len(dev_sets)
    raw_sf = [(p["SFA"].to(dev), p["SFB"].to(dev)) for p in host0]
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(steps):
            d = dev_sets[i % sets]
            for gi, q in enumerate(d):
                binding.nvfp4_gemm_repack_scales(raw_sf[gi][0], q["SFA"], q["M"], q["K"], q["L"], stream)
                binding.nvfp4_gemm_repack_scales(raw_sf[gi][1], q["SFB"], q["N"], q["K"], q["L"], stream)
            launch_grouped(binding, d, stream)
        t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    return {"value": wl.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms, "steps": steps}


def quantize_leg(binding, dev, stream, hbm):
    """Fused quantize + repack (the step that produces B and SFB) on a bf16
    tensor shaped like the skinny workload's B (7168 x 16384); larger than L2."""
    qr, qk, ql = 7168, 16384, 1
    gq = torch.Generator(device=dev).manual_seed(0)
    xq = torch.randn((ql, qr, qk), device=dev, dtype=torch.float32, generator=gq).to(torch.bfloat16)
    qcodes = torch.empty((ql, qr, qk // 2), dtype=torch.uint8, device=dev)
    qsf = torch.empty(binding.nvfp4_gemm_repacked_scales_bytes(qr, qk, ql), dtype=torch.uint8, device=dev)
    for _ in range(3):
        binding.nvfp4_quantize(xq, binding.DTYPE_BF16, qcodes, qsf, qr, qk, ql, stream)
    torch.cuda.synchronize()
    iters = 20
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(iters):
            binding.nvfp4_quantize(xq, binding.DTYPE_BF16, qcodes, qsf, qr, qk, ql, stream)
        t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / iters
    nbytes = ql * qr * qk * 2 + ql * qr * qk // 2 + qsf.numel()
    ach = nbytes / (ms * 1e-3) / 1e9
    return {"shape_LxRxK": [ql, qr, qk], "input": "bf16", "us": ms * 1e3, "algorithmic_bytes": nbytes,
            "achieved": ach, "unit": "GB/s", "peak": hbm, "frac": ach / hbm}


def repack_leg(binding, dev, stream, l2, hbm, rows=7168, K=16384, iters=50):
    """The scale repack alone (a once-per-weight preparation, outside the
    timed step): row-major [rows, K/16] E4M3 scales -> the atom layout, for
    the skinny workload's B scales (7168 x 1024 bytes), rotating over buffer
    pairs larger than L2 together, against a copy of the same bytes."""
    cols = K // 16
    nbytes_in = rows * cols
    nbytes_out = binding.nvfp4_gemm_repacked_scales_bytes(rows, K, 1)
    per = nbytes_in + nbytes_out
    sets = max(2, math.ceil(3 * l2 / per) + 1)
    g = torch.Generator(device=dev).manual_seed(0)
    src = [torch.randint(0, 127, (rows, cols), dtype=torch.uint8, device=dev, generator=g) for _ in range(sets)]
    dst = [torch.empty(nbytes_out, dtype=torch.uint8, device=dev) for _ in range(sets)]
    with torch.cuda.stream(stream):
        for i in range(sets):
            binding.nvfp4_gemm_repack_scales(src[i], dst[i], rows, K, 1, stream)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(iters):
            binding.nvfp4_gemm_repack_scales(src[i % sets], dst[i % sets], rows, K, 1, stream)
        t1.record(stream)
    torch.cuda.synchronize()
    binding.nvfp4_gemm_check_device_status(stream)
    us = t0.elapsed_time(t1) / iters * 1e3
    ach = per / (us * 1e-6) / 1e9
    del src, dst
    copy = size_matched_copy(per, dev, stream, l2)
    return {"rows_x_scale_bytes": [rows, cols], "bytes_read": nbytes_in, "bytes_written": nbytes_out, "us": us,
            "achieved": ach, "unit": "GB/s", "peak": hbm, "frac": ach / hbm, "size_matched_copy": copy,
            "frac_of_size_matched_copy": ach / copy["achieved"],
            "l2": "rotating %d buffer pairs, %.0f MB > 3 x L2" % (sets, sets * per / 1e6)}


def e2e_leg(binding, host0, steps, dev, stream, flops):
    """The metric through the C ABI with host buffers: per step H2D of A, B
    and the row-major scales from pinned memory, two repacks, the GEMM, D2H of
    C, all inside the timed region."""
    hp = []
    h2d = d2h = 0
    for p in host0:
        e = {k: p[k].pin_memory() for k in ("A", "B", "SFA", "SFB")}
        e["Cout"] = [torch.empty((p["L"], p["M"], p["N"]), dtype=torch.float16).pin_memory() for _ in range(2)]
        h2d += sum(e[k].numel() * e[k].element_size() for k in ("A", "B", "SFA", "SFB"))
        d2h += e["Cout"][0].numel() * 2
        hp.append(e)

    def device_buffers():
        out = []
        for p in host0:
            M, N, K, L = p["M"], p["N"], p["K"], p["L"]
            out.append(dict(M=M, N=N, K=K, L=L, A=torch.empty_like(p["A"], device=dev),
                            B=torch.empty_like(p["B"], device=dev), SFAraw=torch.empty_like(p["SFA"], device=dev),
                            SFBraw=torch.empty_like(p["SFB"], device=dev),
                            SFA=torch.empty(binding.nvfp4_gemm_repacked_scales_bytes(M, K, L), dtype=torch.uint8,
                                            device=dev),
                            SFB=torch.empty(binding.nvfp4_gemm_repacked_scales_bytes(N, K, L), dtype=torch.uint8,
                                            device=dev),
                            C=torch.empty((L, M, N), dtype=torch.float16, device=dev)))
        return out

    # Two device buffer sets and three streams: step i+1's host-to-device
    # copies (copy stream) and step i's device-to-host readback (readback
    # stream) overlap step i+1's repacks and GEMM (compute stream); every step
    # still copies its own inputs in and its own result out inside the timed
    # region, and a set is refilled only after its previous result was read.
    ed_sets = [device_buffers(), device_buffers()]
    copy_stream = torch.cuda.Stream(device=dev)
    read_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    computed = [torch.cuda.Event(), torch.cuda.Event()]
    freed = [torch.cuda.Event(), torch.cuda.Event()]

    def step(i):
        j = i % 2
        ed = ed_sets[j]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(freed[j])  # the set's previous result has been read back
            for e, q in zip(hp, ed):
                q["A"].copy_(e["A"], non_blocking=True)
                q["B"].copy_(e["B"], non_blocking=True)
                q["SFAraw"].copy_(e["SFA"], non_blocking=True)
                q["SFBraw"].copy_(e["SFB"], non_blocking=True)
            copied[j].record(copy_stream)
        stream.wait_event(copied[j])
        with torch.cuda.stream(stream):
            for q in ed:
                binding.nvfp4_gemm_repack_scales(q["SFAraw"], q["SFA"], q["M"], q["K"], q["L"], stream)
                binding.nvfp4_gemm_repack_scales(q["SFBraw"], q["SFB"], q["N"], q["K"], q["L"], stream)
            launch_grouped(binding, ed, stream)
            computed[j].record(stream)
        read_stream.wait_event(computed[j])
        with torch.cuda.stream(read_stream):
            for e, q in zip(hp, ed):
                e["Cout"][j].copy_(q["C"], non_blocking=True)
            freed[j].record(read_stream)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)  # no copy of the timed steps starts before the clock does
    for i in range(steps):
        step(i)
    stream.wait_event(freed[(steps - 1) % 2])  # the clock stops once the last result is on the host
    if steps > 1:
        stream.wait_event(freed[(steps - 2) % 2])
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    binding.nvfp4_gemm_check_device_status(stream)
    return {"value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms, "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "includes": "H2D of A, B, row-major SFA/SFB; 2 repacks; GEMM; D2H of C; two buffer sets, "
                        "step i+1's copies in and step i's readback overlapping step i+1's work"}


# ------------------------------------------------------------------ our arm
def main(argv=None):
    args = parse(argv)
    if one_gpu_only(args):
        return
    if args.impl == "reference":
        return run_reference(args)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from block_scaled_fp4_nvfp4_gb300 import binding
    binding.load_library()
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024)
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(dev)

    if args.configs == "all":
        configs = list(workloads.WORKLOAD_ORDER)
    elif args.configs == "none":
        configs = []
    else:
        configs = [c for c in args.configs.split(",") if c]
    if args.workload not in configs:
        configs.append(args.workload)

    sampler = ClockSampler(0)
    sampler.start()
    per_config = {}
    head = head_inputs = None
    for name in configs:
        res, host0, dev_sets = measure_workload(binding, name, args, dev, stream, l2, peaks, peak_src)
        per_config[name] = res
        if name == args.workload:
            head, head_inputs = res, (host0, dev_sets)
        else:
            del dev_sets
        torch.cuda.empty_cache()
    wl = workloads.WORKLOADS[args.workload]

    extra = {}
    host0, dev_sets = head_inputs
    if not args.no_repack_step:
        extra["step_with_repack"] = repack_step(binding, host0, dev_sets, min(args.steps, 200), dev, stream, wl)
    del dev_sets
    torch.cuda.empty_cache()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    extra["quantize"] = None if args.no_quantize else quantize_leg(binding, dev, stream, hbm)
    extra["repack"] = None if args.no_repack_step else repack_leg(binding, dev, stream, l2, hbm)
    e2e = e2e_leg(binding, host0, args.e2e_steps, dev, stream, wl.flops)
    sampler.stop()

    cpu = None
    if not args.no_cpu_baseline:
        v, dt, threads, desc = time_oracle(args.workload, args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": desc + ", %.1f s" % dt}

    # clocks of each workload (the sampler ran across every timed region and
    # every back-to-back window): the back-to-back window's samples, the first
    # and last 50 ms left out, where there is one; the timed region's beside it
    for res in per_config.values():
        timed = sampler.window(*res.pop("_wall"))
        load = res.pop("_load_wall")
        if load is None:
            res["clocks"] = timed
            continue
        lw0, lw1, n = load
        clocks = sampler.window(lw0, lw1, margin=-0.05,
                                label="%d untimed back-to-back steps (%.2f s) right after the timed ones"
                                      % (n, lw1 - lw0))
        clocks["timed_region"] = timed
        res["clocks"] = clocks
    line = {
        "metric": METRIC, "value": head["tflops"], "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["us_per_launch"] / 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4", "data": "synthetic",
        "config": {"workload": wl.name, "shapes_MNKL": wl.shapes, "seed": 0, "l2": head["l2"],
                   "parallelism": "single GPU"},
        "roofline": head["roofline"],
        "roofline_fraction_min_time": head["roofline_fraction_min_time"],
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": head["clocks"],
        "per_config": {n: {k: v for k, v in r.items() if k not in ("workload",)} for n, r in per_config.items()},
    }
    line.update(extra)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
