#!/usr/bin/env python3
"""NVFP4 block-scaled GEMM benchmark: device-timed TFLOP/s and roofline fraction.

One step = one pass of the hot path over one batch of synthetic input:
``nvfp4_gemm_run_grouped`` on inputs already resident in HBM with scales already
repacked (the repack is a once-per-weight preparation, timed separately in
``step_with_repack``).  Default workload: the skinny-M problem
M=128 N=7168 K=16384 (HBM-bound on B).

Timing: W untimed warm-up steps, then exactly K steps between a barrier and a
device synchronisation on both sides, timed with CUDA events on the launching
stream; the step cycles through R independent input sets whose total size is
more than three times the L2 cache, so no step finds its operands in L2.
``e2e`` is the same metric through the C ABI with host buffers: every step
copies the step's inputs from pinned host memory, repacks both scale tensors,
runs the GEMM and copies C back, all inside the timed region (two device buffer
sets, so one step's host-to-device copies overlap the previous step's work).

``--impl reference`` times the CPU oracle (the only reference this method has)
on a bounded sample of the same workload.

Multi-GPU: launched under torchrun, every rank runs the same workload on its own
GPU (weak scaling; the problems are independent, there is no exchange), the
time is the max over ranks and ``value`` counts the work of all ranks.
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
DEFAULT_WORKLOAD = "skinny_128x7168x16384"
FP4_OVER_BF16 = 13.5 / 2.25   # nominal dense ratio, used to scale the measured bf16 peak
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["gemm_kernel.cu", "gemm_params.h", "ptx.cuh", "descriptors.h", "schedule.h"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(workloads.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target oracle sample time")
    ap.add_argument("--check", action="store_true", help="oracle check of set 0 (sampled)")
    ap.add_argument("--no-quantize", action="store_true", help="skip the fused quantize + repack leg")
    return ap.parse_args()


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


class ClockSampler:
    """nvidia-smi clocks / throttle reasons at 100 ms, for the timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
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

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[2]), float(parts[3]), parts[4], parts[5:]))
            except (ValueError, IndexError):
                continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        window = "timed"
        if not inside:
            # timed region shorter than the sampling period: nearest samples
            inside = sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:3]
            window = "adjacent (timed region %.3f s, shorter than the 0.1 s sampling period)" % (t1 - t0)
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            flags = r[4][1:5]
            for n, fl in zip(names, flags):
                if fl.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": max(r[2] for r in inside),
                "power_w_max": max(float(r[3]) if r[3].replace(".", "", 1).isdigit() else 0.0 for r in inside),
                "reasons": sorted(reasons), "samples": len(inside), "window": window}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    """Largest value over all ranks (the job takes as long as its slowest rank)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step, steps, elapsed_ms_max, world):
    """Whole-job TFLOP/s under weak scaling: every rank ran `steps` steps of
    the same workload; the job took the slowest rank's time."""
    return flops_per_step * steps * world / (elapsed_ms_max * 1e-3) / 1e12


# ------------------------------------------------------------------ CPU oracle timing
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


def _oracle_columns(p, ncols, threads):
    import oracle
    t0 = time.perf_counter()
    oracle.gemm(p["A"], p["B"][:, :ncols].contiguous(), p["SFA"], p["SFB"][:, :ncols].contiguous(),
                p["M"], ncols, p["K"], 1, nthreads=threads)
    return time.perf_counter() - t0


def _oracle_sample(wl, seed=0):
    import oracle
    probs = workloads.make_inputs(wl, seed=seed)
    p = max(probs, key=lambda q: q["N"] * q["K"])
    p = dict(p, A=p["A"][:1], B=p["B"][:1], SFA=p["SFA"][:1], SFB=p["SFB"][:1])
    return p, oracle.max_threads()


def time_oracle(wl, target_s, seed=0):
    """Time the oracle (as it stands) on whole output columns of the workload's
    largest group, growing the sample until it takes about target_s.  Returns
    (TFLOP/s, seconds, threads, description)."""
    p, threads = _oracle_sample(wl, seed)
    M, N, K = p["M"], p["N"], p["K"]
    ncols = 8
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
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = workloads.WORKLOADS[args.workload]
    p, threads = _oracle_sample(args.workload)
    M, N, K = p["M"], p["N"], p["K"]
    t1 = _oracle_columns(p, 1, threads)
    t8 = _oracle_columns(p, 8, threads)
    per_col = max((t8 - t1) / 7.0, 1e-6)
    budget = 120.0 / max(1, args.steps + args.warmup)
    ncols = int(max(1, min(N, (budget - t1) / per_col + 1)))
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
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "shapes_MNKL": wl.shapes, "seed": 0},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm
def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from block_scaled_fp4_nvfp4_gb300 import binding
    binding.load_library()

    wl = workloads.WORKLOADS[args.workload]
    G = len(wl.shapes)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024)
    sets = max(2, math.ceil(3 * l2 / wl.bytes) + 1)

    # ---- inputs: R independent seeded sets, resident in HBM, scales repacked
    host_sets = []
    dev_sets = []
    for r in range(sets):
        probs = workloads.make_inputs(wl, seed=r)
        if r == 0:
            host_sets.append(probs)
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

    def launch(d, stream=None):
        binding.nvfp4_gemm_run_grouped(
            G, [q["A"] for q in d], [q["B"] for q in d], [q["SFA"] for q in d], [q["SFB"] for q in d],
            [q["C"] for q in d], [q["M"] for q in d], [q["N"] for q in d], [q["K"] for q in d],
            [q["L"] for q in d], stream)

    # All launches go to one dedicated stream: the warm-up sizes the library's
    # per-stream split-K workspace before the timed steps are captured.
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, sets)):
            launch(dev_sets[i % sets])
    torch.cuda.synchronize()
    binding.nvfp4_gemm_check_device_status()

    if args.check and rank == 0:
        import oracle
        for gi, p in enumerate(host_sets[0]):
            C = dev_sets[0][gi]["C"]
            rng = np.random.default_rng(gi)
            n = 2000
            ls, ms, ns = rng.integers(0, p["L"], n), rng.integers(0, p["M"], n), rng.integers(0, p["N"], n)
            ref, absacc = oracle.gemm_points(p["A"], p["B"], p["SFA"], p["SFB"], p["M"], p["N"], p["K"],
                                             ls, ms, ns, L=p["L"])
            g = C[torch.as_tensor(ls), torch.as_tensor(ms), torch.as_tensor(ns)].cpu().numpy()
            ok, worst, _ = oracle.compare(g, ref, absacc)
            print("check group %d: ok=%s worst=%.3g" % (gi, ok, worst), file=sys.stderr)

    # ---- the K timed steps are replayed from CUDA graphs (one graph holds one
    # pass over the R input sets, a second one the remainder), so the host's
    # launch rate does not limit the device.
    full, rem = divmod(args.steps, sets)
    graphs = []
    for count, reps in ((sets, full), (rem, 1)):
        if count == 0 or reps == 0:
            continue
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(count):
                launch(dev_sets[i % sets])
        graphs.append((g, reps))
    torch.cuda.synchronize()
    for g, _ in graphs:          # one untimed replay of each graph
        g.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    start_all = torch.cuda.Event(enable_timing=True)
    end_all = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        start_all.record(stream)
        for g, reps in graphs:
            for _ in range(reps):
                g.replay()
        end_all.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(world)
    time.sleep(0.15)
    clocks = sampler.stop(t_wall0, t_wall1)
    binding.nvfp4_gemm_check_device_status(stream)
    elapsed_ms = max_over_ranks(start_all.elapsed_time(end_all), world)
    # back-to-back launches: the average launch duration includes the short
    # gaps between graph nodes, so it slightly understates the kernel's rate
    launch_ms = elapsed_ms / args.steps

    # ---- repack inside the step (for reference, not the headline)
    rp_steps = min(args.steps, 2000)
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    raw_sf = []
    for p in host_sets[0]:
        raw_sf.append((p["SFA"].to(dev), p["SFB"].to(dev)))
    torch.cuda.synchronize()
    torch.cuda.set_stream(stream)
    t0e.record(stream)
    for i in range(rp_steps):
        d = dev_sets[i % sets]
        for gi, q in enumerate(d):
            binding.nvfp4_gemm_repack_scales(raw_sf[gi][0], q["SFA"], q["M"], q["K"], q["L"])
            binding.nvfp4_gemm_repack_scales(raw_sf[gi][1], q["SFB"], q["N"], q["K"], q["L"])
        launch(d)
    t1e.record(stream)
    torch.cuda.synchronize()
    rp_ms = t0e.elapsed_time(t1e) / rp_steps

    # ---- fused quantize + repack (the step that produces B and SFB) on a
    # bf16 tensor shaped like group 0's B; larger than L2, so it streams HBM
    quant = None
    if not args.no_quantize:
        q0 = host_sets[0][0]
        qr, qk, ql = q0["N"], q0["K"], q0["L"]
        gq = torch.Generator(device=dev).manual_seed(0)
        xq = torch.randn((ql, qr, qk), device=dev, dtype=torch.float32, generator=gq).to(torch.bfloat16)
        qcodes = torch.empty((ql, qr, qk // 2), dtype=torch.uint8, device=dev)
        qsf = torch.empty(binding.nvfp4_gemm_repacked_scales_bytes(qr, qk, ql), dtype=torch.uint8, device=dev)
        for _ in range(3):
            binding.nvfp4_quantize(xq, binding.DTYPE_BF16, qcodes, qsf, qr, qk, ql, stream)
        torch.cuda.synchronize()
        q_iters = 20
        t0q, t1q = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0q.record(stream)
        for _ in range(q_iters):
            binding.nvfp4_quantize(xq, binding.DTYPE_BF16, qcodes, qsf, qr, qk, ql, stream)
        t1q.record(stream)
        torch.cuda.synchronize()
        q_ms = t0q.elapsed_time(t1q) / q_iters
        q_bytes = ql * qr * qk * 2 + ql * qr * qk // 2 + qsf.numel()
        quant = {"shape_LxRxK": [ql, qr, qk], "input": "bf16", "us": q_ms * 1e3,
                 "algorithmic_bytes": q_bytes, "achieved": q_bytes / (q_ms * 1e-3) / 1e9, "unit": "GB/s"}
        del xq, qcodes, qsf

    # ---- e2e: host buffers through the C ABI
    hp = []
    h2d = 0
    d2h = 0
    for p in host_sets[0]:
        e = {k: p[k].pin_memory() for k in ("A", "B", "SFA", "SFB")}
        e["Cout"] = torch.empty((p["L"], p["M"], p["N"]), dtype=torch.float16).pin_memory()
        h2d += sum(e[k].numel() * e[k].element_size() for k in ("A", "B", "SFA", "SFB"))
        d2h += e["Cout"].numel() * 2
        hp.append(e)

    def device_buffers():
        out = []
        for p in host_sets[0]:
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

    # Two device buffer sets: the host->device copies of step i+1 (on their own
    # stream) overlap the repacks, GEMM and readback of step i; every step still
    # copies its own inputs and reads back its own result inside the timed region.
    ed_sets = [device_buffers(), device_buffers()]
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    freed = [torch.cuda.Event(), torch.cuda.Event()]

    def e2e_step(i):
        ed = ed_sets[i % 2]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(freed[i % 2])  # the set's previous step is done with it
            for e, q in zip(hp, ed):
                q["A"].copy_(e["A"], non_blocking=True)
                q["B"].copy_(e["B"], non_blocking=True)
                q["SFAraw"].copy_(e["SFA"], non_blocking=True)
                q["SFBraw"].copy_(e["SFB"], non_blocking=True)
            copied[i % 2].record(copy_stream)
        stream.wait_event(copied[i % 2])
        with torch.cuda.stream(stream):
            for q in ed:
                binding.nvfp4_gemm_repack_scales(q["SFAraw"], q["SFA"], q["M"], q["K"], q["L"])
                binding.nvfp4_gemm_repack_scales(q["SFBraw"], q["SFB"], q["N"], q["K"], q["L"])
            launch(ed, stream)
            for e, q in zip(hp, ed):
                e["Cout"].copy_(q["C"], non_blocking=True)
            freed[i % 2].record(stream)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    copy_stream.wait_event(e0)  # no copy of the timed steps starts before the clock does
    for i in range(args.e2e_steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, world)
    binding.nvfp4_gemm_check_device_status()

    # ---- numbers
    flops = wl.flops
    ms_per_step = elapsed_ms / args.steps
    value = job_throughput(flops, args.steps, elapsed_ms, world)
    peaks, peak_src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    fp4_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])) * FP4_OVER_BF16
    t_hbm = wl.bytes / (hbm * 1e9)
    t_fp4 = flops / (fp4_peak * 1e12)
    bound = "hbm" if t_hbm >= t_fp4 else "tensor"
    launch_s = launch_ms * 1e-3
    if bound == "hbm":
        achieved, peak, unit = wl.bytes / launch_s / 1e9, hbm, "GB/s"
    else:
        achieved, peak, unit = flops / launch_s / 1e12, fp4_peak, "TFLOP/s"

    copy_ref = size_matched_copy(wl.bytes, dev, stream, l2) if bound == "hbm" else None

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, dt, threads, desc = time_oracle(args.workload, args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": desc + ", %.1f s" % dt}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4", "data": "synthetic",
            "config": {"workload": wl.name, "shapes_MNKL": wl.shapes, "seed": 0,
                       "l2": "rotating %d input sets, %.0f MB > 3 x L2 (%.0f MB)" % (
                           sets, sets * wl.bytes / 1e6, l2 / 1e6),
                       "parallelism": "replica per GPU" if world > 1 else "single GPU"},
            "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                         "frac": achieved / peak, "traffic": ncu_traffic(wl.name),
                         "peak_source": "%s (%s)" % (peak_src, "hbm_gbs" if bound == "hbm" else
                                                     "bf16_tflops x 6 nominal fp4/bf16"),
                         "algorithmic_bytes_per_launch": wl.bytes, "flops_per_launch": flops,
                         "avg_launch_us": launch_ms * 1e3,
                         "size_matched_copy": copy_ref,
                         "frac_of_size_matched_copy": None if copy_ref is None else achieved / copy_ref["achieved"]},
            "roofline_fraction_min_time": max(t_hbm, t_fp4) / launch_s,
            "cpu_baseline": cpu,
            "e2e": {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "ms_per_step": e2e_ms, "steps": args.e2e_steps, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "includes": "H2D of A, B, row-major SFA/SFB; 2 repacks; GEMM; D2H of C; two buffer "
                                "sets, step i+1's copies overlapping step i"},
            "step_with_repack": {"value": flops / (rp_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                                 "ms_per_step": rp_ms},
            "quantize": None if quant is None else dict(quant, peak=hbm, frac=quant["achieved"] / hbm),
            "gpu_launches": args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
