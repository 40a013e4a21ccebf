#!/usr/bin/env python
"""Throughput of y = FP16(x . W^T) + b on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

A step is one call of poot_linear_f16 on one batch of seeded synthetic
inputs already resident in HBM.  The default workload is the MLP
up-projection (M=8192, N=14336, K=4096), the largest configured shape; its
x + W + y (416 MB) exceed the 129 MB L2, so no flush is needed between
steps.  Under torchrun (N > 1) every rank runs an independent replica on
its own GPU (weak scaling, no data-path collective); the step time is the
maximum over ranks.

Reported beside the device-timed value:
  roofline      the GEMM kernel's achieved TFLOP/s (algorithmic 2MNK per
                launch / mean CUDA-event duration on its stream) against the
                measured dense bf16 peak (the fp16 tensor rate is the same);
                traffic = DRAM bytes per launch from the committed ncu
                summary when it matches the current kernel source, else null
  e2e           same metric through the C ABI with host buffers: every step
                copies its x, W, b host->device (pinned) and its y back,
                inside the timed region; consecutive steps overlap on three
                streams (upload / compute / download)
  cpu_baseline  the CPU oracle timed on a bounded row sample on the host
                cores (a reported baseline, not the target)
  clocks        nvidia-smi samples taken during the timed region
``--impl reference`` times the CPU oracle alone on the same workload.
"""
from __future__ import annotations

import argparse
import csv
import datetime as _dt
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024
METRIC = "TFLOP/s of y=FP16(x·Wᵀ)+b per M×N×K; % of FP16 tensor peak / HBM BW"
CPU_SAMPLE_SECONDS = 10.0


# Widened-contraction forms for --contract: (head dtype, out_f32, bias, steps);
# a step is an activation name or (op, "r") for an [M,N] operand drawn N(0,1).
CONTRACT_FORMS = {
    "bf16": ("bf16", False, True, []),
    "f32out": ("f16", True, True, []),
    "nobias": ("f16", False, False, []),
    "silu": ("f16", False, True, ["silu"]),
    "gelu_tanh": ("f16", False, True, ["gelu_tanh"]),
    "gelu_erf": ("f16", False, True, ["gelu_erf"]),
    "residual": ("f16", False, True, [("add", "r")]),
    "swiglu": ("f16", False, True, ["silu", ("mul", "r")]),
    "bf16_swiglu": ("bf16", False, True, ["silu", ("mul", "r")]),
}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--workload", default="mlp_up")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    p.add_argument("--cpu-seconds", type=float, default=CPU_SAMPLE_SECONDS)
    p.add_argument("--variant", default="auto", help="force a kernel variant (auto, gemm_tma, gemv, ...)")
    p.add_argument("--tile-n", type=int, default=0, help="GEMM output tile width (0 = automatic)")
    p.add_argument("--group-m", type=int, default=0, help="GEMM tile-order group (0 = automatic)")
    p.add_argument("--no-graph", action="store_true", help="launch the timed steps eagerly")
    p.add_argument("--k-chunk", type=int, default=0, help="GEMM TMEM chunk along K (0 = automatic)")
    p.add_argument("--contract", default="", choices=[""] + sorted(CONTRACT_FORMS),
                   help="time a widened-contraction form (poot_contract) instead of the plain linear")
    p.add_argument("--groups", type=int, default=1,
                   help="with --contract: G groups of M/G rows, each with its own W (poot_contract_grouped)")
    a = p.parse_args()
    if a.warmup < 3:
        p.error("--warmup must be >= 3")
    if a.steps < 1:
        p.error("--steps must be >= 1")
    return a


# ---- distributed plumbing (replicas only) ------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, use_cuda):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group("nccl" if use_cuda else "gloo")
    return dist


def max_over_ranks(dist, value, device):
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---- peaks, clocks, profiles ----------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi samples (SM clock, reasons) with host timestamps."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 f"-lms={period_ms}"], stdout=self.fh, stderr=subprocess.DEVNULL)
            deadline = time.time() + 5.0
            while time.time() < deadline and os.path.getsize(self.path) == 0:
                time.sleep(0.02)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self, t0: float, t1: float):
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as fh:
            for r in csv.reader(fh):
                if len(r) < 10:
                    continue
                try:
                    ts = _dt.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(r[2]), float(r[3]), r[4].strip(), [s.strip() for s in r[5:10]]))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 <= r[0] <= t1]
        used = inside if inside else sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:3]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in used for i in range(4) if r[4][i + 1].lower() == "active"})
        power = []
        for r in used:
            try:
                power.append(float(r[3]))
            except ValueError:
                pass
        return {"sm_mhz": statistics.median(r[1] for r in used), "sm_max_mhz": max(r[2] for r in used),
                "sm_min_mhz": min(r[1] for r in used), "reasons": reasons,
                "power_w_median": statistics.median(power) if power else None,
                "power_w_max": max(power) if power else None,
                "samples": len(used), "samples_in_timed_region": len(inside)}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_fp16_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as fh:
                h.update(name.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from profiles/traffic.json if it matches the source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            entries = json.load(fh)
    except (OSError, ValueError):
        return None
    src = kernel_source_hash()
    for e in entries:
        if e.get("kernel") == kernel and e.get("workload") == workload and e.get("source_hash") == src:
            return e.get("dram_bytes_per_launch")
    return None


# ---- CPU oracle sample ----------------------------------------------------------
def cpu_oracle_sample(x, w, b, seconds: float, y_gpu=None):
    """Time the oracle on a row sample sized to about `seconds` of work."""
    import numpy as np
    import oracle
    M, K = x.shape
    N = w.shape[0]
    threads = oracle.default_threads()
    xb = x.view(torch_int16()).numpy().view(np.uint16)
    wb = w.view(torch_int16()).numpy().view(np.uint16)
    bb = b.view(torch_int16()).numpy().view(np.uint16)
    # calibrate on one row per thread
    rows = min(M, threads)
    t = time.perf_counter()
    oracle.linear_f16(xb[:rows], wb, bb, nthreads=threads)
    per_row = (time.perf_counter() - t) / rows
    want = int(max(threads, min(M, seconds / max(per_row, 1e-9))))
    want = min(M, want)
    rng = np.random.default_rng(2024)
    sample = np.sort(rng.choice(M, size=want, replace=False))
    t = time.perf_counter()
    y_ref = oracle.linear_f16(np.ascontiguousarray(xb[sample]), wb, bb, nthreads=threads)
    dt = time.perf_counter() - t
    flops = 2.0 * want * N * K
    out = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
           "sample": f"{want} of {M} rows (seeded), all {N} columns, K={K}; {dt:.2f} s on {threads} threads",
           "seconds": round(dt, 3)}
    if y_gpu is not None:
        g = y_gpu[sample]
        same = (g == y_ref)
        out["sample_rows_identical_bits"] = float(same.mean())
    return out, y_ref, sample


def torch_int16():
    import torch
    return torch.int16


# ---- arms -----------------------------------------------------------------------
def run_reference(args, rank, world):
    import torch
    from linear_fp16_gb300 import synth
    if rank != 0:
        return 0
    wl = synth.WORKLOADS[args.workload]
    x, w, b = synth.workload_inputs(args.workload)
    # each step: a bounded row sample of the workload, sized so that the
    # whole run stays within a few minutes
    per_step = max(0.2, min(3.0, 120.0 / (args.steps + args.warmup)))
    vals = []
    last = None
    for i in range(args.warmup + args.steps):
        res, _, _ = cpu_oracle_sample(x, w, b, per_step)
        if i >= args.warmup:
            vals.append(res["value"])
            last = res
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        # a whole step's time at the sampled rate (each step times a row sample)
        "ms_per_step": 2.0 * wl.M * wl.N * wl.K / (value * 1e12) * 1e3 if value > 0 else None,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": wl.name, "M": wl.M, "N": wl.N, "K": wl.K, "dist": wl.dist,
                   "seed": wl.seed, "accumulate": "f32", "sample": "rows",
                   "ms_per_step": "extrapolated from the row sample's rate to the whole workload"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": last["cores"], "kind": "oracle",
                         "sample": last["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, rank, world, local):
    import numpy as np
    import torch
    import linear_fp16_gb300 as L
    from linear_fp16_gb300 import synth

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the CUDA path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(world, True)
    lib = L.load_library()

    wl = synth.WORKLOADS[args.workload]
    M, N, K = wl.M, wl.N, wl.K
    x_h, w_h, b_h = synth.workload_inputs(args.workload, seed_offset=0)
    x = x_h.to(dev)
    w = w_h.to(dev)
    b = b_h.to(dev)
    y = torch.empty((M, N), dtype=torch.float16, device=dev)
    variant = L.VARIANT_AUTO
    if args.variant != "auto":
        variant = {v: k for k, v in L.VARIANT_NAMES.items()}[args.variant]
    chosen = L.variant_for(x, w, b, y) if variant == L.VARIANT_AUTO else variant
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    # Inputs larger than L2 between steps: when one set of x, W, b, y is
    # smaller than 3x L2, rotate through enough copies (same values) that a
    # step never finds its operands in L2 from an earlier step.
    working_set = 2 * (M * K + N * K + N + M * N)
    copies = 1
    if working_set < 3 * L2_BYTES:
        copies = min(64, -(-3 * L2_BYTES // working_set))
    sets = [(x, w, b, y)]
    for _ in range(copies - 1):
        sets.append((x.clone(), w.clone(), b.clone(), torch.empty_like(y)))
    ptr_sets = [(a.data_ptr(), bb.data_ptr(), c.data_ptr(), d.data_ptr()) for (a, bb, c, d) in sets]
    opts = L.options(variant, 0, args.tile_n, args.group_m, args.k_chunk)
    opts_ref = __import__("ctypes").byref(opts)

    def step(i, stream_handle):
        rc = lib.poot_linear_f16_ex(*ptr_sets[i % copies], M, N, K, opts_ref, stream_handle)
        if rc != 0:
            raise RuntimeError(f"poot_linear_f16: {L.poot_linear_status_string(rc)}")

    for i in range(args.warmup):
        step(i, sh)
    torch.cuda.synchronize()
    if L.poot_linear_device_status(sh) != 0:
        raise RuntimeError("device-side wait timed out during warm-up")

    # The K timed steps are captured once into a CUDA graph and replayed, so
    # a short kernel is not timed together with the host's launch overhead.
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cap = torch.cuda.current_stream().cuda_stream
            for i in range(args.steps):
                step(args.warmup + i, cap)
        graph.replay()  # one untimed replay: the graph's own first-launch cost
        torch.cuda.synchronize()

    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local) if rank == 0 else None
    barrier(dist)
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            step(args.warmup + i, sh)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    wall1 = time.time()
    clocks = None
    if sampler is not None:
        sampler.stop()
        clocks = sampler.summary(wall0, wall1)
    total_ms = t_start.elapsed_time(t_end)
    step_ms = max_over_ranks(dist, total_ms / args.steps, dev)
    # one kernel per step (two for GEMM_PACKED: the row copy, then the
    # GEMM): the mean duration of the step's kernels is the step time on the
    # launching stream (graph replay keeps launches back to back)
    kern_ms = step_ms
    launches_per_step = 2 if chosen == L.VARIANT_GEMM_PACKED else 1
    if L.poot_linear_device_status(sh) != 0:
        raise RuntimeError("device-side wait timed out during the timed region")
    y = sets[(args.warmup + args.steps - 1) % copies][3]

    # Per-launch distribution, after (and apart from) the timed region: each
    # call launched eagerly between its own pair of events on the launching
    # stream, rotating the input sets as the timed steps do (so it includes
    # the host's launch latency that the graph-timed value leaves out).
    reps = 200 if M <= L.GEMV_MAX_M else 50
    ev_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for r, (e0, e1) in enumerate(ev_pairs):
        e0.record(stream)
        step(args.warmup + args.steps + r, sh)
        e1.record(stream)
    torch.cuda.synchronize()
    per_launch = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in ev_pairs)
    per_launch_us = {"reps": reps, "median": per_launch[reps // 2], "p10": per_launch[reps // 10],
                     "p90": per_launch[(9 * reps) // 10],
                     "how": "eager launches, each between its own CUDA events (launch latency included)"}

    flops = 2.0 * M * N * K
    value = world * flops / (step_ms * 1e-3) / 1e12

    # ---- end to end through the C ABI with host buffers --------------------
    # Every step uploads its x, W and b from pinned host memory, runs
    # poot_linear_f16 and downloads its y.  Steps are independent, so the
    # upload of step i+1 and the download of step i-1 run on their own
    # streams while step i computes (two device buffer sets).
    e2e = None
    if not args.no_e2e:
        xp, wp, bp = x_h.pin_memory(), w_h.pin_memory(), b_h.pin_memory()
        yps = [torch.empty((M, N), dtype=torch.float16).pin_memory() for _ in range(2)]
        dsets = [(torch.empty_like(x), torch.empty_like(w), torch.empty_like(b), torch.empty_like(y))
                 for _ in range(2)]
        s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        in_done, cmp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

        def e2e_step(i):
            k = i % 2
            xd, wd, bd, yd = dsets[k]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(cmp_done[k])      # set k no longer read
                xd.copy_(xp, non_blocking=True)
                wd.copy_(wp, non_blocking=True)
                bd.copy_(bp, non_blocking=True)
                in_done[k].record(s_in)
            s_cmp.wait_event(in_done[k])
            if i >= 2:
                s_cmp.wait_event(out_done[k])         # y of set k downloaded
            rc = lib.poot_linear_f16(xd.data_ptr(), wd.data_ptr(), bd.data_ptr(), yd.data_ptr(), M, N, K,
                                     s_cmp.cuda_stream)
            if rc != 0:
                raise RuntimeError("poot_linear_f16 failed in e2e")
            cmp_done[k].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(cmp_done[k])
                yps[k].copy_(yd, non_blocking=True)
                out_done[k].record(s_out)

        e2e_steps = max(4, min(args.steps, 50))
        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier(dist)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(s_in)
        s_cmp.wait_event(a0)
        s_out.wait_event(a0)
        for i in range(e2e_steps):
            e2e_step(i)
        s_out.wait_stream(s_in)
        s_out.wait_stream(s_cmp)
        a1.record(s_out)
        torch.cuda.synchronize()
        barrier(dist)
        e2e_ms = max_over_ranks(dist, a0.elapsed_time(a1) / e2e_steps, dev)
        # the copies made it: the last y on the host equals y on the device
        same = bool(torch.equal(yps[(e2e_steps - 1) % 2], y.cpu()))
        e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(2 * (M * K + N * K + N)), "d2h_bytes_per_step": int(2 * M * N),
               "ms_per_step": e2e_ms, "steps": e2e_steps, "host_y_matches_device_y": same,
               "pipelined": "upload i+1 / compute i / download i-1 on three streams"}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    # ---- roofline of the dominant kernel -----------------------------------
    peaks, src = load_peaks()
    gemm = chosen in (L.VARIANT_GEMM_TMA, L.VARIANT_GEMM_CPASYNC, L.VARIANT_GEMM_REG, L.VARIANT_GEMM_PACKED)
    gemv_vec = "gemv_f16_rows_kernel" if M <= 2 else "gemv_f16_mma_kernel"
    kernel_name = {L.VARIANT_GEMM_TMA: "gemm_f16_tcgen05_kernel<tma>",
                   L.VARIANT_GEMM_CPASYNC: "gemm_f16_tcgen05_kernel<cpasync4>",
                   L.VARIANT_GEMM_REG: "gemm_f16_tcgen05_kernel<reg16>",
                   L.VARIANT_GEMM_PACKED: "pack_rows_kernel + gemm_f16_tcgen05_kernel<tma>",
                   L.VARIANT_GEMV: gemv_vec, L.VARIANT_GEMV_SCALAR: "gemv_f16_kernel<scalar>",
                   }.get(chosen, "bias_only_kernel")
    kern_s = kern_ms * 1e-3
    if gemm:
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        achieved = flops / kern_s / 1e12
        sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "peak_source": f"{src} dense bf16 burst (fp16 runs at the bf16 rate)",
                "frac_of_sustained_peak": achieved / sustained}
    else:
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        achieved = wl.algorithmic_bytes / kern_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"{src} STREAM-style copy"}
    roof["traffic"] = committed_traffic(kernel_name, wl.name)
    roof["kernel"] = kernel_name
    roof["kernel_ms"] = kern_ms
    roof["algorithmic_per_launch"] = flops if gemm else wl.algorithmic_bytes
    roof["hbm_gbs_algorithmic"] = wl.algorithmic_bytes / kern_s / 1e9

    cpu = None
    if not args.no_cpu:
        y_bits = y.cpu().view(torch.int16).numpy().view(np.uint16)
        cpu, _, _ = cpu_oracle_sample(x_h, w_h, b_h, args.cpu_seconds, y_gpu=y_bits)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": wl.name, "M": M, "N": N, "K": K, "dist": wl.dist, "seed": wl.seed,
                   "accumulate": "f32", "variant": L.VARIANT_NAMES.get(chosen, str(chosen)),
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": ("inputs larger than L2 (x+W+b+y = %.0f MB > 129 MB)" % (working_set / 1e6))
                   if copies == 1 else
                   "inputs larger than L2: %d rotating copies of x, W, b, y (%.0f MB in all)"
                   % (copies, copies * working_set / 1e6),
                   "timing": "CUDA graph of the K steps, replayed between two events" if graph is not None
                   else "eager launches between two events",
                   "hbm_gbs_algorithmic": wl.algorithmic_bytes / (step_ms * 1e-3) / 1e9},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_step,
        "per_launch_us": per_launch_us,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_contract(args, rank, world, local):
    """Time one widened-contraction form (kernel throughput, graph-timed)."""
    import ctypes
    import torch
    import linear_fp16_gb300 as L
    from linear_fp16_gb300 import synth

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the CUDA path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(world, True)
    dt_name, out_f32, with_bias, steps = CONTRACT_FORMS[args.contract]
    tdt = torch.bfloat16 if dt_name == "bf16" else torch.float16
    wl = synth.WORKLOADS[args.workload]
    M, N, K = wl.M, wl.N, wl.K
    G = max(1, args.groups)
    if M % G:
        raise SystemExit(f"bench.py: M = {M} is not a multiple of --groups {G}")
    x_h, w_h, b_h = synth.workload_inputs(args.workload, seed_offset=0)
    x, w, b = (t.to(dev).to(tdt) for t in (x_h, w_h, b_h))
    if G > 1:
        # G experts: each its own copy of W and b, M/G rows of x
        w = torch.cat([w] * G, dim=0).contiguous()
        b = torch.cat([b] * G, dim=0).contiguous()
    Mg = M // G
    g = torch.Generator(device="cpu").manual_seed(wl.seed + 77)
    n_ops = sum(1 for st in steps if not isinstance(st, str))
    ydt = torch.float32 if out_f32 else tdt
    ybytes = 4 if out_f32 else 2
    working_set = 2 * (M * K + G * N * K + G * N) + ybytes * M * N + 2 * M * N * n_ops
    copies = 1 if working_set >= 3 * L2_BYTES else min(64, -(-3 * L2_BYTES // working_set))
    sets = []
    for c in range(copies):
        xs, ws, bs = (x, w, b) if c == 0 else (x.clone(), w.clone(), b.clone())
        ops = [torch.randn((M, N), generator=g).to(dev).to(tdt) for _ in range(n_ops)]
        spec = L.ContractionSpec()
        spec.dtype = L.DTYPE_BF16 if dt_name == "bf16" else L.DTYPE_F16
        spec.out_f32 = int(out_f32)
        spec.num_steps = len(steps)
        k = 0
        for i, st in enumerate(steps):
            name = st if isinstance(st, str) else st[0]
            spec.steps[i].op = L.binding.EP_CODES[name]
            if not isinstance(st, str):
                spec.steps[i].operand = ops[k].data_ptr()
                spec.steps[i].ld = N
                k += 1
        y = torch.empty((M, N), dtype=ydt, device=dev)
        sets.append((xs, ws, bs if with_bias else None, y, ops, spec))
    opts = L.options(L.VARIANT_AUTO, 0, args.tile_n, args.group_m, args.k_chunk)
    lib = L.load_library()

    def step(i, sh):
        xs, ws, bs, y, _, spec = sets[i % copies]
        bp = bs.data_ptr() if bs is not None else None
        if G > 1:
            rc = lib.poot_contract_grouped(xs.data_ptr(), ws.data_ptr(), bp, y.data_ptr(), G, Mg, N, K,
                                           ctypes.byref(spec), ctypes.byref(opts), sh)
        else:
            rc = lib.poot_contract(xs.data_ptr(), ws.data_ptr(), bp, y.data_ptr(), M, N, K, ctypes.byref(spec),
                                   ctypes.byref(opts), sh)
        if rc != 0:
            raise RuntimeError(f"poot_contract: {L.poot_linear_status_string(rc)}")

    stream = torch.cuda.current_stream(dev)
    for i in range(args.warmup):
        step(i, stream.cuda_stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap = torch.cuda.current_stream().cuda_stream
        for i in range(args.steps):
            step(args.warmup + i, cap)
    graph.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local) if rank == 0 else None
    barrier(dist)
    torch.cuda.synchronize()
    wall0 = time.time()
    t0.record(stream)
    graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    wall1 = time.time()
    clocks = None
    if sampler is not None:
        sampler.stop()
        clocks = sampler.summary(wall0, wall1)
    step_ms = max_over_ranks(dist, t0.elapsed_time(t1) / args.steps, dev)
    if L.poot_linear_device_status(stream.cuda_stream) != 0:
        raise RuntimeError("device-side wait timed out during the timed region")
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0
    flops = 2.0 * M * N * K
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = flops / (step_ms * 1e-3) / 1e12
    alg_bytes = 2 * (M * K + G * N * K + (G * N if with_bias else 0)) + ybytes * M * N + 2 * M * N * n_ops
    if M // G <= L.GEMV_MAX_M:
        # M <= 16 per group: the widened GEMV, bound by the W stream
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        gbs = alg_bytes / (step_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                "peak_source": f"{src} STREAM-style copy", "traffic": None,
                "kernel": "gemv_f16_rows_kernel<wide>" if M // G <= 2 else "gemv_f16_mma_kernel<wide>",
                "kernel_ms": step_ms, "algorithmic_per_launch": alg_bytes}
    else:
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_source": f"{src} dense bf16 burst",
                "traffic": None, "kernel": "gemm_f16_tcgen05_kernel<tma, widened>",
                "kernel_ms": step_ms, "algorithmic_per_launch": flops}
    line = {
        "metric": METRIC, "value": world * achieved, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dt_name, "data": "synthetic",
        "config": {"workload": wl.name, "M": M, "N": N, "K": K, "dist": wl.dist, "seed": wl.seed,
                   "accumulate": "f32", "contract": args.contract, "groups": G, "out": "f32" if out_f32 else dt_name,
                   "bias": with_bias, "steps": [st if isinstance(st, str) else st[0] for st in steps],
                   "l2": "inputs larger than L2" if copies == 1 else f"{copies} rotating copies",
                   "timing": "CUDA graph of the K steps, replayed between two events",
                   "hbm_gbs_algorithmic": alg_bytes / (step_ms * 1e-3) / 1e9},
        "roofline": roof,
        "cpu_baseline": None,
        "e2e": None,
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.contract:
        return run_contract(args, rank, world, local)
    return run_ours(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
