#!/usr/bin/env python
"""Throughput of y = FP16(x . W^T) + b on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

A step is one call of poot_linear_f16 on one batch of seeded synthetic
inputs already resident in HBM.  The default workload is the MLP
up-projection (M=8192, N=14336, K=4096), the largest configured shape; its
x + W + y (416 MB) exceed the 129 MB L2, so no flush is needed between
steps.  Exactly K steps are timed (a CUDA graph of the K calls, replayed once
between two events on the launching stream).  Under torchrun (N > 1) every
rank runs an independent replica on its own GPU (weak scaling, no data-path
collective); the step time is the maximum over ranks.

Reported beside the device-timed value:
  roofline      the dominant kernel's achieved TFLOP/s (algorithmic 2MNK per
                launch / mean CUDA-event duration on its stream) against the
                measured dense bf16 burst peak (the fp16 tensor rate is the
                same); traffic = DRAM bytes per launch from the committed ncu
                summary when it matches the current kernel source, else null
  sustained     the same graph replayed back to back for about half a
                second: time per step, clocks in that window, and the
                fraction of the measured sustained (power-capped) peak
  workloads     every other configured shape: graph-timed time per call
                (a burst of about 10 ms, like the headline's K steps),
                its roofline fraction, the kernel that dominates it, and the
                parity of the device result with the CPU oracle under the
                contract's rule (full output, or sampled rows on the largest
                shapes)
  e2e           same metric through the C ABI with host buffers: every step
                copies its x, W, b host->device (pinned) and its y back,
                inside the timed region; consecutive steps overlap on three
                streams (upload / compute / download)
  cpu_baseline  the CPU oracle timed on a bounded row sample on all host
                cores (a reported baseline, not the target), plus one-core
                timings of every workload; the sample's rows are compared
                with the device result under the contract's rule
  clocks        SM clock and throttle reasons sampled (NVML, every 2 ms)
                during the timed region
``--impl reference`` times the CPU oracle alone on the same workload.
"""
from __future__ import annotations

import argparse
import csv
import ctypes
import datetime as _dt
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024
METRIC = "TFLOP/s of y=FP16(x·Wᵀ)+b per M×N×K; % of FP16 tensor peak / HBM BW"
CPU_SAMPLE_SECONDS = 10.0
WORKLOAD_ORDER = ["toy", "ragged_exact", "gemv_m1", "gemv_m8", "prefill", "mlp_up"]
# rows of the oracle compared on the shapes too large for a full CPU pass
PARITY_SAMPLE_ROWS = 256
# one-core oracle timing: these shapes in full, the others on a row subset
SINGLE_CORE_FULL = {"toy", "ragged_exact", "gemv_m1", "gemv_m8"}
SINGLE_CORE_ROWS = 64
# beyond-2-ulp elements (each inside the FP32-accumulation interval) allowed
# per element compared, as in the GPU tests
MAX_BEYOND = 1e-5


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
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline and its parity check")
    p.add_argument("--no-workloads", action="store_true", help="skip the other configured shapes")
    p.add_argument("--cpu-seconds", type=float, default=CPU_SAMPLE_SECONDS)
    p.add_argument("--sustain-seconds", type=float, default=0.5,
                   help="length of the back-to-back replay behind the sustained figure (0 = skip)")
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
    """SM clock, power and throttle reasons with host timestamps, sampled in
    the background: NVML through ctypes every ``period_s`` (reads only), else
    ``nvidia-smi -lms``.  ``summary(t0, t1)`` describes one window."""

    NVML_CLOCK_SM = 1
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    SMI_QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, cuda_index: int, period_s: float = 0.002):
        self.rows = []  # (host time, sm MHz, reason names, power W or None)
        self.max_mhz = None
        self.period_s = period_s
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        if self._init_nvml(cuda_index):
            self._thread = threading.Thread(target=self._run_nvml, daemon=True)
            self._thread.start()
            self.source = f"NVML every {period_s * 1e3:.0f} ms"
        else:
            self._init_smi(cuda_index)

    # NVML, read-only queries
    def _init_nvml(self, cuda_index: int) -> bool:
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return False
            h = ctypes.c_void_p()
            ok = False
            try:
                import torch
                pr = torch.cuda.get_device_properties(cuda_index)
                bus = "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
                ok = lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
            except (AttributeError, RuntimeError):
                ok = False
            if not ok:
                ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(cuda_index), ctypes.byref(h)) == 0
            if not ok:
                return False
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
            if reasons is None:
                reasons = lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint(0)
            if lib.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(self.NVML_CLOCK_SM), ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self._nvml, self._h, self._reasons = lib, h, reasons
            return True
        except (OSError, AttributeError):
            return False

    def _run_nvml(self):
        lib, h = self._nvml, self._h
        clk, rs, pw = ctypes.c_uint(0), ctypes.c_ulonglong(0), ctypes.c_uint(0)
        n = 0
        while not self._stop.is_set():
            t = time.time()
            if lib.nvmlDeviceGetClockInfo(h, ctypes.c_int(self.NVML_CLOCK_SM), ctypes.byref(clk)) == 0:
                names = []
                if self._reasons(h, ctypes.byref(rs)) == 0:
                    names = [v for bit, v in self.REASON_BITS.items() if rs.value & bit]
                power = None
                if n % 8 == 0 and lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0:
                    power = pw.value / 1000.0
                self.rows.append((t, float(clk.value), names, power))
            n += 1
            self._stop.wait(self.period_s)

    # nvidia-smi fallback
    def _init_smi(self, cuda_index: int):
        try:
            fd, self._path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self._fh = open(self._path, "w")
            self._proc = subprocess.Popen(
                ["nvidia-smi", f"--id={cuda_index}", f"--query-gpu={self.SMI_QUERY}",
                 "--format=csv,noheader,nounits", "-lms=5"], stdout=self._fh, stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi -lms 5"
            deadline = time.time() + 5.0
            while time.time() < deadline and os.path.getsize(self._path) == 0:
                time.sleep(0.02)
        except OSError:
            self._proc = None

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        with open(self._path) as fh:
            for r in csv.reader(fh):
                if len(r) < 10:
                    continue
                try:
                    ts = _dt.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    act = [names[i] for i in range(4) if r[6 + i].strip().lower() == "active"]
                    try:
                        power = float(r[4])
                    except ValueError:
                        power = None
                    rows.append((ts, float(r[2]), act, power))
                    self.max_mhz = float(r[3])
                except ValueError:
                    continue
        self.rows = rows

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=2)
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
            self._fh.close()
            self._read_smi()
            os.unlink(self._path)
            self._proc = None

    def summary(self, t0: float, t1: float):
        if self._proc is not None:
            self._read_smi()
        if self.source is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"], "samples_in_timed_region": 0}
        rows = list(self.rows)
        inside = [r for r in rows if t0 <= r[0] <= t1]
        used = inside if inside else sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:3]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"],
                    "samples_in_timed_region": 0, "source": self.source}
        reasons = sorted({n for r in used for n in r[2]})
        power = [r[3] for r in used if r[3] is not None]
        return {"sm_mhz": statistics.median(r[1] for r in used), "sm_max_mhz": self.max_mhz,
                "sm_min_mhz": min(r[1] for r in used), "reasons": reasons,
                "power_w_median": statistics.median(power) if power else None,
                "power_w_max": max(power) if power else None,
                "samples": len(used), "samples_in_timed_region": len(inside),
                "window_ms": round((t1 - t0) * 1e3, 3), "source": self.source}


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


def l2_policy(wl):
    """(copies of x, W, b, y rotated between steps, the statement for `config`)."""
    working_set = 2 * (wl.M * wl.K + wl.N * wl.K + wl.N + wl.M * wl.N)
    if working_set >= 3 * L2_BYTES:
        return 1, "inputs larger than L2 (x+W+b+y = %.0f MB > 129 MB)" % (working_set / 1e6)
    copies = min(64, -(-3 * L2_BYTES // working_set))
    return copies, ("inputs larger than L2: %d rotating copies of x, W, b, y (%.0f MB in all)"
                    % (copies, copies * working_set / 1e6))


def workload_config(wl, world):
    """The `config` object of both arms: what the workload is, nothing measured."""
    return {"workload": wl.name, "M": wl.M, "N": wl.N, "K": wl.K, "dist": wl.dist, "seed": wl.seed,
            "accumulate": "f32", "parallelism": "replicas" if world > 1 else "single",
            "l2": l2_policy(wl)[1]}


# ---- CPU oracle -------------------------------------------------------------------
def _u16(t):
    import numpy as np
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def cpu_oracle_sample(x, w, b, seconds: float):
    """Time the oracle (all host cores) on a seeded row sample sized to about
    `seconds` of work; returns (baseline dict, y_ref, p_ref, rows)."""
    import numpy as np
    import oracle
    M, K = x.shape
    N = w.shape[0]
    threads = oracle.default_threads()
    xb, wb, bb = _u16(x), _u16(w), _u16(b)
    # calibrate on one row per thread
    rows = min(M, threads)
    t = time.perf_counter()
    oracle.linear_f16(xb[:rows], wb, bb, nthreads=threads)
    per_row = (time.perf_counter() - t) / rows
    want = int(max(threads, min(M, seconds / max(per_row, 1e-9))))
    want = min(M, want)
    rng = np.random.default_rng(2024)
    sample = np.sort(rng.choice(M, size=want, replace=False))
    xs = np.ascontiguousarray(xb[sample])
    t = time.perf_counter()
    y_ref, p_ref = oracle.linear_f16(xs, wb, bb, nthreads=threads, want_proj=True)
    dt = time.perf_counter() - t
    flops = 2.0 * want * N * K
    out = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
           "sample": f"{want} of {M} rows (seeded), all {N} columns, K={K}; {dt:.2f} s on {threads} threads",
           "seconds": round(dt, 3)}
    return out, y_ref, p_ref, sample


def single_core_timings():
    """The oracle on one core: the small workloads in full, the two largest on
    a seeded row subset, extrapolated linearly in rows (and labelled so)."""
    import numpy as np
    import oracle
    from linear_fp16_gb300 import synth
    out = {}
    for name in WORKLOAD_ORDER:
        wl = synth.WORKLOADS[name]
        x, w, b = synth.workload_inputs(name)
        xb, wb, bb = _u16(x), _u16(w), _u16(b)
        if name in SINGLE_CORE_FULL:
            rows = np.arange(wl.M)
        else:
            rows = np.sort(np.random.default_rng(77).choice(wl.M, size=SINGLE_CORE_ROWS, replace=False))
        xs = np.ascontiguousarray(xb[rows])
        t = time.perf_counter()
        oracle.linear_f16(xs, wb, bb, nthreads=1)
        dt = time.perf_counter() - t
        full_s = dt * wl.M / len(rows)
        out[name] = {"rows": int(len(rows)), "of_rows": wl.M, "seconds": round(dt, 3),
                     "seconds_whole_workload": round(full_s, 3),
                     "extrapolated": len(rows) != wl.M,
                     "tflops": 2.0 * len(rows) * wl.N * wl.K / dt / 1e12}
    return out


def parity_rows(name, M):
    """Rows compared with the oracle: all of them, or on the largest shapes a
    seeded sample that includes the first and last row of every 128-row
    block boundary it can reach and the ragged last row."""
    import numpy as np
    if name in SINGLE_CORE_FULL:
        return None
    rng = np.random.default_rng(4040)
    edges = [0, 127, 128, 255, 256, 383, 384, M - 129, M - 128, M - 1]
    rest = rng.choice(M, size=PARITY_SAMPLE_ROWS - len(edges), replace=False)
    return np.unique(np.concatenate([np.array(edges), rest]))


def parity_check(name, x, w, b, y_bits, exact, rows=None, y_ref=None, p_ref=None):
    """The contract's rule on the device result (``oracle.parity``)."""
    import numpy as np
    from oracle import parity
    xb, wb, bb = _u16(x), _u16(w), _u16(b)
    xs = xb if rows is None else np.ascontiguousarray(xb[rows])
    yg = y_bits if rows is None else y_bits[rows]
    if y_ref is None:
        import oracle
        y_ref, p_ref = oracle.linear_f16(xs, wb, bb, want_proj=True)
    ok, rep = parity.judge(yg, y_ref, p_ref, xs, wb, bb, exact, max_outside=MAX_BEYOND)
    rep = {k: v for k, v in rep.items() if k != "first_bad" or not ok}
    rep["rule"] = ("bit-exact (small-integer inputs: every FP32 partial sum is exact)" if exact else
                   "|y - y_ref| <= 2 ulp16(max(|p_ref|, |y_ref|)); beyond that only inside the interval of "
                   "round-to-nearest FP32 accumulations in any order (u = 2^-24) and at most 1e-5 of the elements")
    rep["rows"] = "all" if rows is None else f"{len(rows)} of {x.shape[0]} (seeded, block edges included)"
    rep["ok"] = bool(ok)
    return rep


# ---- the GPU arm -------------------------------------------------------------------
def kernel_name(L, variant, M):
    return {L.VARIANT_GEMM_TMA: "gemm_f16_tcgen05_kernel<tma>",
            L.VARIANT_GEMM_CPASYNC: "gemm_f16_tcgen05_kernel<cpasync4>",
            L.VARIANT_GEMM_REG: "gemm_f16_tcgen05_kernel<reg16>",
            L.VARIANT_GEMM_PACKED: "gemm_f16_tcgen05_kernel<tma> (after pack_rows_kernel)",
            L.VARIANT_GEMV: "gemv_f16_rows_kernel" if M <= 2 else "gemv_f16_mma_kernel",
            L.VARIANT_GEMV_SCALAR: "gemv_f16_kernel<scalar>",
            }.get(variant, "bias_only_kernel")


class Operands:
    """One workload's x, W, b, y on the device, in as many identical copies as
    it takes to rotate past L2, and the C-ABI call on copy i % copies."""

    def __init__(self, L, lib, wl, dev, opts):
        import torch
        from linear_fp16_gb300 import synth
        self.L, self.lib, self.wl = L, lib, wl
        self.x_h, self.w_h, self.b_h = synth.workload_inputs(wl.name)
        x, w, b = self.x_h.to(dev), self.w_h.to(dev), self.b_h.to(dev)
        y = torch.empty((wl.M, wl.N), dtype=torch.float16, device=dev)
        self.copies, self.l2 = l2_policy(wl)
        self.sets = [(x, w, b, y)]
        for _ in range(self.copies - 1):
            self.sets.append((x.clone(), w.clone(), b.clone(), torch.empty_like(y)))
        self.ptrs = [tuple(t.data_ptr() for t in s) for s in self.sets]
        self.opts = opts
        self.opts_ref = ctypes.byref(opts)
        self.variant = L.variant_for(x, w, b, y) if opts.variant == L.VARIANT_AUTO else opts.variant
        self.kernel = kernel_name(L, self.variant, wl.M)
        self.launches_per_call = 2 if self.variant == L.VARIANT_GEMM_PACKED else 1

    def call(self, i, stream_handle):
        wl = self.wl
        rc = self.lib.poot_linear_f16_ex(*self.ptrs[i % self.copies], wl.M, wl.N, wl.K, self.opts_ref,
                                         stream_handle)
        if rc != 0:
            raise RuntimeError(f"poot_linear_f16: {self.L.poot_linear_status_string(rc)}")

    def graph(self, n, first):
        import torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cap = torch.cuda.current_stream().cuda_stream
            for i in range(n):
                self.call(first + i, cap)
        g.replay()  # one untimed replay: the graph's own first-launch cost
        torch.cuda.synchronize()
        return g

    def y_bits(self):
        return _u16(self.sets[0][3].cpu())


def gemm_plan(L, wl):
    """The GEMM's automatic tile plan for this shape on this device (host logic)."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    rc, plan = L.poot_linear_gemm_plan(wl.M, wl.N, wl.K, sms)
    return plan if rc == 0 else None


def roofline_for(wl, variant, L, seconds_per_call, peaks, src, sustained=False):
    gemm = variant in (L.VARIANT_GEMM_TMA, L.VARIANT_GEMM_CPASYNC, L.VARIANT_GEMM_REG, L.VARIANT_GEMM_PACKED)
    if gemm:
        key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
        peak = float(peaks.get(key, FALLBACK_PEAKS[key]))
        achieved = wl.flops / seconds_per_call / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{src} dense bf16 {'sustained' if sustained else 'burst'} "
                               "(fp16 runs at the bf16 rate)"}
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved = wl.algorithmic_bytes / seconds_per_call / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "peak_source": f"{src} STREAM-style copy"}


def measure_workload(L, lib, name, dev, sampler, peaks, src, replay_ms=2.0, max_calls=200, reps=5, check=True):
    """Graph-timed time per call of one configured shape, its roofline
    fraction, and the parity of the device result with the oracle.

    Timed like the headline, as a burst of about reps * replay_ms: a graph
    of as many calls as fill replay_ms (20 .. max_calls), replayed `reps`
    times, the median replay reported.  Longer windows enter the power
    cap's regime (prefill: 82.4 µs per call in the first 33 ms, 89 µs after
    70 ms), which the headline's `sustained` figure covers."""
    import torch
    from linear_fp16_gb300 import synth
    wl = synth.WORKLOADS[name]
    ops = Operands(L, lib, wl, dev, L.options(L.VARIANT_AUTO))
    stream = torch.cuda.current_stream(dev)
    for i in range(5):
        ops.call(i, stream.cuda_stream)
    torch.cuda.synchronize()
    if L.poot_linear_device_status(stream.cuda_stream) != 0:
        raise RuntimeError(f"{name}: device-side wait timed out")
    probe = ops.graph(20, 5)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    probe.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    calls = max(20, min(max_calls, int(replay_ms / (e0.elapsed_time(e1) / 20))))
    del probe
    g = ops.graph(calls, 5)
    times = []
    time.sleep(0.2)  # let the clock settle after the previous measurement
    w0 = time.time()
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / calls)
    w1 = time.time()
    if L.poot_linear_device_status(stream.cuda_stream) != 0:
        raise RuntimeError(f"{name}: device-side wait timed out")
    ms = statistics.median(times)
    roof = roofline_for(wl, ops.variant, L, ms * 1e-3, peaks, src)
    entry = {"M": wl.M, "N": wl.N, "K": wl.K, "dist": wl.dist, "us_per_call": ms * 1e3,
             "us_per_call_min": min(times) * 1e3, "us_per_call_each_replay": [round(t * 1e3, 3) for t in times],
             "calls_per_replay": calls, "replays": reps,
             "tflops": wl.flops / (ms * 1e-3) / 1e12, "gbs_algorithmic": wl.algorithmic_bytes / (ms * 1e-3) / 1e9,
             "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac", "peak_source")},
             "kernel": ops.kernel, "variant": L.VARIANT_NAMES.get(ops.variant), "launches_per_call":
                 ops.launches_per_call, "l2": ops.l2, "clocks": sampler.summary(w0, w1) if sampler else None}
    if ops.launches_per_call > 1:
        entry["roofline"]["note"] = "time per call covers both launches (operand copy + GEMM)"
    entry["gemm_plan"] = gemm_plan(L, wl) if wl.M > L.GEMV_MAX_M else None
    if check:
        exact = wl.dist == "smallint"
        entry["parity"] = parity_check(name, ops.x_h, ops.w_h, ops.b_h, ops.y_bits(), exact,
                                       rows=parity_rows(name, wl.M))
    del g, ops
    torch.cuda.empty_cache()
    return entry


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
    sampler = ClockSampler(local) if rank == 0 else None

    wl = synth.WORKLOADS[args.workload]
    M, N, K = wl.M, wl.N, wl.K
    variant = L.VARIANT_AUTO
    if args.variant != "auto":
        variant = {v: k for k, v in L.VARIANT_NAMES.items()}[args.variant]
    ops = Operands(L, lib, wl, dev, L.options(variant, 0, args.tile_n, args.group_m, args.k_chunk))
    chosen = ops.variant
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    for i in range(args.warmup):
        ops.call(i, sh)
    torch.cuda.synchronize()
    if L.poot_linear_device_status(sh) != 0:
        raise RuntimeError("device-side wait timed out during warm-up")

    # The K timed steps are captured once into a CUDA graph and replayed, so
    # a short kernel is not timed together with the host's launch overhead.
    graph = None if args.no_graph else ops.graph(args.steps, args.warmup)

    def timed_region():
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(args.steps):
                ops.call(args.warmup + i, sh)
        t1.record(stream)
        return t0, t1

    # ---- burst: exactly K steps ------------------------------------------
    barrier(dist)
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start, t_end = timed_region()
    torch.cuda.synchronize()
    barrier(dist)
    wall1 = time.time()
    total_ms = t_start.elapsed_time(t_end)
    step_ms = max_over_ranks(dist, total_ms / args.steps, dev)
    if L.poot_linear_device_status(sh) != 0:
        raise RuntimeError("device-side wait timed out during the timed region")

    # ---- every other configured shape ---------------------------------------
    # (measured before the sustained replay, which leaves the GPU at its power
    # cap for a while; only on rank 0)
    peaks, src = load_peaks()
    workloads = None
    if not args.no_workloads and rank == 0:
        workloads = {}
        for name in WORKLOAD_ORDER:
            if name == wl.name:
                continue
            workloads[name] = measure_workload(L, lib, name, dev, sampler, peaks, src, check=not args.no_cpu)
        torch.cuda.synchronize()

    # ---- sustained: the same K steps back to back for about half a second
    sustained = None
    if args.sustain_seconds > 0:
        reps = max(1, int(args.sustain_seconds / max(total_ms * 1e-3, 1e-6)) + 1)
        barrier(dist)
        torch.cuda.synchronize()
        sw0 = time.time()
        s0, s1 = timed_region()
        for _ in range(reps - 1):
            _, s1 = timed_region()
        torch.cuda.synchronize()
        barrier(dist)
        sw1 = time.time()
        sus_ms = max_over_ranks(dist, s0.elapsed_time(s1) / (reps * args.steps), dev)
        sustained = {"ms_per_step": sus_ms, "steps": reps * args.steps, "seconds": round(sw1 - sw0, 3),
                     "value": world * wl.flops / (sus_ms * 1e-3) / 1e12, "unit": "TFLOP/s"}
        if sampler is not None:
            sustained["clocks"] = sampler.summary(sw0, sw1)
        if L.poot_linear_device_status(sh) != 0:
            raise RuntimeError("device-side wait timed out during the sustained replay")

    # Per-launch distribution, after (and apart from) the timed region: each
    # call launched eagerly between its own pair of events on the launching
    # stream (so it includes the host's launch latency that the graph-timed
    # value leaves out).
    reps_l = 200 if M <= L.GEMV_MAX_M else 50
    ev_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps_l)]
    for r, (e0, e1) in enumerate(ev_pairs):
        e0.record(stream)
        ops.call(args.warmup + args.steps + r, sh)
        e1.record(stream)
    torch.cuda.synchronize()
    per_launch = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in ev_pairs)
    per_launch_us = {"reps": reps_l, "median": per_launch[reps_l // 2], "p10": per_launch[reps_l // 10],
                     "p90": per_launch[(9 * reps_l) // 10],
                     "how": "eager launches, each between its own CUDA events (launch latency included)"}

    value = world * wl.flops / (step_ms * 1e-3) / 1e12
    y = ops.sets[0][3]

    # ---- end to end through the C ABI with host buffers --------------------
    # Every step uploads its x, W and b from pinned host memory, runs
    # poot_linear_f16 and downloads its y.  Steps are independent, so the
    # upload of step i+1 and the download of step i-1 run on their own
    # streams while step i computes (two device buffer sets).
    e2e = None
    if not args.no_e2e:
        x, w, b = ops.sets[0][:3]
        xp, wp, bp = ops.x_h.pin_memory(), ops.w_h.pin_memory(), ops.b_h.pin_memory()
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
        e2e = {"value": world * wl.flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(2 * (M * K + N * K + N)), "d2h_bytes_per_step": int(2 * M * N),
               "ms_per_step": e2e_ms, "steps": e2e_steps, "host_y_matches_device_y": same,
               "pipelined": "upload i+1 / compute i / download i-1 on three streams"}
        del dsets, yps

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    # ---- roofline of the dominant kernel -----------------------------------
    roof = roofline_for(wl, chosen, L, step_ms * 1e-3, peaks, src)
    roof["traffic"] = committed_traffic(ops.kernel, wl.name)
    roof["kernel"] = ops.kernel
    roof["kernel_ms"] = step_ms
    roof["algorithmic_per_launch"] = wl.flops if roof["bound"] == "tensor" else wl.algorithmic_bytes
    roof["hbm_gbs_algorithmic"] = wl.algorithmic_bytes / (step_ms * 1e-3) / 1e9
    roof["gemm_plan"] = gemm_plan(L, wl) if M > L.GEMV_MAX_M else None
    if sustained is not None:
        sr = roofline_for(wl, chosen, L, sustained["ms_per_step"] * 1e-3, peaks, src, sustained=True)
        sustained["roofline"] = {k: sr[k] for k in ("bound", "achieved", "peak", "unit", "frac", "peak_source")}

    y_bits = ops.y_bits()
    x_h, w_h, b_h = ops.x_h, ops.w_h, ops.b_h
    del ops, graph
    torch.cuda.empty_cache()

    cpu = None
    parity = None
    if not args.no_cpu:
        cpu, y_ref, p_ref, sample = cpu_oracle_sample(x_h, w_h, b_h, args.cpu_seconds)
        exact = wl.dist == "smallint"
        parity = parity_check(wl.name, x_h, w_h, b_h, y_bits, exact, rows=sample, y_ref=y_ref, p_ref=p_ref)
        parity["rows"] = f"the CPU baseline's sample: {len(sample)} of {M} rows (seeded)"
        cpu["single_core"] = single_core_timings()
        cpu["single_core_note"] = ("one thread; toy, ragged_exact and both GEMVs in full, prefill and mlp_up on "
                                   f"{SINGLE_CORE_ROWS} seeded rows with the whole-workload time extrapolated "
                                   "linearly in rows")

    clocks = sampler.summary(wall0, wall1) if sampler is not None else None
    if sampler is not None:
        sampler.stop()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": workload_config(wl, world),
        "kernel_variant": L.VARIANT_NAMES.get(chosen, str(chosen)),
        "timing": ("CUDA graph of the K steps, replayed once between two events on the launching stream"
                   if not args.no_graph else "eager launches between two events"),
        "roofline": roof,
        "sustained": sustained,
        "parity": parity,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * (2 if chosen == L.VARIANT_GEMM_PACKED else 1),
        "per_launch_us": per_launch_us,
        "clocks": clocks,
        "workloads": workloads,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


# ---- the reference arm: the CPU oracle ----------------------------------------------
def run_reference(args, rank, world):
    from linear_fp16_gb300 import synth
    if rank != 0:
        return 0
    wl = synth.WORKLOADS[args.workload]
    x, w, b = synth.workload_inputs(args.workload)
    # each step: a bounded row sample of the workload, sized so that the
    # whole run stays within a few minutes
    per_step = max(0.2, min(3.0, 120.0 / (args.steps + args.warmup)))
    vals, secs = [], []
    last = None
    for i in range(args.warmup + args.steps):
        res, _, _, _ = cpu_oracle_sample(x, w, b, per_step)
        if i >= args.warmup:
            vals.append(res["value"])
            secs.append(res["seconds"])
            last = res
    value = statistics.mean(vals)
    step_ms = statistics.mean(secs) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        # the measured time of a step: one bounded row sample of the workload
        "ms_per_step": step_ms,
        "ms_whole_workload_extrapolated": wl.flops / (value * 1e12) * 1e3 if value > 0 else None,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": workload_config(wl, world),
        "timing": "each step: the oracle on a seeded row sample of the workload (all columns, all K), "
                  "perf_counter around the call",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": last["cores"], "kind": "oracle",
                         "sample": last["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
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
