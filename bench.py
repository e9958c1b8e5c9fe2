"""Benchmark of the dense half-precision GEMM (TFLOP/s at M = N = K = 4096).

One step = the 4096^3 GEMM once in bf16 and once in fp16 (A, B row-major,
entries U[-1, 1) from seed 1, fp32 accumulation, C in the input dtype), each
through the C ABI with operands resident in HBM. L2 is flushed before every
GEMM: a 256 MiB device write evicts every operand line, then (the default,
``--l2 clean``) a 256 MiB read of another buffer replaces the write's dirty
lines with clean ones, so the timed GEMM does not pay for writing back the
flush's data. Only the GEMM is inside the CUDA-event interval. `value` =
2MNK x GEMMs / summed GEMM time, over all ranks.

The roofline object names the bound from the workload's arithmetic
intensity (flops per algorithmic byte, 2(MK + KN) + 2MN bytes for 16-bit
operands) against the ridge of the measured peaks: below it the GEMM is
HBM-bound and `achieved` is GB/s of algorithmic bytes, above it tensor-bound
and `achieved` is TFLOP/s; the other roofline is reported beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

`--impl reference` times the CPU oracle instead (the only other place this
file runs the oracle), on a bounded row sample of the same workload.
For N > 1 (torchrun), every rank runs its own independent problem (no
collective on the data path; the barrier and the max over ranks are timing
only): weak scaling.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

# BLAS threads for the oracle legs: every core this process may use.
_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(_CORES))
os.environ.setdefault("OMP_NUM_THREADS", str(_CORES))

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fp16/bf16 GEMM TFLOP/s at M=N=K=4096; % of GB300 dense tensor-core peak"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20
# Bumped whenever the code of the kernel instance a traffic record describes, or its default launch (store
# path), changes, so ncu figures taken on an older kernel are not reported as current.
KERNEL_REV = 15

# name -> list of (M, N, K, dtype, dist, sigma, seed) GEMMs making up one step
WORKLOADS = {
    "square4096": [(4096, 4096, 4096, "bf16", "uniform", 1.0, 1),
                   (4096, 4096, 4096, "f16", "uniform", 1.0, 1)],
    "square8192_bf16": [(8192, 8192, 8192, "bf16", "normal", 1.0, 2)],
    "mlp_up_bf16": [(16384, 14336, 4096, "bf16", "normal", 0.02, 3)],
    "mlp_down_bf16": [(16384, 4096, 14336, "bf16", "normal", 0.02, 3)],
    "mlp_bf16": [(16384, 14336, 4096, "bf16", "normal", 0.02, 3),
                 (16384, 4096, 14336, "bf16", "normal", 0.02, 3)],
    "skinny_bf16": [(128, 8192, 8192, "bf16", "uniform", 1.0, 4)],
    "tails_bf16": [(1000, 4095, 4104, "bf16", "uniform", 1.0, 4)],
    "shortk_bf16": [(4096, 4096, 64, "bf16", "uniform", 1.0, 4)],
    "square256_bf16": [(256, 256, 256, "bf16", "uniform", 1.0, 0)],
    # the TF32 variant: fp32 A, B, C ("f32" inputs multiplied as tf32)
    "tf32_4096": [(4096, 4096, 4096, "f32", "uniform", 1.0, 1)],
    # the FP8 variant: E4M3 operands (uniform over [-8, 8) rounded to E4M3),
    # per-channel scales uniform in [0.5, 2), bf16 C
    "fp8_4096": [(4096, 4096, 4096, "e4m3", "uniform", 8.0, 1)],
    # the block-scaled FP8 variant: the same operands, one fp32 factor per
    # 64 x 64 (or 32 x 32) sub-block of A and of B, uniform in [0.5, 2)
    "fp8bs_4096": [(4096, 4096, 4096, "e4m3", "uniform", 8.0, 1)],
    "fp8bs32_4096": [(4096, 4096, 4096, "e4m3", "uniform", 8.0, 1)],
}
# block-scaled workloads: name -> scale block
BLOCK_SCALED = {"fp8bs_4096": 64, "fp8bs32_4096": 32}
# convolution workloads (im2col + GEMM): name -> (N, H, W, C, R, S, K, stride, pad, dtype, seed)
CONV_WORKLOADS = {
    "conv3x3_resnet": (32, 28, 28, 256, 3, 3, 512, 1, 1, "bf16", 1),
}
DESCRIPTIONS = {
    "square4096": "GEMM M=N=K=4096, once bf16 and once fp16, A/B row-major, U[-1,1) seed 1",
    "tf32_4096": "TF32 GEMM M=N=K=4096, fp32 A/B/C row-major, U[-1,1) seed 1",
    "fp8_4096": "FP8 GEMM M=N=K=4096, E4M3 A/B row-major (U[-8,8) rounded), per-channel scales, bf16 C, seed 1",
    "fp8bs_4096": ("block-scaled FP8 GEMM M=N=K=4096, E4M3 A/B row-major (U[-8,8) rounded), one fp32 factor "
                   "per 64x64 sub-block of A and of B (U[0.5,2)), bf16 C, seed 1"),
    "fp8bs32_4096": ("block-scaled FP8 GEMM M=N=K=4096, E4M3 A/B row-major (U[-8,8) rounded), one fp32 factor "
                     "per 32x32 sub-block of A and of B (U[0.5,2)), bf16 C, seed 1"),
    "conv3x3_resnet": ("conv2d as a GEMM (implicit, TMA im2col): x 32x28x28x256 (NHWC), w 3x3x256x512 (RSCK), "
                       "stride 1, pad 1, bf16, U[-1,1) seed 1"),
}
METRICS = {
    "tf32_4096": "TF32 GEMM TFLOP/s at M=N=K=4096 (fp32 in and out); % of GB300 dense tf32 tensor-core peak",
    "fp8_4096": "FP8 (E4M3) GEMM TFLOP/s at M=N=K=4096 with per-channel scales; % of GB300 dense fp8 tensor-core peak",
    "fp8bs_4096": ("block-scaled FP8 (E4M3, fp32 scale per 64x64 sub-block) GEMM TFLOP/s at M=N=K=4096; "
                   "% of GB300 dense fp8 tensor-core peak"),
    "fp8bs32_4096": ("block-scaled FP8 (E4M3, fp32 scale per 32x32 sub-block) GEMM TFLOP/s at M=N=K=4096; "
                     "% of GB300 dense fp8 tensor-core peak"),
    "conv3x3_resnet": ("conv2d as an implicit GEMM (TMA im2col) TFLOP/s, 2*N*P*Q*K*R*S*C flops; "
                       "% of GB300 dense bf16 tensor-core peak"),
}
# Nominal dense tensor rates relative to bf16 (2.25 PFLOP/s): tf32 1.1 PFLOP/s.
NOMINAL_RATIO = {"bf16": 1.0, "f16": 1.0, "f32": 1.1 / 2.25, "e4m3": 4.5 / 2.25, "e5m2": 4.5 / 2.25}
ESIZE = {"bf16": 2, "f16": 2, "f32": 4, "e4m3": 1, "e5m2": 1}
C_ESIZE = {"bf16": 2, "f16": 2, "f32": 4, "e4m3": 2, "e5m2": 2}
FP8 = ("e4m3", "e5m2")


def flops(M, N, K):
    return 2 * M * N * K


def hbm_bytes(M, N, K, esize=2):
    return esize * (M * K + K * N + M * N)


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------ clocks
# NVML clock-event reason bits (nvmlClocksEventReason*), read only.
_NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class _Nvml:
    """Read-only NVML queries through the driver's libnvidia-ml (ctypes): SM
    clock, maximum SM clock, power and clock-event reasons of one GPU."""

    def __init__(self, cuda_index: int):
        import ctypes

        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.handle = ctypes.c_void_p()
        found = False
        try:  # the GPU this process uses, by UUID (NVML numbers every GPU of the machine)
            import torch
            u = str(torch.cuda.get_device_properties(cuda_index).uuid)
            for name in (u if u.startswith("GPU-") else "GPU-" + u, u):
                if self.lib.nvmlDeviceGetHandleByUUID(name.encode(), ctypes.byref(self.handle)) == 0:
                    found = True
                    break
        except Exception:
            pass
        if not found and self.lib.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(self.handle)) != 0:
            raise OSError("no NVML handle")
        mx = ctypes.c_uint(0)
        self.max_mhz = float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0 \
            else None
        self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        ct = self.ct
        mhz, mw, rs = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        ok = self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ct.byref(mhz)) == 0   # NVML_CLOCK_SM
        pw = float(mw.value) / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.handle, ct.byref(mw)) == 0 else None
        reasons = [n for b, n in _NVML_REASONS.items() if rs.value & b] \
            if self._reasons(self.handle, ct.byref(rs)) == 0 else []
        return (float(mhz.value) if ok else None, pw, reasons)


class ClockSampler:
    """SM clocks, power and throttle reasons sampled during the timed region:
    read-only NVML queries every 5 ms from a thread (ctypes releases the GIL
    during each query), else `nvidia-smi -lms 100`. `sample_now()` adds one
    sample on demand (the launch loop calls it while the GPU is still busy)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_s: float = 0.005):
        self.dev = device_index
        self.period = period_s
        self.proc = None
        self.nvml = None
        self.samples = []      # (sm_mhz, power_w, [reasons])
        self.max_mhz = None
        self.source = None

    def sample_now(self):
        if self.nvml is not None:
            try:
                self.samples.append(self.nvml.sample())
            except Exception:
                pass

    def _loop(self):
        import time as _t
        while not self._stop.is_set():
            self.sample_now()
            _t.sleep(self.period)

    def __enter__(self):
        import threading
        try:
            self.nvml = _Nvml(self.dev)
            self.max_mhz = self.nvml.max_mhz
            self.source = "nvml"
            self._stop = threading.Event()
            self.sample_now()
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()
            return self
        except Exception:
            self.nvml = None
        import shutil
        exe = shutil.which("nvidia-smi") or next(
            (p for p in ("/usr/bin/nvidia-smi", "/usr/local/nvidia/bin/nvidia-smi") if os.path.exists(p)), None)
        if exe is None:
            return self
        try:
            self.proc = subprocess.Popen(
                [exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.nvml is not None:
            self.sample_now()
            self._stop.set()
            self._thread.join(timeout=2)
            return False
        if self.proc is None:
            return False
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            num = lambda v: float(v) if v.replace(".", "").isdigit() else None
            if num(parts[2]) is not None:
                self.max_mhz = max(self.max_mhz or 0.0, num(parts[2]))
            self.samples.append((num(parts[1]), num(parts[3]),
                                 [n for n, v in zip(names, parts[5:9]) if v.lower() == "active"]))
        return False

    def summary(self):
        sm = [s[0] for s in self.samples if s[0] is not None]
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz,
                    "reasons": ["no clock samples (NVML and nvidia-smi unavailable)"], "samples": 0}
        pw = [s[1] for s in self.samples if s[1] is not None]
        reasons = sorted({r for s in self.samples for r in s[2]})
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(sm), "power_w_max": max(pw) if pw else None,
                "source": self.source}


# ------------------------------------------------------- multi-rank timing
def max_over_ranks(values, device, world):
    """Element-wise max of `values` over all ranks (each rank ran its own
    independent problem; the slowest one sets the job time)."""
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as tdist
        tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(world, steps, step_flops, total_ms):
    """Whole-job TFLOP/s: every rank's steps over the slowest rank's time."""
    return world * steps * step_flops / (total_ms * 1e-3) / 1e12


# --------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch

    from half_precision_dense_gb300 import binding as hg
    from half_precision_dense_gb300 import build as hbuild
    from half_precision_dense_gb300 import inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or not os.path.exists(hbuild.LIB_PATH):
        hbuild.build()
    if world > 1:
        torch.distributed.barrier()
    hg.load_library()

    gemms = WORKLOADS.get(args.workload, [])
    ops = []
    if args.workload in CONV_WORKLOADS:
        (cN, cH, cW, cC, cR, cS, cK, cst, cpd, dt, seed) = CONV_WORKLOADS[args.workload]
        cP = (cH + 2 * cpd - cR) // cst + 1
        cQ = (cW + 2 * cpd - cS) // cst + 1
        x = inputs.generate((1, cN * cH * cW * cC), dt, seed, 0).view(cN, cH, cW, cC)
        w = inputs.generate((1, cR * cS * cC * cK), dt, seed, 1).view(cR, cS, cC, cK)
        ops.append(dict(kind="conv", M=cN * cP * cQ, N=cK, K=cR * cS * cC, dt=dt, hA=x, hB=w, A=x.to(dev),
                        B=w.to(dev), sa=None, sb=None, conv=(cN, cH, cW, cC, cK, cR, cS, cst, cpd),
                        C=torch.empty((cN, cP, cQ, cK), dtype=inputs.TORCH_DTYPES[dt], device=dev)))
    bs = BLOCK_SCALED.get(args.workload, 0)
    for (M, N, K, dt, dist, sigma, seed) in gemms:
        if dt in FP8:
            A = torch.from_numpy(inputs.generate_fp8((M, K), dt, seed, 0, sigma))
            B = torch.from_numpy(inputs.generate_fp8((K, N), dt, seed, 1, sigma))
            if bs:
                ga, gb = (-(-M // bs), -(-K // bs)), (-(-K // bs), -(-N // bs))
                sa = torch.from_numpy(inputs.generate_scales(ga[0] * ga[1], seed, 2).reshape(ga)).to(dev)
                sb = torch.from_numpy(inputs.generate_scales(gb[0] * gb[1], seed, 3).reshape(gb)).to(dev)
            else:
                sa = torch.from_numpy(inputs.generate_scales(M, seed, 2)).to(dev)
                sb = torch.from_numpy(inputs.generate_scales(N, seed, 3)).to(dev)
            cdt = torch.bfloat16
        else:
            A = inputs.generate((M, K), dt, seed, 0, dist, sigma)
            B = inputs.generate((K, N), dt, seed, 1, dist, sigma)
            sa = sb = None
            cdt = inputs.TORCH_DTYPES[dt]
        ops.append(dict(M=M, N=N, K=K, dt=dt, hA=A, hB=B, A=A.to(dev), B=B.to(dev), sa=sa, sb=sb,
                        C=torch.empty((M, N), dtype=cdt, device=dev)))
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    clean = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev) if args.l2 == "clean" else None
    sink = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2():
        flush.zero_()                      # a write larger than L2: no operand line stays
        if clean is not None:
            torch.sum(clean, 0, out=sink)  # a read larger than L2: no dirty line of the write stays

    def one_gemm(o):
        if o.get("kind") == "conv":
            hg.hgemm_conv2d(o["A"], o["B"], o["C"], *o["conv"], o["dt"], stream)
        elif o["dt"] in FP8 and bs:
            hg.hgemm_fp8_blockscaled(o["A"], o["B"], o["C"], o["sa"], o["sb"], o["M"], o["N"], o["K"], bs, o["dt"],
                                     None, stream)
        elif o["dt"] in FP8:
            hg.hgemm_fp8(o["A"], o["B"], o["C"], o["sa"], o["sb"], o["M"], o["N"], o["K"], o["dt"], None, stream)
        else:
            hg.hgemm(o["A"], o["B"], o["C"], o["M"], o["N"], o["K"], o["dt"], stream)

    for _ in range(args.warmup):
        for o in ops:
            flush_l2()
            one_gemm(o)
    torch.cuda.synchronize(dev)
    hg.get_device_status(local_rank, reset=True)

    n_ev = args.steps * len(ops)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clk:
        wall0 = time.perf_counter()
        i = 0
        for _ in range(args.steps):
            for o in ops:
                flush_l2()
                starts[i].record(stream)
                one_gemm(o)
                ends[i].record(stream)
                i += 1
        clk.sample_now()                   # the queued GEMMs are still running
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(times_ms)
    st, info = hg.get_device_status(local_rank)
    if st != 0:
        raise RuntimeError(f"kernel status {st} info {info:#x}")

    # per-GEMM-kind averages (the dominant kernel is the GEMM kernel itself)
    per_kind = {}
    for j, o in enumerate(ops):
        ts = times_ms[j::len(ops)]
        per_kind[f"{o['dt']}_{o['M']}x{o['N']}x{o['K']}"] = {
            "ms": statistics.mean(ts),
            "tflops": flops(o["M"], o["N"], o["K"]) / (statistics.mean(ts) * 1e-3) / 1e12}
    step_flops = sum(flops(o["M"], o["N"], o["K"]) for o in ops)

    # e2e: host operands -> device -> GEMM -> host result, through hgemm_host
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    pinned = []
    for o in ops:
        pinned.append((o["hA"].pin_memory(), o["hB"].pin_memory(),
                       torch.empty((o["M"], o["N"]), dtype=o["C"].dtype).pin_memory()))
    def host_step(o, pa, pb, pc):
        if o.get("kind") == "conv" or bs:
            # host x, w -> device, convolution, y -> host, through the binding
            o["A"].copy_(pa, non_blocking=True)
            o["B"].copy_(pb, non_blocking=True)
            one_gemm(o)
            pc.view(o["C"].shape).copy_(o["C"], non_blocking=True)
            stream.synchronize()
        else:
            hg.hgemm_host(pa, pb, pc, o["M"], o["N"], o["K"], o["dt"], o["A"], o["B"], o["C"], stream)

    for o, (pa, pb, pc) in zip(ops, pinned):   # warm the copy path
        host_step(o, pa, pb, pc)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    e0 = time.perf_counter()
    for _ in range(e2e_steps):
        for o, (pa, pb, pc) in zip(ops, pinned):
            host_step(o, pa, pb, pc)
    torch.cuda.synchronize(dev)
    e2e_s = time.perf_counter() - e0

    total_ms, e2e_s, wall = max_over_ranks([total_ms, e2e_s, wall], dev, world)
    if rank != 0:
        return None

    peaks, peak_src = read_peaks()
    value = job_throughput(world, args.steps, step_flops, total_ms)
    step_s = total_ms / args.steps * 1e-3
    achieved = step_flops / step_s / 1e12
    # algorithmic bytes: each operand read once, C written once (for a
    # convolution: x, the filters and y, not the im2col matrix)
    step_bytes = sum(ESIZE[o["dt"]] * (o["hA"].numel() + o["hB"].numel()) + C_ESIZE[o["dt"]] * o["C"].numel()
                     for o in ops)
    achieved_gbs = step_bytes / step_s / 1e9
    dts = {o["dt"] for o in ops}
    ratio = min(NOMINAL_RATIO[d] for d in dts)
    peak = round(float(peaks["bf16_tflops"]) * ratio, 1)
    hbm_peak = float(peaks["hbm_gbs"])
    # the ridge of the two measured peaks: flops per byte where HBM and the
    # tensor cores take equally long
    ridge = peak * 1e12 / (hbm_peak * 1e9)
    intensity = step_flops / step_bytes
    tensor_roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                   "frac": round(achieved / peak, 4)}
    hbm_roof = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved_gbs / hbm_peak, 4),
                "peak_source": f"{peak_src} device copy bandwidth (hbm_gbs)"}
    peak_desc = (f"{peak_src} bf16 dense (cuBLAS burst); fp16 has the same nominal rate (ratio 1)"
                 if ratio == 1.0 else
                 f"{peak_src} bf16 dense (cuBLAS burst) x nominal fp8/bf16 ratio 4.5/2.25" if ratio > 1.0 else
                 f"{peak_src} bf16 dense (cuBLAS burst) x nominal tf32/bf16 ratio 1.1/2.25")
    clocks = clk.summary()
    e2e_value = job_throughput(world, e2e_steps, step_flops, e2e_s * 1e3)
    h2d = sum(ESIZE[o["dt"]] * (o["hA"].numel() + o["hB"].numel()) for o in ops)
    d2h = sum(C_ESIZE[o["dt"]] * o["M"] * o["N"] for o in ops)
    line = {
        "metric": METRICS.get(args.workload, METRIC),
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("f32 in (multiplied as tf32), f32 accumulate and out" if dts == {"f32"} else
                  "+".join(sorted(dts)) + " in, f32 accumulate, bf16 out" if dts <= set(FP8) else
                  "+".join(sorted(dts)) + " in, f32 accumulate"),
        "data": "synthetic (seeded SplitMix64 inputs)",
        "config": {
            "workload": DESCRIPTIONS.get(args.workload, args.workload),
            "gemms_per_step": len(ops),
            "shapes": [[o["M"], o["N"], o["K"], o["dt"]] for o in ops],
            "l2": (f"flushed before every GEMM, outside the timed interval: a {L2_FLUSH_BYTES >> 20} MiB device "
                   f"write" + (f", then a {L2_FLUSH_BYTES >> 20} MiB read of another buffer (no dirty line of "
                               f"the write left to write back)" if args.l2 == "clean" else "")),
            "parallelism": f"independent problem per GPU x{world}" if world > 1 else "single GPU",
        },
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "per_gemm": {k: {"ms": round(v["ms"], 5), "tflops": round(v["tflops"], 1)} for k, v in per_kind.items()},
        "roofline": dict(
            (hbm_roof if intensity < ridge else dict(tensor_roof, peak_source=peak_desc)),
            kernel="hg::hgemm_tc_kernel",
            traffic=None,
            algorithmic_bytes_per_launch=step_bytes // len(ops),
            algorithmic_flops_per_launch=step_flops // len(ops),
            intensity_flop_per_byte=round(intensity, 1),
            ridge_flop_per_byte=round(ridge, 1),
            other=(dict(tensor_roof, peak_source=peak_desc) if intensity < ridge else hbm_roof),
        ),
        "clocks": clocks,
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "path": ("pinned host operands -> device (cudaMemcpyAsync), the GEMM through the binding, "
                         "C -> pinned host, per GEMM" if (bs or args.workload in CONV_WORKLOADS) else
                         "hgemm_host: pinned host A,B -> device, GEMM, C -> pinned host, per GEMM")},
        "gpu_launches": n_ev,
        "wall_s_timed_region": round(wall, 4),
    }
    o = ops[0]
    plan = hg.plan(o["M"], o["N"], o["K"], o["dt"])
    plan_key = [plan["cta_group"], plan["block_n"], plan["sk_tiles"], plan["grid_ctas"]]
    line["roofline"]["plan"] = {"cta_group": plan_key[0], "block_n": plan_key[1],
                                "stream_k_tiles": plan_key[2], "grid_ctas": plan_key[3],
                                "split_k": plan["split_k"], "store_mode": plan["store_mode"],
                                "epi_warps": plan["epi_warps"]}
    if bs:
        # the block-scaled kernel plans its own tiles: 128 columns, a CTA pair
        # per 256-row tile unless there is a single 128-row tile row
        cg = 2 if o["M"] > 128 else 1
        line["roofline"]["kernel"] = "hg::hgemm_fp8bs_kernel"
        line["roofline"]["plan"] = {"cta_group": cg, "block_n": 128, "scale_block": bs}
        plan_key = None
    if args.traffic_file and os.path.exists(args.traffic_file):
        # DRAM bytes from an ncu capture count only while the kernel and plan
        # they were taken on are the ones running now.
        try:
            with open(args.traffic_file) as f:
                tr = json.load(f)
            if (plan_key is not None and tr.get("plan") == plan_key and tr.get("kernel_rev") == KERNEL_REV and
                    tr.get("dtype", "bf16") in {o["dt"] for o in ops}):
                line["roofline"]["traffic"] = tr.get("dram_bytes_per_launch")
                line["roofline"]["traffic_source"] = tr.get("source")
            else:
                line["roofline"]["traffic_source"] = "stale capture (kernel or plan changed); null"
        except (OSError, ValueError):
            pass
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_budget)
    return line


# ---------------------------------------------------- oracle (CPU) timing
def _conv_sample(workload, npts):
    """``npts`` evenly spaced output pixels of a convolution workload, every
    output channel: the oracle evaluates each from the convolution's
    definition (uint16 bit patterns in, one row of K exact sums out)."""
    import numpy as np

    from half_precision_dense_gb300 import inputs

    (N, H, W, C, R, S, K, st, pd, dt, seed) = CONV_WORKLOADS[workload]
    P = (H + 2 * pd - R) // st + 1
    Q = (W + 2 * pd - S) // st + 1
    x = inputs.bits(inputs.generate((1, N * H * W * C), dt, seed, 0)).reshape(N, H, W, C)
    w = inputs.bits(inputs.generate((1, R * S * C * K), dt, seed, 1)).reshape(R, S, C, K)
    idx = np.linspace(0, N * P * Q - 1, max(1, npts)).astype(np.int64)
    pts = [(int(i // (P * Q)), int(i // Q % P), int(i % Q)) for i in idx]
    return ("conv", x, w, dt, st, pd, pts, 2 * len(pts) * K * R * S * C)


def _oracle_sample(workload, rows, cols):
    """A sampled sub-problem of each GEMM of the workload: the C block at
    `rows` evenly spaced rows and `cols` evenly spaced columns, i.e. the rows
    of A and the columns of B it needs (uint16 bit patterns)."""
    import numpy as np

    from half_precision_dense_gb300 import inputs

    out = []
    bs = BLOCK_SCALED.get(workload, 0)
    for (M, N, K, dt, dist, sigma, seed) in WORKLOADS[workload]:
        ri = np.linspace(0, M - 1, min(rows, M)).astype(np.int64)
        ci = np.linspace(0, N - 1, min(cols, N)).astype(np.int64)
        if dt in FP8 and bs:
            # the leading rows x cols block of C (whole scale blocks), with
            # the factor grids of its operands
            r, c = min(M, -(-rows // bs) * bs), min(N, -(-cols // bs) * bs)
            A = inputs.generate_fp8((M, K), dt, seed, 0, sigma)[:r]
            B = inputs.generate_fp8((K, N), dt, seed, 1, sigma)[:, :c]
            ga, gb = (-(-M // bs), -(-K // bs)), (-(-K // bs), -(-N // bs))
            sa = inputs.generate_scales(ga[0] * ga[1], seed, 2).reshape(ga)[: -(-r // bs)]
            sb = inputs.generate_scales(gb[0] * gb[1], seed, 3).reshape(gb)[:, : -(-c // bs)]
            out.append((np.ascontiguousarray(A), np.ascontiguousarray(B), dt, K, ("blocks", sa, sb, bs)))
            continue
        if dt in FP8:
            A = inputs.generate_fp8((M, K), dt, seed, 0, sigma)
            B = inputs.generate_fp8((K, N), dt, seed, 1, sigma)
            scales = (inputs.generate_scales(M, seed, 2)[ri], inputs.generate_scales(N, seed, 3)[ci])
        else:
            conv = (lambda t: t.numpy()) if dt == "f32" else inputs.bits
            A = conv(inputs.generate((M, K), dt, seed, 0, dist, sigma))
            B = conv(inputs.generate((K, N), dt, seed, 1, dist, sigma))
            scales = None
        out.append((np.ascontiguousarray(A[ri]), np.ascontiguousarray(B[:, ci]), dt, K, scales))
    return out


def _oracle_step(sample):
    import oracle
    from oracle import fp8_oracle, tf32_oracle

    if isinstance(sample, tuple) and sample and sample[0] == "conv":
        from oracle import conv_oracle
        _, x, w, dt, st, pd, pts, fl = sample
        oracle.round_rne(conv_oracle.conv_at(x, w, dt, st, pd, pts), dt)
        return fl
    f = 0
    for (a, b, dt, K, scales) in sample:
        if dt == "f32":
            tf32_oracle.gemm(a, b)
        elif dt in FP8 and isinstance(scales[0], str):
            fp8_oracle.gemm_blockscaled(a, b, dt, scales[1], scales[2], scales[3])
        elif dt in FP8:
            fp8_oracle.gemm(a, b, dt, scales[0], scales[1])
        else:
            oracle.gemm(a, b, dt)
        f += flops(a.shape[0], b.shape[1], K)
    return f


def _calibrated_sample(workload, seconds_per_step):
    if workload in CONV_WORKLOADS:
        npts = 64
        for _ in range(3):
            sample = _conv_sample(workload, npts)
            t0 = time.perf_counter()
            _oracle_step(sample)
            el = max(time.perf_counter() - t0, 1e-6)
            new = max(8, min(20000, int(npts * seconds_per_step / el)))
            if abs(new - npts) <= npts // 8:
                break
            npts = new
        return _conv_sample(workload, npts), npts
    side = 256
    for _ in range(3):
        sample = _oracle_sample(workload, side, side)
        t0 = time.perf_counter()
        _oracle_step(sample)
        el = max(time.perf_counter() - t0, 1e-6)
        new = int(side * (seconds_per_step / el) ** 0.5)
        new = max(16, min(4096, new))
        if abs(new - side) <= side // 8:
            break
        side = new
    return _oracle_sample(workload, side, side), side


def _sample_desc(side, workload):
    if workload in CONV_WORKLOADS:
        return (f"each step: {side} evenly spaced output pixels (every output channel) of {workload}, "
                f"computed by the CPU oracle from the convolution's definition (fp64 taps + bit-level RNE)")
    dts = {g[3] for g in WORKLOADS[workload]}
    how = ("numpy fp64 product of the tf32-truncated operands, rounded to fp32" if dts == {"f32"} else
           "fp8 decode, per-sub-block fp32 factors, numpy fp64 product, bit-level RNE to bf16"
           if dts <= set(FP8) and workload in BLOCK_SCALED else
           "fp8 decode, numpy fp64 product, per-channel scales, bit-level RNE to bf16" if dts <= set(FP8) else
           "numpy fp64 product + bit-level RNE")
    return (f"each step: the {side} x {side} block of C at evenly spaced rows and columns of every "
            f"GEMM of {workload}, computed by the CPU oracle ({how})")


def cpu_baseline(workload, budget_s=15.0):
    sample, side = _calibrated_sample(workload, 1.0)
    done = 0
    reps = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s and reps < 200:
        done += _oracle_step(sample)
        reps += 1
    el = time.perf_counter() - t0
    return {"value": round(done / el / 1e12, 6), "unit": UNIT, "cores": _CORES, "kind": "oracle",
            "sample": _sample_desc(side, workload) + f"; {reps} steps in {el:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    budget = min(150.0, max(20.0, 0.5 * (args.steps + args.warmup)))
    sample, side = _calibrated_sample(args.workload, budget / (args.steps + args.warmup))
    for _ in range(args.warmup):
        _oracle_step(sample)
    t0 = time.perf_counter()
    f = 0
    for _ in range(args.steps):
        f += _oracle_step(sample)
    el = time.perf_counter() - t0
    value = f / el / 1e12
    desc = _sample_desc(side, args.workload)
    return {
        "impl": "reference",
        "metric": METRICS.get(args.workload, METRIC),
        "value": round(value, 6),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * el / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 (oracle)",
        "data": "synthetic (seeded SplitMix64 inputs)",
        "config": {"workload": DESCRIPTIONS.get(args.workload, args.workload), "sample": desc},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": _CORES, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(CONV_WORKLOADS), default="square4096")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--traffic-file", default=None,
                    help="ncu DRAM-traffic record (default: profiles/traffic_<workload>.json)")
    ap.add_argument("--l2", choices=["clean", "dirty"], default="clean",
                    help="clean: flush by a write then a read larger than L2; dirty: the write alone")
    args = ap.parse_args()
    if args.traffic_file is None:
        args.traffic_file = os.path.join(ROOT, "profiles", f"traffic_{args.workload}.json")
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        if world == 1 and args.gpus > 1:
            ap.error("for --gpus N > 1 launch under torch.distributed.run with N processes")
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        line = run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as tdist
            tdist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
