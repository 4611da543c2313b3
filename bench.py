#!/usr/bin/env python3
"""Benchmark: causal long-convolution throughput (B*H*N outputs/s) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step is one pass of the whole hot path (kernel spectrum precomputed,
then the fused forward over every (b,h) row) on the workload's synthetic
inputs, which are resident in HBM before timing starts.  Prints one JSON
line on rank 0.  Under torchrun every rank runs its own copy of the
workload (rows are independent: no collective on the data path) and the
value is the sum over ranks divided by the slowest rank's time.

--impl reference runs the oracle (double-precision CPU FFT convolution) on
the host cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from typing import Optional

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = ("long-conv B·H·N outputs/sec on 1 GB300; achieved fraction of "
          "HBM/tensor roofline")
DEFAULT_WORKLOAD = "m2bert-16k"
L2_BYTES = 129 * 1000 * 1000


def canonical_c(N: int) -> int:
    """Canonical Monarch contraction count per complex point (fwd + inv):
    min over factorizations M = prod M_i, M_i in {16, 32, 64}, of
    sum_{i>=2} M_i + M_1/2 (the padded outer stage does half the work)."""
    best = None
    facs = (16, 32, 64)

    def rec(rem, acc, first):
        nonlocal best
        if rem == 1:
            if first is not None:
                c = first // 2 + acc
                best = c if best is None else min(best, c)
            return
        for f in facs:
            if rem % f == 0:
                if first is None:
                    rec(rem // f, acc, f)
                else:
                    rec(rem // f, acc + f, first)

    rec(N, 0, None)
    return best


def algorithmic(w: W.Workload) -> dict:
    """Compulsory bytes and canonical Monarch FLOPs of one pass."""
    s = 2
    per_row = 2 * w.N * s + (2 * w.N * s if w.gated else 0)
    bytes_ = w.rows * per_row + w.H * (w.N + 1) * 4
    flops = 16 * w.N * canonical_c(w.N) * w.rows
    return {"bytes": bytes_, "flops": flops}


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fft_long_convolution_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(workload)
    if not d or d.get("source_hash") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """SM clocks and clock-event (throttle) reasons polled through NVML
    (read-only queries, libnvidia-ml via ctypes) while the timed region runs."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int):
        import ctypes
        import threading
        self.samples = []
        self.reason_bits = 0
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            ok = False
            try:  # match the CUDA device by PCI location when torch exposes it
                import torch
                p = torch.cuda.get_device_properties(device_index)
                bus = "%08x:%02x:%02x.0" % (int(p.pci_domain_id), int(p.pci_bus_id), int(p.pci_device_id))
                ok = nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
            except Exception:
                ok = False
            if not ok and nv.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(h)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) != 0:
                    return
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self._nv, self._h, self._get_reasons = nv, h, get_reasons
        except Exception:
            return

        def poll():
            clk = ctypes.c_uint()
            rs = ctypes.c_ulonglong()
            while not self._stop.is_set():
                if self._nv.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(clk)) == 0:
                    self.samples.append(clk.value)
                if self._get_reasons(self._h, ctypes.byref(rs)) == 0:
                    self.reason_bits |= rs.value
                time.sleep(0.002)

        self._thread = threading.Thread(target=poll, daemon=True)
        self._thread.start()

    def stop(self):
        if self._thread is None:
            return None
        self._stop.set()
        self._thread.join(timeout=2)
        reasons = sorted(v for b, v in self.REASONS.items() if self.reason_bits & b)
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(self.samples),
                "source": "nvml"}


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time (every rank gets it): the step of a weakly
    scaled job ends when its last replica ends."""
    if world <= 1:
        return float(ms)
    import torch
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(outputs_per_rank: int, world: int, ms_slowest: float) -> float:
    """Whole-job outputs/s: every rank convolves its own copy of the workload
    (rows are independent; no collective on the data path)."""
    return world * outputs_per_rank / (ms_slowest * 1e-3)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def cpu_baseline(w: W.Workload, ins: dict, budget_s: float = 12.0, mask=None):
    """The oracle on the host cores over a bounded sample of rows (the
    masked convolution for a frequency-sparse run): one warm-up, then the
    median of three timed runs, each a bounded number of repeats of the
    sample.  When the whole workload fits the host's cores (the 1K case,
    which cannot occupy them all) a one-thread time is reported beside it."""
    import oracle
    cores = os.cpu_count() or 1
    rows = min(w.rows, max(cores, 1))
    threads = rows  # one row per thread
    # the first `rows` rows (b = 0, h = 0..rows-1) of the workload
    sl = {n: (r.f64.reshape(-1, w.N)[:rows] if n != "k" else r.f64) for n, r in ins.items()}

    def run(nthreads):
        if mask is None:
            oracle.causal_conv_batch(sl["u"], sl["k"], sl.get("w_in"), sl.get("w_out"), threads=nthreads)
        else:
            oracle.masked_causal_conv_batch(sl["u"], sl["k"], mask, sl.get("w_in"), sl.get("w_out"),
                                            threads=nthreads)

    def rate(nthreads, budget):
        t0 = time.perf_counter()
        run(nthreads)  # warm-up, also sizes the runs
        dt = time.perf_counter() - t0
        reps = max(1, min(int(budget / 3 / max(dt, 1e-4)), 100000))
        rates = []
        for _ in range(3):
            t0 = time.perf_counter()
            for _ in range(reps):
                run(nthreads)
            rates.append(rows * reps * w.N / (time.perf_counter() - t0))
        return statistics.median(rates), reps

    v, reps = rate(threads, budget_s)
    out = {"value": v, "unit": "outputs/s", "cores": threads, "kind": "oracle",
           "sample": f"{rows} rows of {w.name} (N={w.N}) x {reps} repeats per run, median of 3 runs, "
                     f"{threads} threads of {cores} host cores"}
    if w.rows <= cores:
        v1, reps1 = rate(1, budget_s / 3)
        out["one_thread"] = {"value": v1, "unit": "outputs/s", "cores": 1,
                             "sample": f"{rows} rows x {reps1} repeats per run, median of 3 runs"}
    return out


def _factors(w: W.Workload) -> list:
    import fft_long_convolution_gb300 as F
    return F.query(w.N, F.F16 if w.dtype == "fp16" else F.BF16)["factors"]


def run_reference(args, w: W.Workload):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    small = W.scaled(w, B=1, H=min(w.H, (os.cpu_count() or 1)))
    ins = W.make_inputs(small, seed=0)
    cores = os.cpu_count() or 1
    band = parse_band(args.band)
    mask = band_mask_for(w, band)
    if mask is None:
        fn = lambda: oracle.causal_conv_batch(  # noqa: E731
            ins["u"].f64, ins["k"].f64, ins["w_in"].f64 if w.gated else None,
            ins["w_out"].f64 if w.gated else None, threads=cores)
    else:
        fn = lambda: oracle.masked_causal_conv_batch(  # noqa: E731
            ins["u"].f64, ins["k"].f64, mask, ins["w_in"].f64 if w.gated else None,
            ins["w_out"].f64 if w.gated else None, threads=cores)
    for _ in range(args.warmup):
        fn()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn()
    dt = time.perf_counter() - t0
    outs = small.rows * small.N * args.steps
    v = outs / dt
    sample = f"{small.rows} rows (B=1, H={small.H}) of {w.name} (N={w.N}) per step, {cores} threads"
    config = config_of(w, band, None if band is None else _factors(w))
    config["sample"] = {"B": 1, "H": small.H, "rows_per_step": small.rows,
                        "note": "each step convolves this sample of the workload's rows; value is outputs/s"}
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "outputs/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": v, "unit": "outputs/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "outputs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def path_of(plan_info: dict, pairs_run: Optional[int] = None, pairs_total: Optional[int] = None) -> dict:
    """The kernels one step launches for a plan (names as in the sources);
    pass B is not launched when a frequency-sparse plan skips every pair."""
    if plan_info["path"] == 1:
        nb = 0 if pairs_run == 0 else 1
        skips = pairs_run is not None and pairs_total is not None and pairs_run < pairs_total
        if plan_info["order"] == 4 and plan_info["factors"][3] == 64:  # outer factor RA x 64, one pass per side
            sparse = " (dead sub-rows skipped)" if skips else ""
            return {"kernel": "otc2_pass (A: RA in registers, 64 on tcgen05) + mp_pass_b_tc + otc2_pass (C) "
                              "(the whole step)" + sparse,
                    "launches_per_step": 2 + nb}
        if plan_info["order"] == 3:
            return {"kernel": "otc_pass (A) + mp_pass_b_tc + otc_pass (C) (the whole step)",
                    "launches_per_step": 2 + nb}
        return {"kernel": "mp_pass_a + mp_pass_b + mp_pass_c (the whole step)", "launches_per_step": 2 + nb}
    if plan_info["order"] == 2:
        return {"kernel": "tc64_conv_kernel", "launches_per_step": 1}
    if plan_info["factors"][1] == 64:  # R0 x 64 x 64 on the tensor cores
        return {"kernel": "ftc_conv_kernel", "launches_per_step": 1}
    return {"kernel": "fused_conv_kernel", "launches_per_step": 1}


def config_of(w: W.Workload, band: Optional[list] = None, factors: Optional[list] = None) -> dict:
    c = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "gated": w.gated, "dtype": w.dtype,
         "u": w.u_kind, "k": w.k_kind,
         "l2": "no flush: inputs+outputs exceed L2" if algorithmic(w)["bytes"] > L2_BYTES
         else "L2 flushed between steps"}
    if band is not None:
        # frequency-sparse: kept fraction of the spectrum, prod_j kept_j / N
        kept = 1
        for b, Mj in zip(band, factors):
            kept *= 0 if b <= 0 else min(Mj, 2 * b - 1)
        c["band"] = list(band)
        c["spectrum_kept"] = kept / w.N
    return c


def parse_band(text: Optional[str]) -> Optional[list]:
    return None if not text else [int(x) for x in text.split(",")]


def band_mask_for(w: W.Workload, band: Optional[list]):
    """The oracle's 0/1 pattern for a frequency-sparse run (None: dense)."""
    if band is None:
        return None
    import oracle
    import fft_long_convolution_gb300 as F
    info = F.query(w.N, F.F16 if w.dtype == "fp16" else F.BF16)
    return oracle.band_mask(w.N, info["factors"], band)


def run_backward(args, w: W.Workload):
    """One step = the input gradient (through the forward kernels with the
    adjoint spectrum) and the kernel gradient (float32 spectral path) of the
    workload, inputs and output gradient resident on the device."""
    import torch
    import fft_long_convolution_gb300 as F
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    F.build_library()
    ins = W.make_inputs(w, seed=rank)
    dy_in = W.make_inputs(dataclasses.replace(w, gated=False), seed=rank + 1000)["u"]  # the output gradient
    tdt = torch.float16 if w.dtype == "fp16" else torch.bfloat16

    def dev_t(r):
        if r.dtype == "fp32":
            return torch.from_numpy(r.bits).to(dev)
        return torch.from_numpy(r.bits.view(np.int16)).view(tdt).to(dev)

    plan = F.Plan(w.N, tdt)
    kfa = plan.kernel_fft_adjoint(dev_t(ins["k"]))
    u, dy = dev_t(ins["u"]), dev_t(dy_in)
    wi = dev_t(ins["w_in"]) if w.gated else None
    wo = dev_t(ins["w_out"]) if w.gated else None
    du = torch.empty_like(u)
    dk = torch.empty(w.H, w.N, dtype=torch.float32, device=dev)
    L = F.lib()
    need = int(L.fftconv_backward_dk_scratch_bytes(plan._h, w.B, w.H))
    scratch = torch.empty(need, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        plan.backward_du(dy, kfa, wi, wo, du=du, stream=stream)
        F._check(L.fftconv_backward_dk(plan._h, u.data_ptr(), dy.data_ptr(), F._ptr(wi), F._ptr(wo), dk.data_ptr(),
                                       w.B, w.H, scratch.data_ptr(), need, stream.cuda_stream), "fftconv_backward_dk")

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = max(1, min(args.steps, 50))
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / steps
    assert plan.device_status() == 0
    ms = max_over_ranks(ms, world, dev)
    if rank == 0:
        peaks = measured_peaks()
        s = 2
        rows = w.rows
        nbytes = rows * w.N * s * (3 + (2 if w.gated else 0)) + w.H * w.N * 4 + w.H * (w.N + 1) * 4
        Ld = 2 * w.N
        if Ld <= 8192:  # whole channels in shared memory
            dk_kernels, dk_launches = "dk_channel_smem", 1
        elif Ld <= 65536:  # four-step: batch-summed pairs of sub-rows, then the inverse columns
            dk_kernels, dk_launches = "dk_rows + dk_cols_inv", 2
        else:  # four-step with the column transforms through HBM
            dk_kernels, dk_launches = "dk_colfft_fwd + dk_rows + dk_colfft_inv", 3
        launches = path_of(plan.info)["launches_per_step"] + dk_launches
        achieved = nbytes / (ms * 1e-3) / 1e9
        out = {"metric": METRIC + " (backward: du + dk)", "value": job_value(w.outputs, world, ms),
               "unit": "outputs/s", "n_gpus": world, "steps": steps, "warmup": max(args.warmup, 3),
               "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
               "dtype": {"fp16": "f16", "bf16": "bf16"}[w.dtype], "data": "synthetic",
               "config": config_of(w),
               "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                            "algorithmic_bytes_per_launch": nbytes,
                            "kernel": "du: " + path_of(plan.info)["kernel"] + "; dk: " + dk_kernels},
               "gpu_launches": steps * launches, "clocks": clk}
        print(json.dumps(out))
    if world > 1:
        torch.distributed.destroy_process_group()


def run_circular(args, w: W.Workload):
    """The circular convolution of length C = the workload's N, B, H and
    dtype: the native circular plan (C/2 complex points, every outer row in
    and out) against the windowed form on a causal plan of length 2C (outputs
    [C, 2C) of the causal convolution of [u, u] with [k, 0]).  One line with
    the native time as the value and the windowed time beside it."""
    import torch
    import fft_long_convolution_gb300 as F
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    F.build_library()
    ins = W.make_inputs(w, seed=rank)
    tdt = torch.float16 if w.dtype == "fp16" else torch.bfloat16

    def dev_t(r):
        if r.dtype == "fp32":
            return torch.from_numpy(r.bits).to(dev)
        return torch.from_numpy(r.bits.view(np.int16)).view(tdt).to(dev)

    C = w.N
    k = dev_t(ins["k"])  # C taps
    u = dev_t(ins["u"])
    wi = dev_t(ins["w_in"]) if w.gated else None
    wo = dev_t(ins["w_out"]) if w.gated else None
    y = torch.empty_like(u)
    stream = torch.cuda.current_stream()
    native = F.Plan(C, tdt, circular=True)
    kf_n = native.kernel_fft(k)
    win = F.Plan(2 * C, tdt)
    kf_w = win.kernel_fft_partial(k)

    def step_native():
        if w.gated:
            native.forward_gated(u, wi, wo, kf_n, y=y, stream=stream)
        else:
            native.forward(u, kf_n, y=y, stream=stream)

    def step_windowed():
        win.forward_circular(u, kf_w, wi, wo, y=y, stream=stream)

    def timed(step, steps):
        for _ in range(max(args.warmup, 3)):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    steps = max(1, min(args.steps, 200))
    ms_w = timed(step_windowed, steps)
    clocks = ClockSampler(local)
    ms = timed(step_native, steps)
    clk = clocks.stop()
    assert native.device_status() == 0 and win.device_status() == 0
    ms = max_over_ranks(ms, world, dev)
    if rank == 0:
        peaks = measured_peaks()
        nbytes = w.rows * C * 2 * (2 + (2 if w.gated else 0)) + native.kf_bytes(w.H)
        achieved = nbytes / (ms * 1e-3) / 1e9
        fac = native.info["factors"]
        fused = native.info["path"] == F.PATH_FUSED
        kern = ("ftc_conv_kernel (circular rows, R0 = 2)" if fused
                else "otc_pass (A, all rows) + mp_pass_b_tc + otc_pass (C, all rows)")
        out = {"metric": METRIC + " (circular convolution)", "value": job_value(w.outputs, world, ms),
               "unit": "outputs/s", "n_gpus": world, "steps": steps, "warmup": max(args.warmup, 3),
               "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
               "dtype": {"fp16": "f16", "bf16": "bf16"}[w.dtype], "data": "synthetic",
               "config": dict(config_of(w), circular_length=C, factors=fac),
               "windowed_2C_ms_per_step": ms_w,
               "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                            "algorithmic_bytes_per_launch": nbytes,
                            "kernel": kern},
               "gpu_launches": steps * (1 if fused else 3), "clocks": clk}
        print(json.dumps(out))
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(W.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--band", default=None,
                    help="frequency-sparse forward: one band per plan factor, comma separated (e.g. 16,33,33)")
    ap.add_argument("--pass", dest="which", default="forward", choices=["forward", "backward", "circular"],
                    help="backward: input and kernel gradients (du + dk) per step; circular: the circular "
                         "convolution of length N (native plan, with the windowed 2N form timed beside it)")
    ap.add_argument("--order", type=int, default=0,
                    help="the plan's factorization order (0: the default per length; see fftconv_plan_query)")
    ap.add_argument("--batch", type=int, default=None,
                    help="run the workload with this batch size instead of its own (small cases for profiler "
                         "captures; the benchmark is quoted on the workload's own size)")
    args = ap.parse_args()
    w = W.WORKLOADS[args.workload]
    if args.batch is not None:
        w = W.scaled(w, B=args.batch)
    if args.impl == "reference":
        run_reference(args, w)
        return
    if args.which == "backward":
        run_backward(args, w)
        return
    if args.which == "circular":
        run_circular(args, w)
        return

    import torch
    import fft_long_convolution_gb300 as F

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    F.build_library()

    ins = W.make_inputs(w, seed=rank)
    tdt = torch.float16 if w.dtype == "fp16" else torch.bfloat16

    def dev_t(r):
        if r.dtype == "fp32":
            return torch.from_numpy(r.bits).to(dev)
        return torch.from_numpy(r.bits.view(np.int16)).view(tdt).to(dev)

    band = parse_band(args.band)
    plan = F.Plan(w.N, tdt, order=args.order, band=band)
    bd = plan.band()
    path = path_of(plan.info, bd["pairs_run"] if band is not None else None,
                   bd["pairs_total"] if band is not None else None)
    k = dev_t(ins["k"])
    kf = plan.kernel_fft(k)
    # the kernel spectrum is computed once per set of weights (outside the
    # step); its time is reported beside the step
    torch.cuda.synchronize()
    kf_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    kf_ev[0].record()
    for _ in range(3):
        plan.kernel_fft(k, k_f=kf)
    kf_ev[1].record()
    torch.cuda.synchronize()
    kernel_fft_ms = kf_ev[0].elapsed_time(kf_ev[1]) / 3
    u = dev_t(ins["u"])
    wi = dev_t(ins["w_in"]) if w.gated else None
    wo = dev_t(ins["w_out"]) if w.gated else None
    y = torch.empty_like(u)
    stream = torch.cuda.current_stream()
    alg = algorithmic(w)
    flush = None if alg["bytes"] > L2_BYTES else torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        if w.gated:
            plan.forward_gated(u, wi, wo, kf, y=y, stream=stream)
        else:
            plan.forward(u, kf, y=y, stream=stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        step()
    barrier()
    clocks = ClockSampler(local)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    kernel_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = t_start.elapsed_time(t_end)
    step_ms = sum(kernel_ms) / len(kernel_ms) if flush is not None else total_ms / args.steps
    assert plan.device_status() == 0
    step_ms_max = max_over_ranks(step_ms, world, dev)
    value = job_value(w.outputs, world, step_ms_max)

    # end to end through the public API with host buffers (pinned)
    hu = torch.from_numpy(ins["u"].bits.view(np.int16)).view(tdt).pin_memory()
    hwi = torch.from_numpy(ins["w_in"].bits.view(np.int16)).view(tdt).pin_memory() if w.gated else None
    hwo = torch.from_numpy(ins["w_out"].bits.view(np.int16)).view(tdt).pin_memory() if w.gated else None
    hy = torch.empty_like(hu).pin_memory()
    h2d = hu.numel() * 2 * (3 if w.gated else 1)
    d2h = hy.numel() * 2

    def e2e_step():  # the library's host-buffer call: chunked copies overlapped with the convolution
        if w.gated:
            plan.forward_host(hu, kf, hwi, hwo, y=hy, stream=stream)
        else:
            plan.forward_host(hu, kf, y=hy, stream=stream)

    for _ in range(2):
        e2e_step()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_steps = max(3, min(args.steps, 10))
    e0.record(stream)
    for _ in range(e_steps):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e_steps
    e2e_value = job_value(w.outputs, world, max_over_ranks(e2e_ms, world, dev))

    if rank == 0:
        peaks = measured_peaks()
        kern_s = (sum(kernel_ms) / len(kernel_ms)) * 1e-3
        achieved = alg["bytes"] / kern_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic(w.name if band is None else f"{w.name}[band={','.join(map(str, band))}]"),
                "peak_source": peaks["source"] + " hbm_gbs (copy)",
                "algorithmic_bytes_per_launch": alg["bytes"],
                "tensor_frac": alg["flops"] / kern_s / 1e12 / peaks["bf16_tflops"],
                "kernel": path["kernel"]}
        out = {
            "metric": METRIC, "value": value, "unit": "outputs/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": step_ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": {"fp16": "f16", "bf16": "bf16"}[w.dtype],
            "data": "synthetic (seeded SplitMix64 / Box-Muller, see workloads/)",
            "config": dict(config_of(w, band, plan.info["factors"]), factors=plan.info["factors"],
                           order=plan.info["order"]), "roofline": roof,
            "gpu_launches": args.steps * path["launches_per_step"],
            "e2e": {"value": e2e_value, "unit": "outputs/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "clocks": clk,
            "kernel_fft_ms": kernel_fft_ms,
        }
        if not args.no_cpu_baseline and world == 1:
            import oracle
            oracle.build()
            out["cpu_baseline"] = cpu_baseline(w, ins, mask=band_mask_for(w, band))
        if band is not None:
            out["config"]["pairs_run"] = bd["pairs_run"]
            out["config"]["pairs_total"] = bd["pairs_total"]
        print(json.dumps(out))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
