"""FusedConv benchmark: one JSON line on stdout.

A step is one pass of the whole FusedConv suite: the eleven synthetic convolutions of
the five benchmark workloads (2-D fp32 3->8; 1-D fp16 dilated SAME_UPPER +B+Z; the
fp16 residual-CNN 3x3 stack at batch 512; the fp16 vision-encoder stem patch-embed,
depthwise 7x7 and strided downsample; the fp16 3-D strided SAME_LOWER conv, dense and
grouped), each auto-planned by the library exactly as a user call would be. Inputs are
resident in HBM; L2 is flushed (a 256 MiB memset) before every step, outside the timed
events. `value` = algorithmic FLOPs of all ranks / the max over ranks of the device time.

Also reported: per-conv TFLOP/s, GB/s and roofline fractions (CUDA events around every
conv launch on the launching stream), the roofline of the dominant launch, the
end-to-end throughput through the public API with pinned host buffers (H2D of every
input and D2H of every output inside the timed region), the CPU oracle's throughput on
the host cores, and SM clocks sampled during the timed region.

`--impl reference` times the CPU oracle (the only reference this operator has) on the
host cores, on bounded batch-1 samples of the same convolutions.
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
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "FusedConv TFLOP/s (fp16/fp32) and % of roofline per config; depthwise GB/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# CUDA-core f32 FMA peak of a GB300: 152 SMs x 128 FMA lanes x 2 FLOP per FMA x the
# maximum SM clock (2070 MHz) = 80.5 TFLOP/s. The depthwise, grouped, direct and transposed
# routes compute on these lanes, so their compute roofline is this one, not the tensor
# cores'.
SMS, FMA_LANES_PER_SM, SM_MAX_MHZ = 152, 128, 2070.0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = dict(json.load(open(p)))
        kind = "measured"
    else:
        d, kind = dict(PEAKS_FALLBACK), "fallback"
    mhz = float(d.get("sm_max_mhz", SM_MAX_MHZ))
    d["alu_f32_tflops"] = SMS * FMA_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
    return d, kind


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks of the initialised process group (a job takes as
    long as its slowest rank). NCCL reduces a tensor on `device`, other backends on the
    host; with one rank (or no process group) the value itself."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    on = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=on)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step: float, ranks: int, steps: int, ms: float) -> float:
    """Whole-job throughput of `ranks` replicas that each ran `steps` steps of
    `flops_per_step` in `ms` milliseconds (the slowest rank's time)."""
    return flops_per_step * ranks * steps / (ms * 1e-3) / 1e12


def copy_link_gbs(dev, h2d_s, d2h_s, mib: int = 256, reps: int = 3) -> float:
    """Host<->device rate (GB/s, both directions together) of pinned copies running at the
    same time on the two copy streams: the bound of the end-to-end step's data movement."""
    import torch
    n = mib << 20
    hs = torch.empty(n, dtype=torch.uint8).pin_memory()
    hd = torch.empty(n, dtype=torch.uint8).pin_memory()
    ds = torch.empty(n, dtype=torch.uint8, device=dev)
    dd = torch.empty(n, dtype=torch.uint8, device=dev)
    cur = torch.cuda.current_stream(dev)

    def both():
        h2d_s.wait_stream(cur)
        d2h_s.wait_stream(cur)
        with torch.cuda.stream(h2d_s):
            ds.copy_(hs, non_blocking=True)
        with torch.cuda.stream(d2h_s):
            hd.copy_(dd, non_blocking=True)
        cur.wait_stream(h2d_s)
        cur.wait_stream(d2h_s)

    both()
    torch.cuda.synchronize()
    best = 0.0
    for _ in range(3):  # the best of three trials: the rate the link sustains
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for _ in range(reps):
            both()
        b.record(cur)
        torch.cuda.synchronize()
        best = max(best, 2.0 * n * reps / (a.elapsed_time(b) * 1e-3) / 1e9)
    return best


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples with host timestamps."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
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

    def summary(self, t0: float, t1: float):
        win = [p for (t, p) in self.samples if t0 <= t <= t1]
        if not win:
            win = [p for (_, p) in self.samples]
        if not win:
            return None

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(win)}


def oracle_tensors(case):
    """Inputs of one conv for the CPU legs (the oracle derives Y's shape for Z)."""
    import oracle
    ys = oracle.output_shape(case.x_shape, case.w_shape, **case.attrs())
    return workloads.make_inputs(case, ys), ys


CUDA_CORE_ROUTES = ("depthwise", "grouped", "direct", "transposed")


def bound_of(flops, bytes_, peaks, route="igemm_tc"):
    """The roofline a launch sits under: its compute units' peak (tensor cores, or the f32
    FMA lanes for the CUDA-core routes) against the measured HBM copy rate."""
    comp = peaks["alu_f32_tflops"] if route in CUDA_CORE_ROUTES else peaks["bf16_tflops"]
    ridge = comp * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if flops / bytes_ < ridge:
        return "hbm"
    return "alu" if route in CUDA_CORE_ROUTES else "tensor"


def compute_peak(bound, peaks):
    return peaks["alu_f32_tflops"] if bound == "alu" else peaks["bf16_tflops"]


# fp32 convolutions on the tensor cores issue three TF32 MMAs per product (3xTF32 split): their
# peak is the TF32 rate (the measured bf16 rate x the nominal TF32/bf16 ratio 1.1/2.25) / 3.
TF32_OVER_BF16 = 1.1 / 2.25


def tf32x3_peak(peaks):
    return peaks["bf16_tflops"] * TF32_OVER_BF16 / 3.0


def dw_streams(case, plan) -> bool:
    """Whether a depthwise plan runs the column-streaming kernel: 2-D, stride 1, dilation 1,
    K in {3, 5, 7}, the same-size left pad modulo 4, rows of X and Y in whole 4-element
    vectors (the library's rule, in either precision; the bench's buffers are aligned)."""
    if len(case.x_shape) != 4:
        return False
    k = case.w_shape[-1]
    ones = lambda v: v is None or all(e == 1 for e in v)
    return (case.w_shape[-2] == k and k in (3, 5, 7) and ones(case.strides)
            and ones(case.dilations) and (plan.pad_begin[2] - (k - 1) // 2) % 4 == 0
            and case.x_shape[3] % 4 == 0 and plan.y_shape[3] % 4 == 0)


def main_kernel_name(case, route, plan=None):
    """The kernel that does the conv's arithmetic (the TMA-fed implicit GEMM takes
    C/group a multiple of 64; other tensor-core convs build A from the input patch)."""
    if route == "igemm_tc":
        return "igemm_tma_kernel" if case.w_shape[1] % 64 == 0 else "igemm_patch_kernel"
    if route == "depthwise":
        return "dw_stream_kernel" if plan is not None and dw_streams(case, plan) else "dw_tile_kernel"
    return {"direct": "direct_conv_kernel", "grouped": "grouped_kernel"}[route]


def measure_next_rows(dev, stream, flush, peaks):
    """Rows beyond the suite, timed after it and outside its value: each workload of
    workloads.TRANSPOSED_CASES through the library's transposed route, L2 flushed before
    every run, CUDA events on the launching stream."""
    import torch
    import activation_implicit_gemm_gb300 as fc
    from activation_implicit_gemm_gb300 import _lib
    rows = []
    for case in workloads.TRANSPOSED_CASES:
        dt = _lib.F16 if case["dtype"] == "f16" else _lib.F32
        plan = fc.FusedConvPlan(dt, case["x_shape"], case["w_shape"], has_bias=True,
                                has_z=True, transposed=True, **case["attrs"])
        t = workloads.make_transposed_inputs(case, plan.y_shape)
        d = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in t.items()}
        y = torch.empty(plan.y_shape, dtype=d["x"].dtype, device=dev)
        reps = 10
        for _ in range(3):
            plan.run(d["x"], d["w"], d["b"], d["z"], y=y, stream=stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            plan.run(d["x"], d["w"], d["b"], d["z"], y=y, stream=stream)
            b.record(stream)
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in ev) / reps
        tf = plan.flops / (ms * 1e-3) / 1e12
        bnd = bound_of(plan.flops, plan.bytes, peaks, plan.route)
        frac = (tf / compute_peak(bnd, peaks) if bnd in ("tensor", "alu")
                else plan.bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"])
        rows.append({"row": "NEXT-4 transposed convolution (gather form)", "conv": case["name"],
                     "route": plan.route, "us": round(ms * 1e3, 2), "tflops": round(tf, 2),
                     "gbs": round(plan.bytes / (ms * 1e-3) / 1e9, 1), "bound": bnd,
                     "frac_of_bound": round(frac, 4), "flops": plan.flops,
                     "bytes": plan.bytes, "kernel": "convt_kernel"})
    # the opt-in half2 row-partial mode of the depthwise kernel on the stem's depthwise conv
    case = workloads.case_by_name("stem_dw_128_k7")
    times = {}
    for prec in ("default", "half2_rows"):
        plan = fc.FusedConvPlan(_lib.F16, case.x_shape, case.w_shape, has_bias=case.has_bias,
                                has_z=case.has_z, precision=prec, **case.attrs())
        if prec == "default":
            t = workloads.make_inputs(case, plan.y_shape)
            d = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in t.items()}
            y = torch.empty(plan.y_shape, dtype=torch.float16, device=dev)
        for _ in range(3):
            plan.run(d["x"], d["w"], d["b"], d["z"], y=y, stream=stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(10)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            plan.run(d["x"], d["w"], d["b"], d["z"], y=y, stream=stream)
            b.record(stream)
        torch.cuda.synchronize()
        times[prec] = (plan, sum(a.elapsed_time(b) for a, b in ev) / 10)
    plan, ms = times["half2_rows"]
    tf = plan.flops / (ms * 1e-3) / 1e12
    rows.append({"row": "NEXT-2 half2 row partials (depthwise, opt-in precision)",
                 "conv": case.name, "route": plan.route, "us": round(ms * 1e3, 2),
                 "tflops": round(tf, 2), "gbs": round(plan.bytes / (ms * 1e-3) / 1e9, 1),
                 "frac_of_hbm": round(plan.bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                 "default_precision_us": round(times["default"][1] * 1e3, 2),
                 "speedup_vs_default": round(times["default"][1] / ms, 3),
                 "kernel": "dw_stream_kernel<__half, 7, 1, true>",
                 "error": "bounded by f16 rounding + 7 * 2^-11 * sum|x*w| (tests/test_gpu_half2.py)"})
    for case in workloads.PATCHIFY_CASES:
        y_shape = fc.FusedConvPlan(_lib.F16, case.x_shape, case.w_shape, has_bias=case.has_bias,
                                   has_z=case.has_z, **case.attrs()).y_shape
        t = workloads.make_inputs(case, y_shape)
        d = {k: (None if v is None else torch.from_numpy(np.ascontiguousarray(v)).to(dev))
             for k, v in t.items()}
        res = {}
        for route, reps in (("auto", 10), ("direct", 2)):
            plan = fc.FusedConvPlan(_lib.F16, case.x_shape, case.w_shape, has_bias=case.has_bias,
                                    has_z=case.has_z, route=route, **case.attrs())
            y = torch.empty(plan.y_shape, dtype=torch.float16, device=dev)
            wsb = (torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
                   if plan.workspace_bytes else None)
            for _ in range(2):
                plan.run(d["x"], d["w"], d["b"], d["z"], y=y, workspace=wsb, stream=stream)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(reps)]
            for a, b in ev:
                flush.zero_()
                a.record(stream)
                plan.run(d["x"], d["w"], d["b"], d["z"], y=y, workspace=wsb, stream=stream)
                b.record(stream)
            torch.cuda.synchronize()
            res[route] = (plan, sum(a.elapsed_time(b) for a, b in ev) / reps)
        plan, ms = res["auto"]
        bnd = bound_of(plan.flops, plan.bytes, peaks, plan.route)
        ach = (plan.flops / (ms * 1e-3) / 1e12 if bnd == "tensor"
               else plan.bytes / (ms * 1e-3) / 1e9)
        pk = peaks["bf16_tflops"] if bnd == "tensor" else peaks["hbm_gbs"]
        rows.append({"row": "NEXT-3 stride == kernel (patchify)", "conv": case.name,
                     "route": plan.route, "us": round(ms * 1e3, 2),
                     "tflops": round(plan.flops / (ms * 1e-3) / 1e12, 2),
                     "gbs": round(plan.bytes / (ms * 1e-3) / 1e9, 1), "bound": bnd,
                     "frac_of_bound": round(ach / pk, 4), "kernel": "igemm_patch_kernel",
                     "cuda_core_route_us": round(res["direct"][1] * 1e3, 2),
                     "speedup_vs_cuda_cores": round(res["direct"][1] / ms, 1)})
    for case in workloads.FP32_TC_CASES:
        t = workloads.make_inputs(case, fc.FusedConvPlan(
            _lib.F32, case.x_shape, case.w_shape, has_bias=case.has_bias, has_z=case.has_z,
            **case.attrs()).y_shape)
        d = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in t.items()}
        res = {}
        for route, reps in (("auto", 10), ("direct", 3)):
            plan = fc.FusedConvPlan(_lib.F32, case.x_shape, case.w_shape, has_bias=True,
                                    has_z=True, route=route, **case.attrs())
            y = torch.empty(plan.y_shape, dtype=torch.float32, device=dev)
            wsb = (torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
                   if plan.workspace_bytes else None)
            for _ in range(2):
                plan.run(d["x"], d["w"], d["b"], d["z"], y=y, workspace=wsb, stream=stream)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(reps)]
            for a, b in ev:
                flush.zero_()
                a.record(stream)
                plan.run(d["x"], d["w"], d["b"], d["z"], y=y, workspace=wsb, stream=stream)
                b.record(stream)
            torch.cuda.synchronize()
            res[route] = (plan, sum(a.elapsed_time(b) for a, b in ev) / reps)
        plan, ms = res["auto"]
        tf = plan.flops / (ms * 1e-3) / 1e12
        pk = tf32x3_peak(peaks)
        rows.append({"row": "NEXT-1 fp32 on the tensor cores (3xTF32)", "conv": case.name,
                     "route": plan.route, "launches": plan.launches, "us": round(ms * 1e3, 2),
                     "tflops": round(tf, 2), "bound": "tensor", "peak_tflops": round(pk, 1),
                     "peak_kind": "measured bf16 x nominal TF32/bf16 (1.1/2.25) / 3 MMAs",
                     "frac_of_bound": round(tf / pk, 4), "flops": plan.flops,
                     "kernel": "igemm_tf32_kernel",
                     "cuda_core_route_us": round(res["direct"][1] * 1e3, 2),
                     "speedup_vs_cuda_cores": round(res["direct"][1] / ms, 1)})
    return rows


def run_ours(args):
    import torch
    import torch.distributed as dist

    ws_n, rank, local = dist_env()
    if ws_n > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import activation_implicit_gemm_gb300 as fc
    from activation_implicit_gemm_gb300 import _lib
    fc.build()
    peaks, peaks_kind = load_peaks()

    convs = []
    cases = workloads.ALL_CASES
    if args.conv:
        cases = [workloads.case_by_name(n) for n in args.conv.split(",")]
    for case in cases:
        dt = _lib.F16 if case.dtype == "f16" else _lib.F32
        plan = fc.FusedConvPlan(dt, case.x_shape, case.w_shape, has_bias=case.has_bias,
                                has_z=case.has_z, device=local, **case.attrs())
        t = workloads.make_inputs(case, plan.y_shape)
        d = {k: (None if v is None else torch.from_numpy(np.ascontiguousarray(v)).to(dev))
             for k, v in t.items()}
        h = {k: (None if v is None else torch.from_numpy(np.ascontiguousarray(v)).pin_memory())
             for k, v in t.items()}
        tdt = torch.float16 if case.dtype == "f16" else torch.float32
        y = torch.empty(plan.y_shape, dtype=tdt, device=dev)
        yh = torch.empty(plan.y_shape, dtype=tdt).pin_memory()
        wsb = (torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
               if plan.workspace_bytes else None)
        convs.append(dict(case=case, plan=plan, d=d, h=h, y=y, yh=yh, ws=wsb))
    total_flops = sum(c["plan"].flops for c in convs)
    launches_per_step = sum(c["plan"].launches for c in convs)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        for i, c in enumerate(convs):
            if evs is not None:
                evs[i].record(stream)
            d = c["d"]
            c["plan"].run(d["x"], d["w"], d["b"], d["z"], y=c["y"], workspace=c["ws"],
                          stream=stream)
        if evs is not None:
            evs[len(convs)].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    K = args.steps
    # the timed steps carry events only at their ends, so each conv's kernels follow the
    # previous conv's as they would in a user's stream (programmatic dependent launch
    # lets a kernel set itself up while its predecessor drains)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if ws_n > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_host0 = time.time()
    for k in range(K):
        flush.zero_()
        step_ev[k][0].record(stream)
        step()
        step_ev[k][1].record(stream)
    torch.cuda.synchronize()
    if ws_n > 1:
        dist.barrier()
    t_host1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    clocks = sampler.summary(t_host0, t_host1)

    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    dev_ms = max_over_ranks(sum(step_ms), dev)
    ms_per_step = dev_ms / K
    value = job_tflops(total_flops, ws_n, K, dev_ms)

    # per-conv breakdown and the dominant launch's roofline, from a separate pass with an
    # event between convs (each conv then starts from an idle stream)
    Kc = min(K, 100)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(convs) + 1)]
          for _ in range(Kc)]
    for k in range(Kc):
        flush.zero_()
        step(ev[k])
    torch.cuda.synchronize()
    per_conv_ms = [sum(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(Kc))
                   for i in range(len(convs))]
    per = []
    for i, c in enumerate(convs):
        p = c["plan"]
        ms = per_conv_ms[i] / Kc
        fl, by = p.flops, p.bytes
        bnd = bound_of(fl, by, peaks, p.route)
        tf = fl / (ms * 1e-3) / 1e12
        gbs = by / (ms * 1e-3) / 1e9
        if bnd in ("tensor", "alu"):
            frac = tf / compute_peak(bnd, peaks)
        else:
            frac = gbs / peaks["hbm_gbs"]
        comp = peaks["alu_f32_tflops"] if p.route in CUDA_CORE_ROUTES else peaks["bf16_tflops"]
        attain = min(comp * 1e12, fl / by * peaks["hbm_gbs"] * 1e9) / 1e12
        per.append({"conv": c["case"].name, "route": p.route, "tile_n": p.tile_n,
                    "split_k": p.split_k, "us": round(ms * 1e3, 2), "tflops": round(tf, 2),
                    "gbs": round(gbs, 1), "bound": bnd, "frac_of_bound": round(frac, 4),
                    "frac_of_fp16_peak": round(tf / peaks["bf16_tflops"], 4),
                    "frac_of_attainable": round(tf / attain, 4)})
    top = max(range(len(convs)), key=lambda i: per_conv_ms[i])
    tp = convs[top]["plan"]
    tms = per_conv_ms[top] / Kc
    tb = bound_of(tp.flops, tp.bytes, peaks, tp.route)
    if tb in ("tensor", "alu"):
        ach, pk, unit = tp.flops / (tms * 1e-3) / 1e12, compute_peak(tb, peaks), "TFLOP/s"
    else:
        ach, pk, unit = tp.bytes / (tms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s"
    traffic = load_traffic(convs[top]["case"].name)
    roofline = {"bound": tb, "achieved": round(ach, 3), "peak": pk, "unit": unit,
                "frac": round(ach / pk, 4), "traffic": traffic,
                "kernel": main_kernel_name(convs[top]["case"], tp.route, tp),
                "launch": convs[top]["case"].name,
                "peak_kind": ("derived: 152 SMs x 128 f32 FMA lanes x 2 FLOP x max SM clock"
                              if tb == "alu" else f"{peaks_kind} (burst)"),
                "algorithmic_flops_per_launch": tp.flops,
                "algorithmic_bytes_per_launch": tp.bytes}

    # end to end through the public API with pinned host buffers
    e2e_steps = max(3, min(20, K))
    h2d = sum(sum(v.numel() * v.element_size() for v in c["h"].values() if v is not None)
              for c in convs)
    d2h = sum(c["yh"].numel() * c["yh"].element_size() for c in convs)

    # Three streams: the inputs of conv i+1 travel host->device and the output of conv i-1
    # device->host while conv i runs. Events order each conv's copies and launch, and keep
    # the next step from overwriting a buffer the previous step still uses.
    h2d_s = torch.cuda.Stream(dev)
    d2h_s = torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in convs]  # conv i's inputs are on the device
    ran = [torch.cuda.Event() for _ in convs]       # conv i has read its inputs, written Y
    out_read = [torch.cuda.Event() for _ in convs]  # conv i's Y has reached the host
    state = {"first": True}

    def e2e_step():
        for i, c in enumerate(convs):
            d, hh = c["d"], c["h"]
            with torch.cuda.stream(h2d_s):
                if not state["first"]:
                    h2d_s.wait_event(ran[i])
                for key in ("x", "w", "b", "z"):
                    if hh[key] is not None:
                        d[key].copy_(hh[key], non_blocking=True)
                in_ready[i].record(h2d_s)
            stream.wait_event(in_ready[i])
            if not state["first"]:
                stream.wait_event(out_read[i])
            c["plan"].run(d["x"], d["w"], d["b"], d["z"], y=c["y"], workspace=c["ws"],
                          stream=stream)
            ran[i].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ran[i])
                c["yh"].copy_(c["y"], non_blocking=True)
                out_read[i].record(d2h_s)
        state["first"] = False

    e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(h2d_s)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(d2h_s)  # after the last output's copy, which follows every other step
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    e2e_value = job_tflops(total_flops, ws_n, e2e_steps, e2e_ms)
    link_gbs = copy_link_gbs(dev, h2d_s, d2h_s)
    # the step cannot end before its bytes have crossed the host link at that rate
    copy_bound = total_flops / ((h2d + d2h) / (link_gbs * 1e9)) / 1e12

    next_rows = [] if args.conv else measure_next_rows(dev, stream, flush, peaks)

    out = {"metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": ws_n,
           "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
           "data": "synthetic (seeded splitmix64/Box-Muller inputs of the benchmark shapes)",
           "config": {"workload": "fusedconv_suite: 11 convs of the 5 benchmark workloads "
                                  "(2-D fp32 3->8 k3; 1-D fp16 64->64 k5 d2 SAME_UPPER +B+Z; "
                                  "3x3 CNN stack N=512 3->64@32, 64->128@16 +Z, 128->256@8, "
                                  "256->512@4 +Z QuickGelu; stem patch k7 s4 +B Gelu, "
                                  "depthwise k7 +B+Z Clip, downsample k2 s2; 3-D k3 s2 "
                                  "SAME_LOWER +B HardSwish, dense and group 4 +Z)",
                      "flops_per_step": total_flops, "l2": "flushed before every step "
                      "(256 MiB memset outside the timed events)",
                      "parallelism": f"replicas x{ws_n} (no data-path collective)",
                      "fp32_convs": "the 2-D 3->8 conv computes in fp32",
                      "per_conv_timing": "separate pass of min(steps, 100) steps with an event "
                                         "between convs"},
           "per_conv": per, "roofline": roofline,
           "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s",
                   "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                   "steps": e2e_steps, "api": "FusedConvPlan.run (C ABI fconv_run)",
                   "overlap": "conv i+1's inputs upload and conv i-1's output downloads "
                              "while conv i runs (copy streams ordered by events)",
                   "copy_link_gbs": round(link_gbs, 1),
                   "copy_bound_tflops": round(copy_bound, 3),
                   "frac_of_copy_bound": round(e2e_value / copy_bound, 4),
                   "copy_link": "pinned 256 MiB host->device and device->host copies at the "
                                "same time on the two copy streams, best of three trials in "
                                "this run"},
           "gpu_launches": launches_per_step * K, "clocks": clocks}
    if next_rows:
        out["next_rows"] = next_rows
    if args.conv:
        out["config"]["workload"] = "subset: " + args.conv
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline and not args.conv:
        out["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws_n > 1:
        dist.destroy_process_group()


def strip_comments(src: str) -> str:
    """C/C++/CUDA source without its comments and blank lines (string and character
    literals kept), so that editing a comment does not count as changing a kernel."""
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
        else:
            out.append(c)
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).split("\n")]
    return "\n".join(ln for ln in lines if ln.strip())


def kernel_sources_digest():
    """Digest of the library's code (comments excluded): the committed DRAM counters are
    reported only for the code they were measured on."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "activation_implicit_gemm_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h", ".cpp")):
            h.update(f.encode() + b"\0")
            h.update(strip_comments(open(os.path.join(csrc, f)).read()).encode())
    return h.hexdigest()[:16]


def load_traffic(conv_name):
    """DRAM bytes of one launch of this conv's main kernel from the committed ncu summary,
    or None when there is none or the kernel sources changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_sources_sha256_16") != kernel_sources_digest():
        return None
    return d.get("per_launch_bytes", {}).get(conv_name)


def cpu_baseline():
    """The oracle, as it stands, on the host cores over the whole suite (one pass)."""
    import oracle
    flops = 0.0
    secs = 0.0
    for case in workloads.ALL_CASES:
        t, _ = oracle_tensors(case)
        t0 = time.perf_counter()
        y, _ = oracle.fused_conv(t["x"], t["w"], t["b"], t["z"], **case.attrs())
        secs += time.perf_counter() - t0
        flops += 2.0 * y.size * np.prod(case.w_shape[1:])
        if secs > 60.0:
            break
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s",
            "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"one pass over the suite's convolutions at full size "
                      f"({flops / 1e9:.1f} GFLOP, {secs:.1f} s, fp64 direct loops, OpenMP)"}


def run_reference(args):
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    cases = workloads.ALL_CASES
    samples = []
    for case in cases:
        ys = oracle.output_shape(case.x_shape, case.w_shape, **case.attrs())
        t = workloads.make_inputs(case, ys, batch=1)
        samples.append((case, t))
    flops = 0.0
    secs = 0.0
    for k in range(args.warmup + args.steps):
        case, t = samples[k % len(samples)]
        t0 = time.perf_counter()
        y, _ = oracle.fused_conv(t["x"], t["w"], t["b"], t["z"], **case.attrs())
        dt = time.perf_counter() - t0
        if k >= args.warmup:
            secs += dt
            flops += 2.0 * y.size * np.prod(case.w_shape[1:])
    value = flops / secs / 1e12
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
           "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(secs * 1e3 / args.steps, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded, same generator as the GPU arm)",
           "config": {"workload": "fusedconv_suite: 11 convs of the 5 benchmark workloads; "
                                  "each step one conv, batch-1 sample, round robin"},
           "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s",
                            "cores": oracle.max_threads(), "kind": "oracle",
                            "sample": "batch-1 sample of one suite conv per step"},
           "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--conv", default="",
                    help="comma-separated conv names: time only these (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
