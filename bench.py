#!/usr/bin/env python3
"""Benchmark of the strided batched fp32 product on GB300.

One step = the large projection sweep, four products through the C-ABI on one
stream, each over resident synthetic inputs:
    c5a  8192 x 960  -> 2560, W[2560,960] read transposed by strides
    c5b  8192 x 2560 -> 960,  W[960,2560] read transposed by strides
    c5c  4096^3, row-major, accumulate into C
    c5d  4096^3, A and B read transposed by swapped strides, accumulate
(`--workload` selects another workload of the same set instead).

Prints ONE JSON line: GFLOP/s of the timed steps (2*M*N*K*batch per product),
the dominant kernel's roofline fraction, the CPU oracle timed on a bounded
sample, an end-to-end figure with host buffers, and the SM clocks sampled
while the timed steps ran.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--math fp32|tf32]
                    [--workload c5|c1|...] [--impl ours|reference]
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "GFLOP/s of strided batched fp32 GEMM; % of FP32 (or TF32 TC) peak, 1×GB300"
L2_BYTES = 129 * 1024 * 1024
FP32_FLOP_PER_CLK_PER_SM = 256      # 128 FP32 lanes x 2 flop per FMA
TF32_OVER_BF16_NOMINAL = 1.1 / 2.25  # dense nominal tf32 / bf16 tensor rates
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0}

SWEEPS = {"c5": ["c5a", "c5b", "c5c", "c5d"], "c3all": ["c3", "c3gqa"],
          "f1": list(wl.BACKWARD), "f4": ["f4spec", "f4dist"]}
DESCR = {
    "c5": "large projection sweep: 8192x960->2560 (W^T), 8192x2560->960 (W^T), "
          "4096^3 row-major +C, 4096^3 A^T B^T +C",
    "f1": "backward products of the two projection layers: dX = G W (8192x960x2560, "
          "8192x2560x960), dW += G^T X (2560x960x8192, 960x2560x8192)",
    "f4": "spectrogram basis product (64 clips, overlapping 512-sample frames every 128, "
          "x 512x514 windowed DFT basis) and codebook distances (8192 x 4096 x 256)",
}


# ---------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group("gloo")
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(flops_per_step: int, world: int, steps: int, ms_slowest: float) -> float:
    """Whole-job GFLOP/s: every rank runs the full step (replicas), so the job
    does world x steps steps in the slowest rank's time."""
    return flops_per_step * world * steps / (ms_slowest * 1e-3) / 1e9


# ---------------------------------------------------------------- peaks, clocks

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons in the background."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None, period_ms: int = 100):
        self.rows = []
        self.proc = None
        self.marks = []
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
               "-lms", str(period_ms)]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def wait_first(self, timeout=5.0):
        t0 = time.time()
        while self.proc is not None and not self.rows and time.time() - t0 < timeout:
            time.sleep(0.05)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [r for (t, r) in self.rows if t0 <= t <= t1]
        if not rows:
            rows = [r for (_, r) in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if len(r) > 5 + i and r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(rows)}


def gpu_uuid(torch):
    try:
        u = torch.cuda.get_device_properties(torch.cuda.current_device()).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


# ---------------------------------------------------------------- workloads

def workload_cases(name):
    names = SWEEPS.get(name, [name])
    return names, [wl.make(n, "real") for n in names]


def case_args(case, dA, dB, dC):
    return (dA.data_ptr() + 4 * case.A.offset, case.A.rs, case.A.cs, case.A.bs,
            dB.data_ptr() + 4 * case.B.offset, case.B.rs, case.B.cs, case.B.bs,
            dC.data_ptr() + 4 * case.C.offset, case.C.rs, case.C.cs, case.C.bs,
            case.M, case.N, case.K, case.batch, case.alpha, case.accumulate)


def kernel_source_digest(path_name):
    common = ["internal.h", "epilogue.cuh"]
    files = {"gather_ffma": ["ffma_gather.cu"] + common,
             "tma_ffma": ["ffma_tma.cu", "ffma_tma_kernel.cuh", "ffma_tma_256x128.cu", "ffma_tma_128x256.cu",
                          "ffma_tma_512x64.cu", "schedule.cuh", "ptx.cuh"] + common,
             "tma_tf32": ["tf32_tc.cu", "schedule.cuh", "ptx.cuh"] + common,
             "attention": ["attention.cu", "internal.h"],
             "attention_tc": ["attention_tc.cu", "attention_tc.h", "ptx.cuh", "internal.h"],
             "attention_decode": ["attention_decode.cu", "internal.h"]}.get(path_name, [])
    h = hashlib.sha256()
    for f in files:
        p = os.path.join(ROOT, "strided_gemm_gb300", "csrc", f)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(path_name, case_name):
    """DRAM bytes per launch from a committed ncu summary, if its kernel source
    digest still matches the source being timed."""
    p = os.path.join(ROOT, "profiles", f"traffic_{path_name}_{case_name}.txt")
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_source_digest") != kernel_source_digest(path_name):
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- CPU oracle

def host_cpu():
    """The host CPU as /proc/cpuinfo names it (model name, or on Arm the
    implementer and part codes), plus the machine type."""
    fields = {}
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    import platform
    if "model name" in fields:
        name = fields["model name"]
    elif "CPU implementer" in fields:
        name = f"implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    else:
        name = "unknown"
    return f"{name} ({platform.machine()})"


def oracle_sample(cases, seconds_target, threads, rows_override=None):
    """Times the oracle on the first rows of each product.  Returns
    (gflop_per_s, seconds, flops, rows)."""
    import oracle
    oracle.load()

    def run(rows):
        fl = 0
        t0 = time.perf_counter()
        for c in cases:
            r = min(rows, c.M)
            oracle.product(c.A, c.B, c.C, r, c.N, c.K, min(c.batch, 1), c.alpha, c.accumulate,
                           nthreads=threads)
            fl += wl.flops(r, c.N, c.K, min(c.batch, 1))
        return time.perf_counter() - t0, fl

    if rows_override is None:
        dt, fl = run(threads)                         # calibration pass
        rate = fl / max(dt, 1e-6)
        per_row = sum(wl.flops(1, c.N, c.K, 1) for c in cases)
        rows = int(max(threads, min(max(c.M for c in cases),
                                    seconds_target * rate / per_row)))
    else:
        rows = rows_override
    dt, fl = run(rows)
    return fl / dt / 1e9, dt, fl, rows


# ---------------------------------------------------------------- GPU arm

def run_ours(args, world, rank, local, dist):
    import torch
    import strided_gemm_gb300 as sg
    from strided_gemm_gb300 import build as sgbuild

    torch.cuda.set_device(local)
    sgbuild.build()
    sg.load()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    s_handle = stream.cuda_stream
    math = sg.MATH_TF32 if args.math == "tf32" else sg.MATH_FP32
    force = {"auto": sg.PATH_AUTO, "gather": sg.PATH_GATHER_FFMA, "tma": sg.PATH_TMA_FFMA,
             "tf32": sg.PATH_TMA_TF32}[args.path]

    names, cases = workload_cases(args.workload)
    dev_bufs = []
    for c in cases:
        dA = torch.from_numpy(c.A.storage).to(dev)
        dB = torch.from_numpy(c.B.storage).to(dev)
        dC = torch.from_numpy(c.C.storage).to(dev)
        dev_bufs.append((dA, dB, dC))
    calls = [case_args(c, *b) for c, b in zip(cases, dev_bufs)]
    # Caller-owned scratch that lets the planner split the last waves along K.
    ws = None
    ws_kw = {}
    if not args.no_workspace:
        ws = torch.empty(sg.sbgemm_workspace_bytes(local), dtype=torch.uint8, device=dev)
        ws_kw = dict(workspace=ws.data_ptr(), workspace_bytes=ws.numel())
    plans = [sg.sbgemm_plan(*a[:16], c.accumulate, math=math, force_path=force, **ws_kw)
             for c, a in zip(cases, calls)]
    flops_step = sum(c.flops for c in cases)
    bytes_step = sum(wl.alg_bytes(c) for c in cases)
    ws_bytes = sum(c.A.storage.nbytes + c.B.storage.nbytes + c.C.storage.nbytes for c in cases)

    def launch(i, m=None):
        sg.sbgemm_ex(*calls[i], s_handle, math=math if m is None else m,
                     force_path=force if m is None else sg.PATH_AUTO, **ws_kw)

    def step():
        for i in range(len(calls)):
            launch(i)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    sampler = ClockSampler(gpu_uuid(torch))
    sampler.wait_first()
    # Per-launch events for the kernel-level roofline; whole-step events below.
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in calls] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start.record(stream)
    for k in range(args.steps):
        for i in range(len(calls)):
            ev[k][i][0].record(stream)
            launch(i)
            ev[k][i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(dist)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)

    elapsed_ms = start.elapsed_time(end)
    ms_max = max_over_ranks(dist, elapsed_ms)
    ms_per_step = ms_max / args.steps
    value = job_rate(flops_step, world, args.steps, ms_max)

    per = {}
    for i, (n, c) in enumerate(zip(names, cases)):
        ms = [ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(args.steps)]
        avg = sum(ms) / len(ms)
        per[n] = {"ms": round(avg, 4), "gflops": round(c.flops / (avg * 1e-3) / 1e9, 1),
                  "path": plans[i]["path_name"], "tile": [plans[i]["tile_m"], plans[i]["tile_n"]],
                  "stream_k": bool(plans[i]["stream_k"]), "total_ms": sum(ms)}

    # Dominant kernel: the launch (product) with the largest total time.
    dom = max(per, key=lambda n: per[n]["total_ms"])
    dcase = cases[names.index(dom)]
    peaks, peaks_src = measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_max = float(peaks.get("sm_max_mhz") or FALLBACK["sm_max_mhz"])
    dom_path = per[dom]["path"]
    avg_s = per[dom]["ms"] * 1e-3
    if dom_path == "tma_tf32":
        peak = float(peaks.get("bf16_tflops", FALLBACK["bf16_tflops"])) * TF32_OVER_BF16_NOMINAL
        roof = {"bound": "tensor", "achieved": round(dcase.flops / avg_s / 1e12, 2),
                "peak": round(peak, 1), "unit": "TFLOP/s",
                "peak_source": f"{peaks_src} bf16 dense burst x nominal tf32/bf16 ratio "
                               f"{TF32_OVER_BF16_NOMINAL:.3f}"}
    else:
        peak = sms * FP32_FLOP_PER_CLK_PER_SM * sm_max * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": round(dcase.flops / avg_s / 1e12, 2),
                "peak": round(peak, 2), "unit": "TFLOP/s",
                "peak_source": f"{sms} SMs x 256 fp32 flop/clk x {sm_max:.0f} MHz ({peaks_src} max clock)"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    if clocks.get("sm_mhz"):
        roof["frac_at_sampled_clock"] = round(roof["frac"] * sm_max / clocks["sm_mhz"], 4)
    roof["traffic"] = profiled_traffic(dom_path, dom)
    roof["kernel"] = f"{dom_path} ({dom})"
    roof["alg_bytes_per_launch"] = wl.alg_bytes(dcase)
    roof["hbm_frac"] = round(wl.alg_bytes(dcase) / avg_s / 1e9 /
                             float(peaks.get("hbm_gbs", FALLBACK["hbm_gbs"])), 4)

    # End to end through the public API with host buffers: every step copies all
    # of its inputs from pinned host memory, runs the products and reads every
    # C back.  Copies run on two copy streams so that product i+1's inputs move
    # while product i computes and product i's result returns while i+1 runs,
    # and the device operands are double-buffered so that step k+1's inputs
    # move while step k's products run (as a training loop prefetches its next
    # batch).  Every step's copies are inside the timed region.
    e2e = None
    if not args.no_e2e:
        host_in = [(torch.from_numpy(c.A.storage).pin_memory(),
                    torch.from_numpy(c.B.storage).pin_memory(),
                    torch.from_numpy(c.C.storage).pin_memory()) for c in cases]
        host_out = [torch.empty_like(h[2]).pin_memory() for h in host_in]
        h2d = sum(h[0].numel() * 4 + h[1].numel() * 4 + (h[2].numel() * 4 if c.accumulate else 0)
                  for h, c in zip(host_in, cases))
        d2h = sum(h.numel() * 4 for h in host_out)
        n_e2e = max(1, min(args.steps, args.e2e_steps))
        up = torch.cuda.Stream(dev)
        down = torch.cuda.Stream(dev)
        sets = [dev_bufs, [tuple(torch.empty_like(t) for t in bb) for bb in dev_bufs]]
        set_calls = [calls, [case_args(c, *bb) for c, bb in zip(cases, sets[1])]]
        set_free = [None, None]       # the set's last read-back has finished

        def e2e_step(k, start=None):
            bufs, cl = sets[k % 2], set_calls[k % 2]
            if start is not None:
                up.wait_event(start)
            if set_free[k % 2] is not None:
                up.wait_event(set_free[k % 2])
            inputs_ready = []
            with torch.cuda.stream(up):
                for i, c in enumerate(cases):
                    dA, dB, dC = bufs[i]
                    dA.copy_(host_in[i][0], non_blocking=True)
                    dB.copy_(host_in[i][1], non_blocking=True)
                    if c.accumulate:
                        dC.copy_(host_in[i][2], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(up)
                    inputs_ready.append(ev)
            for i, c in enumerate(cases):
                stream.wait_event(inputs_ready[i])
                sg.sbgemm_ex(*cl[i], s_handle, math=math, force_path=force, **ws_kw)
                done = torch.cuda.Event()
                done.record(stream)
                down.wait_event(done)
                with torch.cuda.stream(down):
                    host_out[i].copy_(bufs[i][2], non_blocking=True)
            back = torch.cuda.Event()
            back.record(down)
            set_free[k % 2] = back
            return back

        e2e_step(0)
        e2e_step(1)
        torch.cuda.synchronize()
        barrier(dist)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        last = None
        for k in range(n_e2e):
            last = e2e_step(k, start=e0 if k == 0 else None)
        stream.wait_event(last)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        e_ms = max_over_ranks(dist, e0.elapsed_time(e1))
        e2e = {"value": round(job_rate(flops_step, world, n_e2e, e_ms), 1),
               "unit": "GFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": n_e2e, "ms_per_step": round(e_ms / n_e2e, 3),
               "copies": "pinned host buffers, two copy streams; the device operands are double-buffered, "
                         "so step k+1's inputs upload while step k's products run; every step's inputs "
                         "and every C cross the host link inside the timed region"}
        del sets[1], set_calls[1]

    # The opt-in tensor-core path on the same products (operands TMA cannot
    # fetch fall back to strict fp32 and are reported as such).
    tf32 = None
    if not args.no_tf32 and math == sg.MATH_FP32:
        tf32 = {"per_product": {}}
        reps = max(3, min(args.steps, 20))
        best = None
        for i, (n, c) in enumerate(zip(names, cases)):
            pl = sg.sbgemm_plan(*calls[i][:16], c.accumulate, math=sg.MATH_TF32, **ws_kw)
            for _ in range(3):
                launch(i, sg.MATH_TF32)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(reps):
                launch(i, sg.MATH_TF32)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / reps
            tf32["per_product"][n] = {"ms": round(ms, 4), "gflops": round(c.flops / ms / 1e6, 1),
                                      "path": pl["path_name"]}
            if pl["path_name"] == "tma_tf32" and (best is None or ms > best[1]):
                best = (n, ms, c)
        if best is not None:
            n, ms, c = best
            peak = float(peaks.get("bf16_tflops", FALLBACK["bf16_tflops"])) * TF32_OVER_BF16_NOMINAL
            ach = c.flops / (ms * 1e-3) / 1e12
            tf32["roofline"] = {"bound": "tensor", "kernel": f"tma_tf32 ({n})",
                                "achieved": round(ach, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
                                "frac": round(ach / peak, 4),
                                "peak_source": f"{peaks_src} bf16 dense burst x nominal tf32/bf16 "
                                               f"ratio {TF32_OVER_BF16_NOMINAL:.3f}",
                                "traffic": profiled_traffic("tma_tf32", n)}
            # The rate the hardware demonstrably reaches in tf32, measured
            # here: the vendor library's tf32 GEMM on an 8192^3 row-major
            # product (a comparison denominator only; nothing on the
            # library's path calls it).
            prev = torch.backends.cuda.matmul.allow_tf32
            torch.backends.cuda.matmul.allow_tf32 = True
            try:
                ga = torch.randn(8192, 8192, device=dev)
                gb = torch.randn(8192, 8192, device=dev)
                gc = torch.empty(8192, 8192, device=dev)
                for _ in range(3):
                    torch.matmul(ga, gb, out=gc)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record(stream)
                for _ in range(10):
                    torch.matmul(ga, gb, out=gc)
                e1.record(stream)
                torch.cuda.synchronize()
                lib_tf = 2 * 8192 ** 3 / (e0.elapsed_time(e1) / 10 * 1e-3) / 1e12
                tf32["roofline"]["peak_library_measured"] = round(lib_tf, 1)
                tf32["roofline"]["frac_of_library_measured"] = round(ach / lib_tf, 4)
                tf32["roofline"]["library_measured_source"] = (
                    "torch.matmul tf32 (cuBLAS), 8192^3 fp32, mean of 10 after 3 warm-ups, this run")
                del ga, gb, gc
            finally:
                torch.backends.cuda.matmul.allow_tf32 = prev

    # Backward products of the same layers (dX = G W, dW += G^T X), each with
    # the step's workspace and without it: the long-K weight gradients have
    # fewer tiles than SMs and are split into independent K pieces.
    backward = None
    if not args.no_backward and args.workload == "c5" and math == sg.MATH_FP32:
        backward = {"per_product": {}}
        reps = max(3, min(args.steps, 10))
        for n in wl.BACKWARD:
            c = wl.make(n, "real")
            bufs = tuple(torch.from_numpy(x).to(dev) for x in (c.A.storage, c.B.storage, c.C.storage))
            a = case_args(c, *bufs)
            row = {}
            # "tf32": the opt-in tensor-core path, with the workspace when
            # there is one (the weight gradients have both operands MN-major).
            for label, kw in (("workspace", ws_kw), ("no_workspace", {}),
                              ("tf32", dict(ws_kw, math=sg.MATH_TF32))):
                if label == "workspace" and not kw:
                    continue
                pl = sg.sbgemm_plan(*a[:16], c.accumulate, **kw)
                for _ in range(3):
                    sg.sbgemm_ex(*a, s_handle, **kw)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record(stream)
                for _ in range(reps):
                    sg.sbgemm_ex(*a, s_handle, **kw)
                e1.record(stream)
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1) / reps
                row[label] = {"ms": round(ms, 4), "gflops": round(c.flops / ms / 1e6, 1),
                              "path": pl["path_name"],
                              "stream_k": {0: "none", 1: "chained", 2: "pieces"}[pl["stream_k"]],
                              "ctas": pl["ctas"]}
            backward["per_product"][n] = row
            del bufs
        key = "workspace" if ws_kw else "no_workspace"
        tot_ms = sum(r[key]["ms"] for r in backward["per_product"].values())
        tot_fl = sum(2 * wl.FULL[n]["batch"] * wl.FULL[n]["M"] * wl.FULL[n]["N"] * wl.FULL[n]["K"]
                     for n in wl.BACKWARD)
        backward["gflops"] = round(tot_fl / tot_ms / 1e6, 1)
        slow = max(backward["per_product"], key=lambda n: backward["per_product"][n][key]["ms"])
        ach = backward["per_product"][slow][key]["gflops"] / 1e3
        fp32_peak = sms * FP32_FLOP_PER_CLK_PER_SM * sm_max * 1e6 / 1e12
        backward["roofline"] = {"bound": "alu", "kernel": f"tma_ffma ({slow})",
                                "achieved": round(ach, 2), "peak": round(fp32_peak, 2),
                                "unit": "TFLOP/s", "frac": round(ach / fp32_peak, 4),
                                "traffic": profiled_traffic("tma_ffma", slow)}

    # Fused epilogue on the feed-forward projection (c5a): y = act(x W^T + b)
    # in one launch, against the plain product, on both arithmetic paths.
    epilogue = None
    if not args.no_epilogue and args.workload == "c5" and math == sg.MATH_FP32:
        i5 = names.index("c5a")
        c = cases[i5]
        bias = torch.randn(c.N, generator=torch.Generator().manual_seed(6)).to(dev)
        reps = max(3, min(args.steps, 10))
        epilogue = {"product": "c5a", "bias": "per output column", "per_variant": {}}
        for mname, m in (("fp32", sg.MATH_FP32), ("tf32", sg.MATH_TF32)):
            variants = {"plain": lambda m=m: sg.sbgemm_ex(*calls[i5], s_handle, math=m, **ws_kw)}
            for act in ("relu", "gelu_erf"):
                variants["bias+" + act] = (lambda m=m, a=act: sg.sbgemm_fused(
                    *calls[i5], bias.data_ptr(), 0, 1, 0, sg.ACTIVATIONS[a], s_handle, m, **ws_kw))
            for k, f in variants.items():
                for _ in range(3):
                    f()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record(stream)
                for _ in range(reps):
                    f()
                e1.record(stream)
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1) / reps
                epilogue["per_variant"][f"{mname} {k}"] = {
                    "ms": round(ms, 4), "gflops": round(c.flops / ms / 1e6, 1)}
            base = epilogue["per_variant"][f"{mname} plain"]["ms"]
            for k in ("bias+relu", "bias+gelu_erf"):
                v = epilogue["per_variant"][f"{mname} {k}"]
                v["overhead_vs_plain"] = round(v["ms"] / base - 1.0, 4)

    # Fused attention (row f2): softmax(alpha Q K^T [causal]) V on the c3/c4
    # problems, against the same result computed in three steps (S by this
    # library's product, a library softmax, P V by this library's product).
    attention = None
    if not args.no_attention and args.workload == "c5" and math == sg.MATH_FP32:
        attention = {"per_workload": {}}
        reps = max(3, min(args.steps, 10))
        fp32_peak = sms * FP32_FLOP_PER_CLK_PER_SM * sm_max * 1e6 / 1e12

        def timed(fn):
            for _ in range(3):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / reps

        for n in wl.ATTENTION:
            c = wl.make_attention(n)
            dQ, dK, dV, dO = (torch.from_numpy(op.storage).to(dev) for op in (c.Q, c.K, c.V, c.O))
            a = (dQ.data_ptr(), c.Q.rs, c.Q.cs, c.Q.bs, dK.data_ptr(), c.K.rs, c.K.cs, c.K.bs,
                 dV.data_ptr(), c.V.rs, c.V.cs, c.V.bs, dO.data_ptr(), c.O.rs, c.O.cs, c.O.bs,
                 c.M, c.N, c.D, c.Dv, c.batch, c.alpha, c.causal, c.q_len)
            ms = timed(lambda: sg.sbgemm_attention(*a, s_handle))
            row = {"ms": round(ms, 4), "gflops": round(c.flops / ms / 1e6, 1),
                   "flops": "2*M*N*(D+Dv) per batch entry, every key counted",
                   "causal": bool(c.causal)}
            # The opt-in TF32 kernel (both products on the tensor cores).
            ms_tc = timed(lambda: sg.sbgemm_attention(*a, s_handle, math=sg.MATH_TF32,
                                                      force_path=sg.PATH_TMA_TF32))
            row["tf32"] = {"ms": round(ms_tc, 4), "gflops": round(c.flops / ms_tc / 1e6, 1),
                           "speedup_vs_fp32": round(ms / ms_tc, 2)}
            if not c.causal:
                S = torch.empty(c.batch, c.M, c.N, device=dev)

                def three_steps():
                    sg.sbgemm_ex(dQ.data_ptr(), c.Q.rs, c.Q.cs, c.Q.bs, dK.data_ptr(), c.K.cs, c.K.rs,
                                 c.K.bs, S.data_ptr(), c.N, 1, c.M * c.N, c.M, c.N, c.D, c.batch,
                                 c.alpha, 0, s_handle, **ws_kw)
                    P = torch.softmax(S, dim=-1)
                    sg.sbgemm_ex(P.data_ptr(), c.N, 1, c.M * c.N, dV.data_ptr(), c.V.rs, c.V.cs,
                                 c.V.bs, dO.data_ptr(), c.O.rs, c.O.cs, c.O.bs, c.M, c.Dv, c.N,
                                 c.batch, 1.0, 0, s_handle, **ws_kw)
                ms3 = timed(three_steps)
                row["three_steps_ms"] = round(ms3, 4)
                row["speedup_vs_three_steps"] = round(ms3 / ms, 2)
                del S
                attention["roofline"] = {"bound": "alu", "kernel": f"attention ({n})",
                                         "achieved": round(c.flops / ms / 1e9, 2),
                                         "peak": round(fp32_peak, 2), "unit": "TFLOP/s",
                                         "frac": round(c.flops / ms / 1e9 / fp32_peak, 4),
                                         "traffic": profiled_traffic("attention", n)}
            attention["per_workload"][n] = row

        # A decode step over a paged K / V cache (row f2's paged read): four
        # query heads per KV head against each sequence's whole context, K and
        # V rows read through the block table.  The stream of K and V rows is
        # the work, so the roofline is the measured copy bandwidth.  Beside
        # it, the same step over the same context stored contiguously.
        hbm_peak = float(peaks.get("hbm_gbs", FALLBACK["hbm_gbs"]))
        for n in wl.PAGED:
            c = wl.make_paged(n)
            dQ = torch.from_numpy(c.Q.storage).to(dev)
            dKc = torch.from_numpy(c.K_cache.reshape(-1)).to(dev)
            dVc = torch.from_numpy(c.V_cache.reshape(-1)).to(dev)
            dT = torch.from_numpy(c.block_table).to(dev)
            dL = torch.from_numpy(c.seq_lens).to(dev)
            dO = torch.from_numpy(c.O.storage).to(dev)
            a = (dQ.data_ptr(), c.Q.rs, c.Q.cs, c.Q.bs, dKc.data_ptr(), dVc.data_ptr(),
                 c.K_cache.shape[0], c.block_size, c.n_kv_heads, dT.data_ptr(),
                 c.block_table.shape[1], dL.data_ptr(), dO.data_ptr(), c.O.rs, c.O.cs, c.O.bs,
                 c.M, c.N, c.D, c.D, c.n_seqs, c.alpha, c.causal, c.q_len)
            ms = timed(lambda: sg.sbgemm_attention_paged(*a, s_handle, **ws_kw))
            gbs = c.alg_bytes / ms / 1e6
            row = {"ms": round(ms, 4), "gb_s": round(gbs, 1), "alg_mb": round(c.alg_bytes / 1e6, 2),
                   "keys": c.keys, "gflops": round(c.flops / ms / 1e6, 1),
                   "shape": {"n_seqs": c.n_seqs, "n_kv_heads": c.n_kv_heads, "rows_per_entry": c.M,
                             "head_dim": c.D, "block_size": c.block_size,
                             "context": [int(c.seq_lens.min()), int(c.seq_lens.max())]},
                   "roofline": {"bound": "hbm", "kernel": "attention_decode (paged)",
                                "achieved": round(gbs, 1), "peak": round(hbm_peak, 1),
                                "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                                "traffic": profiled_traffic("attention_decode", n)}}
            del dKc, dVc
            # The same keys stored contiguously, [entry][N][D] padded to N.
            dK = torch.from_numpy(c.K_ctx.reshape(-1)).to(dev)
            dV = torch.from_numpy(c.V_ctx.reshape(-1)).to(dev)
            b = (dQ.data_ptr(), c.Q.rs, c.Q.cs, c.Q.bs, dK.data_ptr(), c.D, 1, c.N * c.D,
                 dV.data_ptr(), c.D, 1, c.N * c.D, dO.data_ptr(), c.O.rs, c.O.cs, c.O.bs,
                 c.M, c.N, c.D, c.D, c.batch, c.alpha, c.causal, c.q_len)
            ms_c = timed(lambda: sg.sbgemm_attention(*b, s_handle, **ws_kw))
            row["contiguous_padded_ms"] = round(ms_c, 4)
            row["contiguous_note"] = ("every entry padded to the longest context (keys past it are "
                                      "masked but still read), the layout a gather into one buffer "
                                      "gives")
            attention["per_workload"][n] = row
            del dK, dV

    # Every other config of the workload list, each against its own roofline,
    # min(peak compute, algorithmic bytes x HBM bandwidth): median of 21 timed
    # launches after 5 warm-ups, and the mean of back-to-back launches (1000
    # for the latency-bound c1 / c2, 200 for c3 / c4, whose working sets exceed
    # the L2).
    configs = None
    if not args.no_configs and args.workload == "c5" and math == sg.MATH_FP32:
        configs = {}
        hbm = float(peaks.get("hbm_gbs", FALLBACK["hbm_gbs"]))
        fp32_peak = sms * FP32_FLOP_PER_CLK_PER_SM * sm_max * 1e6 / 1e12
        tf32_peak = float(peaks.get("bf16_tflops", FALLBACK["bf16_tflops"])) * TF32_OVER_BF16_NOMINAL
        # The floor of the single-launch figure: two events recorded back to
        # back with nothing between them (the host's event-record calls and
        # the GPU's timestamp latency, which every single-launch median
        # below includes on top of the call and the kernel).
        floor = []
        for _ in range(41):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            e1.record(stream)
            e1.synchronize()
            floor.append(e0.elapsed_time(e1) * 1e3)
        configs["single_launch_event_floor_us"] = round(statistics.median(floor), 2)
        for n in ("c1", "c2a", "c2b", "c3", "c3gqa", "c4"):
            c = wl.make(n, "real")
            bufs = tuple(torch.from_numpy(x).to(dev) for x in (c.A.storage, c.B.storage, c.C.storage))
            a = case_args(c, *bufs)
            row = {"gflop": round(c.flops / 1e9, 4), "alg_mb": round(wl.alg_bytes(c) / 1e6, 2)}
            for mname, m in (("fp32", sg.MATH_FP32), ("tf32", sg.MATH_TF32)):
                pl = sg.sbgemm_plan(*a[:16], c.accumulate, math=m, **ws_kw)
                if m == sg.MATH_TF32 and pl["path_name"] != "tma_tf32":
                    continue
                for _ in range(5):
                    sg.sbgemm_ex(*a, s_handle, math=m, **ws_kw)
                times = []
                for _ in range(21):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    sg.sbgemm_ex(*a, s_handle, math=m, **ws_kw)
                    e1.record(stream)
                    e1.synchronize()
                    times.append(e0.elapsed_time(e1))
                ms = statistics.median(times)
                peak = fp32_peak if m == sg.MATH_FP32 else tf32_peak
                roof_c = min(peak, c.flops / wl.alg_bytes(c) * hbm / 1e3)   # TFLOP/s
                ent = {"ms_median": round(ms, 4), "gflops": round(c.flops / ms / 1e6, 1),
                       "path": pl["path_name"],
                       "roof_tflops": round(roof_c, 2),
                       "bound": "compute" if roof_c == peak else "hbm",
                       "frac_of_roof": round(c.flops / ms / 1e9 / roof_c, 4)}
                # Back to back: the launches queue up, so the host's per-call
                # validation and launch cost (a few us) overlaps the kernels.
                # The single-launch median above includes it.
                nb = 1000 if n in ("c1", "c2a", "c2b") else 200
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(nb):
                    sg.sbgemm_ex(*a, s_handle, math=m, **ws_kw)
                e1.record(stream)
                torch.cuda.synchronize()
                us_b2b = e0.elapsed_time(e1) * 1e3 / nb
                ent["us_back_to_back"] = round(us_b2b, 2)
                ent["frac_of_roof_back_to_back"] = round(c.flops / (us_b2b * 1e-6) / 1e12 / roof_c, 4)
                row[mname] = ent
            configs[n] = row
            del bufs

    # The other products the pages route through the kernel (row f4): the
    # spectrogram (frames read as overlapping strided rows) and the tokenizer's
    # codebook distances.
    spectral = None
    if not args.no_f4 and args.workload == "c5" and math == sg.MATH_FP32:
        spectral = {"per_product": {}}
        reps = max(3, min(args.steps, 10))
        for n in ("f4spec", "f4dist"):
            c = wl.make(n, "real")
            bufs = tuple(torch.from_numpy(x).to(dev) for x in (c.A.storage, c.B.storage, c.C.storage))
            a = case_args(c, *bufs)
            pl = sg.sbgemm_plan(*a[:16], c.accumulate, **ws_kw)
            for _ in range(3):
                sg.sbgemm_ex(*a, s_handle, **ws_kw)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(reps):
                sg.sbgemm_ex(*a, s_handle, **ws_kw)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / reps
            spectral["per_product"][n] = {"ms": round(ms, 4), "gflops": round(c.flops / ms / 1e6, 1),
                                          "path": pl["path_name"], "note": c.note}
            del bufs

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        threads = oracle.default_threads()
        g, dt, fl, rows = oracle_sample(cases, args.cpu_seconds, threads)
        cpu = {"value": round(g, 3), "unit": "GFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"first {rows} rows of each product of the step "
                         f"({fl / 1e9:.2f} GFLOP, {dt:.1f} s), fp64 accumulation",
               "cpu": host_cpu()}

    if rank != 0:
        return None
    wsmb = ws_bytes / 2**20
    return {
        "metric": METRIC, "value": round(value, 1), "unit": "GFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if math == sg.MATH_FP32 else "tf32",
        "data": "synthetic (seeded numpy generators, shapes and value distributions of the workload)",
        "config": {"workload": DESCR.get(args.workload, args.workload),
                   "products_per_step": len(cases), "math": args.math, "path": args.path,
                   "gflop_per_step": round(flops_step / 1e9, 3),
                   "alg_mb_per_step": round(bytes_step / 2**20, 1),
                   "l2": f"inputs larger than L2: {wsmb:.0f} MiB resident per step vs "
                         f"{L2_BYTES / 2**20:.0f} MiB L2, no flush",
                   "parallelism": f"replicas x{world} (each GPU runs the whole step)",
                   "workspace_mib": round(ws.numel() / 2**20, 1) if ws is not None else 0},
        "pct_of_peak": round(100 * value / world / 1e3 / roof["peak"], 2)
        if roof["unit"] == "TFLOP/s" else None,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "tf32": tf32,
        "backward": backward,
        "epilogue": epilogue,
        "attention": attention,
        "spectrogram_and_distances": spectral,
        "configs": configs,
        "gpu_launches": len(calls) * args.steps,
        "clocks": clocks,
        "per_product": {n: {k: v for k, v in d.items() if k != "total_ms"} for n, d in per.items()},
    }


def run_reference(args, world, rank):
    """The oracle as it stands on the host cores, one bounded sample of the
    workload per step."""
    if rank != 0:
        return None
    import oracle
    threads = oracle.default_threads()
    names, cases = workload_cases(args.workload)
    _, dt, fl, rows = oracle_sample(cases, args.ref_step_seconds, threads)
    for _ in range(args.warmup):
        oracle_sample(cases, 0, threads, rows_override=rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample(cases, 0, threads, rows_override=rows)
    el = time.perf_counter() - t0
    value = fl * args.steps / el / 1e9
    sample = f"first {rows} rows of each product per step ({fl / 1e9:.3f} GFLOP)"
    return {
        "metric": METRIC, "value": round(value, 3), "unit": "GFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": DESCR.get(args.workload, args.workload), "math": "fp64 oracle"},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 3), "unit": "GFLOP/s", "kind": "oracle",
                         "cores": threads, "sample": sample, "cpu": host_cpu()},
        "e2e": {"value": round(value, 3), "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--math", choices=["fp32", "tf32"], default="fp32")
    ap.add_argument("--workload", default="c5",
                    choices=sorted(set(wl.WORKLOADS) | set(SWEEPS)))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=0.5)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workspace", action="store_true",
                    help="call without scratch (data-parallel schedule only)")
    ap.add_argument("--path", choices=["auto", "gather", "tma", "tf32"], default="auto",
                    help="force one kernel path for the timed products")
    ap.add_argument("--no-tf32", action="store_true",
                    help="skip the opt-in tensor-core measurement")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the backward-product measurement")
    ap.add_argument("--no-epilogue", action="store_true",
                    help="skip the fused-epilogue measurement")
    ap.add_argument("--no-attention", action="store_true",
                    help="skip the fused-attention measurement")
    ap.add_argument("--no-f4", action="store_true",
                    help="skip the spectrogram and distance products")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config measurements of c1-c4")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)     # at least three untimed warm-up steps
    world, rank, local = dist_env()
    if args.impl == "reference":
        out = run_reference(args, world, rank)
    else:
        dist = init_dist(world)
        out = run_ours(args, world, rank, local, dist)
        if dist is not None:
            dist.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
