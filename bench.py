#!/usr/bin/env python
"""Benchmark of the fused low-rank-adapted linear layer on GB300.

Headline step: one forward + backward of the bf16 LoRA linear layer at the LLM attention
projection size (M = 8192 tokens = batch 4 x seq 2048, d_in = d_out = 4096, rank 16, alpha 32),
through the C ABI, inputs resident in HBM.  value = algorithmic TFLOP/s of the whole job.

Also measured in the same run (the "workloads" object): the DoRA-rows layer
(8192 x 4096 -> 11008, r 32), the LoRA SwiGLU MLP (16384 tokens, 4096 -> 14336 -> 4096, r 16)
and the W8A8 + LoRA forward (16384 x 3072 x 3072, r 32), each with its own roofline line.

One JSON line on stdout (rank 0).  Multi-GPU (torchrun): independent replicas, weak scaling.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused LoRA/DoRA linear fwd+bwd TFLOP/s and % bf16 tensor peak (1 GB300)"
HEADLINE = "lora_4096_bf16"


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------------------- flop counts
def lora_flops(M, d_in, d_out, r):
    """Algorithmic flops of one forward + backward (no dW0; W0 frozen)."""
    fwd = 2 * M * d_in * d_out + 2 * M * r * (d_in + d_out)
    bwd = 2 * M * d_in * d_out + 4 * M * r * (d_in + d_out)
    return fwd, bwd


def dora_flops(M, d_in, d_out, r):
    fwd, bwd = lora_flops(M, d_in, d_out, r)
    return fwd + 2 * d_out * d_in * r, bwd + 2 * d_out * d_in * r   # W0 A^T prepass, W0^T (g o B) norm term


def mlp_flops(M, H, I, r):
    proj = 2 * M * H * I
    fwd = 3 * proj + 3 * 2 * M * r * (H + I)
    bwd = 3 * proj + 3 * 4 * M * r * (H + I)
    return fwd, bwd


# ----------------------------------------------------------------------------- clocks
class NvmlSampler:
    """Reads SM clock, max clock, power and clock-event reasons through NVML every ~2 ms.
    Read-only: nothing on the GPU is changed."""
    BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, cuda_index: int):
        import ctypes
        self.samples, self.ok, self._stop = [], False, False
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            import torch
            pr = torch.cuda.get_device_properties(cuda_index)
            self.h = ctypes.c_void_p()
            bus = f"{getattr(pr, 'pci_domain_id', 0):08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0".encode()
            if self.nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(self.h)) != 0:
                if self.nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h)) != 0:
                    return
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def start(self):
        if self.ok:
            threading.Thread(target=self._run, daemon=True).start()

    def _run(self):
        import ctypes
        mhz, mx, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop:
            self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz))
            self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
            self.nv.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(mw))
            self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs))
            self.samples.append((time.time(), mhz.value, mx.value, mw.value / 1e3, rs.value))
            time.sleep(0.002)

    def stop(self):
        self._stop = True

    def summary(self, t0, t1):
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        if not win:
            return None
        reasons = sorted({nm for s in win for b, nm in self.BITS.items() if s[4] & b})
        return {"sm_mhz": statistics.median(s[1] for s in win), "sm_max_mhz": max(s[2] for s in win),
                "reasons": reasons, "samples": len(win), "window": "timed (NVML, 2 ms period)",
                "power_w_max": max(s[3] for s in win)}


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        win = [s for t, s in self.samples if t0 <= t <= t1]
        window = "timed"
        if len(win) < 3:
            win = [s for _, s in self.samples]
            window = "whole run (timed region shorter than the sampling period)"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[0]) for s in win if num(s[0]) is not None]
        mx = [num(s[1]) for s in win if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i in range(4) if len(s) > 4 + i and s[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(win), "window": window,
                "power_w_max": max((num(s[2]) or 0.0) for s in win)}


def clocks_rejected(c):
    """True for a clock record that the measurement rules reject: a hardware or thermal slowdown
    during the timed region, or an SM clock well below its maximum with no reason (a clock lock
    left by someone else).  A power-cap reason alone is kept."""
    if not c or c.get("sm_mhz") is None or not c.get("sm_max_mhz"):
        return False
    if {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"} & set(c.get("reasons") or []):
        return True
    return c["sm_mhz"] < 0.85 * c["sm_max_mhz"] and not c.get("reasons")


# ----------------------------------------------------------------------------- peaks
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------- CPU oracle leg
def oracle_lora_sample(M_s, seed=7):
    """One fwd+bwd of the fp64 oracle on an M_s-row sample of the headline workload."""
    import numpy as np

    import datagen as D
    import oracle as O
    case = D.scaled(D.WORKLOADS[HEADLINE], M=M_s)
    t = D.make_linear(case)
    f = {k: (None if v is None else v.double().numpy()) for k, v in t.items()}
    t0 = time.perf_counter()
    O.lora_linear_fwd(f["X"], f["W0"], f["A"], f["B"], case.s)
    O.lora_linear_bwd(f["X"], f["W0"], f["A"], f["B"], case.s, f["dY"])
    dt = time.perf_counter() - t0
    fwd, bwd = lora_flops(M_s, case.d_in, case.d_out, case.r)
    np.asarray(0)
    return dt, fwd + bwd


def cpu_baseline(budget_s=12.0):
    M_s, dt, fl = 64, 0.0, 0
    while True:
        dt, fl = oracle_lora_sample(M_s)
        if dt * 2 > budget_s or M_s >= 8192:
            break
        M_s *= 2
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{M_s} of the 8192 token rows of the {HEADLINE} workload, forward + backward, fp64 "
                      f"materialised W' = W0 + sBA, {dt:.2f} s"}


def run_reference(args, rank):
    """Reference arm: the fp64 CPU oracle as it stands, timed on the host cores."""
    if rank != 0:
        return
    # calibrate a per-step sample so that (warmup + steps) samples take about two minutes
    dt1, _ = oracle_lora_sample(64)
    per_step = 120.0 / max(1, args.steps + args.warmup)
    M_s = 64
    while M_s < 8192 and dt1 * (M_s * 2 / 64) <= per_step:
        M_s *= 2
    for _ in range(args.warmup):
        oracle_lora_sample(M_s)
    tot_t, tot_f = 0.0, 0
    for _ in range(args.steps):
        dt, fl = oracle_lora_sample(M_s)
        tot_t += dt
        tot_f += fl
    v = tot_f / tot_t / 1e12
    sample = f"each step {M_s} of the 8192 token rows of {HEADLINE}, forward + backward, fp64 oracle"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{HEADLINE}: M=8192 d_in=4096 d_out=4096 r=16 alpha=32, fwd+bwd (row sample)"},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ----------------------------------------------------------------------------- multi-rank
def reduce_max(vals, dist, device):
    """Max over ranks of each timing (the slowest replica sets the job's time)."""
    if dist is None:
        return list(vals)
    import torch
    t = torch.tensor(list(vals), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(flops_per_rank_step, world, ms_max):
    """Whole-job TFLOP/s: the work of all replicas over the slowest replica's step time."""
    return flops_per_rank_step * world / (ms_max * 1e-3) / 1e12


# ----------------------------------------------------------------------------- GPU workloads
def timed(fn, steps, warmup, dist=None):
    import torch
    for _ in range(warmup):
        fn()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    t0 = time.time()
    for _ in range(steps):
        fn()
    e1.record(st)
    torch.cuda.synchronize()
    t1 = time.time()
    if dist is not None:
        dist.barrier()
    return e0.elapsed_time(e1) / steps, t0, t1


def timed_reps(fn, steps, warmup, dist=None, min_s=1.0, max_reps=200):
    """Timed regions of exactly `steps` steps each (barrier and synchronize on both sides), repeated
    until they cover at least min_s seconds: (median ms per step, per-region ms, t0, t1)."""
    per, t_first, t_last = [], None, None
    ms, t0, t1 = timed(fn, steps, warmup, dist)
    per.append(ms)
    t_first, t_last = t0, t1
    if dist is not None:   # every rank runs the same number of regions (each one ends in a barrier)
        import torch
        ms = reduce_max([ms], dist, torch.device("cuda", torch.cuda.current_device()))[0]
    reps = max(1, min(max_reps, int(min_s / max(1e-9, ms * steps * 1e-3))))
    for _ in range(reps - 1):
        ms, _, t1 = timed(fn, steps, 0, dist)
        per.append(ms)
        t_last = t1
    return statistics.median(per), per, t_first, t_last


# DRAM bytes (read + write) per GEMM launch from ncu captures, keyed by workload; a value is
# dropped (None) whenever the kernel changes and is re-measured before it is put back.
# lora_4096_bf16: dram__bytes_read.sum + dram__bytes_write.sum of the forward (CTA pair) and dX
# (one-CTA kernel, no cluster) GEMM launches of the headline step, one full capture of each:
# forward 153.1 + 48.0 MB, dX 119.5 + 43.5 MB, mean 182.1 MB per launch; the algorithmic bytes
# are 64 MiB activation + 32 MiB weight + 64 MiB output = 167.8 MB.
GEMM_TRAFFIC = {"lora_4096_bf16": 182.1e6}


def timed_gemm_events(L, fn, steps, warmup=1):
    """A second timed pass of the same steps with CUDA events around every GEMM launch (the
    library's own timing): returns that pass's ms per step.  The events sit between kernels and
    so cost the step the programmatic-launch overlap at each GEMM boundary; the step time that is
    reported comes from the plain pass, the kernel durations from this one."""
    L.lora_prof_gemm(reset=True)
    L.lora_prof_enable(True)
    try:
        ms, _, _ = timed(fn, steps, warmup)
    finally:
        L.lora_prof_enable(False)
    return ms


def gemm_roofline(L, peaks, ms_step, steps_recorded, sustained, workload):
    """Roofline of the dominant kernel (tcgen05 GEMM) from the library's own event timing, taken in
    the pass of `timed_gemm_events` (ms_step is that pass's step time)."""
    ms, n, fl = L.lora_prof_gemm(reset=True)
    if n == 0 or ms <= 0:
        return None
    ach = fl / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    return {"kernel": "tcgen05 GEMM with fused rank-r tail (tc_pair_kernel, forward and dX)",
            "bound": "tensor",
            "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s", "frac": round(ach / peak, 4),
            "peak_kind": ("sustained" if sustained else "burst") + " bf16, " + peaks["source"] + " (of measured)",
            "launches": n, "avg_launch_ms": round(ms / n, 4),
            "share_of_step": round(ms / (steps_recorded * ms_step), 4),
            "timing": "CUDA events around each GEMM launch in a second pass of the timed steps "
                      f"({ms_step:.4f} ms per step with the events, which cost the programmatic-launch "
                      "overlap at the GEMM boundaries; the step time is from the pass without them)",
            "flops_per_launch": fl / n, "traffic": GEMM_TRAFFIC.get(workload)}


def rank_pass_roofline(L, peaks):
    """HBM roofline of the rank-r passes recorded in the events pass (their algorithmic bytes over
    their event time)."""
    ms, n, by = L.lora_prof_rank(reset=True)
    if n == 0 or ms <= 0:
        return None
    ach = by / (ms * 1e-3) / 1e9
    return {"kernels": "rowproj_kernel / rowcol_kernel / colreduce_kernel (rank-r passes)", "bound": "hbm",
            "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(ach / peaks["hbm_gbs"], 4), "launches": n, "avg_launch_ms": round(ms / n, 4),
            "bytes_per_launch": by / n}


def headline(args, L, ops, dist, world, peaks):
    import torch

    import datagen as D
    case = D.WORKLOADS[HEADLINE]
    t = D.make_linear(case)
    dev = torch.device("cuda", torch.cuda.current_device())
    X, W0, A, B, dY = (t[k].to(dev) for k in ("X", "W0", "A", "B", "dY"))
    M, d_in, d_out, r, s = case.M, case.d_in, case.d_out, case.r, case.s
    sh = L.shape(M, d_in, d_out, r, L.LORA_BF16)
    Ys = [torch.empty(M, d_out, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    Zs = [torch.empty(M, r, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    dXs = [torch.empty_like(X) for _ in range(2)]
    dAs = [torch.empty_like(A) for _ in range(2)]
    dBs = [torch.empty_like(B) for _ in range(2)]
    wsf = torch.zeros(L.lora_workspace_bytes(L.OP_LINEAR_FWD, sh), dtype=torch.uint8, device=dev)
    wsb = torch.zeros(L.lora_workspace_bytes(L.OP_LINEAR_BWD, sh), dtype=torch.uint8, device=dev)

    def fwd(Xb=X, b=0):
        L.lora_linear_fwd(sh, Xb, W0, A, B, None, s, Ys[b], Zs[b], wsf)

    def bwd(Xb=X, dYb=dY, b=0):
        L.lora_linear_bwd(sh, Xb, W0, A, B, Zs[b], dYb, s, dXs[b], dAs[b], dBs[b], None, wsb)

    def step(Xb=X, dYb=dY, b=0):
        fwd(Xb, b)
        bwd(Xb, dYb, b)

    fwd_fl, bwd_fl = lora_flops(M, d_in, d_out, r)
    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    nv = NvmlSampler(torch.cuda.current_device())
    nv.start()
    time.sleep(0.3)
    n0 = L.lora_launch_count()
    ms, per, t0, t1 = timed_reps(step, args.steps, args.warmup, dist, args.min_timed_s)
    launches = L.lora_launch_count() - n0
    # the count includes the warm-up steps: scale it to one timed region of exactly K steps
    gpu_launches = round(launches * args.steps / (args.steps * len(per) + args.warmup))
    clocks = nv.summary(t0, t1) or clk.summary(t0, t1)
    if dist is None and clocks_rejected(clocks):
        # a record the measurement rules reject: take the timed regions once more (one process
        # only: with several ranks the decision would have to be collective)
        first = clocks
        ms, per, t0, t1 = timed_reps(step, args.steps, args.warmup, dist, args.min_timed_s)
        clocks = dict(nv.summary(t0, t1) or clk.summary(t0, t1) or {},
                      remeasured_after=first.get("reasons") or ["SM clock below 85% of max"])
    nv.stop()
    # each direction alone (the same calls), for the split of the step
    ms_fwd, _, _, _ = timed_reps(fwd, args.steps, 2, dist, args.min_timed_s / 4)
    ms_bwd, _, _, _ = timed_reps(bwd, args.steps, 2, dist, args.min_timed_s / 4)
    # a second pass with CUDA events around every GEMM and rank-r launch (the library's tracing)
    L.lora_prof_rank(reset=True)
    ms_ev = timed_gemm_events(L, step, args.steps)
    roof = gemm_roofline(L, peaks, ms_ev, args.steps + 1, False, HEADLINE)
    rank_roof = rank_pass_roofline(L, peaks)
    clk.stop()
    for ws in (wsf, wsb):
        if L.lora_check_device_error(ws) != 0:
            raise RuntimeError("a kernel recorded a timed-out wait during the benchmark")

    # End to end through the same entry points: every step copies its inputs X and dY from pinned
    # host memory and reads its results Y, dX, dA and dB back into pinned host memory.  Device
    # buffers are doubled: step i+1's inputs arrive (copy stream) and step i-1's results leave
    # (second copy stream) while step i computes.
    Xh = t["X"].pin_memory()
    dYh = t["dY"].pin_memory()
    Yh = [torch.empty(M, d_out, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dXh = [torch.empty(M, d_in, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dAh = [torch.empty_like(A, device="cpu").pin_memory() for _ in range(2)]
    dBh = [torch.empty_like(B, device="cpu").pin_memory() for _ in range(2)]
    Xd, dYd = [X, torch.empty_like(X)], [dY, torch.empty_like(dY)]
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(n):
        cur = torch.cuda.current_stream()
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        done = [torch.cuda.Event(), torch.cuda.Event()]
        fdone = [torch.cuda.Event(), torch.cuda.Event()]
        out = [torch.cuda.Event(), torch.cuda.Event()]
        cin.wait_stream(cur)
        cout.wait_stream(cur)
        with torch.cuda.stream(cin):
            Xd[0].copy_(Xh, non_blocking=True)
            dYd[0].copy_(dYh, non_blocking=True)
            copied[0].record(cin)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                with torch.cuda.stream(cin):
                    if i >= 1:
                        cin.wait_event(done[1 - b])     # step i-1 has read that half of the inputs
                    Xd[1 - b].copy_(Xh, non_blocking=True)
                    dYd[1 - b].copy_(dYh, non_blocking=True)
                    copied[1 - b].record(cin)
            cur.wait_event(copied[b])
            if i >= 2:
                cur.wait_event(out[b])                  # step i-2's results have left these buffers
            fwd(Xd[b], b)
            fdone[b].record(cur)
            bwd(Xd[b], dYd[b], b)
            done[b].record(cur)
            with torch.cuda.stream(cout):
                cout.wait_event(fdone[b])
                Yh[b].copy_(Ys[b], non_blocking=True)
                cout.wait_event(done[b])
                dXh[b].copy_(dXs[b], non_blocking=True)
                dAh[b].copy_(dAs[b], non_blocking=True)
                dBh[b].copy_(dBs[b], non_blocking=True)
                out[b].record(cout)
        cur.wait_stream(cout)

    e2e_steps = max(4, min(args.steps, 50))
    e2e_run(3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    q0.record()
    e2e_run(e2e_steps)
    q1.record()
    torch.cuda.synchronize()
    ms_e2e = q0.elapsed_time(q1) / e2e_steps
    if dist is not None:
        dist.barrier()

    context = same_box_context(case, X, W0, A, B, dY, dev, peaks) if dist is None or dist.get_rank() == 0 else None
    ms_all, ms_e2e, ms_fwd, ms_bwd = reduce_max([ms, ms_e2e, ms_fwd, ms_bwd], dist, dev)
    h2d = X.numel() * 2 + dY.numel() * 2
    d2h = Ys[0].numel() * 2 + dXs[0].numel() * 2 + dAs[0].numel() * 2 + dBs[0].numel() * 2
    return {
        "value": job_throughput(fwd_fl + bwd_fl, world, ms_all), "ms_per_step": ms_all, "clocks": clocks,
        "timed_regions": {"regions": len(per), "steps_each": args.steps,
                          "ms_per_step_each": [round(x, 4) for x in per], "ms_per_step": "median of the regions",
                          "seconds": round(t1 - t0, 3)},
        "roofline": roof, "rank_passes": rank_roof, "gpu_launches": gpu_launches,
        "fwd": {"ms": round(ms_fwd, 4), "tflops": round(fwd_fl / (ms_fwd * 1e-3) / 1e12, 1)},
        "bwd": {"ms": round(ms_bwd, 4), "tflops": round(bwd_fl / (ms_bwd * 1e-3) / 1e12, 1)},
        "e2e": {"value": job_throughput(fwd_fl + bwd_fl, world, ms_e2e), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                "copies": "h2d X, dY; d2h Y, dX, dA, dB (pinned host, separate copy streams, double-buffered)"},
        "tokens_per_s": M * world / (ms_all * 1e-3),
        "frac_of_bf16_peak_step": (fwd_fl + bwd_fl) / (ms_all * 1e-3) / 1e12 / peaks["bf16_tflops"],
        "context": context,
    }


def same_box_context(case, X, W0, A, B, dY, dev, peaks, steps=20):
    """Context on the same GPU (not the product): the plain X W0^T product through cuBLAS
    (torch.matmul), and the unfused bypass of eager PyTorch (F.linear plus two low-rank matmuls,
    backward by autograd, W0 frozen) for the same forward + backward."""
    import torch
    M, d_in, d_out, r, s = case.M, case.d_in, case.d_out, case.r, case.s

    def mm():
        torch.matmul(X, W0.t())
    ms_mm, _, _ = timed(mm, steps, 3)
    Ag = A.detach().clone().requires_grad_(True)
    Bg = B.detach().clone().requires_grad_(True)
    Xg = X.detach().clone().requires_grad_(True)

    def eager():
        y = torch.nn.functional.linear(Xg, W0) + s * ((Xg @ Ag.t()) @ Bg.t())
        y.backward(dY)
        Xg.grad = None
        Ag.grad = None
        Bg.grad = None
    ms_eager, _, _ = timed(eager, steps, 3)
    fwd, bwd = lora_flops(M, d_in, d_out, r)
    return {"cublas_matmul_x_w0t": {"ms": round(ms_mm, 4), "tflops": round(2 * M * d_in * d_out / (ms_mm * 1e-3) / 1e12, 1),
                                    "frac_of_bf16_peak": round(2 * M * d_in * d_out / (ms_mm * 1e-3) / 1e12 /
                                                               peaks["bf16_tflops"], 4)},
            "torch_eager_unfused_bypass_fwd_bwd": {"ms": round(ms_eager, 4),
                                                   "tflops": round((fwd + bwd) / (ms_eager * 1e-3) / 1e12, 1)}}


def extra_workloads(args, L, ops, peaks, which=("dora", "mlp", "w8a8", "qkv", "dropout")):
    """DoRA, gated MLP, W8A8, fused-QKV and input-dropout workloads, each a fwd+bwd step (W8A8 also
    fwd alone)."""
    import torch

    import datagen as D
    dev = torch.device("cuda", torch.cuda.current_device())
    out = {}
    steps, warm = max(3, min(args.steps, 20)), 3
    if "dora" in which:
        out.update(_dora_workload(args, L, ops, peaks, D, dev, steps, warm))
    if "mlp" in which:
        out.update(_mlp_workload(args, L, ops, peaks, D, dev, steps, warm))
    if "w8a8" in which:
        out.update(_w8a8_workload(args, L, ops, peaks, D, dev, steps, warm))
    if "qkv" in which:
        out.update(_qkv_workload(args, L, ops, peaks, D, dev, steps, warm))
    if "dropout" in which:
        out.update(_dropout_workload(args, L, ops, peaks, D, dev, steps, warm))
    return out


def _dropout_workload(args, L, ops, peaks, D, dev, steps, warm, p=0.1):
    """The headline LoRA layer with input dropout (keep mask drawn once, p = 0.1), forward +
    backward on the unfused path; the flops counted are the plain layer's."""
    import torch
    case = D.WORKLOADS[HEADLINE]
    t = D.make_linear(case)
    g = {k: v.to(dev) for k, v in t.items() if v is not None}
    mask = D.make_dropout_mask(case.M, case.d_in, p).to(dev)
    keep = 1.0 / (1.0 - p)

    def drop_step():
        Y, Z = ops.lora_linear_dropout_fwd(g["X"], mask, keep, g["W0"], g["A"], g["B"], case.s)
        ops.lora_linear_dropout_bwd(g["X"], mask, keep, g["W0"], g["A"], g["B"], Z, g["dY"], case.s)
    ms, _, _ = timed(drop_step, steps, warm)
    ms_ev = timed_gemm_events(L, drop_step, steps)
    f, b = lora_flops(case.M, case.d_in, case.d_out, case.r)
    name = "lora_dropout_4096_bf16"
    out = {name: {"ms_per_step": ms, "tflops": (f + b) / (ms * 1e-3) / 1e12,
                  "frac_of_bf16_peak": (f + b) / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                  "note": f"keep mask with p = {p}; unfused call: the Z and dA passes read the mask beside X "
                          "(no masked copy of X), the adapter's share of dX is a masked rank-r pass",
                  "roofline": gemm_roofline(L, peaks, ms_ev, steps + 1, False, name)}}
    for buf in ops._WS.values():
        if L.lora_check_device_error(buf) != 0:
            raise RuntimeError("a kernel recorded a timed-out wait in the dropout workload")
    del g, t, mask
    torch.cuda.empty_cache()
    return out


def _qkv_workload(args, L, ops, peaks, D, dev, steps, warm):
    """Fused query/key/value projection with one adapter per leaf, forward + backward."""
    import torch
    case = D.WORKLOADS["qkv_lora_4096_gqa_bf16"]
    t = D.make_qkv(case)
    g = {k: v.to(dev) for k, v in t.items() if v is not None}
    leaves = [(g[f"A{l}"], g[f"B{l}"], case.s[l]) for l in range(len(case.n))]

    def qkv_step():
        Y, Z = ops.lora_qkv_fwd(g["X"], g["W0"], leaves)
        ops.lora_qkv_bwd(g["X"], g["W0"], leaves, Z, g["dY"])
    ms, _, _ = timed(qkv_step, steps, warm)
    ms_ev = timed_gemm_events(L, qkv_step, steps)
    N = sum(case.n)
    f = 2 * case.M * case.d_in * N + 2 * case.M * case.r * len(case.n) * case.d_in + 2 * case.M * case.r * N
    b = 2 * case.M * case.d_in * N + 4 * case.M * case.r * (len(case.n) * case.d_in + N)
    out = {case.name: {"ms_per_step": ms, "tokens_per_s": case.M / (ms * 1e-3),
                       "tflops": (f + b) / (ms * 1e-3) / 1e12,
                       "frac_of_bf16_peak": (f + b) / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                       "roofline": gemm_roofline(L, peaks, ms_ev, steps + 1, False, case.name)}}
    del g, t
    torch.cuda.empty_cache()
    return out


def _dora_workload(args, L, ops, peaks, D, dev, steps, warm):
    out = {}
    case = D.WORKLOADS["dora_4096x11008_bf16"]
    t = D.make_linear(case)
    g = {k: v.to(dev) for k, v in t.items() if v is not None}
    r0 = ops.dora_rownorm2(g["W0"])

    def dora_step():
        Y, Z, n, V = ops.dora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], r0, case.s, case.eps, g["bias"])
        ops.dora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], g["m"], g["bias"], Y, Z, n, V, g["dY"], case.s,
                            case.eps)
    ms, _, _ = timed(dora_step, steps, warm)
    ms_ev = timed_gemm_events(L, dora_step, steps)
    f, b = dora_flops(case.M, case.d_in, case.d_out, case.r)
    out["dora_4096x11008_bf16"] = {"ms_per_step": ms, "tflops": (f + b) / (ms * 1e-3) / 1e12,
                                   "frac_of_bf16_peak": (f + b) / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                                   "roofline": gemm_roofline(L, peaks, ms_ev, steps + 1, False,
                                                             "dora_4096x11008_bf16")}
    del g, t
    # the column variant on the same shapes: magnitude per input column
    case = D.WORKLOADS["dora_cols_4096x11008_bf16"]
    t = D.make_linear(case)
    g = {k: v.to(dev) for k, v in t.items() if v is not None}
    c0 = ops.dora_colnorm2(g["W0"])

    def cols_step():
        Y, Z, n, U = ops.dora_cols_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], c0, case.s, case.eps, g["bias"])
        ops.dora_cols_bwd(g["X"], g["W0"], g["A"], g["B"], g["m"], Z, n, U, g["dY"], case.s, case.eps)
    ms, _, _ = timed(cols_step, steps, warm)
    ms_ev = timed_gemm_events(L, cols_step, steps)
    f, b = dora_flops(case.M, case.d_in, case.d_out, case.r)
    out[case.name] = {"ms_per_step": ms, "tflops": (f + b) / (ms * 1e-3) / 1e12,
                      "frac_of_bf16_peak": (f + b) / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                      "roofline": gemm_roofline(L, peaks, ms_ev, steps + 1, False, case.name)}
    del g, t
    return out


def _mlp_workload(args, L, ops, peaks, D, dev, steps, warm):
    import torch
    out = {}
    case = D.WORKLOADS["mlp_swiglu_4096x14336_bf16"]
    t = D.make_mlp(case)
    g = {k: v.to(dev) for k, v in t.items()}
    P = {p: {"W": g["W" + p], "A": g["A" + p], "B": g["B" + p], "s": case.s} for p in "gud"}

    f, b = mlp_flops(case.M, case.H, case.I, case.r)
    # the same shapes and inputs with each gate activation (SwiGLU, GeGLU with exact GELU)
    for name, act in (("mlp_swiglu_4096x14336_bf16", 0), ("mlp_geglu_4096x14336_bf16", 1)):
        def mlp_step():
            Y, saved = ops.lora_mlp_swiglu_fwd(g["X"], P["g"], P["u"], P["d"], act=act)
            ops.lora_mlp_swiglu_bwd(g["X"], P["g"], P["u"], P["d"], saved, g["dY"], act=act)
        mlp_steps = max(3, steps // 2)
        ms, _, _ = timed(mlp_step, mlp_steps, 2)
        ms_ev = timed_gemm_events(L, mlp_step, mlp_steps)
        out[name] = {"ms_per_step": ms, "tflops": (f + b) / (ms * 1e-3) / 1e12,
                     "frac_of_bf16_peak": (f + b) / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                     "roofline": gemm_roofline(L, peaks, ms_ev, mlp_steps + 1, True, name)}
    del g, t, P
    torch.cuda.empty_cache()
    return out


def _w8a8_workload(args, L, ops, peaks, D, dev, steps, warm):
    """W8A8 + LoRA forward: quantise X (W-1), exact int8 product with the LoRA epilogue."""
    import torch
    out = {}
    case = D.WORKLOADS["w8a8_lora_3072"]
    t = D.make_w8a8(case)
    X = t["X"].to(dev)
    A = t["A"].to(dev)
    B = t["B"].to(dev)
    # the frozen int8 weight with its per-row scales, from the library's own per-row quantiser
    Wq, sw, _ = ops.w8a8_quantize_rows(t["W0"].to(torch.bfloat16).to(dev))

    # the frozen weight laid out once (codes as bf16 for the forward, dequantised copy for the
    # backward), outside the timed steps like loading the model
    Wb, Wd = ops.w8a8_prepack_weight(Wq, sw)

    def w8_step():   # W-1 (codes written as bf16) + the packed product with the LoRA epilogue
        Xc, sx, Z = ops.w8a8_quantize_rows_bf16(X, A)
        ops.w8a8_lora_fwd_packed(Xc, sx, Wb, sw, Z, B, case.s)

    def w8_step_int8():   # the same through the int8 interface (re-lays out codes and weight per call)
        Xq, sx, Z = ops.w8a8_quantize_rows(X, A)
        ops.w8a8_lora_fwd(Xq, sx, Wq, sw, Z, B, case.s)
    ms_int8, _, _ = timed(w8_step_int8, steps, warm)
    ms, _, _ = timed(w8_step, steps, warm)
    ms_ev = timed_gemm_events(L, w8_step, steps)
    gms, gn, gfl = L.lora_prof_gemm(reset=True)
    for buf in ops._WS.values():
        if L.lora_check_device_error(buf) != 0:
            raise RuntimeError("a kernel recorded a timed-out wait in the workload breakdown")
    ops_int8 = 2 * case.M * case.d_in * case.d_out
    lora_fl = 2 * case.M * case.r * (case.d_in + case.d_out)
    rec = {"ms_per_step": ms, "int8_tops": ops_int8 / (ms * 1e-3) / 1e12,
           "lora_tflops": lora_fl / (ms * 1e-3) / 1e12,
           "path": "w8a8_quantize_rows_bf16 + w8a8_lora_fwd_packed (weight prepacked once)",
           "int8_interface_ms_per_step": ms_int8,
           "note": "exact int8 product on the bf16 tcgen05 tensor cores with the codes as bf16 values, "
                   "summed exactly in fp32 over 1024-wide K chunks and added as int32 (sm_103a has no "
                   "tcgen05 int8 kind)"}
    if gn:
        # the method's own work per launch: the int8 product 2 M N K plus the rank-r term 2 M N r,
        # which is also the bf16 tensor work the kernel does
        own = ops_int8 + 2 * case.M * case.d_out * case.r
        ach = own * gn / (gms * 1e-3) / 1e12
        rec["roofline"] = {"kernel": "tc_gemm_kernel (chunked exact W8A8 mode)", "bound": "tensor",
                           "achieved": round(ach, 1), "peak": peaks["bf16_tflops"], "unit": "T-ops/s",
                           "frac": round(ach / peaks["bf16_tflops"], 4), "launches": gn,
                           "avg_launch_ms": round(gms / gn, 4), "share_of_step": round(gms / ((steps + 1) * ms_ev), 4),
                           "ops_per_launch": own, "traffic": None,
                           "tensor_work_per_launch": gfl / gn,
                           "note": "achieved counts the method's own work (2 M N K int8 + 2 M N r bf16) against "
                                   "the bf16 tensor peak, on which it runs",
                           "timing": "CUDA events around each GEMM launch in a second pass of the timed steps"}
    out["w8a8_lora_3072"] = rec

    # backward through the int8 base (dX via the dequantised weight + LoRA dgrad, dA, dB)
    dY = torch.randn(case.M, case.d_out, device=dev, dtype=torch.bfloat16)
    Xq, sx, Z = ops.w8a8_quantize_rows(X, A)

    def w8_bwd_step():   # through the prepacked dequantised weight
        ops.lora_linear_bwd(X, Wd, A, B, Z, dY, case.s)
    ms_b, _, _ = timed(w8_bwd_step, steps, warm)
    fb = 2 * case.M * case.d_in * case.d_out + 4 * case.M * case.r * (case.d_in + case.d_out)
    out["w8a8_lora_3072_bwd"] = {"ms_per_step": ms_b, "tflops": fb / (ms_b * 1e-3) / 1e12,
                                 "frac_of_bf16_peak": fb / (ms_b * 1e-3) / 1e12 / peaks["bf16_tflops"]}
    return out


def profile_steps(args, ops):
    """W + K forward + backward steps of one workload and nothing else (a profiler's view)."""
    import torch

    import datagen as D
    dev = torch.device("cuda", torch.cuda.current_device())
    kw = {"M": args.profile_m} if args.profile_m > 0 else {}
    if args.profile in ("lora", "dora"):
        case = D.scaled(D.WORKLOADS[HEADLINE if args.profile == "lora" else "dora_4096x11008_bf16"], **kw)
        g = {k: v.to(dev) for k, v in D.make_linear(case).items() if v is not None}
        if args.profile == "lora":
            def step():
                Y, Z = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], case.s)
                ops.lora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], Z, g["dY"], case.s)
        else:
            r0 = ops.dora_rownorm2(g["W0"])

            def step():
                Y, Z, n, V = ops.dora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], r0, case.s, case.eps,
                                                 g["bias"])
                ops.dora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], g["m"], g["bias"], Y, Z, n, V, g["dY"], case.s,
                                    case.eps)
    elif args.profile == "mlp":
        case = D.scaled(D.WORKLOADS["mlp_swiglu_4096x14336_bf16"], **kw)
        g = {k: v.to(dev) for k, v in D.make_mlp(case).items()}
        P = {p: {"W": g["W" + p], "A": g["A" + p], "B": g["B" + p], "s": case.s} for p in "gud"}

        def step():
            Y, saved = ops.lora_mlp_swiglu_fwd(g["X"], P["g"], P["u"], P["d"])
            ops.lora_mlp_swiglu_bwd(g["X"], P["g"], P["u"], P["d"], saved, g["dY"])
    elif args.profile == "dropout":
        case = D.scaled(D.WORKLOADS[HEADLINE], **kw)
        g = {k: v.to(dev) for k, v in D.make_linear(case).items() if v is not None}
        mask = D.make_dropout_mask(case.M, case.d_in, 0.1).to(dev)
        keep = 1.0 / 0.9

        def step():
            Y, Z = ops.lora_linear_dropout_fwd(g["X"], mask, keep, g["W0"], g["A"], g["B"], case.s)
            ops.lora_linear_dropout_bwd(g["X"], mask, keep, g["W0"], g["A"], g["B"], Z, g["dY"], case.s)
    elif args.profile == "qkv":
        case = D.scaled(D.WORKLOADS["qkv_lora_4096_gqa_bf16"], **kw)
        g = {k: v.to(dev) for k, v in D.make_qkv(case).items() if v is not None}
        leaves = [(g[f"A{l}"], g[f"B{l}"], case.s[l]) for l in range(len(case.n))]

        def step():
            Y, Z = ops.lora_qkv_fwd(g["X"], g["W0"], leaves)
            ops.lora_qkv_bwd(g["X"], g["W0"], leaves, Z, g["dY"])
    else:
        case = D.scaled(D.WORKLOADS["w8a8_lora_3072"], **kw)
        t = D.make_w8a8(case)
        X, A, B = t["X"].to(dev), t["A"].to(dev), t["B"].to(dev)
        Wq, swd, _ = ops.w8a8_quantize_rows(t["W0"].to(torch.bfloat16).to(dev))
        Wb, Wd = ops.w8a8_prepack_weight(Wq, swd)

        def step():
            Xc, sx, Z = ops.w8a8_quantize_rows_bf16(X, A)
            ops.w8a8_lora_fwd_packed(Xc, sx, Wb, swd, Z, B, case.s)
    for _ in range(args.warmup + args.steps):
        step()
    torch.cuda.synchronize()
    return {"profile": args.profile, "M": case.M, "steps": args.steps, "warmup": args.warmup}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workloads", default="all", choices=["all", "headline"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--min-timed-s", type=float, default=1.0,
                    help="repeat the timed region of K steps until the regions cover this many seconds")
    ap.add_argument("--profile", default=None, choices=["lora", "dora", "mlp", "qkv", "w8a8", "dropout"],
                    help="profiling aid: run only W + K steps of this workload (no timing, no context) so that a "
                         "profiler's launch list holds just those kernels")
    ap.add_argument("--profile-m", type=int, default=0, help="token rows of the --profile workload (0: its own)")
    ap.add_argument("--only", default=None, choices=["dora", "mlp", "w8a8", "qkv", "dropout"],
                    help="time one non-headline workload alone (for profiling) and print its record")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = tdist

    from dora_adapter_linear_gb300.build import build
    if rank == 0:
        build()
    if dist is not None:
        dist.barrier()
    from dora_adapter_linear_gb300 import _lib as L
    from dora_adapter_linear_gb300 import ops

    peaks = measured_peaks()
    if args.profile:
        print(json.dumps(profile_steps(args, ops)), flush=True)
        return
    if args.only:
        print(json.dumps(extra_workloads(args, L, ops, peaks, which=(args.only,))), flush=True)
        return
    h = headline(args, L, ops, dist, world, peaks)
    extra = extra_workloads(args, L, ops, peaks) if args.workloads == "all" and rank == 0 else None
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(h["value"], 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(h["ms_per_step"], 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded Gaussian inputs of the workload's shapes; random-init weights)",
            "config": {"workload": f"{HEADLINE}: LoRA linear fwd+bwd, M=8192 (batch 4 x seq 2048), "
                                   "d_in=d_out=4096, rank 16, alpha 32, no bias",
                       "global_batch": 4 * world, "seq_len": 2048, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2: X, dY 64 MiB each + W0 32 MiB + outputs per step (no flush)",
                       "flops_per_step": sum(lora_flops(8192, 4096, 4096, 16))},
            "tokens_per_s": round(h["tokens_per_s"]), "frac_of_bf16_peak": round(h["frac_of_bf16_peak_step"], 4),
            "timed_regions": h["timed_regions"], "fwd": h["fwd"], "bwd": h["bwd"],
            "peaks": peaks, "roofline": h["roofline"], "rank_passes": h["rank_passes"], "cpu_baseline": cpu,
            "e2e": h["e2e"], "gpu_launches": h["gpu_launches"], "clocks": h["clocks"], "context": h["context"],
            "largest_linear_config": None if not extra else {
                "workload": "dora_4096x11008_bf16 (DoRA rows fwd+bwd, M 8192, 4096 -> 11008, r 32)",
                "tflops": round(extra["dora_4096x11008_bf16"]["tflops"], 1),
                "frac_of_bf16_peak": round(extra["dora_4096x11008_bf16"]["frac_of_bf16_peak"], 4)},
            "workloads": extra,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
