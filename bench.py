#!/usr/bin/env python3
"""Benchmark of the grouped MoE backward GEMMs on one GB300 (or N replicas).

Default workload: MXFP8 grouped wgrad at the wgrad page's default shape,
M = N = K = 8192 tokens/features, E = 8 experts of 1024 tokens.  One step is the
whole hot path for that workload: MXFP8 quantize of g and of x, then the grouped
wgrad.  ``value`` is algorithmic wgrad FLOPs (2*M*N*K) per second of step time.
A secondary object measures the fp32 grouped dgrad (rows 4096, 1024 -> 1024,
E = 8, multinomial split).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def _source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "moe_grouped_gemm_wgrad_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic(kernel: str, src_files) -> float | None:
    """DRAM bytes per launch from a committed ncu summary, if taken on this source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        ent = t[kernel]
        if ent.get("source_hash") == _source_hash(src_files):
            return float(ent["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons, sampled every 50 ms; only the samples whose
    timestamps fall inside the timed window are summarised."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int, path: str | None = None, cmd: list | None = None,
                 settle_s: float = 1.0):
        """Starts sampling GPU ``gpu_index``; the raw lines also go to ``path`` if given.
        ``cmd`` replaces the nvidia-smi command line (same CSV columns)."""
        import threading

        self.proc = None
        self.path = path
        self.windows = {}
        self.lines = []
        try:
            if cmd is None:
                cmd = ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.Q}",
                       "--format=csv,noheader,nounits", "-lms", "50"]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        # drain the pipe continuously so that nvidia-smi never blocks on a full pipe
        self.reader = threading.Thread(target=self._drain, daemon=True)
        self.reader.start()
        time.sleep(settle_s)  # let the sampler come up before the timed region

    def _drain(self):
        for line in self.proc.stdout:
            self.lines.append(line)

    def mark(self, t0: float, t1: float, name: str = "step"):
        self.windows[name] = (t0, t1)

    def stop(self):
        """Stops sampling; returns {window name: summary} (the summary of all samples under
        "all" when no window saw a sample)."""
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.reader.join(timeout=5)
        if self.path is not None:
            with open(self.path, "w") as f:
                f.writelines(self.lines)
        import datetime

        rows = []
        for line in list(self.lines):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), float(parts[4]), parts[6:10]))
            except ValueError:
                continue

        def summary(use, n_inside):
            if not use:
                return None
            reasons = sorted({n for r in use for n, v in zip(self.NAMES, r[4]) if v.lower() == "active"})
            return {"sm_mhz": statistics.median(r[1] for r in use),
                    "sm_max_mhz": max(r[2] for r in use),
                    "power_w_median": statistics.median(r[3] for r in use), "reasons": reasons,
                    "samples": len(use), "samples_in_timed_window": n_inside}

        out = {}
        for name, (t0, t1) in self.windows.items():
            inside = [r for r in rows if t0 <= r[0] <= t1]
            out[name] = summary(inside if inside else rows, len(inside))
        out["all"] = summary(rows, 0)
        return out


# ----------------------------------------------------------------- workloads
def wgrad_case(name):
    from moe_grouped_gemm_wgrad_gb300 import synth

    if name == "moe_ffn_pair":
        return synth.moe_ffn_pair()[0]
    return getattr(synth, name)()


def dgrad_case(name):
    from moe_grouped_gemm_wgrad_gb300 import synth

    if name == "moe_ffn_pair":
        return synth.moe_ffn_pair()[1]
    return getattr(synth, name)()


def run_wgrad(name, steps, warmup, dist_ctx, clocks_csv=None, clock_leg_s=0.6):
    import torch

    from moe_grouped_gemm_wgrad_gb300 import mgw

    case = wgrad_case(name)
    dev = torch.device("cuda", torch.cuda.current_device())
    M, N, K, E = case.M, case.N, case.K, case.E
    flops = 2.0 * M * N * K
    Mcap = mgw.token_capacity(M, E)
    g_host = torch.from_numpy(case.g_bf16.view(np.int16)).view(torch.bfloat16).pin_memory()
    x_host = torch.from_numpy(case.x_bf16.view(np.int16)).view(torch.bfloat16).pin_memory()
    off_host = torch.from_numpy(case.expert_off).pin_memory()
    gather = "hidden_bf16" in case.meta  # x = hidden[token_of_row]: quantize by gather
    if gather:
        x_host = torch.from_numpy(case.meta["hidden_bf16"].view(np.int16)).view(torch.bfloat16).pin_memory()
        rows_host = torch.from_numpy(case.meta["token_of_row"]).pin_memory()
        rows_dev = rows_host.to(dev)
    g = g_host.to(dev)
    x = x_host.to(dev)
    off = off_host.to(dev)
    gq = torch.empty((N, Mcap), dtype=torch.uint8, device=dev)
    xq = torch.empty((K, Mcap), dtype=torch.uint8, device=dev)
    gs = torch.empty((mgw.scale_bytes(N, Mcap),), dtype=torch.uint8, device=dev)
    xs = torch.empty((mgw.scale_bytes(K, Mcap),), dtype=torch.uint8, device=dev)
    out = torch.empty((E * N, K), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def quant_x():
        if gather:
            mgw.mxfp8_quantize_gather(x, rows_dev, off, Mcap, xq, xs, status)
        else:
            mgw.mxfp8_quantize(x, off, Mcap, xq, xs, status)

    def step():
        mgw.mxfp8_quantize(g, off, Mcap, gq, gs, status)
        quant_x()
        mgw.grouped_wgrad_mxfp8(gq, gs, xq, xs, off, M, out, status)

    # raw clock samples go to a CSV only when asked for (one file per rank)
    csv_path = None if clocks_csv is None else f"{clocks_csv}.r{dist_ctx.rank}" if dist_ctx.world > 1 else clocks_csv
    clocks = ClockSampler(dist_ctx.local_rank, csv_path)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    # per-kernel events inside the timed region, on the launching stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    dist_ctx.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    host_t0 = time.time()
    t_start.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        mgw.mxfp8_quantize(g, off, Mcap, gq, gs, status)
        ev[i][1].record(stream)
        quant_x()
        ev[i][2].record(stream)
        mgw.grouped_wgrad_mxfp8(gq, gs, xq, xs, off, M, out, status)
        ev[i][3].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks.mark(host_t0, time.time(), "step")
    dist_ctx.barrier()
    # Clock leg: the wgrad kernel alone, back to back for at least `clock_leg_s` seconds,
    # so that its time carries SM clock samples taken while it ran (the step region above
    # can be shorter than the sampling period).
    leg = None
    if clock_leg_s > 0:
        per = max(1, int(clock_leg_s / 4 / max(statistics.mean(e[2].elapsed_time(e[3]) for e in ev) * 1e-3, 1e-6)))
        la, lb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_leg = 0
        torch.cuda.synchronize()
        h0 = time.time()
        la.record(stream)
        while time.time() - h0 < clock_leg_s:
            for _ in range(per):
                mgw.grouped_wgrad_mxfp8(gq, gs, xq, xs, off, M, out, status)
            n_leg += per
            torch.cuda.synchronize()
        lb.record(stream)
        torch.cuda.synchronize()
        clocks.mark(h0, time.time(), "wgrad_clock_leg")
        leg = {"launches": n_leg, "ms_per_launch": la.elapsed_time(lb) / n_leg,
               "seconds": la.elapsed_time(lb) * 1e-3}
    clk_all = clocks.stop()
    clk = clk_all.get("step") if clk_all else None
    if leg is not None and clk_all:
        c = clk_all.get("wgrad_clock_leg")
        leg["clocks"] = c
        if c:
            leg["tflops"] = flops / (leg["ms_per_launch"] * 1e-3) / 1e12
            leg["us_x_mhz"] = leg["ms_per_launch"] * 1e3 * c["sm_mhz"]
    total_ms = dist_ctx.max(t_start.elapsed_time(t_end))
    wg_ms = [e[2].elapsed_time(e[3]) for e in ev]
    qg_ms = [e[0].elapsed_time(e[1]) for e in ev]
    qx_ms = [e[1].elapsed_time(e[2]) for e in ev]
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")

    # End to end through the public API: every step copies its inputs from pinned host
    # memory and its grad_w back to pinned host memory.  Steps are pipelined the way a
    # training loop would run them: inputs and outputs are double-buffered on the device,
    # and host-to-device copies, the kernels and device-to-host copies run on three streams
    # ordered by events, so step i's grad_w download overlaps step i+1's upload and compute.
    out_host = torch.empty((E * N, K), dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(4, min(steps, 40))
    s_h2d, s_comp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    bufs = []
    for j in range(2):
        bufs.append({
            "g": g if j == 0 else torch.empty_like(g), "x": x if j == 0 else torch.empty_like(x),
            "off": off if j == 0 else torch.empty_like(off),
            "rows": (rows_dev if j == 0 else torch.empty_like(rows_dev)) if gather else None,
            "out": out if j == 0 else torch.empty_like(out),
            "in_free": torch.cuda.Event(), "in_ready": torch.cuda.Event(),
            "out_ready": torch.cuda.Event(), "out_free": torch.cuda.Event()})
    for bf in bufs:  # nothing in flight yet
        bf["in_free"].record(s_comp)
        bf["out_free"].record(s_d2h)

    def e2e_step(i):
        bf = bufs[i % 2]
        with torch.cuda.stream(s_h2d):
            s_h2d.wait_event(bf["in_free"])
            bf["g"].copy_(g_host, non_blocking=True)
            bf["x"].copy_(x_host, non_blocking=True)
            bf["off"].copy_(off_host, non_blocking=True)
            if gather:
                bf["rows"].copy_(rows_host, non_blocking=True)
            bf["in_ready"].record(s_h2d)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(bf["in_ready"])
            s_comp.wait_event(bf["out_free"])
            mgw.mxfp8_quantize(bf["g"], bf["off"], Mcap, gq, gs, status, stream=s_comp)
            if gather:
                mgw.mxfp8_quantize_gather(bf["x"], bf["rows"], bf["off"], Mcap, xq, xs, status, stream=s_comp)
            else:
                mgw.mxfp8_quantize(bf["x"], bf["off"], Mcap, xq, xs, status, stream=s_comp)
            mgw.grouped_wgrad_mxfp8(gq, gs, xq, xs, bf["off"], M, bf["out"], status, stream=s_comp)
            bf["in_free"].record(s_comp)
            bf["out_ready"].record(s_comp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(bf["out_ready"])
            out_host.copy_(bf["out"], non_blocking=True)
            bf["out_free"].record(s_d2h)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    dist_ctx.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_h2d)
    for i in range(e2e_steps):
        e2e_step(i)
    # the timed region ends when the last step's grad_w has reached the host
    s_h2d.wait_stream(s_d2h)
    b.record(s_h2d)
    torch.cuda.synchronize()
    e2e_ms = dist_ctx.max(a.elapsed_time(b)) / e2e_steps
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the end-to-end leg")
    # same inputs, deterministic kernels: the downloaded grad_w equals the device-timed one
    if not torch.equal(out_host[:: max(1, out_host.shape[0] // 64)].to(dev), out[:: max(1, out.shape[0] // 64)]):
        raise RuntimeError("end-to-end grad_w differs from the device-timed grad_w")
    h2d = g_host.numel() * 2 + x_host.numel() * 2 + off_host.numel() * 4 + (rows_host.numel() * 4 if gather else 0)
    d2h = out_host.numel() * 2

    ms_step = total_ms / steps
    wg_avg = statistics.mean(wg_ms)
    bytes_q = lambda C: M * C * 2 + C * Mcap + C * Mcap // 32  # noqa: E731
    # gathered x reads each source row once per routed copy (HBM once, the rest from L2);
    # the bytes counted here are the routed rows, as for the materialised operand
    return {
        "case": case, "flops": flops, "ms_per_step": ms_step, "wgrad_ms": wg_avg,
        "wgrad_ms_median": statistics.median(wg_ms), "quant_g_ms": statistics.mean(qg_ms),
        "quant_x_ms": statistics.mean(qx_ms), "e2e_ms": e2e_ms, "h2d": h2d, "d2h": d2h,
        "clocks": clk, "clock_leg": leg, "launches": 3 * steps, "x_gather": gather,
        "quant_bytes": bytes_q(N) + bytes_q(K),
        "wgrad_min_bytes": N * Mcap + K * Mcap + (N + K) * Mcap // 32 + E * N * K * 2,
    }


def run_dgrad(name, steps, warmup):
    import torch

    from moe_grouped_gemm_wgrad_gb300 import mgw

    case = dgrad_case(name)
    dev = torch.device("cuda", torch.cuda.current_device())
    dy = torch.from_numpy(case.dy).to(dev)
    W = torch.from_numpy(case.W).to(dev)
    off = torch.from_numpy(case.expert_off).to(dev)
    dx = torch.empty((case.rows, case.in_f), dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        mgw.grouped_dgrad_f32(dy, W, off, dx)
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush.fill_(1.0)  # L2 flush between timed launches (256 MB > 129 MB L2)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        mgw.grouped_dgrad_f32(dy, W, off, dx)
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in times]
    flops = 2.0 * case.rows * case.out_f * case.in_f
    return {"workload": name, "tflops": flops / (statistics.mean(ms) * 1e-3) / 1e12,
            "ms": statistics.mean(ms), "ms_median": statistics.median(ms),
            "rows": case.rows, "out_features": case.out_f, "in_features": case.in_f, "experts": case.E,
            "l2": "flushed between launches (256 MB write)"}


def run_mx_pair(name, steps, warmup):
    """The MXFP8 forward and data-gradient GEMMs of the MoE FFN pair: per step the routed
    rows are gathered and quantized along hidden, W is quantized both ways, then
    y = x W[e]^T and dx = dy W[e].  Per-kernel CUDA events; every operand is larger
    than L2 or read once per step."""
    import torch

    from moe_grouped_gemm_wgrad_gb300 import mgw

    from moe_grouped_gemm_wgrad_gb300 import synth

    if name == "moe_ffn_small":  # 2048 tokens x top-8 of 16 experts: a small profiling case
        wg, dg = synth.moe_ffn_pair(tokens=2048, E=16)
    else:
        wg, dg = wgrad_case(name), dgrad_case(name)
    dev = torch.device("cuda", torch.cuda.current_device())
    E, N, K, M = wg.E, wg.N, wg.K, wg.M
    w_off_h = np.arange(E + 1, dtype=np.int32) * N
    hidden = torch.from_numpy(wg.meta["hidden_bf16"].view(np.int16)).to(dev).view(torch.bfloat16)
    tok = torch.from_numpy(wg.meta["token_of_row"]).to(dev)
    dy = torch.from_numpy(wg.g_bf16.view(np.int16)).to(dev).view(torch.bfloat16)
    W = torch.from_numpy(synth.bf16_bits_from_f32(dg.W.reshape(E * N, K)).view(np.int16)).to(dev).view(torch.bfloat16)
    off = torch.from_numpy(wg.expert_off).to(dev)
    w_off = torch.from_numpy(w_off_h).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    Mcap = mgw.token_capacity(M, E)
    xq, xs = mgw.mxfp8_quantize_rows(hidden, off, Mcap, row_index=tok, status=status)
    wq, ws = mgw.mxfp8_quantize_rows(W, w_off, status=status)
    dyq, dys = mgw.mxfp8_quantize_rows(dy, off, Mcap, status=status)
    wtq, wts = mgw.mxfp8_quantize(W, w_off, status=status)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def kernels():
        return [
            lambda: mgw.mxfp8_quantize_rows(hidden, off, Mcap, xq, xs, status, row_index=tok),
            lambda: mgw.mxfp8_quantize_rows(W, w_off, wq.shape[0], wq, ws, status),
            lambda: mgw.grouped_fprop_mxfp8(xq, xs, wq, ws, off, M, N, y, status),
            lambda: mgw.mxfp8_quantize_rows(dy, off, Mcap, dyq, dys, status),
            lambda: mgw.mxfp8_quantize(W, w_off, wtq.shape[1], wtq, wts, status),
            lambda: mgw.grouped_dgrad_mxfp8(dyq, dys, wtq, wts, off, M, dx, status),
        ]

    ks = kernels()
    for _ in range(warmup):
        for k in ks:
            k()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ks) + 1)] for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        for j, k in enumerate(ks):
            k()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    ms = [statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev) for j in range(len(ks))]
    flops = 2.0 * M * N * K
    names = ["quantize_rows_x_gather", "quantize_rows_w", "grouped_fprop_mxfp8", "quantize_rows_dy",
             "quantize_w_along_n", "grouped_dgrad_mxfp8"]
    return {"workload": name, "rows": M, "ffn": N, "hidden": K, "experts": E,
            "kernels_ms": dict(zip(names, ms)),
            "fprop_tflops": flops / (ms[2] * 1e-3) / 1e12, "dgrad_mx_tflops": flops / (ms[5] * 1e-3) / 1e12,
            "launches_per_step": len(ks)}


def run_wgrad_kernels(name, steps, warmup):
    """The static and the load-balanced wgrad kernels on one workload, launches alternated,
    each timed with CUDA events (output larger than L2)."""
    import torch

    from moe_grouped_gemm_wgrad_gb300 import mgw

    case = wgrad_case(name)
    dev = torch.device("cuda", torch.cuda.current_device())
    off = torch.from_numpy(case.expert_off).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    Mcap = mgw.token_capacity(case.M, case.E)
    g = torch.from_numpy(case.g_bf16.view(np.int16)).to(dev).view(torch.bfloat16)
    if "hidden_bf16" in case.meta:
        hidden = torch.from_numpy(case.meta["hidden_bf16"].view(np.int16)).to(dev).view(torch.bfloat16)
        rows = torch.from_numpy(case.meta["token_of_row"]).to(dev)
        xq, xs = mgw.mxfp8_quantize_gather(hidden, rows, off, Mcap, status=status)
    else:
        x = torch.from_numpy(case.x_bf16.view(np.int16)).to(dev).view(torch.bfloat16)
        xq, xs = mgw.mxfp8_quantize(x, off, Mcap, status=status)
    gq, gs = mgw.mxfp8_quantize(g, off, Mcap, status=status)
    out = torch.empty((case.E * case.N, case.K), dtype=torch.bfloat16, device=dev)
    ws = mgw.wgrad_workspace(case.E, case.N, case.K)
    stream = torch.cuda.current_stream()
    kern = {
        "static": lambda: mgw.grouped_wgrad_mxfp8(gq, gs, xq, xs, off, case.M, out, status),
        "balanced": lambda: mgw.grouped_wgrad_mxfp8_balanced(gq, gs, xq, xs, off, case.M, ws, out, status),
    }
    for _ in range(warmup):
        for k in kern.values():
            k()
    torch.cuda.synchronize()
    ev = {n: [] for n in kern}
    for _ in range(steps):
        for n, k in kern.items():
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            k()
            b.record(stream)
            ev[n].append((a, b))
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    flops = 2.0 * case.M * case.N * case.K
    nbytes = (case.N + case.K) * Mcap * (1 + 1 / 32) + case.E * case.N * case.K * 2
    res = {"workload": case.name, "M": case.M, "N": case.N, "K": case.K, "experts": case.E}
    for n in kern:
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev[n])
        res[n] = {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12, "hbm_gbs": nbytes / (ms * 1e-3) / 1e9}
    res["algorithmic_bytes"] = nbytes
    return res


def run_wgrad_step_leg(name, steps, warmup, graph_steps=0):
    """One workload's whole wgrad step -- quantize g, quantize x (gathered from the hidden
    states by the routing map when the workload has one), grouped wgrad -- with CUDA events
    around each launch, steps back to back.  For the tiny workload the step time is
    dominated by launch latency; for the larger ones the output exceeds L2."""
    import torch

    from moe_grouped_gemm_wgrad_gb300 import mgw

    case = wgrad_case(name)
    dev = torch.device("cuda", torch.cuda.current_device())
    M, N, K, E = case.M, case.N, case.K, case.E
    off = torch.from_numpy(case.expert_off).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    Mcap = mgw.token_capacity(M, E)
    g = torch.from_numpy(case.g_bf16.view(np.int16)).to(dev).view(torch.bfloat16)
    gather = "hidden_bf16" in case.meta
    if gather:
        x = torch.from_numpy(case.meta["hidden_bf16"].view(np.int16)).to(dev).view(torch.bfloat16)
        rows = torch.from_numpy(case.meta["token_of_row"]).to(dev)
    else:
        x = torch.from_numpy(case.x_bf16.view(np.int16)).to(dev).view(torch.bfloat16)
    gq = torch.empty((N, Mcap), dtype=torch.uint8, device=dev)
    xq = torch.empty((K, Mcap), dtype=torch.uint8, device=dev)
    gs = torch.empty((mgw.scale_bytes(N, Mcap),), dtype=torch.uint8, device=dev)
    xs = torch.empty((mgw.scale_bytes(K, Mcap),), dtype=torch.uint8, device=dev)
    out = torch.empty((E * N, K), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    ks = [lambda: mgw.mxfp8_quantize(g, off, Mcap, gq, gs, status),
          (lambda: mgw.mxfp8_quantize_gather(x, rows, off, Mcap, xq, xs, status)) if gather
          else (lambda: mgw.mxfp8_quantize(x, off, Mcap, xq, xs, status)),
          lambda: mgw.grouped_wgrad_mxfp8(gq, gs, xq, xs, off, M, out, status)]
    for _ in range(warmup):
        for k in ks:
            k()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ks) + 1)] for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        for j, k in enumerate(ks):
            k()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    ms = [statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev) for j in range(len(ks))]
    step_ms = statistics.mean(e[0].elapsed_time(e[-1]) for e in ev)
    flops = 2.0 * M * N * K
    wg_bytes = N * Mcap + K * Mcap + (N + K) * Mcap // 32 + E * N * K * 2
    graph = None
    if graph_steps > 0:
        # The same launches captured once into a CUDA graph and replayed: the device time
        # of a step without the host's per-call work between launches.
        cg = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for k in ks:  # one eager pass on the capture stream first
                k()
        torch.cuda.synchronize()
        with torch.cuda.graph(cg, stream=side):
            for _ in range(graph_steps):
                for k in ks:
                    k()
        cg.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        cg.replay()
        b.record(stream)
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())} in the graph replay")
        gms = a.elapsed_time(b) / graph_steps
        graph = {"steps_per_graph": graph_steps, "step_ms": gms,
                 "step_tflops": flops / (gms * 1e-3) / 1e12}
    return {"workload": case.name, "M": M, "N": N, "K": K, "experts": E,
            "x": "gathered from hidden[token_of_row]" if gather else "materialised",
            "kernels_ms": {"mxfp8_quantize_g": ms[0],
                           "mxfp8_quantize_gather_x" if gather else "mxfp8_quantize_x": ms[1],
                           "grouped_wgrad": ms[2]},
            "step_ms": step_ms, "step_tflops": flops / (step_ms * 1e-3) / 1e12,
            "wgrad_tflops": flops / (ms[2] * 1e-3) / 1e12,
            "wgrad_hbm_gbs": wg_bytes / (ms[2] * 1e-3) / 1e9, "wgrad_algorithmic_bytes": wg_bytes,
            "launches_per_step": len(ks), "cuda_graph": graph}


def measure_dense_peaks(n: int = 8192, reps: int = 10):
    """Dense GEMM rates of the vendor library on this GPU at n^3, best of ``reps`` with CUDA
    events after three warm-up calls: block-scaled MXFP8 (torch._scaled_mm on e4m3 operands
    with one e8m0 scale per 32 elements of K), TF32 (fp32 torch.matmul with TF32 allowed)
    and bf16.  These are denominators for the roofline fractions, measured beside them."""
    import torch

    dev = torch.device("cuda", torch.cuda.current_device())
    flops = 2.0 * n ** 3
    res = {"n": n, "how": f"best of {reps}, CUDA events, {n}^3, torch {torch.__version__}"}

    def best(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        t = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            t.append((a, b))
        torch.cuda.synchronize()
        return flops / (min(a.elapsed_time(b) for a, b in t) * 1e-3) / 1e12

    A = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    B = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    res["bf16_tflops"] = best(lambda: A @ B)
    a8 = A.to(torch.float8_e4m3fn)
    b8 = B.to(torch.float8_e4m3fn).t().contiguous().t()
    try:
        e8 = torch.float8_e8m0fnu
        sa = torch.full((n * (n // 32),), 127, dtype=torch.uint8, device=dev).view(e8)
        sb = torch.full((n * (n // 32),), 127, dtype=torch.uint8, device=dev).view(e8)
        res["mxfp8_tflops"] = best(lambda: torch._scaled_mm(a8, b8, sa, sb, out_dtype=torch.bfloat16))
    except Exception as exc:  # an older torch without block-scaled MXFP8
        res["mxfp8_error"] = repr(exc)[:200]
    del a8, b8
    Af, Bf = A.float(), B.float()
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        res["tf32_tflops"] = best(lambda: Af @ Bf)
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    del A, B, Af, Bf
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------ CPU baseline
def oracle_wgrad_sample(case, n_sub: int, k_sub: int):
    """Times the oracle (as it stands, single thread) on expert 0's tokens for an
    n_sub x k_sub block of grad_w, including its quantization of that slice.
    Returns (seconds, flops, description)."""
    import oracle

    off = case.expert_off
    e = int(np.argmax(np.diff(off) > 0))
    t0, t1 = int(off[e]), int(off[e + 1])
    g = np.ascontiguousarray(case.g_bf16[t0:t1, :n_sub])
    x = np.ascontiguousarray(case.x_bf16[t0:t1, :k_sub])
    sub_off = [0, t1 - t0]
    oracle.build()
    start = time.perf_counter()
    gq, gs = oracle.mxfp8_quantize(g, sub_off)
    xq, xs = oracle.mxfp8_quantize(x, sub_off)
    oracle.grouped_wgrad(gq, gs, xq, xs, sub_off)
    sec = time.perf_counter() - start
    flops = 2.0 * (t1 - t0) * n_sub * k_sub
    return sec, flops, f"expert {e} ({t1 - t0} tokens), grad_w block {n_sub}x{k_sub}, quantize+wgrad, 1 thread"


def cpu_baseline(case, target_s: float = 16.0):
    """About target_s seconds of oracle work (10-30 s on the hosts measured): a
    1024 x 1024 pilot block, large enough that the quantization of the slice does not
    dominate, then a square block scaled by area."""
    pilot_n, pilot_k = min(1024, case.N), min(1024, case.K)
    sec, _, _ = oracle_wgrad_sample(case, pilot_n, pilot_k)
    scale = max(1.0, (target_s / max(sec, 1e-3)) ** 0.5)
    n_sub = int(min(case.N, max(128, 128 * round(pilot_n * scale / 128))))
    k_sub = int(min(case.K, max(128, 128 * round(pilot_k * scale / 128))))
    sec, flops, desc = oracle_wgrad_sample(case, n_sub, k_sub)
    return {"value": flops / sec / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": desc, "seconds": sec}


# --------------------------------------------------------------- dist glue
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend="nccl"):
        import torch

        if self.world > 1:
            import torch.distributed as dist

            if backend == "nccl":
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if self.pg is None:
            return v
        import torch

        t = torch.tensor([v], dtype=torch.float64,
                         device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mgw", "reference"], default="mgw")
    ap.add_argument("--workload", default="wgrad_8192",
                    choices=["wgrad_tiny", "wgrad_8192", "wgrad_skew", "moe_ffn_pair"])
    ap.add_argument("--dgrad-workloads", default="dgrad_4096,moe_ffn_pair",
                    help="comma list of fp32 dgrad legs (dgrad_4096, moe_ffn_pair; moe_ffn_slice, a "
                         "16-expert slice for profiler captures) or none")
    ap.add_argument("--wgrad-step-workloads", default="wgrad_tiny,moe_ffn_pair",
                    help="comma list of extra whole-step wgrad legs (wgrad_tiny, wgrad_skew, "
                         "moe_ffn_pair) or none")
    ap.add_argument("--mx-workload", default="moe_ffn_pair", choices=["moe_ffn_pair", "moe_ffn_small", "none"])
    ap.add_argument("--skew-workload", default="wgrad_skew",
                    choices=["wgrad_skew", "wgrad_8192", "moe_ffn_pair", "none"])
    ap.add_argument("--clock-leg-s", type=float, default=0.6,
                    help="seconds of back-to-back wgrad launches timed under clock sampling (0: off)")
    ap.add_argument("--no-peak-probe", action="store_true",
                    help="skip measuring the vendor library's MXFP8 / TF32 / bf16 GEMM rates")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-csv", default=None,
                    help="also write the raw nvidia-smi clock samples of the timed step to this CSV")
    args = ap.parse_args()
    peaks = _peaks()
    # Contract denominators: the measured bf16 dense rate times the nominal fp8 : bf16 (4.5 :
    # 2.25) and tf32 : bf16 (1.1 : 2.25, taken as 1/2) ratios; the sustained figure applies to
    # a kernel timed inside a long loop.  The vendor library's own MXFP8 and TF32 rates,
    # measured in this run, are reported beside them.
    mxfp8_burst = 2.0 * peaks["bf16_tflops"]
    mxfp8_sustained = 2.0 * (peaks["bf16_tflops_sustained"] or peaks["bf16_tflops"])
    metric = "MXFP8 grouped wgrad TFLOP/s"
    d = Dist()

    if args.impl == "reference":
        if d.rank != 0:
            return
        case = wgrad_case(args.workload)
        # bounded sample per step: expert 0's tokens, a 256 x 256 block of grad_w
        for _ in range(args.warmup):
            oracle_wgrad_sample(case, 128, 128)
        secs, flops = [], 0.0
        desc = ""
        for _ in range(args.steps):
            s, f, desc = oracle_wgrad_sample(case, 256, 256)
            secs.append(s)
            flops = f
        v = flops * len(secs) / sum(secs) / 1e12
        line = {"impl": "reference", "metric": metric, "value": v, "unit": "TFLOP/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * sum(secs) / len(secs), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": args.workload, "M": case.M, "N": case.N, "K": case.K,
                           "experts": case.E, "sample": desc},
                "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    d.init("nccl")
    torch.cuda.set_device(d.local_rank)
    from moe_grouped_gemm_wgrad_gb300 import build as _build

    _build.build()  # no-op when current
    lst = lambda v: [w for w in v.split(",") if w and w != "none"]  # noqa: E731
    r = run_wgrad(args.workload, args.steps, args.warmup, d, args.clocks_csv, args.clock_leg_s)
    legs_steps, legs_warm = max(5, min(args.steps, 50)), max(3, args.warmup)
    dgs = {w: run_dgrad(w, legs_steps, legs_warm) for w in lst(args.dgrad_workloads)}
    wsteps = {w: run_wgrad_step_leg(w, max(5, min(args.steps, 100 if w == "wgrad_tiny" else 20)), legs_warm,
                                    graph_steps=100 if w == "wgrad_tiny" else 0)
              for w in lst(args.wgrad_step_workloads)}
    sk = None
    if args.skew_workload != "none":
        sk = run_wgrad_kernels(args.skew_workload, legs_steps, legs_warm)
    mx = None
    if args.mx_workload != "none":
        mx = run_mx_pair(args.mx_workload, max(5, min(args.steps, 20)), legs_warm)
    dense = None
    if not args.no_peak_probe:
        dense = measure_dense_peaks()
    case = r["case"]
    value = r["flops"] * d.world / (r["ms_per_step"] * 1e-3) / 1e12
    wg_tflops = r["flops"] / (r["wgrad_ms"] * 1e-3) / 1e12
    # the sustained denominator for a timed region of half a second or more, else burst
    long_region = r["ms_per_step"] * args.steps >= 500.0
    peak_kind = "sustained" if long_region else "burst"
    mxfp8_peak = mxfp8_sustained if peak_kind == "sustained" else mxfp8_burst
    tf32_peak = peaks["bf16_tflops"] / 2.0
    mx_meas = (dense or {}).get("mxfp8_tflops")
    tf32_meas = (dense or {}).get("tf32_tflops")
    cpu = None
    if d.rank == 0 and d.world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(case)
    if d.rank == 0:
        # the CTA-pair kernel serves N % 256 == 0 (every workload here), the single-SM one the rest
        wg_kernel = "grouped_wgrad_pair_kernel" if case.N % 256 == 0 else "grouped_wgrad_kernel"
        note = (f"peak = 2 x measured bf16 dense ({peaks['source']}, MEASURED_PEAKS): burst "
                f"{mxfp8_burst:.1f}, sustained {mxfp8_sustained:.1f} TFLOP/s (fp8:bf16 nominal 2)")
        if mx_meas:
            note += (f"; measured in this run: cuBLAS MXFP8 (torch._scaled_mm, e8m0 32-blocks) "
                     f"{mx_meas:.1f}, cuBLAS TF32 {tf32_meas:.1f} TFLOP/s at 8192^3")
        roof = {"bound": "tensor", "achieved": wg_tflops, "peak": mxfp8_peak,
                "unit": "TFLOP/s", "frac": wg_tflops / mxfp8_peak,
                "traffic": _traffic(wg_kernel, ["wgrad.cu", "ptx.cuh", "common.cuh"]),
                "kernel": wg_kernel, "peak_kind": peak_kind,
                "frac_of_burst": wg_tflops / mxfp8_burst,
                "algorithmic_bytes": r["wgrad_min_bytes"], "peak_note": note}
        if mx_meas:
            roof["frac_of_measured_mxfp8"] = wg_tflops / mx_meas
        line = {
            "metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": d.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "mxfp8-e4m3 (fp32 accumulate, bf16 out)", "data": "synthetic",
            "config": {"workload": case.name, "M": case.M, "N": case.N, "K": case.K, "experts": case.E,
                       "step": ("mxfp8_quantize(g) + mxfp8_quantize_gather(hidden, token_of_row) + grouped_wgrad_mxfp8"
                                if r["x_gather"] else "mxfp8_quantize(g) + mxfp8_quantize(x) + grouped_wgrad_mxfp8"),
                       "l2": "inputs larger than L2 (bf16 g,x 2x134 MB; grad_w 1.07 GB per step)",
                       "parallelism": f"replicas x{d.world} (independent workloads, no collective)"},
            "roofline": roof,
            "kernels_ms": {"mxfp8_quantize_g": r["quant_g_ms"], "mxfp8_quantize_x": r["quant_x_ms"],
                           "grouped_wgrad": r["wgrad_ms"], "grouped_wgrad_median": r["wgrad_ms_median"]},
            "quantize_hbm": {"achieved_gbs": r["quant_bytes"] / ((r["quant_g_ms"] + r["quant_x_ms"]) * 1e-3) / 1e9,
                             "peak_gbs": peaks["hbm_gbs"],
                             "frac": r["quant_bytes"] / ((r["quant_g_ms"] + r["quant_x_ms"]) * 1e-3) / 1e9 / peaks["hbm_gbs"]},
            "e2e": {"value": r["flops"] * d.world / (r["e2e_ms"] * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "ms_per_step": r["e2e_ms"]},
            "gpu_launches": r["launches"],
            "clocks": r["clocks"],
            "cpu_baseline": cpu,
        }
        if r.get("clock_leg"):
            leg = r["clock_leg"]
            if leg.get("tflops"):
                leg["frac"] = leg["tflops"] / mxfp8_sustained
                leg["frac_note"] = "against the sustained denominator (a long back-to-back loop)"
            line["wgrad_clock_leg"] = leg
        if dense is not None:
            line["dense_peaks_measured"] = dense
        for w, dg in dgs.items():
            dg["roofline"] = {"bound": "tensor", "tf32_work_tflops": 3 * dg["tflops"], "peak": tf32_peak,
                              "unit": "TFLOP/s", "frac": 3 * dg["tflops"] / tf32_peak,
                              "note": "3xTF32: three tf32 MMAs per fp32 product; peak = measured bf16 / 2"}
            if tf32_meas:
                dg["roofline"]["frac_of_measured_tf32"] = 3 * dg["tflops"] / tf32_meas
            line["dgrad" if w == "dgrad_4096" else f"dgrad_{w}"] = dg
        for w, ws_ in wsteps.items():
            ws_["wgrad_frac_of_burst"] = ws_["wgrad_tflops"] / mxfp8_burst
            if mx_meas:
                ws_["wgrad_frac_of_measured_mxfp8"] = ws_["wgrad_tflops"] / mx_meas
            ws_["wgrad_hbm_frac"] = ws_["wgrad_hbm_gbs"] / peaks["hbm_gbs"]
            line[f"wgrad_step_{w}"] = ws_
        if sk is not None:
            for k in ("static", "balanced"):
                sk[k]["hbm_frac"] = sk[k]["hbm_gbs"] / peaks["hbm_gbs"]
                sk[k]["tensor_frac_of_burst"] = sk[k]["tflops"] / mxfp8_burst
            line["wgrad_static_vs_balanced"] = sk
        if mx is not None:
            for key in ("fprop_tflops", "dgrad_mx_tflops"):
                mx[key.replace("tflops", "frac_of_burst")] = mx[key] / mxfp8_burst
                if mx_meas:
                    mx[key.replace("tflops", "frac_of_measured_mxfp8")] = mx[key] / mx_meas
            line["mx_forward_dgrad"] = mx
        # the five workload configurations, one line each
        cfgs = {"wgrad_8192": {"wgrad_ms": r["wgrad_ms"], "wgrad_tflops": wg_tflops,
                               "frac_of_burst": wg_tflops / mxfp8_burst}}
        if "wgrad_tiny" in wsteps:
            t = wsteps["wgrad_tiny"]
            cfgs["wgrad_tiny"] = {"step_ms": t["step_ms"], "wgrad_ms": t["kernels_ms"]["grouped_wgrad"],
                                  "wgrad_tflops": t["wgrad_tflops"], "bound": "launch latency",
                                  "graph_step_ms": (t["cuda_graph"] or {}).get("step_ms")}
        if "dgrad_4096" in dgs:
            cfgs["dgrad_4096"] = {"ms": dgs["dgrad_4096"]["ms"], "tflops_fp32": dgs["dgrad_4096"]["tflops"],
                                  "frac_tf32": dgs["dgrad_4096"]["roofline"]["frac"]}
        if sk is not None and sk["workload"] == "wgrad_skew":
            cfgs["wgrad_skew"] = {"static_ms": sk["static"]["ms"], "balanced_ms": sk["balanced"]["ms"],
                                  "balanced_hbm_frac": sk["balanced"]["hbm_frac"]}
        if "moe_ffn_pair" in wsteps or "moe_ffn_pair" in dgs:
            m = {}
            if "moe_ffn_pair" in wsteps:
                t = wsteps["moe_ffn_pair"]
                m.update({"wgrad_ms": t["kernels_ms"]["grouped_wgrad"], "wgrad_tflops": t["wgrad_tflops"],
                          "wgrad_frac_of_burst": t["wgrad_frac_of_burst"]})
            if "moe_ffn_pair" in dgs:
                m.update({"dgrad_f32_ms": dgs["moe_ffn_pair"]["ms"], "dgrad_f32_tflops": dgs["moe_ffn_pair"]["tflops"],
                          "dgrad_f32_frac_tf32": dgs["moe_ffn_pair"]["roofline"]["frac"]})
            cfgs["moe_ffn_pair"] = m
        line["configs"] = cfgs
        print(json.dumps(line))
    d.close()


if __name__ == "__main__":
    main()
