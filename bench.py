#!/usr/bin/env python3
"""Benchmark of the ternary-weight linear layer on GB300.

Headline metric: ternary linear weight GB/s at T = 1 (decode GEMV), as a
fraction of the measured HBM peak; alongside it, int8-operand TOPS of the s8
prefill rung at T = 2048.

Step (N = 1): one T = 1 decode pass over a stack of L layers of the 27B-like
MLP projections (fused gate+up 5120 x 34816, then down 17408 x 5120), weights
resident in HBM, captured once as a CUDA graph and replayed.  The stack holds
L * 71 MB of packed weights (L = 8: 570 MB, more than 4x the 129 MB L2), so a
step streams every weight byte from HBM; no L2 flush is needed.

Inputs are synthetic and seeded (ternary with P(0) = 0.4, log-normal group
scales, N(0,1) activations with 1% outlier channels x20), generated on the
device.  The weights are packed by the library's own tern_pack.

Reference arm (--impl reference): the CPU oracle (the library's test
definition, plain C) timed on this host's cores on a bounded sample of the
same step.  Multi-GPU (torchrun): every rank runs its own replica (the layer
does not shard); value is the sum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

GU = (5120, 2 * 17408)
DN = (17408, 5120)
AI = (5120, 6144)   # attention-like in
AO = (6144, 5120)   # attention-like out
STACK_LAYERS = 64
GROUP = 128


def weight_bytes(K, N):
    return K * N // 4 + N * (K // GROUP) * 2


def algorithmic_bytes(T, K, N):
    """Bytes one call must move at least: packed weights, scales, bf16 x, fp32 y."""
    return weight_bytes(K, N) + 2 * T * K + 4 * T * N


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--profile", choices=["gu", "dn", "s8gu", "s8dn"], default=None,
                    help="only call tern_linear on one projection at T=1 (for profilers)")
    ap.add_argument("--profile-calls", type=int, default=3)
    ap.add_argument("--profile-t", type=int, default=None,
                    help="token count for --profile (default 1 for gu/dn, 2048 for s8gu/s8dn)")
    ap.add_argument("--no-stack", action="store_true",
                    help="skip the 64-layer whole-stack passes")
    ap.add_argument("--formats", action="store_true",
                    help="only time the base-3 weight repack and the Hadamard rotation")
    ap.add_argument("--sweep", action="store_true",
                    help="only time every projection at every token count of the configs")
    return ap.parse_args()


# ---------------------------------------------------------------- helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(ms, world, device):
    """The job's time for a region that every rank timed on its own GPU: the
    largest per-rank figure (each replica runs the same work, so the job ends
    with the slowest one).  world == 1 returns ms unchanged."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world, bytes_per_rank_step, ms_per_step):
    """Aggregate weight GB/s of world independent replicas, each streaming the
    same bytes per step, over the job's (slowest rank's) time per step."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def profile_traffic(kernel_src, summary_name):
    """DRAM bytes per launch recorded by the committed ncu summary, or None if
    the kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", summary_name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_sha = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    if not m_bytes or not m_sha:
        return None
    with open(kernel_src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    return float(m_bytes.group(1)) if sha == m_sha.group(1) else None


# ---------------------------------------------------------------- ours

def make_layer(tl, torch, K, N, gen, dev):
    # ternary weights with P(0) = 0.4, P(+1) = P(-1) = 0.3
    r = torch.randint(0, 10, (N, K), generator=gen, device=dev, dtype=torch.int8)
    W = torch.zeros_like(r)
    W[(r >= 4) & (r < 7)] = 1
    W[r >= 7] = -1
    Wp = tl.tern_pack(W)
    del r, W
    s = torch.exp(torch.randn(N, K // GROUP, generator=gen, device=dev) * 0.3 - 3.5).half()
    return Wp, s


def make_x(torch, T, K, gen, dev):
    x = torch.randn(T, K, generator=gen, device=dev)
    ch = torch.randperm(K, generator=gen, device=dev)[: max(1, round(0.01 * K))]
    x[:, ch] *= 20.0
    return x.bfloat16()


def run_stack(tl, torch, gen, dev, peaks, stream):
    """The whole-stack family: STACK_LAYERS resident layers of (gate+up, down,
    attention-like in and out), one full pass at T = 1, 4 and 2048, each pass
    captured as a CUDA graph and replayed.  Weights at P(0) = 0.4; the kernels
    read zeros like any other code, so the rate does not depend on P(0)."""
    shapes = (GU, DN, AI, AO)
    layers = [[make_layer(tl, torch, K, N, gen, dev) for (K, N) in shapes]
              for _ in range(STACK_LAYERS)]
    wbytes = STACK_LAYERS * sum(weight_bytes(K, N) for K, N in shapes)
    res = {"layers": STACK_LAYERS,
           "projections": "gate+up 5120x34816, down 17408x5120, attn-in 5120x6144, attn-out 6144x5120",
           "weight_bytes": wbytes, "p_zero": 0.4}
    for T in (1, 4, 2048):
        xs = {K: make_x(torch, T, K, gen, dev) for K in sorted({k for k, _ in shapes})}
        ys = {sh: torch.empty(T, sh[1], device=dev) for sh in shapes}
        ws = torch.zeros(max(tl.tern_linear_workspace_bytes(T, K, N) for K, N in shapes),
                         dtype=torch.uint8, device=dev)
        stream.wait_stream(torch.cuda.current_stream())

        def one_pass():
            for lay in layers:
                for sh, (Wp, sc) in zip(shapes, lay):
                    tl.tern_linear(Wp, sc, xs[sh[0]], ys[sh], ws)

        with torch.cuda.stream(stream):
            one_pass()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                one_pass()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        reps = 20 if T < 2048 else 3
        e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        if T < 2048:
            gbs = wbytes / (ms * 1e-3) / 1e9
            res[f"t{T}"] = {"ms_per_pass": round(ms, 4), "GB/s": round(gbs, 1),
                            "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4)}
        else:
            ops = 2.0 * T * STACK_LAYERS * sum(K * N for K, N in shapes)
            tops = ops / (ms * 1e-3) / 1e12
            res[f"t{T}"] = {"ms_per_pass": round(ms, 3), "TOPS": round(tops, 1),
                            "frac_of_bf16_peak": round(tops / peaks.get("bf16_tflops", 1900.0), 4)}
        del g, xs, ys, ws
    if tl.tern_device_status() != 0:
        raise RuntimeError("device error word set in the stack passes")
    del layers
    torch.cuda.empty_cache()
    return res


L2_BYTES = 129 * 2 ** 20
COMPACT_T = {"gate_up": (1, 4, 8, 16, 17, 508, 2048), "down": (1, 4, 8, 16, 17, 508, 2048)}
ROTATED_T = (1, 16, 2048)
BF16_T = (17, 508, 2048)
INT8_DECODE_T = (1, 16)


def rotated_copies(K, N):
    """Distinct weight copies whose packed bytes exceed 4x L2."""
    return -(-4 * L2_BYTES // weight_bytes(K, N))


def time_rotated(tl, torch, layers, K, N, T, gen, dev, reps=10):
    """Per-call time of tern_linear at (T, K, N), cycling over the weight
    copies in `layers` (> 4x L2 of packed weights, so every call streams its
    weights from HBM), all calls captured in one CUDA graph replayed between
    CUDA events on the launching stream.  Returns (us per call, rung,
    kernels launched per call)."""
    copies = len(layers)
    x = make_x(torch, T, K, gen, dev)
    ys = [torch.empty(T, N, device=dev) for _ in range(copies)]
    ws = torch.zeros(tl.tern_linear_workspace_bytes(T, K, N), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    launches = []

    def calls(count=False):
        for (w, sc), y in zip(layers, ys):
            tl.tern_linear(w, sc, x, y, ws)
            if count:
                launches.append(tl.tern_last_launches())

    with torch.cuda.stream(stream):
        calls(count=True)  # library set-up outside capture
    torch.cuda.synchronize()
    rung = tl.tern_last_rung()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            calls()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * copies)
    del g, x, ys, ws
    return us, rung, max(launches)


def compact_sweep(tl, torch, gen, dev, peaks):
    """The configs' token counts on the two 27B-like MLP projections: T = 1
    (decode), 4, 8, 16 (speculative verify) on the bandwidth rungs and 17,
    508, 2048 on s8, each over rotated weight copies; then BF16_T again on
    the exact bf16 prefill rung, and gate+up at ROTATED_T with the fused
    Hadamard rotation switched on."""
    rows = []
    for name, (K, N) in (("gate_up", GU), ("down", DN)):
        layers = [make_layer(tl, torch, K, N, gen, dev) for _ in range(rotated_copies(K, N))]
        for T in COMPACT_T[name]:
            us, rung, nl = time_rotated(tl, torch, layers, K, N, T, gen, dev,
                                        reps=10 if T < 2048 else 4)
            gbs = algorithmic_bytes(T, K, N) / (us * 1e-6) / 1e9
            row = {"proj": name, "K": K, "N": N, "T": T, "rung": rung, "copies": len(layers),
                   "launches_per_call": nl, "us_per_call": round(us, 3)}
            if rung == "s8":
                tops = 2.0 * T * K * N / (us * 1e-6) / 1e12
                row.update({"int8_TOPS": round(tops, 1),
                            "frac_of_bf16_peak": round(tops / peaks["bf16_tflops"], 4)})
            else:
                row.update({"GB/s": round(gbs, 1),
                            "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4)})
            rows.append(row)
        # the exact bf16 prefill rung (TERN_PREFILL=bf16) against s8 on the same calls
        os.environ["TERN_PREFILL"] = "bf16"
        tl.tern_reload_env()
        try:
            for T in BF16_T:
                us, rung, nl = time_rotated(tl, torch, layers, K, N, T, gen, dev,
                                            reps=10 if T < 2048 else 4)
                s8row = next(r for r in rows if r["proj"] == name and r["T"] == T
                             and r["rung"] == "s8")
                tops = 2.0 * T * K * N / (us * 1e-6) / 1e12
                rows.append({"proj": name, "K": K, "N": N, "T": T, "rung": rung,
                             "copies": len(layers), "launches_per_call": nl,
                             "us_per_call": round(us, 3), "TOPS": round(tops, 1),
                             "frac_of_bf16_peak": round(tops / peaks["bf16_tflops"], 4),
                             "vs_s8": round(us / s8row["us_per_call"], 3)})
        finally:
            os.environ.pop("TERN_PREFILL", None)
            tl.tern_reload_env()
        # the int8-activation decode variant (TERN_DECODE_ACT=int8) on the T <= 16 rungs
        os.environ["TERN_DECODE_ACT"] = "int8"
        tl.tern_reload_env()
        try:
            for T in INT8_DECODE_T:
                us, rung, nl = time_rotated(tl, torch, layers, K, N, T, gen, dev)
                plain = next(r for r in rows if r["proj"] == name and r["T"] == T
                             and r["rung"] not in ("bf16",) and not r.get("int8_decode"))
                rows.append({"proj": name, "K": K, "N": N, "T": T, "rung": rung,
                             "int8_decode": True, "copies": len(layers),
                             "launches_per_call": nl, "us_per_call": round(us, 3),
                             "vs_exact": round(us / plain["us_per_call"], 3)})
        finally:
            os.environ.pop("TERN_DECODE_ACT", None)
            tl.tern_reload_env()
        if name == "gate_up":
            # the fused Hadamard rotation (TERN_ROTATE=1) against the plain calls above
            os.environ["TERN_ROTATE"] = "1"
            tl.tern_reload_env()
            try:
                for T in ROTATED_T:
                    us, rung, nl = time_rotated(tl, torch, layers, K, N, T, gen, dev,
                                                reps=10 if T < 2048 else 4)
                    plain = next(r for r in rows if r["proj"] == name and r["T"] == T
                                 and r["rung"] != "bf16" and not r.get("int8_decode"))
                    rows.append({"proj": name, "K": K, "N": N, "T": T, "rung": rung,
                                 "rotated": True, "copies": len(layers),
                                 "launches_per_call": nl, "us_per_call": round(us, 3),
                                 "vs_plain": round(us / plain["us_per_call"], 3)})
            finally:
                os.environ.pop("TERN_ROTATE", None)
                tl.tern_reload_env()
        del layers
        torch.cuda.empty_cache()
    return rows


def run_ours(args, rank, world, local):
    import torch
    import ternary_weight_linear_gb300 as tl

    tl.build()
    tl.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    peaks, peak_kind = load_peaks()

    L = args.layers
    layers = [(make_layer(tl, torch, *GU, gen, dev), make_layer(tl, torch, *DN, gen, dev))
              for _ in range(L)]
    T = 1
    x_gu = make_x(torch, T, GU[0], gen, dev)
    x_dn = make_x(torch, T, DN[0], gen, dev)
    y_gu = [torch.empty(T, GU[1], device=dev) for _ in range(L)]
    y_dn = [torch.empty(T, DN[1], device=dev) for _ in range(L)]
    ws_bytes = max(tl.tern_linear_workspace_bytes(T, *GU), tl.tern_linear_workspace_bytes(T, *DN))
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)  # sync area must start zeroed
    step_bytes = L * (weight_bytes(*GU) + weight_bytes(*DN))

    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())  # inputs and the zeroed workspace

    step_launches = []

    def step_calls(count=False):
        for i, ((gw, gs), (dw, ds)) in enumerate(layers):
            tl.tern_linear(gw, gs, x_gu, y_gu[i], ws)
            if count:
                step_launches.append(tl.tern_last_launches())
            tl.tern_linear(dw, ds, x_dn, y_dn[i], ws)
            if count:
                step_launches.append(tl.tern_last_launches())

    with torch.cuda.stream(stream):
        step_calls(count=True)  # library init outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            step_calls()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    if tl.tern_device_status() != 0:
        raise RuntimeError("device error word set after warm-up")

    # ---- timed region: K graph replays
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.2)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    if world > 1:
        torch.distributed.barrier()
    ms_per_step = ms / args.steps
    value = whole_job_gbs(world, step_bytes, ms_per_step)

    # ---- per-call legs over rotated weight copies (> 4x L2): the configs'
    # token counts on both MLP projections; the T = 1 rows give the roofline
    # of the dominant kernel (gate+up) and of the down projection
    sweep = compact_sweep(tl, torch, gen, dev, peaks)

    def roofline_of(proj, summary):
        row = next(r for r in sweep_plain if r["proj"] == proj and r["T"] == 1)
        K, N = row["K"], row["N"]
        alg = algorithmic_bytes(1, K, N)
        gbs = alg / (row["us_per_call"] * 1e-6) / 1e9
        traffic = profile_traffic(
            os.path.join(ROOT, "ternary_weight_linear_gb300", "csrc", "tern_smallt.cu"), summary)
        return {"bound": "hbm", "kernel": f"tern_linear T=1 {proj} {K}x{N} (smallt_kernel<1>)",
                "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "peak_kind": peak_kind,
                "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                "traffic": traffic, "algorithmic_bytes_per_launch": alg,
                "avg_launch_us": row["us_per_call"], "launches_per_call": row["launches_per_call"],
                "rotation": f"{row['copies']} weight copies (> 4x L2)"}

    sweep_plain = [r for r in sweep if not r.get("rotated") and not r.get("int8_decode")
                   and r["rung"] != "bf16"]
    roofline = roofline_of("gate_up", "smallt_kernel_gu_t1.md")
    roofline_dn = roofline_of("down", "smallt_kernel_dn_t1.md")
    s8_rows = [r for r in sweep_plain if r["T"] == 2048]
    s8_us = sum(r["us_per_call"] for r in s8_rows)
    s8_tops = sum(2.0 * r["T"] * r["K"] * r["N"] for r in s8_rows) / (s8_us * 1e-6) / 1e12
    # The s8 rung contracts every int8 product as two e4m3 products (the
    # activation split into two exact pieces), so its ceiling in int8 ops is
    # half the e4m3 tensor rate, i.e. the bf16 rate: e4m3 runs at twice bf16
    # (nominal ratio), and the measured bf16 peak is the denominator.
    # DRAM bytes of one pass (both launches) from the committed ncu summaries
    s8_src = os.path.join(ROOT, "ternary_weight_linear_gb300", "csrc", "tern_s8.cu")
    s8_parts = [profile_traffic(s8_src, f) for f in ("s8tc_kernel_gu_t2048.md",
                                                     "s8tc_kernel_dn_t2048.md")]
    s8_traffic = sum(s8_parts) if all(v is not None for v in s8_parts) else None
    s8 = {"metric": "int8 TOPS at T=2048 (s8 rung, gate+up + down)", "value": round(s8_tops, 1),
          "unit": "TOPS", "us_per_pass": round(s8_us, 1),
          "roofline": {"bound": "tensor", "achieved": round(s8_tops, 1),
                       "peak": peaks.get("bf16_tflops", 1900.0), "peak_kind": peak_kind + " bf16",
                       "unit": "TOPS", "frac": round(s8_tops / peaks.get("bf16_tflops", 1900.0), 4),
                       "traffic": s8_traffic, "traffic_unit": "bytes per pass (gate+up + down)"}}

    # ---- whole-stack family (64 resident layers) at T = 1, 4, 2048
    stack = run_stack(tl, torch, gen, dev, peaks, stream) if not args.no_stack else None

    # ---- end to end through the C ABI with host buffers
    import numpy as np
    xh_gu = x_gu.cpu().pin_memory()
    xh_dn = x_dn.cpu().pin_memory()
    yh = torch.empty(T, DN[1], dtype=torch.float32).pin_memory()
    e2e_steps = max(10, min(200, args.steps // 10))
    h2d = (xh_gu.numel() * 2 + xh_dn.numel() * 2) * L
    d2h = yh.numel() * 4
    torch.cuda.synchronize()
    ee0, ee1 = torch.cuda.Event(True), torch.cuda.Event(True)
    with torch.cuda.stream(stream):
        ee0.record(stream)
        for _ in range(e2e_steps):
            for i, ((gw, gs), (dw, ds)) in enumerate(layers):
                x_gu.copy_(xh_gu, non_blocking=True)
                tl.tern_linear(gw, gs, x_gu, y_gu[i], ws)
                x_dn.copy_(xh_dn, non_blocking=True)
                tl.tern_linear(dw, ds, x_dn, y_dn[i], ws)
            yh.copy_(y_dn[-1], non_blocking=True)
        ee1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(ee0.elapsed_time(ee1), world, dev) / e2e_steps
    e2e_val = whole_job_gbs(world, step_bytes, e2e_ms)
    if not np.isfinite(yh.numpy()).all():
        raise RuntimeError("non-finite output")
    if tl.tern_device_status() != 0:
        raise RuntimeError("device error word set")

    launches = args.steps * sum(step_launches)  # counted by the library, per call
    out = {
        "metric": "ternary linear weight GB/s at T=1 (frac of HBM peak); int8 TOPS at T=2048",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 x as three exact e5m2 pieces times e4m3 ternary codes (tcgen05 kind::f8f6f4), "
                 "fp32 accumulation",
        "data": "synthetic",
        "config": {"workload": f"decode GEMV T=1 over {L} layers x (gate+up 5120x34816, down 17408x5120), "
                               "27B-like MLP shapes",
                   "layers": L, "T": T, "weight_bytes_per_step": step_bytes,
                   "l2": "inputs larger than L2 (weights per step > 4x L2, no flush)",
                   "parallelism": f"replicas x{world}", "graph": "CUDA graph per step"},
        "frac_of_hbm_peak": round(value / world / peaks["hbm_gbs"], 4),
        "roofline": roofline,
        "roofline_down": roofline_dn,
        "sweep": sweep,
        "s8_t2048": s8,
        "stack_c4": stack,
        "e2e": {"value": round(e2e_val, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "path": "pinned host x -> device copy, tern_linear via the C ABI (eager), y -> pinned host"},
        "clocks": clk,
        "gpu_launches": launches,
    }
    if rank == 0:
        out["cpu_baseline"] = cpu_baseline(sample_layers=1)
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------- oracle timing

def cpu_baseline(sample_layers=1):
    """The CPU oracle on one layer of the same step (gate+up then down, T = 1),
    on this host's cores.  Returns weight GB/s."""
    import numpy as np
    import oracle
    import synth

    oracle.build()
    cg = synth.config_decode("gu")
    cd = synth.config_decode("dn")
    wpg, _ = oracle.pack(cg.W)
    wpd, _ = oracle.pack(cd.W)
    del cg.W, cd.W
    # repeat the layer pass for about 10 s of CPU work
    t0 = time.perf_counter()
    passes = 0
    while passes < sample_layers or time.perf_counter() - t0 < 10.0:
        oracle.linear_f64(wpg, cg.scales, cg.x, 1, *GU)
        oracle.linear_f64(wpd, cd.scales, cd.x, 1, *DN)
        passes += 1
    dt = time.perf_counter() - t0
    b = passes * (weight_bytes(*GU) + weight_bytes(*DN))
    return {"value": round(b / dt / 1e9, 3), "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"{passes} passes over one layer of the step (gate+up and down at T=1, "
                      "full outputs), about 10 s"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    import synth

    oracle.build()
    cg = synth.config_decode("gu")
    cd = synth.config_decode("dn")
    wpg, _ = oracle.pack(cg.W)
    wpd, _ = oracle.pack(cd.W)
    # bounded sample per step: 2048 rows of gate+up and 512 rows of down
    rows_g, rows_d = 2048, 512
    wg, sg = wpg[:rows_g], cg.scales[:rows_g]
    wd, sd = wpd[:rows_d], cd.scales[:rows_d]
    per_step = weight_bytes(GU[0], rows_g) + weight_bytes(DN[0], rows_d)
    for _ in range(args.warmup):
        oracle.linear_f64(wg, sg, cg.x, 1, GU[0], rows_g)
        oracle.linear_f64(wd, sd, cd.x, 1, DN[0], rows_d)
    steps = max(1, args.steps)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.linear_f64(wg, sg, cg.x, 1, GU[0], rows_g)
        oracle.linear_f64(wd, sd, cd.x, 1, DN[0], rows_d)
    dt = (time.perf_counter() - t0) / steps
    value = per_step / dt / 1e9
    out = {"impl": "reference",
           "metric": "ternary linear weight GB/s at T=1 (frac of HBM peak); int8 TOPS at T=2048",
           "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": steps,
           "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": "decode GEMV T=1, gate+up 5120x34816 and down 17408x5120 "
                                  "bounded row sample per step",
                      "rows_per_step": {"gate_up": rows_g, "down": rows_d}},
           "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": oracle.num_threads(),
                            "kind": "oracle",
                            "sample": f"{rows_g} gate+up rows + {rows_d} down rows per step, T=1"},
           "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_profile(args):
    """A few calls on one synthetic projection, nothing else: the command a
    profiler wraps to capture one kernel.  gu / dn: T = 1 (decode) unless
    --profile-t says otherwise; s8gu / s8dn: T = 2048 by default."""
    import torch
    import ternary_weight_linear_gb300 as tl

    tl.build()
    tl.load()
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    K, N = GU if args.profile.endswith("gu") else DN
    T = args.profile_t or (2048 if args.profile.startswith("s8") else 1)
    Wp, s = make_layer(tl, torch, K, N, gen, dev)
    x = make_x(torch, T, K, gen, dev)
    y = torch.empty(T, N, device=dev)
    ws = torch.zeros(tl.tern_linear_workspace_bytes(T, K, N), dtype=torch.uint8, device=dev)
    for _ in range(args.profile_calls):
        tl.tern_linear(Wp, s, x, y, ws)
    torch.cuda.synchronize()
    status = tl.tern_device_status()
    print(json.dumps({"profile": args.profile, "T": T, "rung": tl.tern_last_rung(),
                      "calls": args.profile_calls, "status": status}))
    if status != 0:
        sys.exit(1)


def run_formats(args):
    """Time tern_repack_t5 (gate+up stored as base-3 bytes) and tern_rotate_bf16
    (T = 2048 x 17408 prefill activations, and a decode-sized T = 4 x 5120
    call) with CUDA events.  Several input copies, each launch on the next, so
    that the big launches read from HBM, not L2.  Prints one JSON line."""
    import torch
    import ternary_weight_linear_gb300 as tl

    tl.build()
    tl.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, peak_kind = load_peaks()
    gen = torch.Generator(device=dev)
    gen.manual_seed(4321)

    def timed_us(fn, reps):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(reps):
            fn(i)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    def entry(us, nbytes):
        gbs = nbytes / (us * 1e-6) / 1e9
        return {"us": round(us, 3), "bytes": nbytes, "GB/s": round(gbs, 1),
                "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4)}

    out = {}
    K, N = GU
    copies = 4  # 4 x (36 MB in + 45 MB out)
    P = [torch.randint(0, 243, (N, K // 128 * 26), dtype=torch.uint8, device=dev, generator=gen)
         for _ in range(copies)]
    Wp = [torch.empty((N, K // 16), dtype=torch.int32, device=dev) for _ in range(copies)]
    us = timed_us(lambda i: tl.tern_repack_t5(P[i % copies], K, Wp[i % copies]), 40)
    out["repack_t5_gate_up"] = entry(us, N * K // 128 * 26 + N * K // 4)
    del P, Wp

    T, Kr = 2048, DN[0]
    copies = 3  # 3 x (71 MB in + 71 MB out)
    xs = [torch.randn(T, Kr, device=dev, generator=gen).to(torch.bfloat16) for _ in range(copies)]
    ys = [torch.empty_like(xs[0]) for _ in range(copies)]
    us = timed_us(lambda i: tl.tern_rotate_bf16(xs[i % copies], ys[i % copies]), 40)
    out["rotate_bf16_t2048_k17408"] = entry(us, 2 * T * Kr * 2)
    del xs, ys

    x4 = torch.randn(4, GU[0], device=dev, generator=gen).to(torch.bfloat16)
    y4 = torch.empty_like(x4)
    us = timed_us(lambda i: tl.tern_rotate_bf16(x4, y4), 200)
    out["rotate_bf16_t4_k5120"] = {"us": round(us, 3),
                                   "note": "eager calls from Python back to back: host-bound, "
                                           "an upper bound on the kernel's time"}
    status = tl.tern_device_status()
    print(json.dumps({"formats": out, "peak_hbm_gbs": peaks["hbm_gbs"], "peak_kind": peak_kind,
                      "status": status}), flush=True)
    if status != 0:
        sys.exit(1)


SWEEP_T = (1, 2, 3, 4, 8, 9, 12, 16, 17, 508, 2048)


def run_sweep(args):
    """Per-call time of the four projections at every token count of the
    configs: T = 1..16 on the bandwidth rungs, T = 17, 508 and 2048 on s8.
    Each (projection, T) is timed over enough distinct weight copies to exceed
    4x L2, all calls captured in one CUDA graph that is replayed between CUDA
    events.  Prints one JSON line."""
    import torch
    import ternary_weight_linear_gb300 as tl

    tl.build()
    tl.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, peak_kind = load_peaks()
    gen = torch.Generator(device=dev)
    gen.manual_seed(99)
    rows = []
    for name, (K, N) in (("gate_up", GU), ("down", DN), ("attn_in", AI), ("attn_out", AO)):
        copies = -(-4 * L2_BYTES // weight_bytes(K, N))
        layers = [make_layer(tl, torch, K, N, gen, dev) for _ in range(copies)]
        for T in SWEEP_T:
            x = make_x(torch, T, K, gen, dev)
            ys = [torch.empty(T, N, device=dev) for _ in range(copies)]
            ws = torch.zeros(tl.tern_linear_workspace_bytes(T, K, N), dtype=torch.uint8,
                             device=dev)
            stream = torch.cuda.Stream(device=dev)
            stream.wait_stream(torch.cuda.current_stream())

            def calls():
                for (w, sc), y in zip(layers, ys):
                    tl.tern_linear(w, sc, x, y, ws)

            with torch.cuda.stream(stream):
                calls()  # library set-up outside capture
            torch.cuda.synchronize()
            rung = tl.tern_last_rung()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(g, stream=stream):
                    calls()
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            reps = 10
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (reps * copies)
            gbs = algorithmic_bytes(T, K, N) / (us * 1e-6) / 1e9
            tops = 2.0 * T * K * N / (us * 1e-6) / 1e12
            rows.append({"proj": name, "K": K, "N": N, "T": T, "rung": rung, "copies": copies,
                         "us_per_call": round(us, 3), "GB/s": round(gbs, 1),
                         "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4),
                         "int8_TOPS" if rung == "s8" else "TOPS": round(tops, 1),
                         "frac_of_bf16_peak": round(tops / peaks["bf16_tflops"], 4)})
            del g, x, ys, ws
        del layers
        torch.cuda.empty_cache()
    status = tl.tern_device_status()
    print(json.dumps({"sweep": rows, "peak_hbm_gbs": peaks["hbm_gbs"],
                      "peak_bf16_tflops": peaks["bf16_tflops"], "peak_kind": peak_kind,
                      "status": status}), flush=True)
    if status != 0:
        sys.exit(1)


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.sweep:
        run_sweep(args)
        return
    if args.formats:
        run_formats(args)
        return
    if args.profile:
        run_profile(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
