#!/usr/bin/env python3
"""Benchmark of one routed MoE layer's forward pass on GB300.

Workload (default): the decode layer of a Qwen3-35B-A3B-shaped model --
d_model 2048, 128 experts, top-8, d_ff 768, MXFP4 weights, 47 cache slots
(37% of the experts) filled from pinned host memory -- run at 1, 4 and 16
tokens per step on AR(1) hidden states (rho 0.9).  A step is one moe_forward:
router, permutation, LRU update, miss fills, expert FFN, combine.  Misses are
filled the library's default way (at batch 1 and 4 the expert GEMV reads them
from host memory itself, at batch 16 a copy kernel on 12 reserved SMs does);
the other fill modes are timed beside it per batch, and so is an all-resident
warm run (n_slots = E, every expert installed: no fills, HBM bytes only).

Timing: W warm-up steps, then K timed steps per batch size, each bracketed by
CUDA events on the launching stream; the L2 is flushed (a 512 MiB write)
between timed steps, outside the events.  `value` = tokens / summed step time
over the three batch sizes, inputs resident in HBM.  `e2e` repeats the run
through the C ABI with pinned host x / y buffers (copies inside the timed
call, host wall clock).  The roofline entry is the expert FFN phase-1 kernel
(gate/up GEMV), timed with the library's per-launch CUDA events in a second
pass over the same steps (the events cost host time per launch, so the pass
behind `value` runs without them).

--impl reference times the CPU oracle (FP64, numpy) on a bounded sample of the
same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (decode, prefill); % of HBM BW / % of dense FP4 tensor peak"
FALLBACK_HBM_GBS = 6800.0


FALLBACK_BF16_TFLOPS = 1900.0
FP4_PER_BF16 = 6.0        # nominal dense ratio: 13.5 PF/s FP4 vs 2.25 PF/s bf16


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _fp4_peak():
    """Dense FP4 TF/s: measured bf16 GEMM burst x the nominal FP4/bf16 ratio."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            return float(json.load(fh)["bf16_tflops"]) * FP4_PER_BF16, "measured bf16 x 6"
    except Exception:
        return FALLBACK_BF16_TFLOPS * FP4_PER_BF16, "fallback bf16 x 6"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.out.name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- workload

def decode_tokens(wl, spec, seed, batch, steps):
    x, _ = wl.ar1_tokens(seed, batch, steps, spec.d_model, 0.9)
    return x


def gateup_bytes(spec, layout, n_experts, n_tokens):
    """Algorithmic bytes of phase 1 for one step: the gate and up codes and
    scales of each expert read once, x read, W_g x and W_u x written (fp32)."""
    d, f = spec.d_model, spec.d_ff
    w = 2 * (f * d // 2 + f * d // spec.block)
    rows = n_tokens * spec.k + (n_tokens if spec.has_shared else 0)
    return n_experts * w + n_tokens * d * 2 + rows * 2 * f * 4


def traffic_ratio(kernel, workload):
    """DRAM bytes / algorithmic bytes of a launch, from the ncu capture listed
    in profiles/traffic.txt (None when the kernel has no current capture)."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles", "traffic.txt")
    try:
        for line in open(path):
            f = line.split()
            if len(f) >= 5 and not line.startswith("#") and f[0] == kernel and f[1] == workload:
                return float(f[4])
    except OSError:
        pass
    return None


def run_decode(args, batch, torch, capi, wl, build_layer, flush, st, profile, fill=None):
    """K timed decode steps after W warm-up steps on a fresh layer (cold cache).
    profile=False: the clean pass behind `value`; profile=True: the same steps
    with the library's per-launch events on (kernel times for the roofline)."""
    spec = wl.DECODE_35B.layer
    seed = wl.DECODE_35B.seed
    W, K = args.warmup, args.steps
    x_host = decode_tokens(wl, spec, seed + batch, batch, W + K)
    xs = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).cuda()
    L = build_layer(spec, seed, batch)
    if fill is not None:
        capi.moe_set_fill_mode(L.h, fill)
    y = torch.empty(batch, spec.d_model, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(st):
        for t in range(W):
            L.forward(xs[t], y, stream=st)
    torch.cuda.synchronize()
    stats0 = capi.moe_stats(L.h)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    capi.moe_profile(L.h, profile)
    launches = 0
    fill_b = 0
    ffn_bytes = 0
    with torch.cuda.stream(st):
        for t in range(K):
            flush.zero_()
            ev[t][0].record(st)
            _, info = L.forward(xs[W + t], y, stream=st)
            ev[t][1].record(st)
            launches += info.n_launches
            fill_b += info.fill_bytes
            ffn_bytes += gateup_bytes(spec, L.layout, info.n_distinct, batch)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = sum(step_ms)
    prof = capi.moe_profile_read(L.h)
    capi.moe_profile(L.h, False)
    stats1 = capi.moe_stats(L.h)
    L.close()
    d_misses, d_distinct = stats1[3] - stats0[3], stats1[1] - stats0[1]
    return dict(batch=batch, steps=K, ms=ms, step_ms_p50=statistics.median(step_ms), tokens=K * batch,
                launches=launches,
                misses=d_misses, distinct=d_distinct, fill_bytes=fill_b, prof=prof,
                gateup_bytes=ffn_bytes)


def run_decode_resident(args, batch, torch, capi, wl, build_layer, flush, st):
    """The same decode steps with every expert resident (n_slots = E, expert e
    installed in slot e): no misses and no fills, so a step moves only HBM
    bytes.  Returns the step time and the step's algorithmic bytes: the
    distinct experts' weights (B_e = 3 d f (1/2 + 1/32) each), W_r in fp32
    (4 E d) and x in / y out (4 N d)."""
    import dataclasses
    spec = dataclasses.replace(wl.DECODE_35B.layer, n_slots=wl.DECODE_35B.layer.E)
    seed = wl.DECODE_35B.seed
    W, K = args.warmup, args.steps
    x_host = decode_tokens(wl, spec, seed + batch, batch, W + K)
    xs = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).cuda()
    L = build_layer(spec, seed, batch, install_all=True)
    y = torch.empty(batch, spec.d_model, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(st):
        for t in range(W):
            L.forward(xs[t], y, stream=st)
    torch.cuda.synchronize()
    stats0 = capi.moe_stats(L.h)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with torch.cuda.stream(st):
        for t in range(K):
            flush.zero_()
            ev[t][0].record(st)
            L.forward(xs[W + t], y, stream=st)
            ev[t][1].record(st)
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in ev)
    stats1 = capi.moe_stats(L.h)
    L.close()
    d, f, E = spec.d_model, spec.d_ff, spec.E
    b_e = 3 * d * f * (1 / 2 + 1 / spec.block)
    nbytes = (stats1[1] - stats0[1]) * b_e + K * (4 * E * d + 4 * batch * d)
    return dict(batch=batch, steps=K, ms=ms, tokens=K * batch, bytes=nbytes,
                misses=stats1[3] - stats0[3])


def measure_h2d(torch, nbytes=256 << 20):
    """Host-to-device GB/s of one copy from pinned memory (best of 3): the
    ceiling the miss fills are held against."""
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    best = None
    for _ in range(4):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        t = a.elapsed_time(b)
        best = t if best is None else min(best, t)
    return nbytes / (best / 1000.0) / 1e9


def run_decode_e2e(args, batch, torch, capi, wl, build_layer, flush):
    spec = wl.DECODE_35B.layer
    seed = wl.DECODE_35B.seed
    W, K = args.warmup, args.steps
    x_host = decode_tokens(wl, spec, seed + batch, batch, W + K)
    xs = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).pin_memory()
    ys = torch.empty(W + K, batch, spec.d_model, dtype=torch.bfloat16).pin_memory()
    L = build_layer(spec, seed, batch)
    for t in range(W):
        capi.moe_forward(L.h, xs[t], batch, ys[t], None, capi.MOE_REGIME_AUTO)
    torch.cuda.synchronize()
    total = 0.0
    for t in range(K):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        capi.moe_forward(L.h, xs[W + t], batch, ys[W + t], None, capi.MOE_REGIME_AUTO)
        total += time.perf_counter() - t0
    L.close()
    return dict(batch=batch, s=total, tokens=K * batch,
                h2d=K * batch * spec.d_model * 2, d2h=K * batch * spec.d_model * 2)


def run_prefill(args, work, torch, capi, wl, build_layer, flush, st):
    """One prefill chunk per step, every expert resident (slot e = expert e).
    Tokens/s from a pass without per-kernel events, kernel times from a second
    instrumented pass."""
    spec, N, seed = work.layer, work.n_tokens, work.seed
    x_host, _ = wl.iid_tokens(seed, N, spec.d_model)
    x = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).cuda()
    L = build_layer(spec, seed, N, install_all=True)
    y = torch.empty(N, spec.d_model, dtype=torch.bfloat16, device="cuda")
    W, K = max(3, args.warmup // 4), max(3, args.prefill_steps)
    with torch.cuda.stream(st):
        for _ in range(W):
            L.forward(x, y, stream=st, regime=capi.MOE_REGIME_PREFILL)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for profile in (False, True):
        capi.moe_profile(L.h, profile)
        launches = 0
        with torch.cuda.stream(st):
            for t in range(K):
                flush.zero_()
                ev[t][0].record(st)
                _, info = L.forward(x, y, stream=st, regime=capi.MOE_REGIME_PREFILL)
                ev[t][1].record(st)
                launches += info.n_launches
        torch.cuda.synchronize()
        if not profile:
            ms = sum(a.elapsed_time(b) for a, b in ev)
    prof = capi.moe_profile_read(L.h)
    capi.moe_profile(L.h, False)
    L.close()
    rows = N * spec.k + (N if spec.has_shared else 0)
    d, f = spec.d_model, spec.d_ff
    flops1, flops2 = 2.0 * rows * d * 2 * f, 2.0 * rows * f * d
    return dict(workload=work.name, steps=K, ms=ms, tokens=K * N, launches=launches, prof=prof,
                flops1=flops1 * K, flops2=flops2 * K)


def prefill_summary(r, fp4_peak):
    p = r["prof"]
    g_ms, g_n = p["gateup"]
    d_ms, d_n = p["down"]
    t1 = r["flops1"] / (g_ms / 1000.0) / 1e12 if g_ms else None
    t2 = r["flops2"] / (d_ms / 1000.0) / 1e12 if d_ms else None
    tboth = (r["flops1"] + r["flops2"]) / ((g_ms + d_ms) / 1000.0) / 1e12 if g_ms + d_ms else None
    return {
        "workload": r["workload"], "tokens_per_s": r["tokens"] / (r["ms"] / 1000.0),
        "ms_per_step": r["ms"] / r["steps"],
        "gemm_tflops": {"gateup": t1, "down": t2, "both": tboth},
        "frac_fp4_peak": (tboth / fp4_peak) if tboth else None,
        "kernel_ms_per_step": {k: v[0] / r["steps"] for k, v in p.items() if v[1]},
    }


# ---------------------------------------------------------------- CPU oracle

def cpu_oracle_sample(budget_s: float):
    """Time the oracle on the decode workload (batch 1, 4, 16 in turn) until
    the budget is spent; returns (tokens/s, tokens, steps, seconds, cores)."""
    from oracle import layer as olayer
    from routed_expert_layer_gemv_gb300 import workloads as wl
    spec = wl.DECODE_35B.layer
    seed = wl.DECODE_35B.seed
    W_r, b = wl.router_weights(spec, seed)
    O = olayer.Layer(spec, lambda e: wl.expert_weights(spec, seed, e), W_r, b)
    tokens = steps = 0
    t0 = time.perf_counter()
    per_batch = budget_s / 3.0
    for batch in (1, 4, 16):
        xb = decode_tokens(wl, spec, seed + batch, batch, 8)
        tb = time.perf_counter()
        t = 0
        while time.perf_counter() - tb < per_batch and t < len(xb):
            O.forward(wl.bf16_bits_to_f64(xb[t]), "decode")
            tokens += batch
            steps += 1
            t += 1
    el = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    return tokens / el, tokens, steps, el, cores


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batches", default="1,4,16")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="decode35b",
                    choices=["decode35b", "prefill35b", "prefill753b"],
                    help="decode35b = the headline decode configuration; the prefill ones "
                         "print that prefill chunk's line instead")
    ap.add_argument("--prefill-steps", type=int, default=8)
    ap.add_argument("--no-prefill", action="store_true", help="skip the secondary prefill result")
    ap.add_argument("--fill-modes", default="memcpy,device,kernel,fused",
                    help="fill modes timed beside the default per batch ('none': skip them)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    ws, rank, local = _dist()
    batches = [int(b) for b in args.batches.split(",")]

    if args.impl == "reference":
        if rank != 0:
            return
        v, tok, steps, el, cores = cpu_oracle_sample(args.cpu_budget)
        cfg = {"workload": "decode_35b_a3b_d2048_e128_top8_f768_mxfp4_s47", "batches": batches}
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
                "n_gpus": 0, "steps": steps, "warmup": 0, "ms_per_step": 1000.0 * el / max(1, steps),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": cfg,
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": "%d decode steps (%d tokens) of batches 1/4/16, %.1f s" % (steps, tok, el)},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    from routed_expert_layer_gemv_gb300 import capi
    from routed_expert_layer_gemv_gb300 import workloads as wl
    from routed_expert_layer_gemv_gb300.layer import build_layer
    capi.lib()

    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    st = torch.cuda.Stream()
    clocks = ClockSampler(local)
    if args.workload != "decode35b":
        work = wl.PREFILL_35B if args.workload == "prefill35b" else wl.PREFILL_753B
        clocks.start()
        r = run_prefill(args, work, torch, capi, wl, build_layer, flush, st)
        clk = clocks.stop()
        fp4, fp4_kind = _fp4_peak()
        sm = prefill_summary(r, fp4)
        tboth = sm["gemm_tflops"]["both"]
        line = {"metric": METRIC, "value": sm["tokens_per_s"] * ws, "unit": "tokens/s", "n_gpus": ws,
                "steps": r["steps"], "warmup": max(3, args.warmup // 4), "ms_per_step": sm["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "fp4(e2m1)xfp4(e2m1)->f32", "data": "synthetic (seeded i.i.d. hidden states, random FP4 weights)",
                "config": {"workload": work.name, "l2": "flushed (512 MiB write) between timed steps",
                           "detail": sm},
                "roofline": {"bound": "tensor", "kernel": "prefill grouped GEMM (gate/up + down)",
                             "achieved": tboth, "peak": fp4, "unit": "TFLOP/s",
                             "frac": (tboth / fp4) if tboth else None, "traffic": None,
                             "peak_kind": fp4_kind},
                "gpu_launches": r["launches"], "clocks": clk}
        if rank == 0:
            print(json.dumps(line))
        return
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    runs = [run_decode(args, b, torch, capi, wl, build_layer, flush, st, False) for b in batches]
    torch.cuda.synchronize()
    clk = clocks.stop()
    # the instrumented pass fills with the SM copy kernel, so every gate/up
    # launch reads HBM-resident weights (the fused mode streams misses over
    # the host link inside the GEMV, which is not an HBM roofline)
    pruns = [run_decode(args, b, torch, capi, wl, build_layer, flush, st, True, capi.MOE_FILL_KERNEL)
             for b in batches]
    modes = {"memcpy": capi.MOE_FILL_MEMCPY, "device": capi.MOE_FILL_DEVICE, "kernel": capi.MOE_FILL_KERNEL,
             "fused": capi.MOE_FILL_FUSED}
    modes = {m: modes[m] for m in args.fill_modes.split(",") if m in modes}
    fruns = {name: [run_decode(args, b, torch, capi, wl, build_layer, flush, st, False, m) for b in batches]
             for name, m in modes.items()}
    e2e_runs = [run_decode_e2e(args, b, torch, capi, wl, build_layer, flush) for b in batches]
    rruns = [run_decode_resident(args, b, torch, capi, wl, build_layer, flush, st) for b in batches]
    h2d = measure_h2d(torch)

    ms = sum(r["ms"] for r in runs)
    tokens = sum(r["tokens"] for r in runs)
    e2e_s = sum(r["s"] for r in e2e_runs)
    if ws > 1:
        t = torch.tensor([ms, e2e_s], dtype=torch.float64, device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms, e2e_s = float(t[0]), float(t[1])
    if rank != 0:
        torch.distributed.barrier() if ws > 1 else None
        return
    value = ws * tokens / (ms / 1000.0)
    e2e_value = ws * tokens / e2e_s

    peak, peak_kind = _peaks()
    g_ms = sum(r["prof"]["gateup"][0] for r in pruns)
    g_n = sum(r["prof"]["gateup"][1] for r in pruns)
    g_bytes = sum(r["gateup_bytes"] for r in pruns)
    achieved = (g_bytes / max(g_n, 1)) / ((g_ms / max(g_n, 1)) / 1000.0) / 1e9 if g_ms > 0 else None
    ratio = traffic_ratio("gemv_gateup", "decode35b")
    roof = {"bound": "hbm", "kernel": "gemv_gateup (expert FFN phase 1)", "achieved": achieved,
            "peak": peak, "unit": "GB/s", "frac": (achieved / peak) if achieved else None,
            "traffic": ratio * g_bytes / max(g_n, 1) if ratio else None, "peak_kind": peak_kind,
            "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one captured launch "
                              "(profiles/gemv_stream_decode35b_b16.md) scaled to this run's bytes per launch"
                              if ratio else None,
            "bytes_per_launch": g_bytes / max(g_n, 1), "ms_per_launch": g_ms / max(g_n, 1)}

    per_batch = {}
    for i, (r, e, pr, rr) in enumerate(zip(runs, e2e_runs, pruns, rruns)):
        p = pr["prof"]
        per_batch[str(r["batch"])] = {
            "tokens_per_s": r["tokens"] / (r["ms"] / 1000.0),
            "e2e_tokens_per_s": e["tokens"] / e["s"],
            "ms_per_step": r["ms"] / r["steps"],
            "ms_per_step_median": r["step_ms_p50"],
            "miss_rate": r["misses"] / max(1, r["distinct"]),
            "fill_GB_per_s": pr["fill_bytes"] / max(1e-9, p["fill"][0] / 1000.0) / 1e9 if p["fill"][0] else None,
            "kernel_ms_per_step": {k: v[0] / r["steps"] for k, v in p.items() if v[1]},
            "tokens_per_s_by_fill_mode": {name: fr[i]["tokens"] / (fr[i]["ms"] / 1000.0)
                                          for name, fr in fruns.items()},
            "all_resident": {
                "tokens_per_s": rr["tokens"] / (rr["ms"] / 1000.0),
                "ms_per_step": rr["ms"] / rr["steps"],
                "hbm_GB_per_s": rr["bytes"] / (rr["ms"] / 1000.0) / 1e9,
                "frac_of_measured_hbm": rr["bytes"] / (rr["ms"] / 1000.0) / 1e9 / peak,
                "misses": rr["misses"]},
        }
    prefill = None
    if not args.no_prefill:
        fp4, _ = _fp4_peak()
        prefill = prefill_summary(run_prefill(args, wl.PREFILL_35B, torch, capi, wl, build_layer,
                                              flush, st), fp4)
    cpu = None
    if not args.no_cpu_baseline:
        v, tok, steps, el, cores = cpu_oracle_sample(args.cpu_budget)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": "%d decode steps (%d tokens) of batches 1/4/16, %.1f s" % (steps, tok, el)}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps * len(batches), "warmup": args.warmup,
        "ms_per_step": ms / (args.steps * len(batches)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp4(e2m1)xbf16->f32",
        "data": "synthetic (seeded AR(1) hidden states, random FP4 weights)",
        "config": {"workload": "decode_35b_a3b_d2048_e128_top8_f768_mxfp4_s47",
                   "batches": batches, "l2": "flushed (512 MiB write) between timed steps",
                   "fill": "the library default MOE_FILL_AUTO: misses streamed from host memory by the "
                           "expert GEMV itself (MOE_FILL_FUSED) at batch 1 and 4, a copy kernel on 12 "
                           "reserved SMs (MOE_FILL_KERNEL) at batch 16; per_batch times every mode",
                   "timing": "value from a pass without per-kernel events; kernel times and "
                             "roofline from a second, instrumented pass of the same steps with "
                             "MOE_FILL_KERNEL fills",
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "h2d_GB_per_s_measured": h2d,
                   "all_resident": "per_batch.all_resident: the same steps with n_slots = E and every "
                                   "expert installed (no fills); bytes = distinct experts' weights + "
                                   "W_r (fp32) + x / y per step",
                   "per_batch": per_batch},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s",
                "h2d_bytes_per_step": sum(e["h2d"] for e in e2e_runs) / (args.steps * len(batches)),
                "d2h_bytes_per_step": sum(e["d2h"] for e in e2e_runs) / (args.steps * len(batches))},
        "gpu_launches": sum(r["launches"] for r in runs),
        "clocks": clk,
        "prefill_35b_a3b_n8192": prefill,
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
