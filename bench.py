#!/usr/bin/env python3
"""Benchmark of one routed MoE layer's forward pass on GB300.

Default workload (the headline line): the decode layer of a Qwen3-35B-A3B-
shaped model -- d_model 2048, 128 experts, top-8, d_ff 768, MXFP4 weights, 47
cache slots (37% of the experts) filled from pinned host memory -- at 1, 4
and 16 tokens per step on AR(1) hidden states (rho 0.9).  A step is one
moe_forward: router, permutation, LRU update, miss fills, expert FFN,
combine, in the library's default modes (a decode step of <= 16 tokens whose
misses the expert FFN itself can fill runs as one fused launch; batch 16,
whose distinct experts outnumber the slots, fills with a copy kernel on 12
reserved SMs and runs the chain of launches).

Beside it, in the same JSON line:
  * per batch: miss rate of the timed steps and of the whole 512-step trace,
    e2e, kernel times, every fill mode, and an all-resident run (n_slots = E,
    no fills: HBM bytes only) -- the roofline entry is the fused decode step
    kernel on those all-resident steps;
  * decode_284b_a13b: the DeepSeek-V4-Flash-shaped decode layer (d 4096, 256
    experts, top-8 + shared, d_ff 2048, 28 slots) at batch 1 and 8, the same
    figures;
  * prefill_35b_a3b_n8192 and prefill_753b_n16384: the two prefill chunks
    (tokens/s, grouped-GEMM TFLOP/s against the dense FP4 peak);
  * cpu_baseline: the C++ FP64 oracle on the host cores (and one thread).

Timing: W warm-up steps, then K timed steps per batch size, each bracketed by
CUDA events on the launching stream; the L2 is flushed (a 512 MiB write)
between timed steps, outside the events.  `value` = tokens / summed step time
over the three batch sizes, inputs resident in HBM.  `e2e` repeats the run
through the C ABI with pinned host x / y buffers (copies inside the timed
call, host wall clock).  Kernel times come from a second, instrumented pass
(the library's per-launch events cost host time, so the pass behind `value`
runs without them).

--impl reference times the CPU oracle (C++, FP64, OpenMP) on a bounded sample
of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
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


def _measured():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh)
    except Exception:
        return None


def _peaks():
    d = _measured()
    if d and "hbm_gbs" in d:
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def _dtype_peak(fmt):
    """Dense tensor TF/s of the prefill MMAs of a weight format: the measured
    bf16 GEMM burst x the nominal ratio (FP4 13.5 : 2.25, FP8 4.5 : 2.25)."""
    d = _measured()
    ratio = {"mxfp4": FP4_PER_BF16, "nvfp4": FP4_PER_BF16, "mxfp8": 2.0, "bf16": 1.0}[fmt]
    if d and "bf16_tflops" in d:
        return float(d["bf16_tflops"]) * ratio, "measured bf16 x %g" % ratio
    return FALLBACK_BF16_TFLOPS * ratio, "fallback bf16 x %g" % ratio


def _fp4_peak():
    """Dense FP4 TF/s: measured bf16 GEMM burst x the nominal FP4/bf16 ratio."""
    d = _measured()
    if d and "bf16_tflops" in d:
        return float(d["bf16_tflops"]) * FP4_PER_BF16, "measured bf16 x 6"
    return FALLBACK_BF16_TFLOPS * FP4_PER_BF16, "fallback bf16 x 6"


def _dist():
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), \
        int(os.environ.get("LOCAL_RANK", "0"))


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


# ---------------------------------------------------------------- helpers

def expert_bytes(spec):
    """Weight bytes of one expert: B_e = 3 d f (code bits / 8 + 1 / B), B the
    elements per block scale (no scale term for BF16)."""
    from routed_expert_layer_gemv_gb300.workloads import CODE_BITS
    per = CODE_BITS[spec.fmt] / 8 + (1 / spec.block if spec.block else 0)
    return 3 * spec.d_model * spec.d_ff * per


def step_bytes(spec, n_distinct, n_tokens):
    """Algorithmic HBM bytes of one decode step: each distinct routed expert's
    weights once (B_e, expert_bytes), the shared expert's, W_r in fp32
    (4 E d) and x in / y out (2 N d each)."""
    d, E = spec.d_model, spec.E
    return (n_distinct + (1 if spec.has_shared else 0)) * expert_bytes(spec) + 4 * E * d + 4 * n_tokens * d


def traffic_ratio(kernel, workload):
    """DRAM bytes / algorithmic bytes of a launch, from the ncu capture listed
    in profiles/traffic.txt (None when the kernel has no current capture)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        for line in open(path):
            f = line.split()
            if len(f) >= 5 and not line.startswith("#") and f[0] == kernel and f[1] == workload:
                return float(f[4])
    except OSError:
        pass
    return None


def gemm_traffic(workload):
    """DRAM bytes of one chunk's two GEMM launches (phase 1 + phase 2) from
    the ncu capture listed in profiles/traffic.txt, or None without one."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    got = {}
    try:
        for line in open(path):
            f = line.split()
            if len(f) >= 5 and not line.startswith("#") and f[0] in ("gemm_ws_phase1", "gemm_ws_phase2") \
                    and f[1] == workload + "_n8192":
                got[f[0]] = float(f[2])
    except OSError:
        pass
    return sum(got.values()) if len(got) == 2 else None


class Ctx:
    """What every run needs: torch, the binding, the generator, a flush
    buffer, the stream, and one packed host pool per workload."""

    def __init__(self, args):
        import torch
        from routed_expert_layer_gemv_gb300 import capi
        from routed_expert_layer_gemv_gb300 import workloads as wl
        from routed_expert_layer_gemv_gb300.layer import build_layer, make_desc, pack_pool
        self.torch, self.capi, self.wl, self.args = torch, capi, wl, args
        self.build_layer, self.make_desc, self.pack_pool = build_layer, make_desc, pack_pool
        capi.lib()
        self.flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")
        self.st = torch.cuda.Stream()
        self.pools = {}

    def layer(self, work, max_tokens, n_slots=None, install_all=False):
        spec = work.layer if n_slots is None else dataclasses.replace(work.layer, n_slots=n_slots)
        key = work.name
        if key not in self.pools:
            lay = self.capi.moe_expert_layout_for(self.make_desc(spec, max_tokens))
            self.pools[key] = self.pack_pool(lay, spec.E, lambda e: self.wl.expert_weights(spec, work.seed, e))
        return self.build_layer(spec, work.seed, max_tokens, install_all=install_all, pool=self.pools[key]), spec

    def tokens(self, work, batch, steps, device="cuda"):
        x, _ = self.wl.ar1_tokens(work.seed + batch, batch, steps, work.layer.d_model, work.rho)
        t = self.torch.from_numpy(x.view(np.int16)).view(self.torch.bfloat16)
        return t.cuda() if device == "cuda" else t


def run_decode(c, work, batch, profile=False, fill=None, resident=None):
    """K timed decode steps after W warm-up steps on a fresh layer (cold
    cache), or on `resident` = (layer, spec), a layer that holds every
    expert.  profile: the library's per-launch events on (kernel times)."""
    torch, capi = c.torch, c.capi
    W, K = c.args.warmup, c.args.steps
    xs = c.tokens(work, batch, W + K)
    L, spec = resident or c.layer(work, batch)
    if fill is not None:
        capi.moe_set_fill_mode(L.h, fill)
    y = torch.empty(batch, spec.d_model, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(c.st):
        for t in range(W):
            L.forward(xs[t], y, stream=c.st)
    torch.cuda.synchronize()
    s0 = capi.moe_stats(L.h)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    capi.moe_profile(L.h, profile)
    launches = fused = 0
    with torch.cuda.stream(c.st):
        for t in range(K):
            c.flush.zero_()
            ev[t][0].record(c.st)
            _, info = L.forward(xs[W + t], y, stream=c.st)
            ev[t][1].record(c.st)
            launches += info.n_launches
            fused += info.fused_step
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    prof = capi.moe_profile_read(L.h)
    capi.moe_profile(L.h, False)
    s1 = capi.moe_stats(L.h)
    if resident is None:
        L.close()
    distinct, misses = s1[1] - s0[1], s1[3] - s0[3]
    return dict(batch=batch, steps=K, ms=sum(step_ms), p50=statistics.median(step_ms), tokens=K * batch,
                launches=launches, fused_steps=fused, distinct=distinct, misses=misses, prof=prof,
                bytes=K * step_bytes(spec, 0, batch) + distinct * expert_bytes(spec))


def trace_miss_rate(c, work, batch):
    """Miss rate over the workload's whole trace (its configured number of
    steps from a cold cache), untimed."""
    torch, capi = c.torch, c.capi
    steps = c.args.trace_steps or work.steps
    xs = c.tokens(work, batch, steps)
    L, spec = c.layer(work, batch)
    y = torch.empty(batch, spec.d_model, dtype=torch.bfloat16, device="cuda")
    for t in range(steps):
        L.forward(xs[t], y)
    torch.cuda.synchronize()
    s = capi.moe_stats(L.h)
    L.close()
    return s[3] / max(1, s[1]), steps


def run_e2e(c, work, batch):
    torch, capi = c.torch, c.capi
    W, K = c.args.warmup, c.args.steps
    xs = c.tokens(work, batch, W + K, device="cpu").pin_memory()
    ys = torch.empty(W + K, batch, work.layer.d_model, dtype=torch.bfloat16).pin_memory()
    L, spec = c.layer(work, batch)
    for t in range(W):
        capi.moe_forward(L.h, xs[t], batch, ys[t], None, capi.MOE_REGIME_AUTO)
    torch.cuda.synchronize()
    total = 0.0
    for t in range(K):
        c.flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        capi.moe_forward(L.h, xs[W + t], batch, ys[W + t], None, capi.MOE_REGIME_AUTO)
        total += time.perf_counter() - t0
    L.close()
    nb = K * batch * spec.d_model * 2
    return dict(batch=batch, s=total, tokens=K * batch, h2d=nb, d2h=nb)


def run_prefill(c, work):
    """One prefill chunk per step, every expert resident (slot e = expert e).
    Tokens/s from a pass without per-kernel events, kernel times from a second
    instrumented pass."""
    torch, capi, wl = c.torch, c.capi, c.wl
    spec, N = work.layer, work.n_tokens
    x_host, _ = wl.iid_tokens(work.seed, N, spec.d_model)
    x = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).cuda()
    L, _ = c.layer(work, N, n_slots=spec.E, install_all=True)
    y = torch.empty(N, spec.d_model, dtype=torch.bfloat16, device="cuda")
    W, K = max(3, c.args.warmup // 4), max(3, c.args.prefill_steps)
    with torch.cuda.stream(c.st):
        for _ in range(W):
            L.forward(x, y, stream=c.st, regime=capi.MOE_REGIME_PREFILL)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for profile in (False, True):
        capi.moe_profile(L.h, profile)
        launches = 0
        with torch.cuda.stream(c.st):
            for t in range(K):
                c.flush.zero_()
                ev[t][0].record(c.st)
                _, info = L.forward(x, y, stream=c.st, regime=capi.MOE_REGIME_PREFILL)
                ev[t][1].record(c.st)
                launches += info.n_launches
        torch.cuda.synchronize()
        if not profile:
            ms = sum(a.elapsed_time(b) for a, b in ev)
    prof = capi.moe_profile_read(L.h)
    capi.moe_profile(L.h, False)
    L.close()
    rows = N * spec.k + (N if spec.has_shared else 0)
    d, f = spec.d_model, spec.d_ff
    return dict(workload=work.name, steps=K, warmup=W, ms=ms, tokens=K * N, launches=launches, prof=prof,
                flops1=2.0 * rows * d * 2 * f * K, flops2=2.0 * rows * f * d * K)


def prefill_summary(r, fp4_peak):
    p = r["prof"]
    g_ms, d_ms = p["gateup"][0], p["down"][0]
    t1 = r["flops1"] / (g_ms / 1000.0) / 1e12 if g_ms else None
    t2 = r["flops2"] / (d_ms / 1000.0) / 1e12 if d_ms else None
    tboth = (r["flops1"] + r["flops2"]) / ((g_ms + d_ms) / 1000.0) / 1e12 if g_ms + d_ms else None
    return {
        "workload": r["workload"], "tokens_per_s": r["tokens"] / (r["ms"] / 1000.0),
        "ms_per_step": r["ms"] / r["steps"], "steps": r["steps"],
        "gemm_tflops": {"gateup": t1, "down": t2, "both": tboth},
        "frac_fp4_peak": (tboth / fp4_peak) if tboth else None,
        "kernel_ms_per_step": {k: v[0] / r["steps"] for k, v in p.items() if v[1]},
        # DRAM bytes of the two GEMM launches per chunk (ncu capture of this workload)
        "gemm_dram_bytes_ncu": gemm_traffic("prefill35b") if r["workload"].startswith("prefill_35b") and
        r["workload"].endswith("_mxfp4") else None,
    }


def h2d_rate(c):
    """Pinned host -> device copy rate of one 256 MB copy (GB/s): the ceiling
    every fill runs against."""
    torch = c.torch
    src = torch.empty(256 << 20, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        dst.copy_(src, non_blocking=True)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(4):
        dst.copy_(src, non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    return 4 * (256 << 20) / (a.elapsed_time(b) / 1000.0) / 1e9


def run_stack(c, n_layers, batches, link_gbs):
    """The 35B-A3B layer shape as a stack of n_layers layers (layer l: the
    seeded weights of seed + l) sharing one slot pool and one LRU table.
    Decode: n_layers x 47 slots (the single layer's 47 of 128, 37%), batches
    from a cold cache, W warm-up and K timed stack steps each.  Prefill: one
    8192-token chunk per step through every layer, 2 E slots, with each
    prefetch mode (none: each layer fills its own misses; serial: whole-layer
    prefetch between layers; overlap: layer l + 1 streams in while layer l
    computes)."""
    torch, capi, wl = c.torch, c.capi, c.wl
    from routed_expert_layer_gemv_gb300.layer import MoEStack
    work, pwork = wl.DECODE_35B, wl.PREFILL_35B
    spec0 = work.layer
    E, d, f = spec0.E, spec0.d_model, spec0.d_ff
    b_e = 3 * d * f * (1 / 2 + 1 / spec0.block)
    lay = c.capi.moe_expert_layout_for(c.make_desc(spec0, 16))
    pools = [c.pack_pool(lay, E, lambda e, l=l: wl.expert_weights(spec0, work.seed + l, e)) for l in range(n_layers)]
    W, K = c.args.warmup, c.args.steps
    out = {"layers": n_layers, "layer": "35B-A3B shape (d 2048, E 128, top-8, d_ff 768, MXFP4)",
           "decode": {}, "prefill": {}}
    S_dec = n_layers * spec0.n_slots
    spec = dataclasses.replace(spec0, n_slots=S_dec)
    for b in batches:
        st = MoEStack(spec, n_layers, work.seed, b, pools=pools)
        xs = c.tokens(work, b, W + K)
        y = torch.empty(b, d, dtype=torch.bfloat16, device="cuda")
        with torch.cuda.stream(c.st):
            for t in range(W):
                st.forward(xs[t], y, stream=c.st, regime=capi.MOE_REGIME_DECODE)
        torch.cuda.synchronize()
        s0 = [capi.moe_stats(L.h) for L in st.layers]
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        launches = fused = 0
        with torch.cuda.stream(c.st):
            for t in range(K):
                c.flush.zero_()
                ev[t][0].record(c.st)
                _, info = st.forward(xs[W + t], y, stream=c.st, regime=capi.MOE_REGIME_DECODE)
                ev[t][1].record(c.st)
                launches += info.n_launches
                fused += info.fused_step
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(bb) for a, bb in ev)
        s1 = [capi.moe_stats(L.h) for L in st.layers]
        st.close()
        dist = sum(x1[1] - x0[1] for x0, x1 in zip(s0, s1))
        miss = sum(x1[3] - x0[3] for x0, x1 in zip(s0, s1))
        out["decode"][str(b)] = {
            "tokens_per_s": K * b / (ms / 1000.0), "ms_per_step": ms / K, "us_per_layer_step": 1000.0 * ms / K / n_layers,
            "miss_rate": miss / max(1, dist), "fill_GB_per_s": miss * b_e / (ms / 1000.0) / 1e9,
            "layers_fused_per_step": fused / K, "gpu_launches_per_step": launches / K}
    out["decode_slots"] = S_dec
    N = pwork.n_tokens
    xp, _ = wl.iid_tokens(pwork.seed, N, d)
    x = torch.from_numpy(xp.view(np.int16)).view(torch.bfloat16).cuda()
    yp = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
    spec_p = dataclasses.replace(spec0, n_slots=2 * E)
    Kp, Wp = max(3, c.args.prefill_steps // 2), 1
    names = {"none": (capi.MOE_PREFETCH_NONE, capi.MOE_FILL_KERNEL),
             "serial": (capi.MOE_PREFETCH_SERIAL, capi.MOE_FILL_KERNEL),
             "overlap": (capi.MOE_PREFETCH_OVERLAP, capi.MOE_FILL_KERNEL),
             "serial_memcpy": (capi.MOE_PREFETCH_SERIAL, capi.MOE_FILL_MEMCPY),
             "overlap_memcpy": (capi.MOE_PREFETCH_OVERLAP, capi.MOE_FILL_MEMCPY)}
    for name, (mode, copy) in names.items():
        st = MoEStack(spec_p, n_layers, work.seed, N, pools=pools)
        capi.moe_stack_set_prefetch(st.h, mode)
        capi.moe_stack_set_prefetch_copy(st.h, copy)
        with torch.cuda.stream(c.st):
            for _ in range(Wp):
                st.forward(x, yp, stream=c.st, regime=capi.MOE_REGIME_PREFILL)
        torch.cuda.synchronize()
        s0 = [capi.moe_stats(L.h) for L in st.layers]
        p0 = capi.moe_stack_prefetch_stats(st.h)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Kp)]
        with torch.cuda.stream(c.st):
            for t in range(Kp):
                c.flush.zero_()
                ev[t][0].record(c.st)
                st.forward(x, yp, stream=c.st, regime=capi.MOE_REGIME_PREFILL)
                ev[t][1].record(c.st)
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(bb) for a, bb in ev)
        s1 = [capi.moe_stats(L.h) for L in st.layers]
        p1 = capi.moe_stack_prefetch_stats(st.h)
        st.close()
        miss = sum(x1[3] - x0[3] for x0, x1 in zip(s0, s1)) + (p1[3] - p0[3])
        gbs = miss * b_e / (ms / 1000.0) / 1e9
        out["prefill"][name] = {"tokens_per_s": Kp * N / (ms / 1000.0), "ms_per_chunk": ms / Kp,
                                "ms_per_layer": ms / Kp / n_layers, "misses_per_chunk": miss / Kp,
                                "link_GB_per_s": gbs, "frac_of_measured_link": gbs / link_gbs if link_gbs else None}
    out["prefill_slots"] = 2 * E
    out["prefill_tokens"] = N
    ov, se = out["prefill"]["overlap"]["ms_per_chunk"], out["prefill"]["serial"]["ms_per_chunk"]
    out["prefill"]["serial_over_overlap"] = se / ov
    return out


def run_formats(c, batches, peak):
    """The 35B-A3B layer shape with FP8 (MXFP8) and BF16 expert weights, every
    expert resident: decode steps at each batch size (A16; tokens/s and the
    step's HBM bytes over its time) and one prefill chunk of 8192 tokens (W8A8,
    W16A16; GEMM TFLOP/s against the dtype's dense tensor peak); then the
    MXFP4 layer's chunk as W4A8 (GEMM against the FP8 peak) and as W4A16
    (through the decode regime)."""
    wl = c.wl
    out = {}
    for fmt in (wl.MXFP8, wl.BF16):
        work = dataclasses.replace(wl.DECODE_35B, name="%s_%s" % (wl.DECODE_35B.name, fmt),
                                   layer=dataclasses.replace(wl.DECODE_35B.layer, fmt=fmt))
        resident = c.layer(work, max(batches), n_slots=work.layer.E, install_all=True)
        dec = {}
        for b in batches:
            r = run_decode(c, work, b, resident=resident)
            dec[str(b)] = {"tokens_per_s": r["tokens"] / (r["ms"] / 1000.0), "ms_per_step": r["ms"] / r["steps"],
                           "frac_of_measured_hbm": r["bytes"] / (r["ms"] / 1000.0) / 1e9 / peak,
                           "fused_steps": r["fused_steps"]}
        resident[0].close()
        pwork = dataclasses.replace(wl.PREFILL_35B, name="%s_%s" % (wl.PREFILL_35B.name, fmt),
                                    layer=dataclasses.replace(wl.PREFILL_35B.layer, fmt=fmt))
        c.pools[pwork.name] = c.pools[work.name]    # the same weights (same seed and shape)
        dpeak, dkind = _dtype_peak(fmt)
        pre = prefill_summary(run_prefill(c, pwork), dpeak)
        pre["peak_TFLOP_s"] = dpeak
        pre["peak_kind"] = dkind
        out[fmt] = {"expert_bytes": expert_bytes(work.layer), "decode_all_resident": dec, "prefill_n8192": pre}
        c.pools.clear()
    # W4A8 on the prefill chunk: the MXFP4 layer with MXFP8 activations
    # (tcgen05 kind::mxf8f6f4, E4M3 x E2M1, at the FP8 rate)
    pw8 = dataclasses.replace(wl.PREFILL_35B, name=wl.PREFILL_35B.name + "_w4a8",
                              layer=dataclasses.replace(wl.PREFILL_35B.layer, prefill_act=wl.MXFP8))
    dpeak, dkind = _dtype_peak("mxfp8")
    pre = prefill_summary(run_prefill(c, pw8), dpeak)
    pre["peak_TFLOP_s"] = dpeak
    pre["peak_kind"] = dkind
    out["w4a8_prefill_n8192"] = pre
    c.pools.clear()
    # W4A16 on a prefill chunk: the MXFP4 layer's 8192-token chunk through the
    # decode regime (FP4 weights x bf16-class activations, mma.sync GEMV),
    # next to its W4A4 tcgen05 prefill
    torch, capi = c.torch, c.capi
    pw = wl.PREFILL_35B
    N = pw.n_tokens
    xp, _ = wl.iid_tokens(pw.seed, N, pw.layer.d_model)
    x = torch.from_numpy(xp.view(np.int16)).view(torch.bfloat16).cuda()
    L, spec = c.layer(pw, N, n_slots=pw.layer.E, install_all=True)
    y = torch.empty(N, spec.d_model, dtype=torch.bfloat16, device="cuda")
    L.forward(x, y, regime=capi.MOE_REGIME_DECODE)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 2
    a.record()
    for _ in range(reps):
        L.forward(x, y, regime=capi.MOE_REGIME_DECODE)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    L.close()
    c.pools.clear()
    out["w4a16_prefill_n8192"] = {"workload": pw.name, "regime": "decode (A16) on the prefill chunk",
                                  "tokens_per_s": N / (ms / 1000.0), "ms_per_chunk": ms}
    return out


def decode_workload(c, work, batches, peak, with_modes=True, timed=None):
    """Everything reported for one decode workload: the timed default pass
    (`timed`, when already run), kernel times, fill modes, e2e, miss rates and
    the all-resident pass whose fused step is the roofline kernel."""
    capi = c.capi
    runs = timed or [run_decode(c, work, b) for b in batches]
    pruns = [run_decode(c, work, b, profile=True) for b in batches]
    modes = {}
    if with_modes:
        names = {"memcpy": capi.MOE_FILL_MEMCPY, "device": capi.MOE_FILL_DEVICE, "kernel": capi.MOE_FILL_KERNEL,
                 "fused": capi.MOE_FILL_FUSED}
        modes = {n: [run_decode(c, work, b, fill=names[n]) for b in batches]
                 for n in c.args.fill_modes.split(",") if n in names}
    e2e = [run_e2e(c, work, b) for b in batches]
    resident = c.layer(work, max(batches), n_slots=work.layer.E, install_all=True)
    res = [run_decode(c, work, b, resident=resident) for b in batches]            # tokens/s
    pres = [run_decode(c, work, b, profile=True, resident=resident) for b in batches]   # kernel times
    resident[0].close()
    trace = [trace_miss_rate(c, work, b) for b in batches]
    per = {}
    for i, b in enumerate(batches):
        r, pr, e, rr, tr = runs[i], pruns[i], e2e[i], res[i], trace[i]
        st_ms, st_n = pres[i]["prof"]["step"]
        per[str(b)] = {
            "tokens_per_s": r["tokens"] / (r["ms"] / 1000.0),
            "e2e_tokens_per_s": e["tokens"] / e["s"],
            "ms_per_step": r["ms"] / r["steps"],
            "ms_per_step_median": r["p50"],
            "miss_rate": r["misses"] / max(1, r["distinct"]),
            "miss_rate_full_trace": tr[0],
            "trace_steps": tr[1],
            "fused_step_share": r["fused_steps"] / r["steps"],
            "kernel_ms_per_step": {k: v[0] / pr["steps"] for k, v in pr["prof"].items() if v[1]},
            "tokens_per_s_by_fill_mode": {n: fr[i]["tokens"] / (fr[i]["ms"] / 1000.0) for n, fr in modes.items()},
            "all_resident": {
                "tokens_per_s": rr["tokens"] / (rr["ms"] / 1000.0),
                "ms_per_step": rr["ms"] / rr["steps"],
                "step_kernel_us": 1000.0 * st_ms / max(1, st_n),
                "hbm_GB_per_s": rr["bytes"] / (rr["ms"] / 1000.0) / 1e9,
                "frac_of_measured_hbm": rr["bytes"] / (rr["ms"] / 1000.0) / 1e9 / peak,
                "kernel_frac_of_measured_hbm":
                    pres[i]["bytes"] / (st_ms / 1000.0) / 1e9 / peak if st_n == pres[i]["steps"] and st_ms else None,
                "kernel_ms_per_step": {k: v[0] / pres[i]["steps"] for k, v in pres[i]["prof"].items() if v[1]},
                "misses": rr["misses"]},
        }
    return dict(runs=runs, e2e=e2e, res=res, pres=pres, per_batch=per)


# ---------------------------------------------------------------- CPU oracle

def cpu_oracle_sample(budget_s: float, threads: int = 0, batches=(1, 4, 16), work_name="decode35b"):
    """Time the C++ FP64 oracle on decode steps of the workload (each batch
    size in turn) until the budget is spent; returns (tokens/s, tokens,
    steps, seconds, threads)."""
    from oracle import native
    from oracle.native import layer as olayer
    from routed_expert_layer_gemv_gb300 import workloads as wl
    work = wl.DECODE_35B if work_name == "decode35b" else wl.TINY
    spec = work.layer
    W_r, b = wl.router_weights(spec, work.seed)
    native.set_threads(threads)
    used = native.threads()
    O = olayer.Layer(spec, lambda e: wl.expert_weights(spec, work.seed, e), W_r, b)
    tokens = steps = 0
    t0 = time.perf_counter()
    per = budget_s / len(batches)
    for batch in batches:
        if work_name == "decode35b":
            xb, _ = wl.ar1_tokens(work.seed + batch, batch, 8, spec.d_model, work.rho)
        else:
            xb = wl.iid_tokens(work.seed, work.n_tokens, spec.d_model)[0][None]
        tb = time.perf_counter()
        t = 0
        while time.perf_counter() - tb < per and t < len(xb):
            O.forward(wl.bf16_bits_to_f64(xb[t]), "decode")
            tokens += xb[t].shape[0]
            steps += 1
            t += 1
    el = time.perf_counter() - t0
    native.set_threads(0)
    return tokens / el, tokens, steps, el, used


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batches", default="1,4,16")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="decode35b", choices=["decode35b", "prefill35b", "prefill753b"],
                    help="decode35b = the headline decode configuration; the prefill ones "
                         "print that prefill chunk's line instead")
    ap.add_argument("--prefill-steps", type=int, default=8)
    ap.add_argument("--stack-layers", type=int, default=8,
                    help="layers of the multi-layer stack measured as an extra key (0: none)")
    ap.add_argument("--formats-only", action="store_true",
                    help="measure only the FP8 / BF16 weight formats and print their object")
    ap.add_argument("--stack-only", action="store_true",
                    help="measure only the multi-layer stack (decode and prefill) and print its object")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the 284B-class decode and the two prefill chunks")
    ap.add_argument("--fill-modes", default="memcpy,device,kernel,fused",
                    help="fill modes timed beside the default per batch ('none': skip them)")
    ap.add_argument("--trace-steps", type=int, default=0,
                    help="steps of the untimed full-trace miss-rate replay (0: the workload's own count)")
    ap.add_argument("--resident-only", action="store_true",
                    help="time only all-resident decode steps of the headline layer (a short run for "
                         "profiler captures)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    ws, rank, local = _dist()
    batches = [int(b) for b in args.batches.split(",")]

    if args.impl == "reference":
        if rank != 0:
            return
        v, tok, steps, el, cores = cpu_oracle_sample(args.cpu_budget)
        cfg = {"workload": "decode_35b_a3b_d2048_e128_top8_f768_mxfp4_s47", "batches": batches}
        sample = "%d decode steps (%d tokens) of batches 1/4/16, %.1f s, C++ FP64 oracle" % (steps, tok, el)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
                "n_gpus": 0, "steps": steps, "warmup": 0, "ms_per_step": 1000.0 * el / max(1, steps),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": cfg,
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    c = Ctx(args)
    wl, capi = c.wl, c.capi
    peak, peak_kind = _peaks()
    fp4, fp4_kind = _fp4_peak()
    clocks = ClockSampler(local)

    if args.workload != "decode35b":
        work = wl.PREFILL_35B if args.workload == "prefill35b" else wl.PREFILL_753B
        clocks.start()
        r = run_prefill(c, work)
        clk = clocks.stop()
        sm = prefill_summary(r, fp4)
        tboth = sm["gemm_tflops"]["both"]
        line = {"metric": METRIC, "value": sm["tokens_per_s"] * ws, "unit": "tokens/s", "n_gpus": ws,
                "steps": r["steps"], "warmup": r["warmup"], "ms_per_step": sm["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "fp4(e2m1)xfp4(e2m1)->f32",
                "data": "synthetic (seeded i.i.d. hidden states, random FP4 weights)",
                "config": {"workload": work.name, "l2": "flushed (512 MiB write) between timed steps",
                           "detail": sm},
                "roofline": {"bound": "tensor", "kernel": "prefill grouped GEMM (gate/up + down)",
                             "achieved": tboth, "peak": fp4, "unit": "TFLOP/s",
                             "frac": (tboth / fp4) if tboth else None, "traffic": gemm_traffic(args.workload),
                             "peak_kind": fp4_kind},
                "gpu_launches": r["launches"], "clocks": clk}
        if rank == 0:
            print(json.dumps(line))
        return

    work = wl.DECODE_35B
    if args.stack_only:
        print(json.dumps({"stack": run_stack(c, max(1, args.stack_layers), batches, h2d_rate(c))}))
        return
    if args.formats_only:
        print(json.dumps({"formats": run_formats(c, batches, peak)}))
        return
    if args.resident_only:
        resident = c.layer(work, max(batches), n_slots=work.layer.E, install_all=True)
        rr = [run_decode(c, work, b, resident=resident) for b in batches]
        resident[0].close()
        out = {str(r["batch"]): {"tokens_per_s": r["tokens"] / (r["ms"] / 1000.0), "ms_per_step": r["ms"] / r["steps"],
                                 "frac_of_measured_hbm": r["bytes"] / (r["ms"] / 1000.0) / 1e9 / peak,
                                 "fused_steps": r["fused_steps"]} for r in rr}
        print(json.dumps({"workload": work.name + "_all_resident", "steps": args.steps, "warmup": args.warmup,
                          "per_batch": out}))
        return
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    c.layer(work, 16)[0].close()      # pack the host pool before the timed region
    clocks.start()
    runs = [run_decode(c, work, b) for b in batches]
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = sum(r["ms"] for r in runs)
    tokens = sum(r["tokens"] for r in runs)
    dec = decode_workload(c, work, batches, peak, timed=runs)
    e2e_s = sum(r["s"] for r in dec["e2e"])
    if ws > 1:
        t = torch.tensor([ms, e2e_s], dtype=torch.float64, device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms, e2e_s = float(t[0]), float(t[1])
    if rank != 0:
        torch.distributed.barrier() if ws > 1 else None
        return
    value = ws * tokens / (ms / 1000.0)
    e2e_value = ws * tokens / e2e_s

    # roofline: the fused decode step kernel on the all-resident steps of the
    # batches that ran fused (one launch per step, so its per-launch events
    # time exactly the kernel)
    fb = [r for r in dec["pres"] if r["prof"]["step"][1] == r["steps"]]
    r_bytes = sum(r["bytes"] for r in fb)
    r_ms = sum(r["prof"]["step"][0] for r in fb)
    r_n = sum(r["prof"]["step"][1] for r in fb)
    achieved = (r_bytes / max(r_n, 1)) / ((r_ms / max(r_n, 1)) / 1000.0) / 1e9 if r_ms > 0 else None
    ratio = traffic_ratio("step_kernel", "decode35b_resident_b4")
    roof = {"bound": "hbm", "kernel": "fused decode step (step_kernel), all-resident decode 35B-A3B steps of "
                                      "batches %s" % "/".join(str(r["batch"]) for r in fb),
            "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": (achieved / peak) if achieved else None,
            "traffic": ratio * r_bytes / max(r_n, 1) if ratio else None, "peak_kind": peak_kind,
            "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of the fused step kernel, "
                              "decode 35B-A3B batch 4 all-resident, scaled to this run's bytes per launch"
                              if ratio else None,
            "bytes_per_launch": r_bytes / max(r_n, 1), "ms_per_launch": r_ms / max(r_n, 1),
            "launches": r_n}

    link = h2d_rate(c)
    extra = {}
    if not args.no_extra:
        w3 = wl.DECODE_284B
        d3 = decode_workload(c, w3, list(w3.batches), peak, with_modes=False)
        t3 = sum(r["tokens"] for r in d3["runs"])
        m3 = sum(r["ms"] for r in d3["runs"])
        extra["decode_284b_a13b"] = {
            "workload": w3.name, "batches": list(w3.batches), "steps": args.steps,
            "tokens_per_s": t3 / (m3 / 1000.0),
            "e2e_tokens_per_s": t3 / sum(r["s"] for r in d3["e2e"]),
            "miss_rate": sum(r["misses"] for r in d3["runs"]) / max(1, sum(r["distinct"] for r in d3["runs"])),
            "per_batch": d3["per_batch"]}
        c.pools.clear()
        for key, w in (("prefill_35b_a3b_n8192", wl.PREFILL_35B), ("prefill_753b_n16384", wl.PREFILL_753B)):
            extra[key] = prefill_summary(run_prefill(c, w), fp4)
            c.pools.clear()
        if args.stack_layers > 0:
            extra["stack_35b_a3b_l%d" % args.stack_layers] = run_stack(c, args.stack_layers, batches, link)
        extra["formats_35b_a3b"] = run_formats(c, batches, peak)

    cpu = None
    if not args.no_cpu_baseline:
        v, tok, steps, el, cores = cpu_oracle_sample(args.cpu_budget)
        v1, tok1, steps1, el1, _ = cpu_oracle_sample(min(10.0, args.cpu_budget / 2), threads=1)
        v0, tok0, steps0, el0, _ = cpu_oracle_sample(3.0, threads=1, batches=(64,), work_name="tiny")
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": "%d decode steps (%d tokens) of batches 1/4/16 of the decode 35B-A3B layer, %.1f s, "
                         "C++ FP64 oracle on %d threads" % (steps, tok, el, cores),
               "one_thread": {"decode_35b_a3b": {"value": v1, "unit": "tokens/s", "steps": steps1},
                              "tiny_n64": {"value": v0, "unit": "tokens/s", "steps": steps0}}}
    fused = sum(r["fused_steps"] for r in runs)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / (args.steps * len(batches)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp4(e2m1)xbf16->f32",
        "data": "synthetic (seeded AR(1) hidden states, random FP4 weights)",
        "config": {"workload": work.name, "batches": batches,
                   "steps_per_batch": args.steps,
                   "miss_rate_per_batch": {b: dec["per_batch"][b]["miss_rate"] for b in dec["per_batch"]},
                   "l2": "flushed (512 MiB write) between timed steps",
                   "path": "library defaults: a step with misses possible runs the chain of launches -- at "
                           "batch 1 and 4 the expert FFN reads misses over the host link and writes them to their "
                           "slots, at batch 16 (distinct experts > slots) a copy kernel on 12 reserved SMs fills "
                           "them; %d of %d timed steps ran as one fused launch (only a layer holding every expert "
                           "fuses its small steps)" % (fused, args.steps * len(batches)),
                   "h2d_GB_per_s_measured": link,
                   "timing": "value from a pass without per-kernel events; kernel times and roofline from "
                             "instrumented passes of the same steps",
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "per_batch": dec["per_batch"]},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s",
                "h2d_bytes_per_step": sum(e["h2d"] for e in dec["e2e"]) / (args.steps * len(batches)),
                "d2h_bytes_per_step": sum(e["d2h"] for e in dec["e2e"]) / (args.steps * len(batches))},
        "gpu_launches": sum(r["launches"] for r in runs),
        "clocks": clk,
    }
    line.update(extra)
    print(json.dumps(line))


if __name__ == "__main__":
    main()
