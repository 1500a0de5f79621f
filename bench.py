#!/usr/bin/env python3
"""Benchmark of the mixed-adapter LoRA delta on one GB300 (or N replicas).

One step = one pass of the whole hot path over one batch: lora_build_segments
(routing metadata) followed, for every projection of the workload, by the
kernels of lora_apply_shrink_expand (the fused decode kernel, the tensor
shrink and the tensor expand).  Inputs are resident in HBM before timing
starts.  Between timed steps y is restored and L2 is flushed (a 256 MiB
write), both outside the CUDA events that time the step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0): the headline workload (cont_batch by default)
and, under "per_workload", every configuration with its step, apply-only and
segment-build times, per-kernel times, roofline fractions and the oracle's
single-thread and all-core rates.  Under torchrun every rank runs its own
batch on its own GPU (no data exchange; weak scaling); times are max-reduced.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from adapter_gemv_lora_gb300 import workloads as W  # noqa: E402

METRIC = "LoRA-delta tokens/s; HBM GB/s (decode) & TFLOP/s (prefill) as % roofline"
TC_MIN_QLEN = 64  # documented tensor-path threshold of the library (own sequence length)
STAGES = ["decode", "tc_shrink", "tc_expand"]  # lora_apply_stage 1, 2, 3
KERNEL_NAMES = {"decode": "dec_fused_kernel", "tc_shrink": "tc_shrink_kernel", "tc_expand": "tc_expand_kernel",
                "seg_build": "seg_build_kernel"}
KERNEL_SOURCES = {"decode": "decode.cu", "tc_shrink": "tensor.cu", "tc_expand": "tensor.cu"}
L2_FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------- helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), float(d.get("bf16_tflops", 1900.0)), "measured"
    return 6800.0, 1900.0, "fallback"


def algorithmic_units(wl: W.Workload):
    """Per projection and per kernel: algorithmic bytes and flops of one step.

    Per active row: 2*d_in bytes of x and 8*D bytes of y (fp32 read + write;
    the decode kernel moves both, the tensor shrink x and the tensor expand
    y).  Per (slot, lane) present on a kernel's rows: 2*r*d_in bytes of A
    (decode kernel, tensor shrink) and 2*r*d_out bytes of B (decode kernel,
    tensor expand), true rank only; a slot with rows on both paths is read by
    both paths' kernels, so each kernel counts its own factor reads.  Base
    rows and rank-0 lanes cost nothing.  flops = sum over active rows and
    loaded lanes of 2*r*(d_in + d_out)."""
    slot = np.repeat(wl.adapter_ids, wl.q_seq_lens)
    qlen = np.repeat(wl.q_seq_lens, wl.q_seq_lens)
    cls = (qlen >= TC_MIN_QLEN).astype(np.int64)
    out = []
    for proj in wl.projections:
        u = {s: {"bytes": 0, "flops": 0, "rows": 0} for s in STAGES}
        for c in (0, 1):
            rows = (slot != 0) & (cls == c)
            ks = slot[rows]
            sh, ex = ("decode", "decode") if c == 0 else ("tc_shrink", "tc_expand")
            for k in np.unique(ks):
                n = int((ks == k).sum())
                loaded = [l for l in range(proj.num_lanes) if proj.rank[k, l] > 0]
                for l in loaded:
                    r = int(proj.rank[k, l])
                    u[sh]["bytes"] += 2 * r * proj.d_in
                    u[ex]["bytes"] += 2 * r * proj.lane_d_out[l]
                    u[sh]["flops"] += n * 2 * r * proj.d_in
                    u[ex]["flops"] += n * 2 * r * proj.lane_d_out[l]
                if loaded:
                    u[sh]["bytes"] += n * 2 * proj.d_in
                    u[ex]["bytes"] += n * 8 * sum(proj.lane_d_out[l] for l in loaded)
                    u[sh]["rows"] += n
                    if ex != sh:
                        u[ex]["rows"] += n
        out.append(u)
    return out


def step_bytes(wl: W.Workload):
    """Algorithmic bytes and flops of the whole step: every active row's x and
    y once, and every present (slot, lane)'s factors once, whichever paths its
    rows take."""
    slot = np.repeat(wl.adapter_ids, wl.q_seq_lens)
    total, flops = 0, 0
    for proj in wl.projections:
        for k in np.unique(slot[slot != 0]):
            n = int((slot == k).sum())
            loaded = [l for l in range(proj.num_lanes) if proj.rank[k, l] > 0]
            for l in loaded:
                r = int(proj.rank[k, l])
                total += 2 * r * (proj.d_in + proj.lane_d_out[l])
                flops += n * 2 * r * (proj.d_in + proj.lane_d_out[l])
            if loaded:
                total += n * (2 * proj.d_in + 8 * sum(proj.lane_d_out[l] for l in loaded))
    return total, flops


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0].split()[0]))
                mx.append(float(parts[1].split()[0]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def traffic_from_profile(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it still matches the kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for ln in open(path):
        if ":" in ln and not ln.startswith("#"):
            k, v = ln.split(":", 1)
            vals[k.strip()] = v.strip()
    src = os.path.join(ROOT, "adapter_gemv_lora_gb300", "csrc",
                       "tensor.cu" if kernel.startswith("tc_") else
                       "segments.cu" if kernel.startswith("seg_") else
                       "fused.cu" if kernel.startswith("fused_") else "decode.cu")
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if vals.get("source_sha256_16") != sha:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def truncate_workload(wl, n_seqs: int):
    """The first n_seqs sequences of a workload (same adapters and factors)."""
    n_seqs = min(n_seqs, wl.S)
    T = int(wl.q_seq_lens[:n_seqs].sum())
    out = W.Workload(wl.name + f"[:{n_seqs}]", wl.adapter_ids[:n_seqs].copy(), wl.q_seq_lens[:n_seqs].copy(),
                     wl.num_slots)
    for p in wl.projections:
        out.projections.append(W.Projection(p.name, p.d_in, p.lane_d_out, p.rank, p.scale, p.A, p.B,
                                            p.x[:T].copy(), p.y0[:T].copy(), p.max_rank))
    return out


# ------------------------------------------------------------ our arm

def setup_device_workload(wl, dev):
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    T = wl.T
    projs = []
    for proj in wl.projections:
        pool = LD.LoraPool(wl.num_slots, proj.max_rank, proj.d_in, proj.lane_d_out, T, device=dev)
        for k in range(1, wl.num_slots):
            for l in range(proj.num_lanes):
                r = int(proj.rank[k, l])
                if r > 0:
                    A = torch.from_numpy(proj.A[k][l].view(np.int16)).to(dev)
                    B = torch.from_numpy(proj.B[k][l].view(np.int16)).to(dev)
                    pool.load(k, l, A, B, float(proj.scale[k, l]))
                    torch.cuda.synchronize()
        x = torch.from_numpy(proj.x.view(np.int16)).to(dev)
        y0 = torch.from_numpy(proj.y0).to(dev)
        y = y0.clone()
        projs.append({"proj": proj, "pool": pool, "x": x, "y0": y0, "y": y})
    seg = LD.LoraSegments(wl.S, T, wl.num_slots, device=dev)
    ids = torch.from_numpy(wl.adapter_ids.astype(np.int32)).to(dev)
    lens = torch.from_numpy(wl.q_seq_lens.astype(np.int32)).to(dev)
    return projs, seg, ids, lens


def setup_device_moe(wl, dev):
    """Pools (every expert's copy of every adapter at lora_moe_slot), the
    dispatched rows' x / y and the routing tensors of an MoE workload."""
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    N = 1 + wl.num_experts * wl.num_adapters
    projs = []
    for mp in wl.projections:
        pool = LD.LoraPool(N, mp.max_rank, mp.d_in, mp.lane_d_out, wl.R, device=dev)
        for e in range(wl.num_experts):
            for a in range(1, wl.num_adapters + 1):
                k = LD.lora_moe_slot(e, a, wl.num_adapters)
                for l in range(mp.num_lanes):
                    if mp.rank[a, l] > 0:
                        A = torch.from_numpy(mp.A[e][a][l].view(np.int16)).to(dev)
                        B = torch.from_numpy(mp.B[e][a][l].view(np.int16)).to(dev)
                        pool.load(k, l, A, B, float(mp.scale[a, l]))
            torch.cuda.synchronize()
        x = torch.from_numpy(mp.x.view(np.int16)).to(dev)
        y0 = torch.from_numpy(mp.y0).to(dev)
        projs.append({"proj": mp, "pool": pool, "x": x, "y0": y0, "y": y0.clone()})
    seg = LD.LoraSegments(min(wl.R, 4096), wl.R, N, device=dev)
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v, dtype=np.int32)).to(dev)
    routing = (t(wl.row_expert), t(wl.row_adapter), t(wl.row_seq))
    return projs, seg, routing


def moe_units(wl):
    """Algorithmic bytes and flops of one MoE step: every dispatched row with
    an adapter moves its x (2 d_in) and its y (8 D) once; every present
    (expert, adapter, lane) its factors once (2 r (d_in + d_out))."""
    total, flops = 0, 0
    act = wl.row_adapter != 0
    pairs = np.unique(np.stack([wl.row_expert[act], wl.row_adapter[act]], axis=1), axis=0) if act.any() else []
    for mp in wl.projections:
        n = int(act.sum())
        total += n * (2 * mp.d_in + 8 * mp.D)
        for e, a in pairs:
            n_ea = int(((wl.row_expert == e) & (wl.row_adapter == a)).sum())
            for l in range(mp.num_lanes):
                r = int(mp.rank[a, l])
                total += 2 * r * (mp.d_in + mp.lane_d_out[l])
                flops += n_ea * 2 * r * (mp.d_in + mp.lane_d_out[l])
    return total, flops


def time_ours(wl, steps, warmup, dev, sampler_index):
    """Device times of one workload's step.

    * eager pass: CUDA events between every kernel (lora_apply_stage) on the
      launching stream -> per-kernel and segment-build times;
    * the step as a serving engine runs it (lora_build_segments +
      lora_apply_shrink_expand per projection) captured once in a CUDA graph
      and replayed -> step time (the headline), checked bit for bit against
      an eager step;
    * the applies alone (segments built once before) and the build alone,
      each captured and replayed the same way -> apply-only and build times.
    y is restored and L2 flushed before every timed replay, outside the events."""
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    moe = isinstance(wl, W.MoeWorkload)
    if moe:
        projs, seg, routing = setup_device_moe(wl, dev)
        ids = lens = None
        T = wl.R
    else:
        projs, seg, ids, lens = setup_device_workload(wl, dev)
        T = wl.T
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    n_ev = 2 + len(STAGES) * len(projs)

    def reset():
        for pr in projs:
            pr["y"].copy_(pr["y0"])
        flush.fill_(1)

    def build():
        if moe:
            LD.lora_build_segments_moe(seg.handle, routing[0].data_ptr(), routing[1].data_ptr(),
                                       routing[2].data_ptr(), T, wl.num_experts, wl.num_adapters,
                                       torch.cuda.current_stream().cuda_stream)
        else:
            LD.lora_build_segments(seg.handle, ids.data_ptr(), lens.data_ptr(), wl.S, T,
                                   torch.cuda.current_stream().cuda_stream)

    def applies():
        for pr in projs:
            LD.apply(pr["pool"], seg, pr["x"], pr["y"])

    def public_step():
        build()
        applies()

    def one_eager(evs):
        evs[0].record(stream)
        build()
        evs[1].record(stream)
        i = 2
        for pr in projs:
            for stage in range(1, len(STAGES) + 1):
                LD.apply_stage(pr["pool"], seg, pr["x"], pr["y"], stage)
                evs[i].record(stream)
                i += 1

    evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(steps)]
    warm = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    for _ in range(warmup):
        reset()
        one_eager(warm)
    torch.cuda.synchronize()
    assert seg.status() == 0, LD.lora_status_string(seg.status())
    barrier()
    torch.cuda.synchronize()
    n0 = LD.lora_launch_count()
    for st in range(steps):
        reset()
        one_eager(evsets[st])
    n1 = LD.lora_launch_count()
    torch.cuda.synchronize()
    barrier()
    assert seg.status() == 0, LD.lora_status_string(seg.status())
    stage_ms = []
    for p in range(len(projs)):
        per = {}
        for j, name in enumerate(STAGES):
            a, b = 1 + len(STAGES) * p + j, 2 + len(STAGES) * p + j
            per[name] = statistics.mean(ev[a].elapsed_time(ev[b]) for ev in evsets)
        stage_ms.append(per)
    res = {"step_ms_eager": statistics.mean(ev[0].elapsed_time(ev[-1]) for ev in evsets),
           "seg_ms_eager": statistics.mean(ev[0].elapsed_time(ev[1]) for ev in evsets),
           "stage_ms": stage_ms, "launches_eager": n1 - n0}

    # reference bits: one eager public step from the restored inputs
    reset()
    public_step()
    torch.cuda.synchronize()
    y_eager = [pr["y"].clone() for pr in projs]

    def graph_loop(fn, check, sampled):
        g = torch.cuda.CUDAGraph()
        n_cap0 = LD.lora_launch_count()
        with torch.cuda.graph(g):
            fn()
        per_replay = LD.lora_launch_count() - n_cap0
        if check:
            reset()
            g.replay()
            torch.cuda.synchronize()
            for pr, ye in zip(projs, y_eager):
                assert torch.equal(pr["y"].view(torch.int32), ye.view(torch.int32)), "graph replay differs from eager"
        for _ in range(warmup):
            reset()
            g.replay()
        torch.cuda.synchronize()
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        sampler = ClockSampler(sampler_index) if sampled else None
        if sampler:
            # the clock samples cover sustained replays of this graph: about
            # 0.6 s of untimed replays right before the timed ones
            sampler.__enter__()
            t_end = time.perf_counter() + 0.6
            while time.perf_counter() < t_end:
                for _ in range(20):
                    reset()
                    g.replay()
                torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        for st in range(steps):
            reset()
            gev[st][0].record(stream)
            g.replay()
            gev[st][1].record(stream)
        torch.cuda.synchronize()
        barrier()
        if sampler:
            sampler.__exit__()
        ms = [a.elapsed_time(b) for a, b in gev]
        return ms, per_replay * steps, (sampler.summary() if sampler else None)

    gms, launches, clocks = graph_loop(public_step, True, True)
    ams, _, _ = graph_loop(applies, True, False)  # segments were built by the eager step above
    sms, _, _ = graph_loop(build, False, False)
    assert seg.status() == 0, LD.lora_status_string(seg.status())
    res.update({"step_ms": statistics.mean(gms), "step_ms_median": statistics.median(gms),
                "apply_ms": statistics.mean(ams), "seg_ms": statistics.mean(sms), "graph": True,
                "launches": launches, "clocks": clocks})
    del flush
    return res, (projs, seg, ids, lens)


def time_e2e(wl, ctx, steps, warmup, dev):
    """Same step through the public API with pinned host buffers: every step copies
    its x, y and routing ids host -> device, builds + applies, and copies y back,
    all inside the timed region.  Steps are double-buffered the way a serving loop
    runs them: step i's host -> device copies (one stream) and step i-1's
    device -> host copy (another) overlap step i's kernels; each step still moves
    all of its own bytes."""
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    projs, seg, ids, lens = ctx
    T = wl.T
    host = []
    for pr in projs:
        host.append({"x": torch.from_numpy(pr["proj"].x.view(np.int16)).pin_memory(),
                     "y0": torch.from_numpy(pr["proj"].y0).pin_memory(),
                     "out": [torch.empty(pr["y"].shape, dtype=torch.float32).pin_memory() for _ in range(2)]})
    ids_h = torch.from_numpy(wl.adapter_ids.astype(np.int32)).pin_memory()
    lens_h = torch.from_numpy(wl.q_seq_lens.astype(np.int32)).pin_memory()
    h2d = sum(h["x"].numel() * 2 + h["y0"].numel() * 4 for h in host) + ids_h.numel() * 4 + lens_h.numel() * 4
    d2h = sum(h["out"][0].numel() * 4 for h in host)
    # two device buffer sets: step i uses set i % 2
    dbuf = [{"ids": ids, "lens": lens, "x": [pr["x"] for pr in projs], "y": [pr["y"] for pr in projs]},
            {"ids": torch.empty_like(ids), "lens": torch.empty_like(lens),
             "x": [torch.empty_like(pr["x"]) for pr in projs], "y": [torch.empty_like(pr["y"]) for pr in projs]}]
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    started = [False, False]

    def one(i):
        b = i % 2
        d = dbuf[b]
        with torch.cuda.stream(s_in):
            if started[b]:
                s_in.wait_event(ev_out[b])  # the step that last used this set has been copied out
            d["ids"].copy_(ids_h, non_blocking=True)
            d["lens"].copy_(lens_h, non_blocking=True)
            for j, h in enumerate(host):
                d["x"][j].copy_(h["x"], non_blocking=True)
                d["y"][j].copy_(h["y0"], non_blocking=True)
            ev_in[b].record(s_in)
        comp.wait_event(ev_in[b])
        LD.lora_build_segments(seg.handle, d["ids"].data_ptr(), d["lens"].data_ptr(), wl.S, T, comp.cuda_stream)
        for j, pr in enumerate(projs):
            LD.apply(pr["pool"], seg, d["x"][j], d["y"][j])
        ev_comp[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            for j, h in enumerate(host):
                h["out"][b].copy_(d["y"][j], non_blocking=True)
            ev_out[b].record(s_out)
        started[b] = True

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record(comp)
    s_in.wait_event(e0)
    for i in range(steps):
        one(warmup + i)
    comp.wait_event(ev_out[(warmup + steps - 1) % 2])
    e1.record(comp)
    torch.cuda.synchronize()
    barrier()
    ms = e0.elapsed_time(e1) / steps
    for h in host:  # both buffer sets computed the same step: their copied-out results agree bit for bit
        assert torch.equal(h["out"][0].view(torch.int32), h["out"][1].view(torch.int32)), "e2e outputs differ"
        assert not torch.equal(h["out"][0], h["y0"]), "e2e step changed nothing"
    return ms, h2d, d2h


def fused_units(wl):
    """Algorithmic flops and bytes of the fused projection (y = x W^T + delta)
    per projection: 2 T D d_in flops of the base product plus the delta's;
    bytes = x and W read once, y written once (4 B per element), the present
    factors once."""
    out = []
    slot = np.repeat(wl.adapter_ids, wl.q_seq_lens)
    for proj in wl.projections:
        T, D, K = wl.T, proj.D, proj.d_in
        flops = 2 * T * D * K
        byts = 2 * T * K + 2 * D * K + 4 * T * D
        for k in np.unique(slot[slot != 0]):
            n = int((slot == k).sum())
            for l in range(proj.num_lanes):
                r = int(proj.rank[k, l])
                if r > 0:
                    flops += n * 2 * r * (K + proj.lane_d_out[l])
                    byts += 2 * r * (K + proj.lane_d_out[l])
        out.append({"flops": int(flops), "bytes": int(byts)})
    return out


def _library_mm(xb, wb, y):
    """y = x W^T by the library GEMM (cuBLAS through torch), fp32 output when
    torch offers it; returns a label of what ran."""
    import torch
    try:
        torch.mm(xb, wb.t(), out_dtype=torch.float32, out=y)
        return "torch.mm bf16 x bf16 -> fp32 (cuBLAS)"
    except (TypeError, RuntimeError):
        y.copy_(torch.mm(xb, wb.t()))
        return "torch.mm bf16 x bf16 -> bf16 (cuBLAS), copied to fp32 y"


def time_fused(wl, steps, warmup, dev):
    """The fused projection of every projection of a workload (graph replays
    with L2 flushed between them): the whole step (build + fused projections),
    the GEMM kernel alone, and, for comparison, the library GEMM (cuBLAS) with
    the separate delta apply after it."""
    import torch
    from adapter_gemv_lora_gb300 import lora_delta as LD
    projs, seg, ids, lens = setup_device_workload(wl, dev)
    for i, pr in enumerate(projs):
        pr["W"] = torch.from_numpy(W.projection_weight(pr["proj"], seed=1 + i).view(np.int16)).to(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    T = wl.T

    def build():
        LD.lora_build_segments(seg.handle, ids.data_ptr(), lens.data_ptr(), wl.S, T, stream.cuda_stream)

    def fused_step():
        build()
        for pr in projs:
            LD.fused_projection(pr["pool"], seg, pr["W"], pr["x"], pr["y"])

    def gemm_only():
        for pr in projs:
            LD.fused_projection_stage(pr["pool"], seg, pr["W"], pr["x"], pr["y"], 3)

    label = [None]

    def library_step():
        build()
        for pr in projs:
            label[0] = _library_mm(pr["x"].view(torch.bfloat16), pr["W"].view(torch.bfloat16), pr["y"])
            LD.apply(pr["pool"], seg, pr["x"], pr["y"])

    def library_gemm():
        for pr in projs:
            _library_mm(pr["x"].view(torch.bfloat16), pr["W"].view(torch.bfloat16), pr["y"])

    # eager reference bits of the fused step
    fused_step()
    torch.cuda.synchronize()
    assert seg.status() == 0, LD.lora_status_string(seg.status())
    y_eager = [pr["y"].clone() for pr in projs]
    library_step()  # warms cuBLAS outside any capture
    torch.cuda.synchronize()

    def graph_ms(fn, check=False):
        g = torch.cuda.CUDAGraph()
        n0 = LD.lora_launch_count()
        with torch.cuda.graph(g):
            fn()
        launches = LD.lora_launch_count() - n0
        if check:
            g.replay()
            torch.cuda.synchronize()
            for pr, ye in zip(projs, y_eager):
                assert torch.equal(pr["y"].view(torch.int32), ye.view(torch.int32)), "fused replay differs"
        for _ in range(warmup):
            flush.fill_(1)
            g.replay()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            flush.fill_(1)
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in evs), launches

    f_ms, f_launch = graph_ms(fused_step, check=True)
    fused_step()  # u' of this step in the pools for the GEMM-only replays
    g_ms, _ = graph_ms(gemm_only)
    l_ms, _ = graph_ms(library_step)
    lg_ms, _ = graph_ms(library_gemm)
    assert seg.status() == 0, LD.lora_status_string(seg.status())
    del flush, projs
    torch.cuda.empty_cache()
    return {"step_ms": f_ms, "gemm_ms": g_ms, "library_step_ms": l_ms, "library_gemm_ms": lg_ms,
            "launches_per_step": f_launch, "library": label[0]}


def fused_record(wl, fr, bf16_peak, hbm_peak):
    units = fused_units(wl)
    flops = sum(u["flops"] for u in units)
    byts = sum(u["bytes"] for u in units)
    g = fr["gemm_ms"] * 1e-3
    return {"step_ms": round(fr["step_ms"], 5), "gemm_ms": round(fr["gemm_ms"], 5),
            "tokens_per_s": round(wl.T / (fr["step_ms"] * 1e-3), 1),
            "alg_flops": int(flops), "alg_bytes": int(byts),
            "gemm_tflops": round(flops / g / 1e12, 2), "gemm_frac_bf16": round(flops / g / 1e12 / bf16_peak, 4),
            "gemm_gbs": round(byts / g / 1e9, 1), "gemm_frac_hbm": round(byts / g / 1e9 / hbm_peak, 4),
            "library_step_ms": round(fr["library_step_ms"], 5), "library_gemm_ms": round(fr["library_gemm_ms"], 5),
            "library": fr["library"],
            "speedup_vs_library_step": round(fr["library_step_ms"] / fr["step_ms"], 3),
            "launches_per_step": fr["launches_per_step"],
            "note": "y = x W^T + delta with the delta in the GEMM's accumulator (one y write); library_step = "
                    "the library GEMM then the separate delta apply (y written, read and written again)"}


def cpu_oracle_rates(wl, threads: int, target_s: float, runs: int = 3, seed: int = 0):
    """The oracle (as it is) on `threads` host threads (0 = all cores).

    The metadata phase (single-threaded code) is timed on the whole step; the
    delta phase on a seeded random sample of the step's rows, sized so that
    one run takes about target_s.  Each phase is the median of `runs` runs.
    tokens/s = T / (metadata time + T * delta time per row)."""
    import oracle
    oracle.build()
    # all cores = the host's usable cores (a 1-thread run leaves OpenMP's
    # default thread count at 1, so it is not asked)
    cores = len(os.sched_getaffinity(0)) if threads <= 0 else threads
    rng = np.random.default_rng(seed)
    meta_t = []
    for _ in range(runs):
        t0 = time.perf_counter()
        meta = oracle.segments(wl.adapter_ids, wl.q_seq_lens, wl.T, wl.num_slots, TC_MIN_QLEN, 128, 8)
        meta_t.append(time.perf_counter() - t0)
    slot = meta["slot"]
    flats = [oracle.flatten_factors(p) for p in wl.projections]

    def run(n):
        rows = np.sort(rng.choice(wl.T, size=n, replace=False))
        t = time.perf_counter()
        for p, fl in zip(wl.projections, flats):
            oracle.delta(p, slot, rows=rows, num_threads=cores, _flat=fl)
        return time.perf_counter() - t

    n = min(16, wl.T)
    dt = run(n)
    while dt < 0.3 * target_s and n < wl.T:
        n = min(wl.T, max(2 * n, int(n * target_s / max(dt, 1e-4) * 0.8)))
        dt = run(n)
    delta_t = sorted(run(n) for _ in range(runs))[runs // 2]
    meta_s = sorted(meta_t)[runs // 2]
    per_row = delta_t / n
    total = meta_s + wl.T * per_row
    return {"tokens_per_s": round(wl.T / total, 2), "threads": cores, "meta_ms": round(1e3 * meta_s, 3),
            "delta_us_per_row": round(1e6 * per_row, 3), "delta_rows_per_s": round(1.0 / per_row, 2),
            "step_s": round(total, 4), "sample_rows": n, "runs": runs,
            "sample": f"metadata on all {wl.T} rows; delta on {n} of {wl.T} rows (seeded uniform sample), "
                      f"fp64, {cores} thread(s), median of {runs}"}


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(v: float) -> float:
    import torch
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return v


def workload_config(wl, ws):
    """The config dict of a bench line (the same for both arms)."""
    active = int((np.repeat(wl.adapter_ids, wl.q_seq_lens) != 0).sum())
    return {"workload": wl.name, "tokens": wl.T, "active_tokens": active, "sequences": wl.S,
            "slots": wl.num_slots,
            "projections": [{"name": p.name, "d_in": p.d_in, "lanes": p.lane_d_out, "max_rank": p.max_rank}
                            for p in wl.projections],
            "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write, outside the events)",
            "timing": "CUDA-graph replay of build_segments + apply per step (checked bit-exact against "
                      "an eager step); per-kernel times from an eager pass with events between kernels",
            "parallelism": f"replicas x{ws} (no exchange)"}


def workload_record(wl, res, hbm_peak, bf16_peak):
    """Times, algorithmic bytes and roofline fractions of one workload."""
    units = algorithmic_units(wl)
    kernels = {}
    for p, (u, sm) in enumerate(zip(units, res["stage_ms"])):
        for name in STAGES:
            ms = sm[name]
            b, f = u[name]["bytes"], u[name]["flops"]
            key = name if len(units) == 1 else f"{wl.projections[p].name}.{name}"
            kernels[key] = {"ms": round(ms, 5), "alg_bytes": int(b), "flops": int(f),
                            "gbs": round(b / (ms * 1e-3) / 1e9, 1) if ms > 0 and b else 0.0,
                            "frac_hbm": round(b / (ms * 1e-3) / 1e9 / hbm_peak, 4) if ms > 0 and b else 0.0,
                            "tflops": round(f / (ms * 1e-3) / 1e12, 2) if ms > 0 and f else 0.0}
    sb, sf = step_bytes(wl)
    step_ms, apply_ms = res["step_ms"], res["apply_ms"]
    return {"tokens": wl.T, "active_tokens": int((np.repeat(wl.adapter_ids, wl.q_seq_lens) != 0).sum()),
            "ms_per_step": round(step_ms, 5), "ms_per_step_median": round(res["step_ms_median"], 5),
            "ms_per_step_eager": round(res["step_ms_eager"], 5),
            "tokens_per_s": round(wl.T / (step_ms * 1e-3), 1),
            "apply_ms": round(apply_ms, 5), "seg_build_ms": round(res["seg_ms"], 5),
            "alg_bytes": int(sb), "flops": int(sf),
            "gbs_step": round(sb / (step_ms * 1e-3) / 1e9, 1),
            "frac_hbm_step": round(sb / (step_ms * 1e-3) / 1e9 / hbm_peak, 4),
            "gbs_apply": round(sb / (apply_ms * 1e-3) / 1e9, 1),
            "frac_hbm_apply": round(sb / (apply_ms * 1e-3) / 1e9 / hbm_peak, 4),
            "tflops_apply": round(sf / (apply_ms * 1e-3) / 1e12, 2),
            "frac_bf16_apply": round(sf / (apply_ms * 1e-3) / 1e12 / bf16_peak, 5),
            "kernels": kernels}


def run_fused_only(args):
    """The fused projection of one workload alone (a diagnostic line, e.g.
    for a profiler capture on a smaller case via --max-seqs)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device("cuda:0")
    wl = W.make_workload(args.workload, seed=args.seed)
    if args.max_seqs:
        wl = truncate_workload(wl, args.max_seqs)
    hbm_peak, bf16_peak, _ = measured_peaks()
    rec = fused_record(wl, time_fused(wl, args.steps, args.warmup, "cuda:0"), bf16_peak, hbm_peak)
    print(json.dumps({"mode": "fused_projection", "workload": wl.name, "tokens": wl.T, **rec}), flush=True)


def run_ours(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = f"cuda:{local}"
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    wl = W.make_workload(args.workload, seed=args.seed + rank)
    if args.max_seqs:
        wl = truncate_workload(wl, args.max_seqs)
    res, ctx = time_ours(wl, args.steps, args.warmup, dev, local)
    step_ms = max_over_ranks(res["step_ms"])
    hbm_peak, bf16_peak, peak_src = measured_peaks()
    rec = workload_record(wl, res, hbm_peak, bf16_peak)
    kernels = rec["kernels"]
    dom_key = max(kernels, key=lambda k: kernels[k]["ms"])
    dom = kernels[dom_key]
    stage_name = dom_key.split(".")[-1]
    traffic = traffic_from_profile(KERNEL_NAMES[stage_name], args.workload)
    T = wl.T
    tokens_per_s = T * ws / (step_ms * 1e-3)
    e2e = None
    if not args.no_e2e:
        e2e_ms, h2d, d2h = time_e2e(wl, ctx, max(8, args.steps // 2), 3, dev)
        e2e_ms = max_over_ranks(e2e_ms)
        e2e = {"value": round(T * ws / (e2e_ms * 1e-3), 1), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 4),
               "overlap": "double-buffered: a step's host-to-device copies, kernels and device-to-host copy "
                          "overlap the neighbouring steps' on three streams"}
    del ctx
    torch.cuda.empty_cache()
    cpu, per_workload = None, None
    if rank == 0 and ws == 1 and not args.no_cpu:
        c_all = cpu_oracle_rates(wl, 0, args.cpu_seconds)
        cpu = {"value": c_all["tokens_per_s"], "unit": "tokens/s", "cores": c_all["threads"], "kind": "oracle",
               "sample": c_all["sample"], "seconds": c_all["step_s"]}
    if rank == 0 and not args.headline_only:
        per_workload = per_workload_summary(args, dev, hbm_peak, bf16_peak, (wl.name, res, cpu is not None))
    sb, sf = step_bytes(wl)
    line = {
        "metric": METRIC,
        "value": round(tokens_per_s, 1),
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 in, fp32 accumulate / fp32 y",
        "data": "synthetic (seeded PCG64; random-init adapters)",
        "config": workload_config(wl, ws),
        "roofline": {"kernel": KERNEL_NAMES[stage_name] + (f" ({dom_key})" if "." in dom_key else ""),
                     "bound": "hbm", "achieved": dom["gbs"], "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(dom["gbs"] / hbm_peak, 4), "traffic": traffic,
                     "peak_source": f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)" if peak_src == "measured"
                     else "fallback 6.8 TB/s"},
        "step_roofline": {"alg_bytes": int(sb), "flops": int(sf), "step_ms": round(step_ms, 5),
                          "gbs": round(sb / (step_ms * 1e-3) / 1e9, 1),
                          "frac_hbm": round(sb / (step_ms * 1e-3) / 1e9 / hbm_peak, 4),
                          "apply_ms": rec["apply_ms"], "frac_hbm_apply": rec["frac_hbm_apply"],
                          "seg_build_ms": rec["seg_build_ms"],
                          "tflops": round(sf / (step_ms * 1e-3) / 1e12, 2),
                          "frac_bf16": round(sf / (step_ms * 1e-3) / 1e12 / bf16_peak, 5)},
        "kernels": kernels,
        "gpu_launches": int(res["launches"]),
        "ms_per_step_eager": rec["ms_per_step_eager"],
        "ms_per_step_median": rec["ms_per_step_median"],
        "clocks": res["clocks"],
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if per_workload is not None:
        line["per_workload"] = per_workload
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def per_workload_summary(args, dev, hbm_peak, bf16_peak, headline):
    """Every configuration: device times and rooflines, and the oracle's
    single-thread and all-core rates (the headline's timings are reused)."""
    import torch
    out = {}
    h_name, h_res, with_cpu = headline
    only = [n for n in args.only.split(",") if n]
    for name in W.CONFIG_NAMES:
        if only and name not in only:
            continue
        wl = W.make_workload(name, seed=args.seed)
        if name == h_name and not args.max_seqs:
            res = h_res
        else:
            res, ctx = time_ours(wl, args.steps, args.warmup, dev, 0)
            del ctx
            torch.cuda.empty_cache()
        rec = workload_record(wl, res, hbm_peak, bf16_peak)
        rec["clocks"] = res["clocks"]
        if not args.no_fused:
            rec["fused_projection"] = fused_record(wl, time_fused(wl, args.steps, args.warmup, dev), bf16_peak,
                                                   hbm_peak)
        if with_cpu:
            rec["cpu_oracle"] = {"threads_1": cpu_oracle_rates(wl, 1, args.cpu_seconds_detail),
                                 "threads_all": cpu_oracle_rates(wl, 0, args.cpu_seconds_detail)}
        out[name] = rec
    for name in W.MOE_CONFIG_NAMES:
        if only and name not in only:
            continue
        # MoE expert LoRA (not one of the five reference configurations)
        wl = W.make_moe_workload(name, seed=args.seed)
        res, ctx = time_ours(wl, args.steps, args.warmup, dev, 0)
        del ctx
        torch.cuda.empty_cache()
        b, f = moe_units(wl)
        sm, am = res["step_ms"], res["apply_ms"]
        out[name] = {"dispatched_rows": wl.R, "tokens": wl.T, "experts": wl.num_experts, "top_k": wl.top_k,
                     "adapters": wl.num_adapters,
                     "projections": [{"name": p.name, "d_in": p.d_in, "lanes": p.lane_d_out} for p in wl.projections],
                     "ms_per_step": round(sm, 5), "apply_ms": round(am, 5), "seg_build_ms": round(res["seg_ms"], 5),
                     "rows_per_s": round(wl.R / (sm * 1e-3), 1), "alg_bytes": int(b), "flops": int(f),
                     "frac_hbm_step": round(b / (sm * 1e-3) / 1e9 / hbm_peak, 4),
                     "frac_hbm_apply": round(b / (am * 1e-3) / 1e9 / hbm_peak, 4),
                     "stage_ms": [{k: round(v, 5) for k, v in st.items()} for st in res["stage_ms"]],
                     "clocks": res["clocks"], "note": "expert LoRA on dispatched rows (MoE layer); not one of the "
                                                      "five reference configurations"}
    return out


# ------------------------------------------------------ reference arm

def run_reference(args):
    """The CPU oracle, as it is, on the host cores; rank 0 only."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    wl = W.make_workload(args.workload, seed=args.seed, draw_xy=True)
    per_step_s = max(0.5, min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_oracle_rates(wl, 0, per_step_s * 0.5, runs=1)
    rates, secs, last = [], [], None
    for st in range(args.steps):
        last = cpu_oracle_rates(wl, 0, per_step_s, runs=1, seed=st)
        rates.append(last["tokens_per_s"])
        secs.append(last["step_s"])
    value = statistics.mean(rates)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * wl.T / value, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded PCG64; random-init adapters)",
        "config": workload_config(wl, ws),
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": last["threads"], "kind": "oracle",
                         "sample": f"each step: {last['sample']}"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="cont_batch", choices=W.CONFIG_NAMES)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=3.0,
                    help="oracle delta-phase time per run for the headline cpu_baseline (and the reference arm)")
    ap.add_argument("--cpu-seconds-detail", type=float, default=0.5,
                    help="oracle delta-phase time per run for each configuration's 1-thread / all-core rates")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--headline-only", action="store_true", help="skip the per_workload records of all configs")
    ap.add_argument("--no-fused", action="store_true", help="skip the fused-projection records")
    ap.add_argument("--fused-only", action="store_true",
                    help="time only the fused projection of --workload (one diagnostic JSON line)")
    ap.add_argument("--only", default="", help="per_workload: only these comma-separated configurations")
    ap.add_argument("--max-seqs", type=int, default=0,
                    help="keep only the first N sequences of the workload (smaller case for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.fused_only:
        run_fused_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
