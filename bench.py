#!/usr/bin/env python
"""Benchmark: fwd+bwd tokens/s of chunkwise gated linear attention on one GB300.

One step = the whole path on one batch of the workload: forward_prepare,
compose_prefix, forward_apply, backward_prepare, compose_suffix,
backward_apply (forward only for forward-only workloads), all through the
C ABI on the current stream, inputs resident in HBM.  The forward is also
timed as the one-launch rm_cp_forward_fused (fwd_path_roofline.fused_us).

Prints ONE JSON line (rank 0).  Besides the step throughput it reports:
  roofline      the dominant kernel's algorithmic bytes per launch over its
                CUDA-event launch time, against the measured HBM copy peak;
  path_roofline the whole step against max(flops / bf16 peak, bytes / HBM peak);
  e2e           the same metric with pinned host buffers copied in and out
                inside every timed step;
  cpu_baseline  the fp64 CPU oracle timed on a bounded sample of the workload;
  clocks        nvidia-smi samples taken during the timed region.

--impl reference times the fp64 CPU oracle itself as the reference arm.
Multi-GPU (torchrun): independent replicas, one per GPU, weak scaling.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from state_summary_scan_gb300.workloads import (GDR_WORKLOADS, SSD_WORKLOADS, WORKLOADS,  # noqa: E402
                                                 make_gdr_inputs, make_inputs, make_ssd_inputs)

METRIC = "fwd+bwd tokens/sec on 1 GB300; % of bf16 tensor/HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 2 ** 20
PHASES_FWD = ("forward_prepare", "compose_prefix", "forward_apply")
PHASES_FUSED = ("forward_fused",)  # rm_cp_forward_fused: the same forward in one launch
PHASES_BWD = ("backward_prepare", "compose_suffix", "backward_apply")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ accounting

def kernel_bytes(w, phase):
    """Algorithmic bytes of one launch: each input read once, each output
    written once (tokens: [B,T,H] rows; summaries: [nseg,B,H] states).  With
    vector gates the gate, its gradient, M and the per-token workspace value
    carry one fp32 per key dimension (f bytes)."""
    e = 4 if w.dtype == "f32" else 2
    ntok = w.B * w.T * w.H
    nsum = w.num_segments * w.B * w.H
    st = 4 * w.Dk * w.Dv
    Dk, Dv = w.Dk, w.Dv
    f = 4 * (Dk if getattr(w, "vector_gates", False) else 1)
    if phase == "forward_prepare":
        return ntok * (e * (Dk + Dv) + f) + nsum * (st + f)
    if phase == "compose_prefix":
        return nsum * (2 * st + f)
    if phase == "forward_apply":
        return ntok * (e * (2 * Dk + Dv) + f + e * Dv) + nsum * st
    if phase == "backward_prepare":
        return ntok * (e * (2 * Dk + 2 * Dv) + f + e * Dk + f) + nsum * 2 * st
    if phase == "compose_suffix":
        return nsum * (2 * st + f)
    if phase == "backward_apply":
        return ntok * (e * (2 * Dk + 2 * Dv) + f + f + e * (Dk + Dv) + f) + nsum * 2 * st
    if phase == "forward_fused":  # the three forward calls' inputs and outputs
        return sum(kernel_bytes(w, ph) for ph in PHASES_FWD)
    raise KeyError(phase)


# fp32 FMA throughput of the CUDA cores: 152 SMs x 128 FP32 lanes x 2 flops x
# 2070 MHz (the generic kernels walk tokens one by one in fp32 and are bound by it)
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12


def kernel_alu_flops(w, phase):
    """fp32 flops one launch of the generic token-walking kernels performs
    (multiply-add = 2): the state update k v^T and the readouts, per token and
    head, as the kernels run them."""
    ntok = w.B * w.T * w.H
    kd = w.Dk * w.Dv
    per = {"forward_prepare": 2 * kd, "forward_apply": 4 * kd, "backward_prepare": 6 * kd,
           "backward_apply": 6 * kd, "compose_prefix": 0, "compose_suffix": 0,
           "forward_fused": 6 * kd}[phase]
    return ntok * per


def path_roofline(w, peaks):
    """Roofline of one step of the method (chunk C): algorithmic flops and
    bytes per token and head, plus summary traffic per segment, row and head."""
    e = 4 if w.dtype == "f32" else 2
    C, Dk, Dv = w.chunk, w.Dk, w.Dv
    ntok = w.B * w.T * w.H
    nsum = w.num_segments * w.B * w.H
    f = 4 * (Dk if getattr(w, "vector_gates", False) else 1)  # gate (and dg) bytes per token-head
    flops = ntok * (C * (Dk + Dv) + 4 * Dk * Dv)
    byts = ntok * (e * (2 * Dk + Dv) + f + e * Dv) + nsum * (16 * Dk * Dv + 2 * f)
    if w.backward:
        flops += ntok * (C * (3 * Dk + 2 * Dv) + 8 * Dk * Dv)
        byts += ntok * (2 * e * (2 * Dk + Dv) + e * Dv + 2 * f) + nsum * (16 * Dk * Dv + 2 * f)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = byts / (peaks["hbm_gbs"] * 1e9)
    return dict(flops=flops, bytes=byts, t_tc_us=t_tc * 1e6, t_hbm_us=t_hbm * 1e6,
                bound="hbm" if t_hbm >= t_tc else "tensor", t_roofline_us=max(t_tc, t_hbm) * 1e6)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ CPU oracle

def oracle_sample_run(w, inp, ntok, threads=0):
    """fp64 oracle fwd (+bwd) on the first ntok tokens of every row and head."""
    import oracle
    cores = oracle.set_threads(threads)
    sl = slice(0, ntok)
    q, k, v, g = inp.q[:, sl], inp.k[:, sl], inp.v[:, sl], inp.g[:, sl]
    si = None
    if inp.cu_seqlens is not None:
        md = oracle.packed_metadata(inp.cu_seqlens, w.T, oracle.equal_segments(w.T, w.num_segments))
        si = md["seq_idx"][:ntok]
    args = [oracle._f64(x) for x in (q, k, v, g)]
    dO = oracle._f64(inp.dO[:, sl]) if w.backward else None
    fwd, bwd = ((oracle.vg_forward, oracle.vg_backward) if getattr(w, "vector_gates", False)
                else (oracle.forward, oracle.backward))
    t0 = time.perf_counter()
    fwd(*args, w.scale, si)
    if w.backward:
        bwd(*args, dO, w.scale, si)
    return time.perf_counter() - t0, cores


def calibrate_oracle(w, inp, target_s):
    """Number of tokens (per row) whose oracle run takes about target_s."""
    ntok = 64
    dt, _ = oracle_sample_run(w, inp, ntok)
    per_tok = max(dt / ntok, 1e-9)
    n = int(target_s / per_tok)
    return max(64, min(w.T, n - n % 64))


def cpu_baseline(w, inp, target_s=12.0):
    ntok = calibrate_oracle(w, inp, target_s)
    dt, cores = oracle_sample_run(w, inp, ntok)
    value = w.B * ntok / dt
    return {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 oracle {'fwd+bwd' if w.backward else 'fwd'} on the first {ntok} of "
                      f"{w.T} tokens of all {w.B} rows x {w.H} heads, {dt:.1f} s wall",
            "seconds": dt}


def workload_of(args):
    """The chosen workload; --T keeps its segment length and shrinks T (a
    smaller case of the same kernels for profiling captures, named as such)."""
    w = WORKLOADS[args.workload]
    if args.T:
        if args.T % w.seg_len or w.packed:
            raise SystemExit(f"--T must be a multiple of {w.seg_len} (and the workload not packed)")
        w = w.replace(T=args.T, num_segments=args.T // w.seg_len, name=f"{w.name}-T{args.T}")
    return w


# ------------------------------------------------------------------ replicas

def replica_time(ms_local: float, world: int, device) -> float:
    """Max over ranks of a per-rank time (the slowest replica sets the step);
    a no-op on one process.  Uses whatever backend the process group has
    (NCCL with a CUDA device, gloo with the CPU)."""
    if world <= 1:
        return float(ms_local)
    t = torch.tensor([float(ms_local)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, tokens_per_step: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every replica processes tokens_per_step per step."""
    return world * tokens_per_step / (ms_per_step / 1e3)


# ------------------------------------------------------------------ GPU arm

# The headline is the largest single-GPU configuration (256k, fwd+bwd); the
# other configurations of the metric are measured in the same run and
# reported under "workloads".
HEADLINE = "256k"
SUB_WORKLOADS = ("32k", "packed64k", "fwd4k", "vg32k")


def measure_workload(w, args, rank, world, dev, peaks, peak_src, with_e2e, with_cpu):
    """Times one workload: `steps` whole steps (fwd+bwd, or fwd for forward-only
    workloads) with per-phase CUDA events, then `steps` forward-only steps.
    Returns the workload's fields of the JSON line."""
    from state_summary_scan_gb300 import _capi as C
    from state_summary_scan_gb300 import api

    inp = make_inputs(w)
    q, k, v, g = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.g))
    dO = inp.dO.to(dev) if w.backward else None
    plan = api.make_plan(w.B, w.T, w.H, w.Dk, w.Dv, w.num_segments, w.chunk, w.scale,
                         q.dtype, inp.cu_seqlens, dev, w.backward, vector_gates=w.vector_gates)
    o = torch.empty_like(v)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dg = torch.empty_like(g)
    s = plan.spec
    stream = torch.cuda.current_stream(dev)
    phases = PHASES_FWD + (PHASES_BWD if w.backward else ())
    fns = {
        "forward_fused": lambda: C.rm_cp_forward_fused(s, q, k, v, g, plan.M, plan.dS, plan.S_in, o,
                                                       plan.ws, stream),
        "forward_prepare": lambda: C.rm_cp_forward_prepare(s, k, v, g, plan.M, plan.dS, plan.ws, stream),
        "compose_prefix": lambda: C.rm_cp_compose_prefix(s, plan.M, plan.dS, plan.S_in, stream),
        "forward_apply": lambda: C.rm_cp_forward_apply(s, q, k, v, g, plan.S_in, o, plan.ws, stream),
        "backward_prepare": lambda: C.rm_cp_backward_prepare(s, q, k, v, g, plan.S_in, dO, plan.gamma,
                                                             dq, plan.ws, stream),
        "compose_suffix": lambda: C.rm_cp_compose_suffix(s, plan.M, plan.gamma, plan.dS_out, stream),
        "backward_apply": lambda: C.rm_cp_backward_apply(s, q, k, v, g, dO, plan.S_in, plan.dS_out,
                                                         dk, dv, dg, plan.ws, stream),
    }

    def step(events=None, which=phases):
        for i, ph in enumerate(which):
            if events is not None:
                events[i].record(stream)
            fns[ph]()
        if events is not None:
            events[len(which)].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local_rank_of(dev))
    clocks.start()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(phases) + 1)]
          for _ in range(args.steps)]
    l0 = C.rm_cp_launch_count()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(ev[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    launches = C.rm_cp_launch_count() - l0
    # forward-only steps, timed the same way: the three calls, and the same
    # forward as the one-launch rm_cp_forward_fused for comparison
    fstart = torch.cuda.Event(enable_timing=True)
    fend = torch.cuda.Event(enable_timing=True)
    fstart.record(stream)
    for i in range(args.steps):
        step(None, PHASES_FWD)
    fend.record(stream)
    f3start = torch.cuda.Event(enable_timing=True)
    f3end = torch.cuda.Event(enable_timing=True)
    f3start.record(stream)
    for i in range(args.steps):
        step(None, PHASES_FUSED)
    f3end.record(stream)
    # the same step and forward captured once as CUDA graphs (api.StepGraph)
    # and replayed: one graph launch a step instead of one launch a call
    g_step = api.StepGraph(plan, q, k, v, g, dO) if w.backward else None
    g_fwd = api.StepGraph(plan, q, k, v, g)
    gtimes = {}
    for name, gr in (("step", g_step), ("fwd", g_fwd)):
        if gr is None:
            continue
        for _ in range(3):
            gr.replay()
        a_ev = torch.cuda.Event(enable_timing=True)
        b_ev = torch.cuda.Event(enable_timing=True)
        a_ev.record(stream)
        for _ in range(args.steps):
            gr.replay()
        b_ev.record(stream)
        gtimes[name] = (a_ev, b_ev)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms_per_step = replica_time(start.elapsed_time(end), world, dev) / args.steps
    fwd_ms = replica_time(fstart.elapsed_time(fend), world, dev) / args.steps
    fwd3_ms = replica_time(f3start.elapsed_time(f3end), world, dev) / args.steps
    g_fwd_ms = replica_time(gtimes["fwd"][0].elapsed_time(gtimes["fwd"][1]), world, dev) / args.steps
    g_ms = (replica_time(gtimes["step"][0].elapsed_time(gtimes["step"][1]), world, dev) / args.steps
            if "step" in gtimes else g_fwd_ms)
    del g_step, g_fwd
    tok_per_step = w.B * w.T
    value = replica_throughput(world, tok_per_step, ms_per_step)
    fwd_value = replica_throughput(world, tok_per_step, fwd_ms)

    phase_ms = {ph: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps))
                for j, ph in enumerate(phases)}
    dom = max(phase_ms, key=phase_ms.get)
    dom_bytes = kernel_bytes(w, dom)
    achieved = dom_bytes / (phase_ms[dom] / 1e3) / 1e9
    roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
            "traffic": load_traffic(w.name, dom), "algorithmic_bytes": dom_bytes,
            "launch_us": phase_ms[dom] * 1e3, "peak_source": peak_src}
    if w.vector_gates and C.rm_cp_path(s) != 1:
        # the generic kernels walk tokens one by one in fp32: bound by the CUDA cores
        fl = kernel_alu_flops(w, dom)
        ach = fl / (phase_ms[dom] / 1e3) / 1e12
        roof = {"bound": "alu", "kernel": dom, "achieved": ach, "peak": FP32_ALU_TFLOPS,
                "unit": "TFLOP/s", "frac": ach / FP32_ALU_TFLOPS,
                "traffic": load_traffic(w.name, dom), "alu_flops": fl,
                "algorithmic_bytes": dom_bytes, "launch_us": phase_ms[dom] * 1e3,
                "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 flop x 2070 MHz"}
    pr = path_roofline(w, peaks)
    path = {"bound": pr["bound"], "t_roofline_us": pr["t_roofline_us"],
            "t_measured_us": ms_per_step * 1e3, "frac": pr["t_roofline_us"] / (ms_per_step * 1e3),
            "flops": pr["flops"], "bytes": pr["bytes"], "peak_source": peak_src,
            "phases_us": {ph: round(t * 1e3, 2) for ph, t in phase_ms.items()},
            "phase_frac_of_hbm": {ph: round(kernel_bytes(w, ph) / (phase_ms[ph] / 1e3) / 1e9
                                            / peaks["hbm_gbs"], 4) for ph in phases}}
    fpr = path_roofline(w.replace(backward=False), peaks)
    fwd_path = {"bound": fpr["bound"], "t_roofline_us": fpr["t_roofline_us"],
                "t_measured_us": fwd_ms * 1e3, "frac": fpr["t_roofline_us"] / (fwd_ms * 1e3),
                "calls": "forward_prepare, compose_prefix, forward_apply",
                "fused_us": fwd3_ms * 1e3,
                "fused_frac": fpr["t_roofline_us"] / (fwd3_ms * 1e3)}

    # ---- end to end through rm_cp_step_host: pinned host buffers in, results
    # out, every step.  Two device buffer sets and two copy streams: the
    # host->device copy of step i+1 and the device->host copy of step i-1 run
    # while step i's kernels do, as a training loop that prefetches its next
    # batch would; every step's copies are inside the timed region.
    e2e = None
    if with_e2e:
        names_in = ("q", "k", "v", "g") + (("dO",) if w.backward else ())
        host = {n: getattr(inp, n).pin_memory() for n in names_in}
        outs0 = {"o": o}
        if w.backward:
            outs0.update(dq=dq, dk=dk, dv=dv, dg=dg)
        host.update({n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in outs0.items()})
        pipe = api.HostPipeline(plan, host, dev)

        def e2e_run(n):
            pipe.begin(stream)
            for _ in range(n):
                pipe.step(stream)
            pipe.join(stream)

        e2e_run(max(2, min(args.warmup, 3)))
        torch.cuda.synchronize(dev)
        n_e2e = max(3, min(args.steps // 2, 30))
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_run(n_e2e)
        b.record(stream)
        torch.cuda.synchronize(dev)
        pipe.close()
        e_ms = replica_time(a.elapsed_time(b) / n_e2e, world, dev)
        e2e = {"value": replica_throughput(world, tok_per_step, e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": sum(host[n].numel() * host[n].element_size() for n in names_in),
               "d2h_bytes_per_step": sum(host[n].numel() * host[n].element_size() for n in outs0),
               "ms_per_step": e_ms, "steps": n_e2e, "call": "rm_cp_step_host",
               "pipeline": "2 device buffer sets; h2d of step i+1 and d2h of step i-1 overlap step i"}
        del host, pipe

    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, g) + ((dO,) if dO is not None else ()))
    cpu = cpu_baseline(w, inp, args.cpu_seconds) if with_cpu else None
    path_kind = C.rm_cp_path(s)
    out = {
        "value": value, "fwd_value": fwd_value, "unit": "tokens/s", "ms_per_step": ms_per_step,
        "fwd_ms_per_step": fwd_ms, "mode": "fwd+bwd" if w.backward else "fwd",
        "dtype": "bf16" if (w.dtype == "bf16" and path_kind == 1) else "f32",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "Dk": w.Dk, "Dv": w.Dv,
                   "num_segments": w.num_segments, "chunk": w.chunk, "storage": w.dtype,
                   "mode": "fwd+bwd" if w.backward else "fwd", "packed": w.packed,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": (f"inputs larger than L2 ({in_bytes / 2**20:.0f} MiB > 129 MiB), no flush"
                          if in_bytes > L2_BYTES else
                          f"inputs ({in_bytes / 2**20:.0f} MiB) fit in L2: no flush, warm-L2 figure"),
                   "kernel_path": "tcgen05" if path_kind == 1 else "simt-fp32",
                   "gates": "per key dimension" if w.vector_gates else "per head"},
        "roofline": roof, "path_roofline": path, "fwd_path_roofline": fwd_path,
        "graph": {"value": replica_throughput(world, tok_per_step, g_ms), "ms_per_step": g_ms,
                  "fwd_value": replica_throughput(world, tok_per_step, g_fwd_ms), "fwd_ms_per_step": g_fwd_ms,
                  "frac": path["t_roofline_us"] / (g_ms * 1e3),
                  "how": "the same calls captured once as a CUDA graph (api.StepGraph) and replayed"},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches), "clocks": clk,
    }
    del q, k, v, g, dO, o, dq, dk, dv, dg, plan, inp
    torch.cuda.empty_cache()
    return out


def local_rank_of(dev) -> int:
    return dev.index if dev.index is not None else 0


def run_ours(args, rank, world, local_rank):
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks, peak_src = load_peaks()
    w = workload_of(args)
    head = measure_workload(w, args, rank, world, dev, peaks, peak_src,
                            with_e2e=not args.no_e2e,
                            with_cpu=rank == 0 and world == 1 and not args.no_cpu_baseline)
    line = {
        "metric": METRIC, "value": head["value"], "fwd_value": head["fwd_value"], "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"], "fwd_ms_per_step": head["fwd_ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
        "data": "synthetic (seeded: q,k,v,dO ~ N(0,1), k L2-normalised, g = logsigmoid(N(0,1)+c))",
    }
    for key in ("config", "roofline", "path_roofline", "fwd_path_roofline", "graph", "cpu_baseline",
                "e2e", "gpu_launches", "clocks"):
        line[key] = head[key]
    if args.workload == HEADLINE and not args.T and not args.headline_only:
        subs = {}
        for name in SUB_WORKLOADS + tuple(GDR_WORKLOADS):
            if name in GDR_WORKLOADS:
                r = measure_gdr(GDR_WORKLOADS[name], args, rank, world, dev, peaks, peak_src, False)
            else:
                r = measure_workload(WORKLOADS[name], args, rank, world, dev, peaks, peak_src,
                                     with_e2e=False, with_cpu=False)
            subs[name] = {key: r[key] for key in ("value", "fwd_value", "unit", "mode", "ms_per_step",
                                                 "fwd_ms_per_step", "dtype", "config", "roofline",
                                                 "path_roofline", "fwd_path_roofline", "graph", "e2e",
                                                 "gpu_launches", "clocks") if key in r}
        line["workloads"] = subs
        line["gpu_launches"] = head["gpu_launches"]
    return line


# ------------------------------------------------------------------ Mamba2 SSD

SSD_PHASES = ("ssd_map_inputs",) + PHASES_FWD + ("ssd_finish_forward",) + PHASES_BWD + (
    "ssd_finish_backward",)


def ssd_core_workload(w):
    """The gated-recurrence problem the SSD scan runs as (Dk = N, Dv = P)."""
    from state_summary_scan_gb300.workloads import Workload
    return Workload(w.name, B=w.B, T=w.T, H=w.H, Dk=w.N, Dv=w.P, dtype=w.dtype,
                    num_segments=w.num_segments, chunk=w.chunk, gate_shift=0.0)


def ssd_kernel_bytes(w, phase):
    """Algorithmic bytes of one launch (each input read once, each output
    written once); the six path calls as for the gated recurrence."""
    e = 4 if w.dtype == "f32" else 2
    ntok = w.B * w.T * w.H
    shared = 2 * e * w.N * w.B * w.T * w.G  # B and C, once per group
    if phase == "ssd_map_inputs":
        return ntok * (4 + e * w.N + 4) + shared // 2 + 4 * w.H
    if phase == "ssd_finish_forward":
        return ntok * 3 * e * w.P + 4 * w.H
    if phase == "ssd_finish_backward":
        return (ntok * (2 * e * w.N + 8 + 4 + 4 * e * w.P + 4 + 12) + e * w.N * w.B * w.T * w.G
                + 2 * e * w.N * w.B * w.T * w.G + 12 * w.H)
    return kernel_bytes(ssd_core_workload(w), phase)


def ssd_path_roofline(w, peaks):
    """The SSD scan's own step: read x, dt, B, C (B and C once per group), write
    y; backward also reads dy and writes dx, ddt, dB, dC; the summary traffic
    and the flops are those of the recurrence it runs as."""
    e = 4 if w.dtype == "f32" else 2
    core = path_roofline(ssd_core_workload(w), peaks)
    ntok = w.B * w.T * w.H
    nsum = w.num_segments * w.B * w.H
    bc = w.B * w.T * w.G * e * w.N
    byts = (ntok * (2 * e * w.P + 4) + 2 * bc + nsum * (16 * w.N * w.P + 8)
            + ntok * (3 * e * w.P + 8) + 4 * bc + nsum * (16 * w.N * w.P + 8))
    flops = core["flops"]
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = byts / (peaks["hbm_gbs"] * 1e9)
    return dict(flops=flops, bytes=byts, bound="hbm" if t_hbm >= t_tc else "tensor",
                t_roofline_us=max(t_tc, t_hbm) * 1e6)


def ssd_cpu_baseline(w, inp, target_s=12.0):
    import oracle
    cores = oracle.set_threads(0)

    def run(n):
        sl = slice(0, n)
        t0 = time.perf_counter()
        oracle.ssd_forward(inp.x[:, sl], inp.dt[:, sl], inp.A, inp.Bm[:, sl], inp.Cm[:, sl], inp.D)
        oracle.ssd_backward(inp.x[:, sl], inp.dt[:, sl], inp.A, inp.Bm[:, sl], inp.Cm[:, sl],
                            inp.dy[:, sl], inp.D)
        return time.perf_counter() - t0

    per_tok = max(run(64) / 64, 1e-9)
    n = max(64, min(w.T, int(target_s / per_tok) // 64 * 64))
    dt = run(n)
    return {"value": w.B * n / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 SSD oracle fwd+bwd on the first {n} of {w.T} tokens of all {w.B} rows x "
                      f"{w.H} heads, {dt:.1f} s wall", "seconds": dt}


def run_ssd(args, rank, world, local_rank):
    from state_summary_scan_gb300 import _capi as C
    from state_summary_scan_gb300 import api

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = SSD_WORKLOADS[args.workload]
    peaks, peak_src = load_peaks()
    inp = make_ssd_inputs(w)
    x, dt, A, Bm, Cm, D, dy = (t.to(dev) for t in (inp.x, inp.dt, inp.A, inp.Bm, inp.Cm, inp.D, inp.dy))
    sp = api.make_ssd_plan(w.B, w.T, w.H, w.G, w.N, w.P, w.num_segments, w.chunk, w.torch_dtype,
                           device=dev)
    plan, s = sp.core, sp.core.spec
    y = torch.empty_like(x)
    dq, dk, dv = torch.empty_like(sp.k), torch.empty_like(sp.k), torch.empty_like(x)
    dg = torch.empty_like(sp.g)
    ddt = torch.empty_like(dt)
    dA = torch.empty_like(A)
    dD = torch.empty_like(D)
    dB, dC = torch.empty_like(Bm), torch.empty_like(Cm)
    stream = torch.cuda.current_stream(dev)
    fns = {
        "ssd_map_inputs": lambda: C.rm_ssd_map_inputs(s, w.G, dt, A, Bm, None, None, sp.k, sp.g, stream),
        "forward_fused": lambda: C.rm_cp_forward_fused(s, Cm, sp.k, x, sp.g, plan.M, plan.dS, plan.S_in, y,
                                                       plan.ws, stream),
        "forward_prepare": lambda: C.rm_cp_forward_prepare(s, sp.k, x, sp.g, plan.M, plan.dS, plan.ws, stream),
        "compose_prefix": lambda: C.rm_cp_compose_prefix(s, plan.M, plan.dS, plan.S_in, stream),
        "forward_apply": lambda: C.rm_cp_forward_apply(s, Cm, sp.k, x, sp.g, plan.S_in, y, plan.ws, stream),
        "ssd_finish_forward": lambda: C.rm_ssd_finish_forward(s, x, D, y, stream),
        "backward_prepare": lambda: C.rm_cp_backward_prepare(s, Cm, sp.k, x, sp.g, plan.S_in, dy,
                                                             plan.gamma, dq, plan.ws, stream),
        "compose_suffix": lambda: C.rm_cp_compose_suffix(s, plan.M, plan.gamma, plan.dS_out, stream),
        "backward_apply": lambda: C.rm_cp_backward_apply(s, Cm, sp.k, x, sp.g, dy, plan.S_in,
                                                         plan.dS_out, dk, dv, dg, plan.ws, stream),
        "ssd_finish_backward": lambda: C.rm_ssd_finish_backward(s, w.G, x, dt, A, Bm, dy, D, dq, dk, dv,
                                                                dg, ddt, dA, dB, dC, dD, sp.ws, stream),
    }

    def step(events=None):
        for i, ph in enumerate(SSD_PHASES):
            if events is not None:
                events[i].record(stream)
            fns[ph]()
        if events is not None:
            events[len(SSD_PHASES)].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local_rank)
    clocks.start()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(SSD_PHASES) + 1)]
          for _ in range(args.steps)]
    l0 = C.rm_cp_launch_count()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(ev[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    launches = C.rm_cp_launch_count() - l0
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms_per_step = replica_time(start.elapsed_time(end), world, dev) / args.steps
    tok_per_step = w.B * w.T
    value = replica_throughput(world, tok_per_step, ms_per_step)
    phase_ms = {ph: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps))
                for j, ph in enumerate(SSD_PHASES)}
    dom = max(phase_ms, key=phase_ms.get)
    dom_bytes = ssd_kernel_bytes(w, dom)
    achieved = dom_bytes / (phase_ms[dom] / 1e3) / 1e9
    roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": load_traffic(w.name, dom),
            "algorithmic_bytes": dom_bytes, "launch_us": phase_ms[dom] * 1e3, "peak_source": peak_src}
    pr = ssd_path_roofline(w, peaks)
    path = {"bound": pr["bound"], "t_roofline_us": pr["t_roofline_us"], "t_measured_us": ms_per_step * 1e3,
            "frac": pr["t_roofline_us"] / (ms_per_step * 1e3), "flops": pr["flops"], "bytes": pr["bytes"],
            "peak_source": peak_src, "phases_us": {ph: round(t * 1e3, 2) for ph, t in phase_ms.items()},
            "phase_frac_of_hbm": {ph: round(ssd_kernel_bytes(w, ph) / (phase_ms[ph] / 1e3) / 1e9
                                            / peaks["hbm_gbs"], 4) for ph in SSD_PHASES}}
    e2e = None
    if not args.no_e2e:
        e2e = host_e2e(stream, dev, dict(x=x, dt=dt, A=A, B=Bm, C=Cm, D=D, dy=dy),
                       dict(y=y, dx=dv, ddt=ddt, dA=dA, dB=dB, dC=dC, dD=dD), step,
                       max(3, min(args.steps // 2, 20)), tok_per_step, world,
                       "rm_ssd_map_inputs, the six calls and the two finish calls (bench.run_ssd's step)")
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = ssd_cpu_baseline(w, inp, args.cpu_seconds)
    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded Mamba2 SSD inputs)",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "G": w.G, "N": w.N, "P": w.P,
                   "num_segments": w.num_segments, "chunk": w.chunk, "mode": "fwd+bwd",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2, no flush", "kernel_path": "tcgen05"},
        "roofline": roof, "path_roofline": path, "cpu_baseline": cpu,
        "e2e": e2e, "gpu_launches": int(launches), "clocks": clk,
    }


def reference_budget(args) -> float:
    """Seconds of oracle work per reference step: the whole --steps/--warmup
    run stays near two and a half minutes of CPU time (at least 50 ms, the
    smallest sample being 64 tokens of every row and head)."""
    return max(0.05, min(8.0, 150.0 / max(1, args.steps + args.warmup)))


# ------------------------------------------------------------------ gated delta rule

GDR_PHASES_FWD = ("gdr_forward_prepare", "gdr_compose_prefix", "gdr_forward_apply")
GDR_PHASES_BWD = ("gdr_backward_prepare", "gdr_compose_suffix", "gdr_backward_apply")


def gdr_kernel_alu_flops(w, phase):
    """fp32 flops one launch of the generic gated-delta-rule kernels performs,
    per token and head as the kernels run them (multiply-add = 2): the state
    step is k^T S then the rank-one correction (about 6 Dk Dv), the prepare
    also walks M's Dk columns, the reverse sweep rebuilds the states S_{t-1} of
    each group of four tokens once from the state saved every 16 tokens (2.25
    steps a token) and forms its gradients (about 18 Dk Dv)."""
    ntok = w.B * w.T * w.H
    kd = w.Dk * w.Dv
    per = {"gdr_forward_prepare": 6 * w.Dk * (w.Dv + w.Dk), "gdr_forward_apply": 8 * kd,
           "gdr_backward_prepare": 16 * kd, "gdr_backward_apply": 32 * kd,
           "gdr_compose_prefix": 0, "gdr_compose_suffix": 0}[phase]
    return ntok * per


def gdr_kernel_bytes(w, phase):
    """Algorithmic bytes of one gated-delta-rule call on the tensor-core
    sweeps: its inputs read once and its outputs written once (token tensors,
    gates, summaries) plus its share of the workspace: the forward prepare
    writes each 64-token chunk's two bf16 [64][64] factors, the apply and
    the backward prepare read T, the backward apply reads both; the backward
    prepare writes, and the apply reads, one fp32 state per chunk."""
    e = 4 if w.dtype == "f32" else 2
    Dk, Dv = w.Dk, w.Dv
    ntok = w.B * w.T * w.H
    nsum = w.num_segments * w.B * w.H
    st, mt = 4 * Dk * Dv, 4 * Dk * Dk
    nch = ntok // 64
    ckpt = nch * st
    tf = nch * 64 * 64 * 2  # one bf16 factor tile a chunk
    return {
        "gdr_forward_prepare": ntok * (e * (Dk + Dv) + 8) + nsum * (mt + st) + 2 * tf,
        "gdr_compose_prefix": nsum * (mt + 2 * st),
        "gdr_forward_apply": ntok * (e * (2 * Dk + Dv) + 8 + e * Dv) + nsum * st + tf,
        "gdr_backward_prepare": ntok * (e * (2 * Dk + 2 * Dv) + 8 + e * Dk) + 2 * nsum * st + ckpt + tf,
        "gdr_compose_suffix": nsum * (mt + 2 * st),
        "gdr_backward_apply": ntok * (e * (2 * Dk + 2 * Dv) + 8 + e * (Dk + Dv) + 8) + nsum * st + ckpt + 2 * tf,
    }[phase]


def gdr_step_bytes(w, tc):
    """Device bytes one gated-delta-rule step touches: q, k, v, dO, g, beta;
    o, dq, dk, dv, dg, dbeta; M, delta_S, S_in, gamma, dS_out; the saved
    states (one every 64 tokens on the tensor cores, every 16 otherwise)."""
    e = 4 if w.dtype == "f32" else 2
    ntok = w.B * w.T * w.H
    nsum = w.num_segments * w.B * w.H
    qk = ntok * w.Dk * e
    vv = ntok * w.Dv * e
    return (2 * (2 * qk + 2 * vv) + 4 * ntok * 4 + nsum * (w.Dk * w.Dk + 4 * w.Dk * w.Dv) * 4
            + (ntok // (64 if tc else 16)) * w.Dk * w.Dv * 4)


def gdr_kernel_tc_flops(w, phase):
    """Tensor-core flops of one call on the tensor-core sweeps: 64 x 64 x 64
    products per 64-token chunk and head (K K^T and the walk's 6 in the
    forward prepare, 7 in the apply, 7 + 6 in the backward prepare's dq and
    gamma walks, 6 + 15 in the backward apply's adjoint walk and chunk pass)."""
    per = {"gdr_forward_prepare": 7, "gdr_forward_apply": 7, "gdr_backward_prepare": 13,
           "gdr_backward_apply": 21}.get(phase, 0)
    return (w.B * w.T * w.H // 64) * per * 2 * 64 ** 3


def gdr_path_roofline(w, peaks):
    """The method's step: read q, k, v, g, beta (and dO), write o (and dq, dk,
    dv, dg, dbeta); summaries M (Dk x Dk) and delta_S written, read by the
    fold, S_in written and read (both directions).  Flops: the chunkwise form
    of the scalar gate plus the per-chunk K K^T and triangular solve of the
    delta rule (2 C Dk a token each way)."""
    e = 4 if w.dtype == "f32" else 2
    C, Dk, Dv = w.chunk, w.Dk, w.Dv
    ntok = w.B * w.T * w.H
    nsum = w.num_segments * w.B * w.H
    summ = 16 * Dk * Dv + 8 * Dk * Dk
    byts = (ntok * (e * (2 * Dk + Dv) + 8 + e * Dv) + nsum * summ
            + ntok * (2 * e * (2 * Dk + Dv) + e * Dv + 16) + nsum * summ)
    flops = ntok * (C * (3 * Dk + Dv) + 4 * Dk * Dv) + ntok * (C * (5 * Dk + 2 * Dv) + 8 * Dk * Dv)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = byts / (peaks["hbm_gbs"] * 1e9)
    fwd_b = ntok * (e * (2 * Dk + Dv) + 8 + e * Dv) + nsum * summ
    return dict(flops=flops, bytes=byts, bound="hbm" if t_hbm >= t_tc else "tensor",
                t_roofline_us=max(t_tc, t_hbm) * 1e6, t_fwd_roofline_us=fwd_b / (peaks["hbm_gbs"] * 1e9) * 1e6)


def gdr_cpu_baseline(w, inp, target_s=12.0):
    import oracle
    cores = oracle.set_threads(0)

    def run(n):
        sl = slice(0, n)
        args = [oracle._f64(x[:, sl]) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta)]
        dO = oracle._f64(inp.dO[:, sl])
        t0 = time.perf_counter()
        oracle.gdr_forward(*args, w.scale)
        oracle.gdr_backward(*args, dO, w.scale)
        return time.perf_counter() - t0

    per_tok = max(run(64) / 64, 1e-9)
    n = max(64, min(w.T, int(target_s / per_tok) // 64 * 64))
    dt = run(n)
    return {"value": w.B * n / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 gated-delta-rule oracle fwd+bwd on the first {n} of {w.T} tokens of all "
                      f"{w.B} rows x {w.H} heads, {dt:.1f} s wall", "seconds": dt}


def measure_gdr(w, args, rank, world, dev, peaks, peak_src, with_cpu):
    from state_summary_scan_gb300 import _capi as C
    from state_summary_scan_gb300 import api

    inp = make_gdr_inputs(w)
    q, k, v, g, beta, dO = (t.to(dev) for t in (inp.q, inp.k, inp.v, inp.g, inp.beta, inp.dO))
    plan = api.make_gdr_plan(w.B, w.T, w.H, w.Dk, w.Dv, w.num_segments, w.chunk, w.scale,
                             w.torch_dtype, device=dev)
    s = plan.spec
    o = torch.empty_like(v)
    dq, dk, dv = torch.empty_like(k), torch.empty_like(k), torch.empty_like(v)
    dg, db = torch.empty_like(g), torch.empty_like(beta)
    stream = torch.cuda.current_stream(dev)
    fns = {
        "gdr_forward_prepare": lambda: C.rm_gdr_forward_prepare(s, k, v, g, beta, plan.M, plan.dS, plan.ws,
                                                                stream),
        "gdr_compose_prefix": lambda: C.rm_gdr_compose_prefix(s, plan.M, plan.dS, plan.S_in, stream),
        "gdr_forward_apply": lambda: C.rm_gdr_forward_apply(s, q, k, v, g, beta, plan.S_in, o, plan.ws, stream),
        "gdr_backward_prepare": lambda: C.rm_gdr_backward_prepare(s, q, k, v, g, beta, plan.S_in, dO,
                                                                  plan.gamma, dq, plan.ws, stream),
        "gdr_compose_suffix": lambda: C.rm_gdr_compose_suffix(s, plan.M, plan.gamma, plan.dS_out, stream),
        "gdr_backward_apply": lambda: C.rm_gdr_backward_apply(s, q, k, v, g, beta, dO, plan.dS_out, dk, dv,
                                                              dg, db, plan.ws, stream),
    }
    phases = GDR_PHASES_FWD + GDR_PHASES_BWD
    steps = max(3, min(args.steps, 50))  # about a millisecond a step (several on the generic kernels)
    for _ in range(args.warmup):
        for ph in phases:
            fns[ph]()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local_rank_of(dev))
    clocks.start()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(phases) + 1)] for _ in range(steps)]
    l0 = C.rm_cp_launch_count()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        for j, ph in enumerate(phases):
            ev[i][j].record(stream)
            fns[ph]()
        ev[i][len(phases)].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    launches = C.rm_cp_launch_count() - l0
    fs, fe = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fs.record(stream)
    for _ in range(steps):
        for ph in GDR_PHASES_FWD:
            fns[ph]()
    fe.record(stream)
    # the same step and forward captured once as CUDA graphs and replayed
    g_step = api.GdrStepGraph(plan, q, k, v, g, beta, dO)
    g_fwd = api.GdrStepGraph(plan, q, k, v, g, beta)
    gtimes = {}
    for name, gr in (("step", g_step), ("fwd", g_fwd)):
        for _ in range(3):
            gr.replay()
        a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_ev.record(stream)
        for _ in range(steps):
            gr.replay()
        b_ev.record(stream)
        gtimes[name] = (a_ev, b_ev)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms = replica_time(start.elapsed_time(end), world, dev) / steps
    fwd_ms = replica_time(fs.elapsed_time(fe), world, dev) / steps
    g_ms = replica_time(gtimes["step"][0].elapsed_time(gtimes["step"][1]), world, dev) / steps
    g_fwd_ms = replica_time(gtimes["fwd"][0].elapsed_time(gtimes["fwd"][1]), world, dev) / steps
    del g_step, g_fwd
    phase_ms = {ph: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps))
                for j, ph in enumerate(phases)}
    dom = max(phase_ms, key=phase_ms.get)
    e2e = None
    if not args.no_e2e:
        def gdr_step():
            for ph in phases:
                fns[ph]()
        e2e = host_e2e(stream, dev, dict(q=q, k=k, v=v, g=g, beta=beta, dO=dO),
                       dict(o=o, dq=dq, dk=dk, dv=dv, dg=dg, dbeta=db), gdr_step, steps, w.B * w.T, world,
                       "the six rm_gdr_* calls")
    tc = C.rm_gdr_path(s) == 1
    if tc:
        # the tensor-core sweeps: bytes bound them (their flops take less time at peak)
        kb, kf = gdr_kernel_bytes(w, dom), gdr_kernel_tc_flops(w, dom)
        ach = kb / (phase_ms[dom] / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "kernel_bytes": kb, "tensor_flops": kf,
                "tensor_frac": kf / (phase_ms[dom] / 1e3) / (peaks["bf16_tflops"] * 1e12),
                "launch_us": phase_ms[dom] * 1e3, "traffic": load_traffic(w.name, dom),
                "peak_source": peak_src}
    else:
        fl = gdr_kernel_alu_flops(w, dom)
        ach = fl / (phase_ms[dom] / 1e3) / 1e12
        roof = {"bound": "alu", "kernel": dom, "achieved": ach, "peak": FP32_ALU_TFLOPS,
                "unit": "TFLOP/s", "frac": ach / FP32_ALU_TFLOPS, "alu_flops": fl,
                "launch_us": phase_ms[dom] * 1e3, "traffic": load_traffic(w.name, dom),
                "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 flop x 2070 MHz"}
    pr = gdr_path_roofline(w, peaks)
    tok = w.B * w.T
    return {
        "value": replica_throughput(world, tok, ms), "fwd_value": replica_throughput(world, tok, fwd_ms),
        "unit": "tokens/s", "mode": "fwd+bwd", "ms_per_step": ms, "fwd_ms_per_step": fwd_ms,
        "dtype": "bf16" if tc else "f32",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "Dk": w.Dk, "Dv": w.Dv,
                   "num_segments": w.num_segments, "storage": w.dtype, "mode": "fwd+bwd",
                   "recurrence": "gated delta rule",
                   "kernel_path": "tcgen05 sweeps, fp32 folds" if tc else "simt-fp32", "steps": steps,
                   "l2": f"a step touches {gdr_step_bytes(w, tc) / 1e6:.0f} MB (inputs, outputs, summaries, saved "
                         f"states), more than the 129 MB L2; no flush"},
        "roofline": roof,
        "path_roofline": {"bound": pr["bound"], "t_roofline_us": pr["t_roofline_us"],
                          "t_measured_us": ms * 1e3, "frac": pr["t_roofline_us"] / (ms * 1e3),
                          "flops": pr["flops"], "bytes": pr["bytes"], "peak_source": peak_src,
                          "phases_us": {ph: round(t * 1e3, 2) for ph, t in phase_ms.items()}},
        "fwd_path_roofline": {"t_roofline_us": pr["t_fwd_roofline_us"], "t_measured_us": fwd_ms * 1e3,
                              "frac": pr["t_fwd_roofline_us"] / (fwd_ms * 1e3)},
        "graph": {"value": replica_throughput(world, tok, g_ms), "ms_per_step": g_ms,
                  "fwd_value": replica_throughput(world, tok, g_fwd_ms), "fwd_ms_per_step": g_fwd_ms,
                  "frac": pr["t_roofline_us"] / (g_ms * 1e3),
                  "how": "the same calls captured once as a CUDA graph (api.GdrStepGraph) and replayed"},
        "cpu_baseline": gdr_cpu_baseline(w, inp, args.cpu_seconds) if with_cpu else None,
        "e2e": e2e, "gpu_launches": int(launches), "clocks": clk,
    }


def run_gdr(args, rank, world, local_rank):
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks, peak_src = load_peaks()
    r = measure_gdr(GDR_WORKLOADS[args.workload], args, rank, world, dev, peaks, peak_src,
                    rank == 0 and world == 1 and not args.no_cpu_baseline)
    line = {"metric": METRIC, "n_gpus": world, "steps": r["config"]["steps"], "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "data": "synthetic (seeded gated-delta-rule inputs)"}
    line.update(r)
    return line


def run_reference(args):
    """The fp64 CPU oracle as the reference arm, timed per step on host cores."""
    if args.workload in GDR_WORKLOADS:
        w = GDR_WORKLOADS[args.workload]
        inp = make_gdr_inputs(w)
        budget = reference_budget(args)
        runs = [gdr_cpu_baseline(w, inp, budget) for _ in range(args.steps)]
        value = statistics.mean(r["value"] for r in runs)
        return {
            "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * w.B * w.T / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "Dk": w.Dk,
                                            "Dv": w.Dv, "num_segments": w.num_segments, "mode": "fwd+bwd",
                                            "recurrence": "gated delta rule"},
            "cpu_baseline": dict(runs[-1], value=value),
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0,
        }
    if args.workload in SSD_WORKLOADS:
        w = SSD_WORKLOADS[args.workload]
        inp = make_ssd_inputs(w)
        budget = reference_budget(args)
        runs = [ssd_cpu_baseline(w, inp, budget) for _ in range(args.steps)]
        value = statistics.mean(r["value"] for r in runs)
        return {
            "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * w.B * w.T / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "G": w.G,
                                            "N": w.N, "P": w.P, "num_segments": w.num_segments,
                                            "mode": "fwd+bwd"},
            "cpu_baseline": dict(runs[-1], value=value),
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0,
        }
    w = workload_of(args)
    inp = make_inputs(w)
    budget = reference_budget(args)
    ntok = calibrate_oracle(w, inp, budget)
    for _ in range(args.warmup):
        oracle_sample_run(w, inp, ntok)
    times = []
    cores = 1
    for _ in range(args.steps):
        dt, cores = oracle_sample_run(w, inp, ntok)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = w.B * ntok / (ms / 1e3)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "Dk": w.Dk, "Dv": w.Dv,
                   "num_segments": w.num_segments, "chunk": w.chunk,
                   "mode": "fwd+bwd" if w.backward else "fwd"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"fp64 oracle on the first {ntok} of {w.T} tokens of all "
                                   f"{w.B} rows x {w.H} heads per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def host_e2e(stream, dev, dev_in, dev_out, step_fn, steps, tok_per_step, world, call):
    """End to end through the calls with host buffers: every step copies its
    inputs from pinned host memory into the device buffers the calls read,
    runs the calls, and copies the outputs back into pinned host memory, all
    on one stream and inside the timed region (no overlap between steps)."""
    host_in = {n: t.detach().to("cpu").pin_memory() for n, t in dev_in.items()}
    host_out = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in dev_out.items()}

    def one():
        for n, t in dev_in.items():
            t.copy_(host_in[n], non_blocking=True)
        step_fn()
        for n, t in dev_out.items():
            host_out[n].copy_(t, non_blocking=True)

    for _ in range(2):
        one()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        one()
    b.record(stream)
    torch.cuda.synchronize(dev)
    e_ms = replica_time(a.elapsed_time(b) / steps, world, dev)
    return {"value": replica_throughput(world, tok_per_step, e_ms), "unit": "tokens/s",
            "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host_in.values()),
            "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in host_out.values()),
            "ms_per_step": e_ms, "steps": steps, "call": call,
            "pipeline": "one stream: h2d, the calls, d2h, step after step"}


def load_traffic(workload, kernel):
    """DRAM bytes per launch from a committed ncu capture, if one matches."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        table = json.load(f)
    entry = table.get(workload, {}).get(kernel)
    return None if entry is None else entry.get("bytes_per_launch")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE,
                    choices=sorted(WORKLOADS) + sorted(SSD_WORKLOADS) + sorted(GDR_WORKLOADS))
    ap.add_argument("--headline-only", action="store_true",
                    help="time only the chosen workload (no 'workloads' object)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--T", type=int, default=0,
                    help="shorter T with the same segment length (profiling captures of a smaller case)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if (args.workload in SSD_WORKLOADS or args.workload in GDR_WORKLOADS) and args.T:
        ap.error("--T applies to the gated-recurrence workloads only")

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run = (run_ssd if args.workload in SSD_WORKLOADS
               else run_gdr if args.workload in GDR_WORKLOADS else run_ours)
        line = run(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
