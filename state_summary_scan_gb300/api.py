"""PyTorch-facing entry points: buffer allocation and the call sequence.

The work is the six C-ABI calls, issued in the order of the Megatron-Core
page "core.ssm.context_parallel.chunkwise" (chunkwise_cp_forward:
prepare -> prefix -> apply; chunkwise_cp_backward: prepare -> suffix ->
apply).  PyTorch only provides device memory and the stream.
"""
from __future__ import annotations

import collections
import dataclasses
import math
import threading
from typing import Optional

import torch

from . import _capi as C


@dataclasses.dataclass
class Plan:
    """Problem description plus every intermediate buffer of one step."""
    spec: C.ProblemSpec
    M: torch.Tensor          # [nseg,B,H] fp32
    dS: Optional[torch.Tensor]  # [nseg,B,H,Dk,Dv] fp32 (forward summaries)
    S_in: torch.Tensor       # [nseg,B,H,Dk,Dv] fp32
    gamma: torch.Tensor      # [nseg,B,H,Dk,Dv] fp32 (backward summaries)
    dS_out: torch.Tensor     # [nseg,B,H,Dk,Dv] fp32
    ws: torch.Tensor         # uint8 workspace
    metadata: Optional[dict] = None   # host metadata of a packed problem


_SPEC_CACHE: "collections.OrderedDict" = collections.OrderedDict()
_SPEC_CACHE_MAX = 64
_SPEC_LOCK = threading.Lock()


def cached_spec(B, T, H, Dk, Dv, num_segments, chunk=64, scale=None, dtype=torch.bfloat16,
                cu_seqlens=None, device="cuda", q_heads=0, vector_gates=False):
    """The problem description of a shape, built once: packed metadata is
    computed on the host and copied to the device on the first call only.
    Returns (spec, host metadata or None).  The spec holds no per-call
    buffers, so any number of calls (layers, steps) may share it."""
    if scale is None:
        scale = 1.0 / math.sqrt(Dk)
    cu_key = None if cu_seqlens is None else tuple(int(x) for x in cu_seqlens)
    key = (int(B), int(T), int(H), int(Dk), int(Dv), int(num_segments), int(chunk), float(scale),
           dtype, str(torch.device(device)), cu_key, int(q_heads), bool(vector_gates))
    with _SPEC_LOCK:
        hit = _SPEC_CACHE.get(key)
        if hit is not None:
            _SPEC_CACHE.move_to_end(key)
            return hit
    meta = None
    seq_idx = pre = fol = None
    if cu_seqlens is not None:
        meta = C.rm_cp_build_packed_metadata(cu_key, T, num_segments)
        seq_idx = meta["seq_idx"].to(device)
        pre = meta["preceding_start"].to(device)
        fol = meta["following_stop"].to(device)
    spec = C.ProblemSpec(B, T, H, Dk, Dv, num_segments, chunk, scale, dtype, seq_idx, pre, fol,
                         q_heads=q_heads, vector_gates=int(bool(vector_gates)))
    C.rm_cp_validate(spec)
    entry = (spec, meta)
    with _SPEC_LOCK:
        _SPEC_CACHE[key] = entry
        while len(_SPEC_CACHE) > _SPEC_CACHE_MAX:
            _SPEC_CACHE.popitem(last=False)
    return entry


def make_plan(B, T, H, Dk, Dv, num_segments, chunk=64, scale=None, dtype=torch.bfloat16,
              cu_seqlens=None, device="cuda", backward=True, q_heads=0, vector_gates=False) -> Plan:
    """q_heads > 0: q is [B,T,q_heads,Dk], shared by H / q_heads consecutive heads.
    vector_gates: one gate per key dimension (g [B,T,H,Dk], M [nseg,B,H,Dk])."""
    spec, meta = cached_spec(B, T, H, Dk, Dv, num_segments, chunk, scale, dtype, cu_seqlens,
                             device, q_heads, vector_gates)
    f32 = dict(dtype=torch.float32, device=device)
    ssz = (num_segments, B, H, Dk, Dv)
    M = torch.empty((num_segments, B, H) + ((Dk,) if vector_gates else ()), **f32)
    dS = torch.empty(ssz, **f32)
    S_in = torch.empty(ssz, **f32)
    ws = torch.empty(max(C.rm_cp_workspace_size(spec), 16), dtype=torch.uint8, device=device)
    plan = Plan(spec, M, dS, S_in, torch.empty((0,), **f32), torch.empty((0,), **f32), ws, meta)
    if backward:
        backward_buffers(plan)
    return plan


def backward_buffers(plan: Plan) -> Plan:
    """Allocates the backward's gamma, dS_out and workspace if the plan lacks them."""
    s = plan.spec
    ssz = (s.num_segments, s.B, s.H, s.Dk, s.Dv)
    dev = plan.M.device
    if tuple(plan.gamma.shape) != ssz:
        plan.gamma = torch.empty(ssz, dtype=torch.float32, device=dev)
        plan.dS_out = torch.empty(ssz, dtype=torch.float32, device=dev)
    need = max(C.rm_cp_workspace_size(s), 16)
    if plan.ws.numel() < need:
        plan.ws = torch.empty(need, dtype=torch.uint8, device=dev)
    return plan


def plan_like(q: torch.Tensor, v: torch.Tensor, num_segments: int, chunk: int = 64,
              scale=None, cu_seqlens=None, backward=True, vector_gates=False) -> Plan:
    B, T, H, Dk = q.shape
    return make_plan(B, T, H, Dk, v.shape[-1], num_segments, chunk, scale, q.dtype, cu_seqlens,
                     q.device, backward, vector_gates=vector_gates)


def forward(plan: Plan, q, k, v, g, o=None, stream=None, fused=False) -> torch.Tensor:
    """o = chunkwise gated linear attention; fills plan.M, plan.dS, plan.S_in.
    fused=False: the three calls prepare -> compose_prefix -> apply (the
    faster form on these shapes); fused=True: one rm_cp_forward_fused call
    (one launch on the tensor-core path).  Both give the same values."""
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    if fused:
        C.rm_cp_forward_fused(plan.spec, q, k, v, g, plan.M, plan.dS, plan.S_in, o, plan.ws, stream)
        return o
    C.rm_cp_forward_prepare(plan.spec, k, v, g, plan.M, plan.dS, plan.ws, stream)
    C.rm_cp_compose_prefix(plan.spec, plan.M, plan.dS, plan.S_in, stream)
    C.rm_cp_forward_apply(plan.spec, q, k, v, g, plan.S_in, o, plan.ws, stream)
    return o


def backward(plan: Plan, q, k, v, g, dO, grads=None, stream=None):
    """(dq, dk, dv, dg) of sum(dO * o); needs plan.M and plan.S_in from forward."""
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                 torch.empty(g.shape, dtype=torch.float32, device=g.device))
    dq, dk, dv, dg = grads
    C.rm_cp_backward_prepare(plan.spec, q, k, v, g, plan.S_in, dO, plan.gamma, dq, plan.ws, stream)
    C.rm_cp_compose_suffix(plan.spec, plan.M, plan.gamma, plan.dS_out, stream)
    C.rm_cp_backward_apply(plan.spec, q, k, v, g, dO, plan.S_in, plan.dS_out, dk, dv, dg, plan.ws,
                           stream)
    return dq, dk, dv, dg


class StepGraph:
    """One step captured as a CUDA graph: the forward (the three calls, or the
    one-launch forward with fused=True) and, given dO, the three backward
    calls, on fixed buffers.  replay() re-runs the step on whatever those
    buffers hold; results land in the same tensors (o, the gradients and the
    plan's summaries).  The C calls neither allocate nor synchronise and only
    enqueue on the stream they are given, so they capture as they are; one
    uncaptured run first sets the kernels' launch attributes."""

    def __init__(self, plan: Plan, q, k, v, g, dO=None, fused: bool = False):
        self.plan = plan
        self.q, self.k, self.v, self.g, self.dO = q, k, v, g, dO
        self.fused = fused
        self.o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
        self.grads = None
        if dO is not None:
            backward_buffers(plan)
            self.grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                          torch.empty(g.shape, dtype=torch.float32, device=g.device))
        dev = v.device
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            self._run()
        torch.cuda.current_stream(dev).wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=side):
            self._run()

    def _run(self):
        forward(self.plan, self.q, self.k, self.v, self.g, o=self.o, fused=self.fused)
        if self.dO is not None:
            backward(self.plan, self.q, self.k, self.v, self.g, self.dO, grads=self.grads)

    def replay(self):
        """Runs the captured step on the current stream."""
        self.graph.replay()
        return (self.o,) + (self.grads if self.grads is not None else ())


class ChunkwiseGatedLinearAttention(torch.autograd.Function):
    """Autograd adapter.  The problem description (and a packed problem's
    device metadata) comes from a cache keyed by shape and cu_seqlens, so a
    training loop builds and uploads it once.  Between forward and backward
    each call keeps only what the backward reads, M and S_in, beside the saved
    (q, k, v, g); the forward summaries dS die with the forward, and gamma,
    dS_out and the workspace are taken from PyTorch's caching allocator in the
    backward."""

    @staticmethod
    def forward(ctx, q, k, v, g, num_segments, chunk, scale, cu_seqlens):
        q, k, v, g = (t.contiguous() for t in (q, k, v, g))
        plan = plan_like(q, v, num_segments, chunk, scale, cu_seqlens, backward=False,
                         vector_gates=g.dim() == 4)
        o = forward(plan, q, k, v, g)
        plan.dS = None
        ctx.plan = plan
        ctx.save_for_backward(q, k, v, g)
        return o

    @staticmethod
    def backward(ctx, dO):
        q, k, v, g = ctx.saved_tensors
        plan = backward_buffers(ctx.plan)
        dq, dk, dv, dg = backward(plan, q, k, v, g, dO.contiguous())
        ctx.plan = None
        return dq, dk, dv, dg, None, None, None, None


def chunkwise_gla(q, k, v, g, num_segments: int, chunk: int = 64, scale=None, cu_seqlens=None):
    """Differentiable chunkwise gated linear attention.

    q, k [B,T,H,Dk], v [B,T,H,Dv] (fp32 or bf16, CUDA), g [B,T,H] fp32 log-gates
    (or [B,T,H,Dk]: one gate per key dimension).
    cu_seqlens (host int32 [N+1]) packs several sequences along T."""
    return ChunkwiseGatedLinearAttention.apply(q, k, v, g, num_segments, chunk, scale, cu_seqlens)


class HostPipeline:
    """Steps fed from host memory through rm_cp_step_host: two device buffer
    sets used in turn, each with its three events, and two copy streams, so
    that the copies of one step overlap the kernels of the next.  host maps
    q, k, v, g (and dO) to pinned host inputs and o (and dq, dk, dv, dg) to
    pinned host outputs."""

    def __init__(self, plan: Plan, host: dict, device="cuda", nsets: int = 2):
        self.plan = plan
        self.host = host
        self.backward = host.get("dO") is not None
        names = ("q", "k", "v", "g", "o") + (("dO", "dq", "dk", "dv", "dg") if self.backward else ())
        self.sets = []
        for _ in range(nsets):
            dev = {n: torch.empty(host[n].shape, dtype=host[n].dtype, device=device) for n in names}
            events = tuple(C.rm_cp_event_create() for _ in range(3))
            self.sets.append((dev, events))
        self.h2d = torch.cuda.Stream(device)
        self.d2h = torch.cuda.Stream(device)
        self.state = dict(M=plan.M, dS=plan.dS, S_in=plan.S_in, ws=plan.ws)
        if self.backward:
            self.state.update(gamma=plan.gamma, dS_out=plan.dS_out)
        self.n = 0

    def begin(self, compute=None):
        """Order the copy streams after everything already enqueued on compute."""
        compute = compute if compute is not None else torch.cuda.current_stream()
        self.h2d.wait_stream(compute)
        self.d2h.wait_stream(compute)

    def step(self, compute=None):
        """Enqueue one step (copies in, the path, copies out); returns at once."""
        compute = compute if compute is not None else torch.cuda.current_stream()
        dev, events = self.sets[self.n % len(self.sets)]
        C.rm_cp_step_host(self.plan.spec, self.host, dev, events, self.state, compute, self.h2d,
                          self.d2h)
        self.n += 1

    def join(self, compute=None):
        """Make compute wait for every copy enqueued so far."""
        compute = compute if compute is not None else torch.cuda.current_stream()
        compute.wait_stream(self.h2d)
        compute.wait_stream(self.d2h)

    def close(self):
        torch.cuda.synchronize()
        for _, events in self.sets:
            for e in events:
                C.rm_cp_event_destroy(e)
        self.sets = []


# ------------------------------------------------------------------ Mamba2 SSD

@dataclasses.dataclass
class SsdPlan:
    """The path's plan (Dk = N, Dv = P, scale 1, q_heads = G: the heads of a
    group read C itself as their queries) plus the mapped inputs."""
    core: Plan
    G: int
    k: torch.Tensor   # [B,T,H,N] = dt B
    g: torch.Tensor   # [B,T,H] fp32 = dt A
    ws: torch.Tensor  # workspace of rm_ssd_finish_backward


def make_ssd_plan(B, T, H, G, N, P, num_segments, chunk=64, dtype=torch.bfloat16,
                  cu_seqlens=None, device="cuda", backward=True) -> SsdPlan:
    core = make_plan(B, T, H, N, P, num_segments, chunk, 1.0, dtype, cu_seqlens, device, backward,
                     q_heads=G)
    k = torch.empty((B, T, H, N), dtype=dtype, device=device)
    g = torch.empty((B, T, H), dtype=torch.float32, device=device)
    ws = torch.empty(max(C.rm_ssd_workspace_size(core.spec), 16), dtype=torch.uint8, device=device)
    return SsdPlan(core, G, k, g, ws)


def ssd_forward(sp: SsdPlan, x, dt, A, Bm, Cm, D=None, y=None, stream=None) -> torch.Tensor:
    """y of the Mamba2 SSD scan through the six calls: q = C (shared by a
    group's heads), k = dt B, v = x, g = dt A."""
    C.rm_ssd_map_inputs(sp.core.spec, sp.G, dt, A, Bm, None, None, sp.k, sp.g, stream)
    y = forward(sp.core, Cm, sp.k, x, sp.g, o=y, stream=stream)
    C.rm_ssd_finish_forward(sp.core.spec, x, D, y, stream)
    return y


def ssd_backward(sp: SsdPlan, x, dt, A, Bm, Cm, dy, D=None, stream=None, core=None):
    """(dx, ddt, dA, dB, dC, dD) of sum(dy * y); needs ssd_forward on sp first.
    core: an optional dict that receives the gradients of the gated recurrence
    the scan runs as (dq, dk, dv, dg of q = C, k = dt B, v = x, g = dt A)."""
    B, T, H, _ = x.shape
    grads = (torch.empty_like(sp.k), torch.empty_like(sp.k), torch.empty_like(x),
             torch.empty((B, T, H), dtype=torch.float32, device=x.device))
    dq, dk, dv, dg = backward(sp.core, Cm, sp.k, x, sp.g, dy, grads=grads, stream=stream)
    ddt = torch.empty((B, T, H), dtype=torch.float32, device=x.device)
    dA = torch.empty(H, dtype=torch.float32, device=x.device)
    dD = torch.empty(H, dtype=torch.float32, device=x.device)
    dB = torch.empty(Bm.shape, dtype=Bm.dtype, device=x.device)
    dC = torch.empty_like(dB)
    if core is not None:
        # dv becomes dx in place below; keep the recurrence's own copy
        core.update(dq=dq, dk=dk, dv=dv.clone(), dg=dg)
    C.rm_ssd_finish_backward(sp.core.spec, sp.G, x, dt, A, Bm, dy, D, dq, dk, dv, dg, ddt, dA, dB,
                             dC, dD, sp.ws, stream)
    return dv, ddt, dA, dB, dC, dD


# ------------------------------------------------------------------ gated delta rule

@dataclasses.dataclass
class GdrPlan:
    """Summaries and workspace of the gated delta rule (Dk x Dk transitions)."""
    spec: C.ProblemSpec
    M: torch.Tensor        # [nseg,B,H,Dk,Dk] fp32
    dS: torch.Tensor       # [nseg,B,H,Dk,Dv] fp32
    S_in: torch.Tensor
    gamma: torch.Tensor
    dS_out: torch.Tensor
    ws: torch.Tensor       # the step's workspace: per-chunk factors (tensor cores) and saved states


def make_gdr_plan(B, T, H, Dk, Dv, num_segments, chunk=16, scale=None, dtype=torch.float32,
                  cu_seqlens=None, device="cuda", q_heads=0) -> GdrPlan:
    spec, _ = cached_spec(B, T, H, Dk, Dv, num_segments, chunk, scale, dtype, cu_seqlens, device,
                          q_heads)
    f32 = dict(dtype=torch.float32, device=device)
    ssz = (num_segments, B, H, Dk, Dv)
    ws = torch.empty(max(C.rm_gdr_workspace_size(spec), 16), dtype=torch.uint8, device=device)
    return GdrPlan(spec, torch.empty((num_segments, B, H, Dk, Dk), **f32), torch.empty(ssz, **f32),
                   torch.empty(ssz, **f32), torch.empty(ssz, **f32), torch.empty(ssz, **f32), ws)


def gdr_forward(plan: GdrPlan, q, k, v, g, beta, o=None, stream=None) -> torch.Tensor:
    """o of the gated delta rule: prepare -> compose_prefix -> apply."""
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    C.rm_gdr_forward_prepare(plan.spec, k, v, g, beta, plan.M, plan.dS, plan.ws, stream)
    C.rm_gdr_compose_prefix(plan.spec, plan.M, plan.dS, plan.S_in, stream)
    C.rm_gdr_forward_apply(plan.spec, q, k, v, g, beta, plan.S_in, o, plan.ws, stream)
    return o


def gdr_backward(plan: GdrPlan, q, k, v, g, beta, dO, stream=None, grads=None):
    """(dq, dk, dv, dg, dbeta) of sum(dO * o); needs gdr_forward on plan first.
    grads: optional preallocated (dq, dk, dv, dg, dbeta) to write into."""
    if grads is None:
        grads = (torch.empty_like(k), torch.empty_like(k), torch.empty_like(v), torch.empty_like(g),
                 torch.empty_like(beta))
    dq, dk, dv, dg, db = grads
    C.rm_gdr_backward_prepare(plan.spec, q, k, v, g, beta, plan.S_in, dO, plan.gamma, dq, plan.ws,
                              stream)
    C.rm_gdr_compose_suffix(plan.spec, plan.M, plan.gamma, plan.dS_out, stream)
    C.rm_gdr_backward_apply(plan.spec, q, k, v, g, beta, dO, plan.dS_out, dk, dv, dg, db, plan.ws,
                            stream)
    return dq, dk, dv, dg, db


class GatedDeltaRule(torch.autograd.Function):
    """Autograd adapter of the gated delta rule (the six rm_gdr_* calls).  The
    plan (summaries and the step's workspace) lives from the forward to the
    backward: the backward reads M, S_in and the workspace the forward filled
    (on the tensor cores, each chunk's triangular factors).  q has one row per
    head (shared query rows are a plan option of the direct calls only)."""

    @staticmethod
    def forward(ctx, q, k, v, g, beta, num_segments, chunk, scale, cu_seqlens):
        q, k, v, g, beta = (t.contiguous() for t in (q, k, v, g, beta))
        if q.shape != k.shape:
            raise ValueError("gated_delta_rule: q and k must have the same shape [B,T,H,Dk]")
        B, T, H, Dk = k.shape
        plan = make_gdr_plan(B, T, H, Dk, v.shape[-1], num_segments, chunk, scale, v.dtype, cu_seqlens,
                             v.device)
        o = gdr_forward(plan, q, k, v, g, beta)
        ctx.plan = plan
        ctx.save_for_backward(q, k, v, g, beta)
        return o

    @staticmethod
    def backward(ctx, dO):
        q, k, v, g, beta = ctx.saved_tensors
        grads = gdr_backward(ctx.plan, q, k, v, g, beta, dO.contiguous())
        ctx.plan = None
        return grads + (None, None, None, None)


def gated_delta_rule(q, k, v, g, beta, num_segments: int, chunk: int = 16, scale=None, cu_seqlens=None):
    """Differentiable gated delta rule: S_t = exp(g_t)(I - beta_t k_t k_t^T) S_{t-1}
    + beta_t k_t v_t^T, o_t = scale S_t^T q_t.

    q, k [B,T,H,Dk], v [B,T,H,Dv] (fp32 or bf16, CUDA), g and beta [B,T,H] fp32.
    cu_seqlens (host int32 [N+1]) packs several sequences along T."""
    return GatedDeltaRule.apply(q, k, v, g, beta, num_segments, chunk, scale, cu_seqlens)


class GdrStepGraph:
    """One gated-delta-rule step captured as a CUDA graph: the three forward
    calls and, given dO, the three backward calls, on fixed buffers (as
    StepGraph does for the scalar and vector gates).  replay() returns
    (o,) + (dq, dk, dv, dg, dbeta)."""

    def __init__(self, plan: GdrPlan, q, k, v, g, beta, dO=None):
        self.plan = plan
        self.args = (q, k, v, g, beta)
        self.dO = dO
        self.o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
        self.grads = None
        if dO is not None:
            self.grads = (torch.empty_like(k), torch.empty_like(k), torch.empty_like(v), torch.empty_like(g),
                          torch.empty_like(beta))
        dev = v.device
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            self._run()
        torch.cuda.current_stream(dev).wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=side):
            self._run()

    def _run(self):
        gdr_forward(self.plan, *self.args, o=self.o)
        if self.dO is not None:
            gdr_backward(self.plan, *self.args, self.dO, grads=self.grads)

    def replay(self):
        """Runs the captured step on the current stream."""
        self.graph.replay()
        return (self.o,) + (self.grads if self.grads is not None else ())
