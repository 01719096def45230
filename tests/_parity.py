"""Shared helpers for the GPU-vs-oracle parity tests.

The CUDA side runs through the C ABI (via the thin ctypes binding); the
oracle side runs the fp64 segmented oracle on the same seeded inputs,
restricted to sampled heads when the full problem is too large for the CPU.
Heads are independent, so a sampled head's outputs are exact references.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from state_summary_scan_gb300 import api

FP32_TOL = 1e-4   # max|gpu - ref| <= tol * max|ref|, per tensor
BF16_TOL = 2e-2

GRAD_KEYS = ("dq", "dk", "dv", "dg")
SUMMARY_KEYS_FWD = ("M", "dS", "S_in")
SUMMARY_KEYS_BWD = ("gamma", "dS_out")


def tol_for(dtype: torch.dtype) -> float:
    return FP32_TOL if dtype == torch.float32 else BF16_TOL


def canary_empty(shape, dtype, device, pad=64):
    """Output buffer with a NaN-free sentinel tail; returns (view, full)."""
    n = int(np.prod(shape))
    full = torch.full((n + pad,), 12345.0, dtype=dtype, device=device)
    return full[:n].view(shape), full


def run_gpu(q, k, v, g, dO, num_segments, chunk=64, scale=None, cu_seqlens=None,
            use_metadata=True, canary=True, fused=False):
    """Run the CUDA path on host tensors; returns a dict of CPU float64 tensors."""
    dev = "cuda"
    qd, kd, vd, gd = (t.to(dev).contiguous() for t in (q, k, v, g))
    plan = api.plan_like(qd, vd, num_segments, chunk, scale, cu_seqlens, backward=dO is not None)
    if cu_seqlens is not None and not use_metadata:
        # same problem, but prefixes from segment 0 and suffixes to the end
        s = plan.spec
        plan.spec = type(s)(s.B, s.T, s.H, s.Dk, s.Dv, s.num_segments, s.chunk, s.scale, s.dtype,
                            s._keep[0], None, None)
    fulls = []
    if canary:
        o, f = canary_empty(vd.shape, vd.dtype, dev)
        fulls.append(f)
    else:
        o = None
    o = api.forward(plan, qd, kd, vd, gd, o=o, fused=fused)
    out = dict(o=o, M=plan.M, dS=plan.dS, S_in=plan.S_in)
    if dO is not None:
        dOd = dO.to(dev).contiguous()
        grads = []
        for shape, dt in ((qd.shape, qd.dtype), (kd.shape, kd.dtype), (vd.shape, vd.dtype),
                          (gd.shape, torch.float32)):
            t, f = canary_empty(shape, dt, dev)
            grads.append(t)
            fulls.append(f)
        dq, dk, dv, dg = api.backward(plan, qd, kd, vd, gd, dOd, grads=tuple(grads))
        out.update(dq=dq, dk=dk, dv=dv, dg=dg, gamma=plan.gamma, dS_out=plan.dS_out)
    torch.cuda.synchronize()
    for f in fulls:
        n = f.numel() - 64
        assert torch.all(f[n:] == 12345.0), "kernel wrote past the end of an output"
    return {key: val.detach().to("cpu", torch.float64) for key, val in out.items()}


def run_oracle(q, k, v, g, dO, num_segments, scale, cu_seqlens=None, heads=None):
    """Segmented fp64 oracle on the given heads; dict of float64 numpy arrays."""
    if heads is not None:
        q, k, v, g = q[:, :, heads], k[:, :, heads], v[:, :, heads], g[:, :, heads]
        dO = None if dO is None else dO[:, :, heads]
    T = q.shape[1]
    seg = oracle.equal_segments(T, num_segments)
    si = pre = fol = None
    if cu_seqlens is not None:
        md = oracle.packed_metadata(cu_seqlens, T, seg)
        si, pre, fol = md["seq_idx"], md["preceding_start"], md["following_stop"]
    o, mid = oracle.segmented_forward(q, k, v, g, scale, seg, si, pre)
    out = dict(o=o, **mid)
    if dO is not None:
        grads, bmid = oracle.segmented_backward(q, k, v, g, dO, scale, seg, si, pre, fol,
                                                S_in=mid["S_in"], M=mid["M"])
        out.update(dict(zip(GRAD_KEYS, grads)), gamma=bmid["gamma"], dS_out=bmid["dS_out"])
    return out


def select_heads(gpu: dict, heads):
    """Restrict GPU results to sampled heads (head axis: 2 for tokens, 2 for summaries)."""
    res = {}
    for key, val in gpu.items():
        res[key] = val[:, :, heads].numpy() if heads is not None else val.numpy()
    return res


def compare(gpu: dict, ref: dict, tol: float, keys):
    report = {}
    for key in keys:
        a, b = gpu[key], ref[key]
        assert a.shape == b.shape, (key, a.shape, b.shape)
        assert np.all(np.isfinite(a)), f"{key}: non-finite values"
        scale = float(np.max(np.abs(b)))
        err = float(np.max(np.abs(a - b)))
        report[key] = (err, scale)
        assert err <= tol * scale or (scale == 0.0 and err == 0.0), \
            f"{key}: max|err| {err:.3e} > {tol:g} * max|ref| {scale:.3e}"
    return report
