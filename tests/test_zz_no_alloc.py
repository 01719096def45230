"""rm_cp_backward_noalloc against the workspace form of the backward.

Some callers cannot hand this library device memory: a custom operator
called through a plugin interface whose signature has no workspace, or a
deployment whose device memory is planned once and may not grow afterwards.
For them rm_cp_backward_noalloc runs the backward with scratch held by the
library itself.  These tests call it through the C ABI, twice in a row (the
second call finds the previous call's values in the shared scratch), and
compare every result with rm_cp_backward_prepare + rm_cp_compose_suffix +
rm_cp_backward_apply on the same inputs.  Both run the same kernels in the
same order on the same inputs, so the results must be bit-identical: a
partly stale read of the shared scratch would show up as a difference.
(Parity of either form with the fp64 oracle is covered by the other tests.)
This file is collected last so that a failing run has already run the rest.
"""
import math

import pytest
import torch

from state_summary_scan_gb300 import _capi as C
from state_summary_scan_gb300 import api

pytestmark = pytest.mark.gpu

KEYS = ("dq", "dk", "dv", "dg", "gamma", "dS_out")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    C.load()


def inputs(B, T, H, Dk, Dv, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, T, H, Dk, generator=gen)
    k = torch.randn(B, T, H, Dk, generator=gen)
    k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn(B, T, H, Dv, generator=gen)
    g = torch.nn.functional.logsigmoid(torch.randn(B, T, H, generator=gen) + 3.0)
    dO = torch.randn(B, T, H, Dv, generator=gen)
    return [t.to(dtype).cuda() for t in (q, k, v)] + [g.cuda(), dO.to(dtype).cuda()]


def workspace_backward(plan, q, k, v, g, dO):
    dq, dk, dv, dg = api.backward(plan, q, k, v, g, dO)
    return dict(dq=dq.clone(), dk=dk.clone(), dv=dv.clone(), dg=dg.clone(),
                gamma=plan.gamma.clone(), dS_out=plan.dS_out.clone())


def noalloc_backward(plan, q, k, v, g, dO):
    out = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
               dg=torch.empty_like(g), gamma=torch.empty_like(plan.gamma),
               dS_out=torch.empty_like(plan.dS_out))
    C.rm_cp_backward_noalloc(plan.spec, q, k, v, g, plan.S_in, plan.M, dO, out["gamma"],
                             out["dS_out"], out["dq"], out["dk"], out["dv"], out["dg"])
    return out


def assert_same(a, b):
    for key in KEYS:
        assert torch.equal(a[key], b[key]), \
            f"{key}: max|diff| {float((a[key].double() - b[key].double()).abs().max()):.3e}"


@pytest.mark.parametrize("dtype,Dk,Dv", [
    (torch.bfloat16, 128, 128),   # tensor-core kernels
    (torch.bfloat16, 128, 256),
    (torch.float32, 32, 32),      # generic fp32 kernels
])
def test_noalloc_matches_workspace_backward_twice(dtype, Dk, Dv):
    B, T, H, nseg = 1, 1024, 3, 4
    cu = [0, 100, 101, 700, 1024]
    ref_out = None
    for call, seed in enumerate((11, 12)):
        q, k, v, g, dO = inputs(B, T, H, Dk, Dv, dtype, seed)
        plan = api.plan_like(q, v, nseg, 64, 1.0 / math.sqrt(Dk), cu_seqlens=cu)
        api.forward(plan, q, k, v, g)
        ref_out = workspace_backward(plan, q, k, v, g, dO)
        got = noalloc_backward(plan, q, k, v, g, dO)
        torch.cuda.synchronize()
        assert_same(got, ref_out)


def test_noalloc_matches_workspace_on_a_grid_wider_than_the_gpu():
    """16 segments x 16 heads = 256 (segment, head) sweeps, more than the SMs,
    so the sweeps run in more than one wave, with sequences starting inside
    and across segments: the no-alloc form still equals the workspace form
    bit for bit."""
    q, k, v, g, dO = inputs(1, 4096, 16, 128, 128, torch.bfloat16, 31)
    cu = [0, 1000, 1001, 2300, 4096]
    plan = api.plan_like(q, v, 16, 64, 1.0 / math.sqrt(128), cu_seqlens=cu)
    api.forward(plan, q, k, v, g)
    ref_out = workspace_backward(plan, q, k, v, g, dO)
    got = noalloc_backward(plan, q, k, v, g, dO)
    torch.cuda.synchronize()
    assert_same(got, ref_out)


def test_noalloc_repeated_calls_agree():
    q, k, v, g, dO = inputs(2, 512, 2, 128, 128, torch.bfloat16, 21)
    plan = api.plan_like(q, v, 2, 64, 1.0 / math.sqrt(128))
    api.forward(plan, q, k, v, g)
    first = noalloc_backward(plan, q, k, v, g, dO)
    second = noalloc_backward(plan, q, k, v, g, dO)
    torch.cuda.synchronize()
    assert_same(second, first)


@pytest.mark.parametrize("dtype,Dk,Dv", [
    (torch.bfloat16, 128, 128),   # vector gates on the tensor-core kernels
    (torch.float32, 32, 32),      # and on the generic kernels
])
def test_noalloc_vector_gates(dtype, Dk, Dv):
    """One gate per key dimension: the shared scratch holds Dk values per
    (row, token, head); the no-alloc form equals the workspace form."""
    B, T, H, nseg = 1, 1024, 3, 4
    cu = [0, 100, 101, 700, 1024]
    q, k, v, _, dO = inputs(B, T, H, Dk, Dv, dtype, 41)
    gen = torch.Generator().manual_seed(42)
    g = torch.nn.functional.logsigmoid(torch.randn(B, T, H, Dk, generator=gen) + 3.0).cuda()
    plan = api.plan_like(q, v, nseg, 64, 1.0 / math.sqrt(Dk), cu_seqlens=cu, vector_gates=True)
    assert C.rm_cp_path(plan.spec) == (1 if dtype == torch.bfloat16 else 0)
    api.forward(plan, q, k, v, g)
    ref_out = workspace_backward(plan, q, k, v, g, dO)
    got = noalloc_backward(plan, q, k, v, g, dO)
    torch.cuda.synchronize()
    assert_same(got, ref_out)
