"""CUDA-graph capture of a step (api.StepGraph): the C calls neither allocate
nor synchronise and only enqueue on the stream they are given, so the forward
(three calls, or the one-launch forward) and the backward capture as they
are.  Replaying the graph gives the direct calls' outputs, gradients and
summaries bit for bit (same kernels, same launch shapes, same inputs), also
after new values are written into the captured input buffers."""
import math

import pytest
import torch

from state_summary_scan_gb300 import _capi as C
from state_summary_scan_gb300 import api
from state_summary_scan_gb300.workloads import random_cu_seqlens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    C.load()


def _inputs(B, T, H, Dk, Dv, vg, seed):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, T, H, Dk, generator=gen)
    k = torch.randn(B, T, H, Dk, generator=gen)
    k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn(B, T, H, Dv, generator=gen)
    gshape = (B, T, H, Dk) if vg else (B, T, H)
    g = torch.nn.functional.logsigmoid(torch.randn(*gshape, generator=gen) + 3.0)
    dO = torch.randn(B, T, H, Dv, generator=gen)
    bf = torch.bfloat16
    return [t.to("cuda").contiguous() for t in (q.to(bf), k.to(bf), v.to(bf), g, dO.to(bf))]


@pytest.mark.parametrize("case", ["scalar", "fused", "vector", "packed", "dv256"])
def test_graph_replay_equals_direct_calls(case):
    B, T, H, Dk, nseg = 1, 2048, 4, 128, 4
    Dv = 256 if case == "dv256" else 128
    vg = case == "vector"
    fused = case == "fused"
    cu = random_cu_seqlens(torch.Generator().manual_seed(5), T, 700) if case == "packed" else None

    def plan():
        return api.make_plan(B, T, H, Dk, Dv, nseg, 64, 1 / math.sqrt(Dk), torch.bfloat16, cu, "cuda",
                             vector_gates=vg)

    q, k, v, g, dO = _inputs(B, T, H, Dk, Dv, vg, seed=1)
    pg = plan()
    assert C.rm_cp_path(pg.spec) == 1
    sg = api.StepGraph(pg, q, k, v, g, dO, fused=fused)
    for seed in (1, 2):  # the captured values, then new ones in the same buffers
        if seed == 2:
            for dst, src in zip((q, k, v, g, dO), _inputs(B, T, H, Dk, Dv, vg, seed=2)):
                dst.copy_(src)
        got = list(sg.replay()) + [pg.M, pg.dS, pg.S_in, pg.gamma, pg.dS_out]
        pd = plan()
        o = api.forward(pd, q, k, v, g, fused=fused)
        ref = [o, *api.backward(pd, q, k, v, g, dO), pd.M, pd.dS, pd.S_in, pd.gamma, pd.dS_out]
        torch.cuda.synchronize()
        names = ("o", "dq", "dk", "dv", "dg", "M", "dS", "S_in", "gamma", "dS_out")
        for name, a, b in zip(names, got, ref):
            assert torch.equal(a, b), (case, seed, name)


def test_gdr_graph_replay_equals_direct_calls():
    """The gated delta rule's six calls (tensor-core sweeps: the forward
    prepare's two launches, the apply, the backward's two walks and the
    reverse walk) captured as one graph give the direct calls' results bit for
    bit, also after new inputs are written into the captured buffers."""
    B, T, H, D, nseg = 1, 1024, 4, 64, 4
    gen = torch.Generator().manual_seed(11)

    def inputs():
        q = torch.randn(B, T, H, D, generator=gen)
        k = torch.randn(B, T, H, D, generator=gen)
        k = k / k.norm(dim=-1, keepdim=True)
        v = torch.randn(B, T, H, D, generator=gen)
        g = torch.nn.functional.logsigmoid(torch.randn(B, T, H, generator=gen) + 3.0)
        beta = torch.sigmoid(torch.randn(B, T, H, generator=gen))
        dO = torch.randn(B, T, H, D, generator=gen)
        bf = torch.bfloat16
        return [t.to("cuda").contiguous() for t in (q.to(bf), k.to(bf), v.to(bf), g, beta, dO.to(bf))]

    def plan():
        return api.make_gdr_plan(B, T, H, D, D, nseg, 64, 1 / math.sqrt(D), torch.bfloat16, None, "cuda")

    q, k, v, g, beta, dO = inputs()
    pg = plan()
    assert C.rm_gdr_path(pg.spec) == 1
    sg = api.GdrStepGraph(pg, q, k, v, g, beta, dO)
    for it in range(2):  # the captured values, then new ones in the same buffers
        if it == 1:
            for dst, src in zip((q, k, v, g, beta, dO), inputs()):
                dst.copy_(src)
        got = list(sg.replay()) + [pg.M, pg.dS, pg.S_in, pg.gamma, pg.dS_out]
        pd = plan()
        o = api.gdr_forward(pd, q, k, v, g, beta)
        want = [o] + list(api.gdr_backward(pd, q, k, v, g, beta, dO)) + [pd.M, pd.dS, pd.S_in, pd.gamma,
                                                                           pd.dS_out]
        torch.cuda.synchronize()
        for a, b_ in zip(got, want):
            assert torch.equal(a, b_)


@pytest.mark.parametrize("case", ["scalar", "vector"])
def test_autograd_equals_direct_calls_tensor_cores(case):
    """torch.autograd through chunkwise_gla runs its backward on autograd's
    device thread; on the tensor-core path it gives the direct calls' o and
    gradients bit for bit."""
    B, T, H, Dk, Dv, nseg = 1, 1024, 2, 128, 128, 4
    vg = case == "vector"
    q, k, v, g, dO = _inputs(B, T, H, Dk, Dv, vg, seed=3)
    scale = 1 / math.sqrt(Dk)
    pd = api.make_plan(B, T, H, Dk, Dv, nseg, 64, scale, torch.bfloat16, None, "cuda", vector_gates=vg)
    assert C.rm_cp_path(pd.spec) == 1
    o_ref = api.forward(pd, q, k, v, g)
    g_ref = api.backward(pd, q, k, v, g, dO)
    leaves = [t.clone().requires_grad_(True) for t in (q, k, v, g)]
    o = api.chunkwise_gla(*leaves, nseg, 64, scale)
    o.backward(dO)
    torch.cuda.synchronize()
    assert torch.equal(o.detach(), o_ref)
    for name, leaf, ref in zip(("dq", "dk", "dv", "dg"), leaves, g_ref):
        assert torch.equal(leaf.grad, ref), name


@pytest.mark.parametrize("case", ["scalar", "gdr"])
def test_calls_from_a_thread_without_cuda_context(case):
    """A backward called from a thread that has made no CUDA call (buffers
    preallocated, the stream passed in: autograd's device thread with a warm
    caching allocator is such a thread) gives the same gradients as from the
    main thread: the entry points bind the device's context themselves before
    encoding their tensor maps."""
    import threading

    stream = torch.cuda.current_stream()
    if case == "scalar":
        B, T, H, D, nseg = 1, 1024, 2, 128, 4
        q, k, v, g, dO = _inputs(B, T, H, D, D, False, seed=4)
        plan = api.make_plan(B, T, H, D, D, nseg, 64, 1 / math.sqrt(D), torch.bfloat16, None, "cuda")
        assert C.rm_cp_path(plan.spec) == 1
        api.forward(plan, q, k, v, g)
        call = lambda out: api.backward(plan, q, k, v, g, dO, stream=stream, grads=out)
        out = [torch.empty_like(t) for t in (q, k, v, g)]
    else:
        B, T, H, D, nseg = 1, 512, 2, 64, 4
        q, k, v, g, dO = _inputs(B, T, H, D, D, False, seed=4)
        beta = torch.sigmoid(g)
        plan = api.make_gdr_plan(B, T, H, D, D, nseg, 16, 1 / math.sqrt(D), torch.bfloat16, None, "cuda")
        assert C.rm_gdr_path(plan.spec) == 1
        api.gdr_forward(plan, q, k, v, g, beta)
        call = lambda out: api.gdr_backward(plan, q, k, v, g, beta, dO, stream=stream, grads=out)
        out = [torch.empty_like(t) for t in (q, k, v, g, beta)]
    ref = [torch.empty_like(t) for t in out]
    call(ref)
    torch.cuda.synchronize()
    errors = []

    def worker():
        try:
            call(out)
        except Exception as e:  # reported on the main thread
            errors.append(e)

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for a, b in zip(out, ref):
        assert torch.equal(a, b)
