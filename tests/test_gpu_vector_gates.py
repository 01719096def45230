"""GPU parity of vector (per key dimension) gates against the fp64 oracle.

With g [B,T,H,Dk] the recurrence is S_t = diag(exp(g_t)) S_{t-1} + k_t v_t^T
and each segment's transition is the diagonal M of the Megatron-Core page's
general summary S_out = M S_in + delta_S.  The six calls run with
rm_cp_problem.vector_gates = 1: on the tensor-core kernels for bf16 with
Dk = Dv = 128 and segment lengths that are multiples of 64 (the cases named
tc below), on the generic fp32-arithmetic kernels otherwise; outputs,
gradients and the forward summaries (M, delta_S, S_in) are compared element
by element with oracle.vg_forward / vg_backward / vg_forward_prepare /
vg_compose_prefix: max|gpu - ref| <= tol * max|ref| per tensor, tol = 1e-4
for fp32 storage and 2e-2 for bf16."""
import math

import numpy as np
import pytest
import torch

import oracle
from state_summary_scan_gb300 import _capi as C
from state_summary_scan_gb300 import api

from _parity import compare, tol_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    C.load()


def vg_inputs(B, T, H, Dk, Dv, dtype, seed=0, shift=3.0, gate=None, qh=0, gmod=None):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, T, qh or H, Dk, generator=gen)
    k = torch.randn(B, T, H, Dk, generator=gen)
    k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn(B, T, H, Dv, generator=gen)
    g = torch.nn.functional.logsigmoid(torch.randn(B, T, H, Dk, generator=gen) + shift)
    if gate is not None:
        g = torch.full((B, T, H, Dk), float(gate))
    if gmod is not None:
        gmod(g)
    dO = torch.randn(B, T, H, Dv, generator=gen)
    return q.to(dtype), k.to(dtype), v.to(dtype), g.contiguous(), dO.to(dtype)


def run_case(B, T, H, Dk, Dv, dtype, nseg, chunk=16, cu=None, qh=0, direct_dg=False, **kw):
    q, k, v, g, dO = vg_inputs(B, T, H, Dk, Dv, dtype, qh=qh, **kw)
    scale = 1.0 / math.sqrt(Dk)
    dev = "cuda"
    qd, kd, vd, gd, dOd = (t.to(dev).contiguous() for t in (q, k, v, g, dO))
    plan = api.make_plan(B, T, H, Dk, Dv, nseg, chunk, scale, dtype, cu, dev, q_heads=qh,
                         vector_gates=True)
    o = api.forward(plan, qd, kd, vd, gd)
    grads = (torch.empty_like(kd), torch.empty_like(kd), torch.empty_like(vd), torch.empty_like(gd))
    dq, dk, dv, dg = api.backward(plan, qd, kd, vd, gd, dOd, grads=grads)
    torch.cuda.synchronize()
    gpu = {n: t.detach().to("cpu", torch.float64).numpy() for n, t in
           dict(o=o, dq=dq, dk=dk, dv=dv, dg=dg, M=plan.M, dS=plan.dS, S_in=plan.S_in).items()}
    si = None
    seg = oracle.equal_segments(T, nseg)
    if cu is not None:
        si = oracle.packed_metadata(cu, T, seg)["seq_idx"]
    qf = q.repeat_interleave(H // qh, dim=2) if qh else q
    ref = dict(o=oracle.vg_forward(qf, k, v, g, scale, si))
    ref.update(zip(("dq", "dk", "dv", "dg"), oracle.vg_backward(qf, k, v, g, dO, scale, si,
                                                               direct=direct_dg)))
    ref["M"], ref["dS"] = oracle.vg_forward_prepare(k, v, g, seg, si)
    # M is an fp32 array: its reference is the fp64 value rounded to fp32
    # (strong decays take a segment's product below fp32's range, to 0)
    ref["M"] = ref["M"].astype(np.float32).astype(np.float64)
    if cu is None:  # with resets the prefixes start at preceding_start (M = 0 makes them agree)
        ref["S_in"] = oracle.vg_compose_prefix(ref["M"], ref["dS"])
    keys = ("o", "dq", "dk", "dv", "dg", "M", "dS") + (("S_in",) if cu is None else ())
    return compare(gpu, ref, tol_for(dtype), keys)


DTYPES = [torch.float32, torch.bfloat16]


@pytest.mark.parametrize("dtype", DTYPES)
def test_vector_gates_small(dtype):
    run_case(1, 256, 2, 32, 32, dtype, nseg=4)


@pytest.mark.parametrize("dtype", DTYPES)
def test_vector_gates_wide_heads(dtype):
    # Dk = 128 and Dv = 256: two column blocks of the column-owner sweeps
    run_case(1, 512, 2, 128, 256, dtype, nseg=4, seed=1)


def test_vector_gates_narrow_values():
    # Dv = 16 < Dk = 64: fewer column owners than key dimensions
    run_case(2, 256, 3, 64, 16, torch.float32, nseg=8, seed=2)


@pytest.mark.parametrize("dtype", DTYPES)
def test_vector_gates_packed_resets(dtype):
    cu = [0, 1, 2, 17, 31, 64, 65, 200, 255, 256]
    run_case(1, 256, 2, 32, 32, dtype, nseg=4, cu=cu, seed=3)


def test_vector_gates_strong_decay():
    """alpha = e^-30 in every dimension: dg (~1e-13) is compared with the
    oracle's direct form alpha_t[i] <S_{t-1}[i,:], D_t[i,:]>."""
    run_case(1, 128, 2, 16, 16, torch.float32, nseg=4, gate=-30.0, direct_dg=True)


def test_vector_gates_shared_queries():
    run_case(1, 256, 4, 32, 32, torch.float32, nseg=4, qh=2, seed=4)


def test_vector_gates_autograd():
    """chunkwise_gla takes a [B,T,H,Dk] gate as vector gates."""
    q, k, v, g, dO = vg_inputs(1, 128, 2, 32, 16, torch.float32, seed=5)
    qd, kd, vd, gd = (t.cuda().requires_grad_() for t in (q, k, v, g))
    o = api.chunkwise_gla(qd, kd, vd, gd, 4, 16, 0.2)
    o.backward(dO.cuda())
    torch.cuda.synchronize()
    ref_o = oracle.vg_forward(q, k, v, g, 0.2)
    ref = oracle.vg_backward(q, k, v, g, dO, 0.2)
    for a, b in zip((o, qd.grad, kd.grad, vd.grad, gd.grad), (ref_o,) + tuple(ref)):
        a = a.detach().double().cpu().numpy()
        assert np.max(np.abs(a - b)) <= 1e-4 * np.max(np.abs(b))


# ------------------------------------------------------------ tensor-core path
# bf16, Dk = Dv = 128, 64-token chunks.  A chunk is factored (its decays
# folded into the operand tiles) when no sequence starts inside it and every
# |b_t[i] - b_63[i]| < 60; other chunks take their intra-chunk terms directly.

TC = dict(Dk=128, Dv=128, dtype=torch.bfloat16, chunk=64)


def test_vector_gates_tc_path_selected():
    spec = C.ProblemSpec(1, 1024, 2, 128, 128, 4, 64, 1 / math.sqrt(128), torch.bfloat16,
                         vector_gates=1)
    assert C.rm_cp_path(spec) == 1


@pytest.mark.parametrize("B,T,H,nseg,shift,seed", [
    (1, 1024, 2, 4, 3.0, 10),   # moderate decays: factored chunks (the first starts the row)
    (2, 768, 3, 3, 4.0, 11),    # two rows, three heads, three chunks a segment
    (1, 512, 2, 2, -1.0, 12),   # strong decays: every chunk's range exceeds 60, all direct
    (1, 256, 1, 4, 3.0, 13),    # one chunk a segment
])
def test_vector_gates_tc(B, T, H, nseg, shift, seed):
    run_case(B, T, H, nseg=nseg, seed=seed, shift=shift, **TC)


def _strong_chunks(g):
    # chunks 1 and 4 of every 256 tokens decay fast in 16 dimensions: those
    # chunks are taken directly, their neighbours factored
    for c0 in range(0, g.shape[1], 256):
        for c in (1, 4):
            a = c0 + 64 * c
            if a < g.shape[1]:
                g[:, a:a + 64, :, 40:56] = -2.5


def test_vector_gates_tc_mixed_chunks():
    run_case(1, 1024, 2, nseg=2, seed=14, gmod=_strong_chunks, **TC)


def test_vector_gates_tc_packed_resets():
    # starts at chunk boundaries (64, 512), inside chunks (100, 300, 301, 700)
    # and at the last token (1023)
    cu = [0, 64, 100, 300, 301, 512, 700, 1023, 1024]
    run_case(1, 1024, 2, nseg=4, cu=cu, seed=15, **TC)


def test_vector_gates_tc_shared_queries():
    run_case(1, 512, 4, nseg=2, qh=2, seed=16, **TC)


def test_vector_gates_tc_full_size_sampled_heads():
    """vg32k (T = 32768, 16 heads, 16 segments; 256 CTAs, more than the SMs)
    on the GPU; two heads against the oracle (heads are independent)."""
    from state_summary_scan_gb300.workloads import WORKLOADS, make_inputs
    w = WORKLOADS["vg32k"]
    inp = make_inputs(w)
    dev = "cuda"
    qd, kd, vd, gd, dOd = (t.to(dev).contiguous() for t in (inp.q, inp.k, inp.v, inp.g, inp.dO))
    plan = api.make_plan(w.B, w.T, w.H, w.Dk, w.Dv, w.num_segments, w.chunk, w.scale, w.torch_dtype,
                         None, dev, vector_gates=True)
    assert C.rm_cp_path(plan.spec) == 1
    o = api.forward(plan, qd, kd, vd, gd)
    dq, dk, dv, dg = api.backward(plan, qd, kd, vd, gd, dOd)
    torch.cuda.synchronize()
    heads = [0, 11]
    sl = lambda t: t[:, :, heads].contiguous()
    gpu = {n: sl(t).detach().to("cpu", torch.float64).numpy()
           for n, t in dict(o=o, dq=dq, dk=dk, dv=dv, dg=dg).items()}
    for n, t in dict(M=plan.M, dS=plan.dS, S_in=plan.S_in).items():
        gpu[n] = t[:, :, heads].detach().to("cpu", torch.float64).numpy()
    q, k, v, g, dO = (sl(t) for t in (inp.q, inp.k, inp.v, inp.g, inp.dO))
    ref = dict(o=oracle.vg_forward(q, k, v, g, w.scale))
    ref.update(zip(("dq", "dk", "dv", "dg"), oracle.vg_backward(q, k, v, g, dO, w.scale)))
    seg = oracle.equal_segments(w.T, w.num_segments)
    ref["M"], ref["dS"] = oracle.vg_forward_prepare(k, v, g, seg)
    ref["S_in"] = oracle.vg_compose_prefix(ref["M"], ref["dS"])
    compare(gpu, ref, tol_for(w.torch_dtype), ("o", "dq", "dk", "dv", "dg", "M", "dS", "S_in"))


def test_vector_gates_tc_wide_grid():
    """More (segment, head) CTAs than SMs (the forward then runs two CTAs a SM),
    with sequence starts inside chunks and chunks of strong decay."""
    cu = [0, 100, 1024, 1500, 2048, 2049, 3000, 4096]
    run_case(1, 4096, 40, nseg=4, cu=cu, seed=17, gmod=_strong_chunks, **TC)


def test_vector_gates_tc_step_host_pipeline():
    """rm_cp_step_host with vector gates (g and dg [B,T,H,Dk] copied in and
    out): two steps from pinned host buffers equal the device-buffer calls
    bit for bit (same kernels, same order)."""
    B, T, H, D, nseg = 1, 512, 2, 128, 4
    scale = 1.0 / math.sqrt(D)
    q, k, v, g, dO = vg_inputs(B, T, H, D, D, torch.bfloat16, seed=18)
    dev = "cuda"
    qd, kd, vd, gd, dOd = (t.to(dev).contiguous() for t in (q, k, v, g, dO))
    pd = api.make_plan(B, T, H, D, D, nseg, 64, scale, torch.bfloat16, None, dev, vector_gates=True)
    o = api.forward(pd, qd, kd, vd, gd)
    dq, dk, dv, dg = api.backward(pd, qd, kd, vd, gd, dOd)
    torch.cuda.synchronize()
    ref = {n: t.cpu() for n, t in dict(o=o, dq=dq, dk=dk, dv=dv, dg=dg).items()}
    host = {n: t.contiguous().pin_memory() for n, t in (("q", q), ("k", k), ("v", v), ("g", g), ("dO", dO))}
    plan = api.make_plan(B, T, H, D, D, nseg, 64, scale, torch.bfloat16, None, dev, vector_gates=True)
    outs = [{n: torch.full(t.shape, 7.0, dtype=t.dtype).pin_memory() for n, t in ref.items()} for _ in range(2)]
    pipe = api.HostPipeline(plan, dict(host, **outs[0]))
    pipe.begin()
    for i in range(2):
        pipe.host = dict(host, **outs[i])
        pipe.step()
    pipe.join()
    torch.cuda.synchronize()
    pipe.close()
    for i in range(2):
        for n in ref:
            assert torch.equal(outs[i][n], ref[n]), (i, n)


@pytest.mark.parametrize("seed", range(6))
def test_vector_gates_tc_random_shapes(seed):
    """Seeded random problems on the tensor-core path: rows, heads, segment
    count and length (multiples of 64), packed sequences (one row) with
    starts anywhere, shared query rows, gate shifts from strong to weak decay
    (so that factored and directly taken chunks mix)."""
    rng = np.random.default_rng(300 + seed)
    nseg = int(rng.choice([1, 2, 4]))
    L = 64 * int(rng.integers(1, 4))
    T = nseg * L
    packed = bool(rng.integers(0, 2))
    B = 1 if packed else int(rng.integers(1, 3))
    H = int(rng.choice([1, 2, 4]))
    qh = int(rng.choice([0, 1])) if H > 1 else 0
    cu = None
    if packed:
        cuts = sorted(set(int(x) for x in rng.integers(1, T, size=int(rng.integers(1, 6)))))
        cu = [0] + cuts + [T]
    run_case(B, T, H, nseg=nseg, cu=cu, qh=qh, seed=400 + seed, shift=float(rng.uniform(-1.0, 4.0)), **TC)
