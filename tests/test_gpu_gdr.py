"""GPU parity of the gated delta rule against the fp64 oracle.

S_t = exp(g_t)(I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T, o_t = scale
S_t^T q_t, run through the rm_gdr_* calls: each segment's summary is the
general affine map S_out = M S_in + delta_S of the Megatron-Core page with a
Dk x Dk transition M, composed as M S + dS forward and M^T D + gamma
backward.  Outputs, gradients (q, k, v, g, beta) and the forward summaries
(M, delta_S, S_in) are compared element by element with oracle.gdr_forward /
gdr_backward / gdr_forward_prepare / gdr_compose_prefix: max|gpu - ref| <=
tol * max|ref| per tensor, tol = 1e-4 for fp32 storage and 2e-2 for bf16."""
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


def gdr_inputs(B, T, H, Dk, Dv, dtype, seed=0, qh=0, gshift=3.0, bshift=0.0):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, T, qh or H, Dk, generator=gen)
    k = torch.randn(B, T, H, Dk, generator=gen)
    k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn(B, T, H, Dv, generator=gen)
    g = torch.nn.functional.logsigmoid(torch.randn(B, T, H, generator=gen) + gshift)
    beta = torch.sigmoid(torch.randn(B, T, H, generator=gen) + bshift)
    dO = torch.randn(B, T, H, Dv, generator=gen)
    return q.to(dtype), k.to(dtype), v.to(dtype), g, beta, dO.to(dtype)


def run_case(B, T, H, Dk, Dv, dtype, nseg, cu=None, qh=0, seed=0, gshift=3.0, bshift=0.0):
    q, k, v, g, beta, dO = gdr_inputs(B, T, H, Dk, Dv, dtype, seed, qh, gshift, bshift)
    scale = 1.0 / math.sqrt(Dk)
    dev = "cuda"
    qd, kd, vd, gd, bd, dOd = (t.to(dev).contiguous() for t in (q, k, v, g, beta, dO))
    plan = api.make_gdr_plan(B, T, H, Dk, Dv, nseg, 16, scale, dtype, cu, dev, q_heads=qh)
    o = api.gdr_forward(plan, qd, kd, vd, gd, bd)
    grads = api.gdr_backward(plan, qd, kd, vd, gd, bd, dOd)
    torch.cuda.synchronize()
    gpu = {n: t.detach().to("cpu", torch.float64).numpy() for n, t in
           zip(("o", "dq", "dk", "dv", "dg", "dbeta", "M", "dS", "S_in"),
               (o,) + tuple(grads) + (plan.M, plan.dS, plan.S_in))}
    seg = oracle.equal_segments(T, nseg)
    si = None
    if cu is not None:
        si = oracle.packed_metadata(cu, T, seg)["seq_idx"]
    qf = q.repeat_interleave(H // qh, dim=2) if qh else q
    ref = dict(o=oracle.gdr_forward(qf, k, v, g, beta, scale, si))
    ref.update(zip(("dq", "dk", "dv", "dg", "dbeta"), oracle.gdr_backward(qf, k, v, g, beta, dO, scale, si)))
    ref["M"], ref["dS"] = oracle.gdr_forward_prepare(k, v, g, beta, seg, si)
    # M is stored in fp32: under strong decay its entries fall below fp32's
    # range, so the fp64 reference is rounded to the storage type first
    ref["M"] = np.asarray(ref["M"], np.float32).astype(np.float64)
    keys = ("o", "dq", "dk", "dv", "dg", "dbeta", "M", "dS")
    if cu is None:  # with resets the prefixes start at preceding_start (M = 0 makes them agree)
        ref["S_in"] = oracle.gdr_compose_prefix(ref["M"], ref["dS"])
        keys += ("S_in",)
    return compare(gpu, ref, tol_for(dtype), keys)


def test_gdr_small_fp32():
    run_case(1, 128, 2, 16, 16, torch.float32, nseg=4)


def test_gdr_rectangular_heads_many_blocks():
    # Dv != Dk, 64-token segments (four saved states each), two rows
    run_case(2, 256, 2, 32, 48, torch.float32, nseg=4, seed=1)


def test_gdr_packed_resets():
    cu = [0, 1, 2, 17, 31, 64, 65, 100, 127, 128]
    run_case(1, 128, 2, 16, 16, torch.float32, nseg=4, cu=cu, seed=2)


def test_gdr_single_segment_and_shared_queries():
    run_case(1, 64, 4, 16, 16, torch.float32, nseg=1, qh=2, seed=3)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_gdr_wide(dtype):
    run_case(1, 256, 2, 64, 64, dtype, nseg=4, seed=4)


@pytest.mark.parametrize("dtype,Dv", [(torch.float32, 128), (torch.bfloat16, 64)])
def test_gdr_dk128(dtype, Dv):
    # Dk = 128 on the generic kernels: the fold splits a state row over two
    # lanes, the reverse sweep rebuilds one state at a time (Dv = 128)
    run_case(1, 256, 2, 128, Dv, dtype, nseg=4, seed=14)


def test_gdr_dk128_packed_shared_queries():
    cu = [0, 40, 41, 130, 256]
    run_case(1, 256, 4, 128, 32, torch.float32, nseg=8, cu=cu, qh=2, seed=15)


def test_gdr_rejects_unsupported_shapes():
    bad = C.ProblemSpec(1, 128, 2, 48, 16, 4, 16, 0.1, torch.float32)  # Dk = 48
    t = torch.zeros(16, device="cuda")
    with pytest.raises(C.RmCpError) as e:
        C.rm_gdr_forward_prepare(bad, t, t, t, t, t, t, t)
    assert e.value.status == 4


# ------------------------------------------------------------ tensor-core sweeps
# bf16, Dk = Dv = 64, segment lengths that are multiples of 64: the forward's
# prepare and apply and the backward's prepare (dq walk and gamma walk) and
# apply run the chunkwise WY/UT form on the tensor cores; the two folds stay
# on the generic kernels.  Measured errors on these cases are 2e-3 .. 7e-3 of
# max|ref| for every tensor.

def test_gdr_tc_several_chunks():
    run_case(2, 1024, 3, 64, 64, torch.bfloat16, nseg=4, seed=5)


def test_gdr_tc_packed_resets():
    # starts at chunk boundaries (64, 512), inside chunks (100, 300, 301, 700)
    # and at the last token (1023)
    cu = [0, 64, 100, 300, 301, 512, 700, 1023, 1024]
    run_case(1, 1024, 2, 64, 64, torch.bfloat16, nseg=4, cu=cu, seed=6)


def test_gdr_tc_shared_queries():
    run_case(1, 512, 4, 64, 64, torch.bfloat16, nseg=2, qh=2, seed=7)


def test_gdr_tc_one_long_segment():
    # 32 chunks walked by one CTA each way; gamma of the only segment is unused
    run_case(1, 2048, 2, 64, 64, torch.bfloat16, nseg=1, seed=8)


def test_gdr_tc_strong_decay_saturated_writes():
    # alpha ~ 0.3 (the in-chunk decays reach e^-80) and beta ~ 0.95: the
    # triangular inverse far from the identity, decays far below fp32's range
    run_case(1, 512, 2, 64, 64, torch.bfloat16, nseg=4, seed=9, gshift=-1.0, bshift=3.0)


def test_gdr_tc_many_segments_long_sequences():
    # 32 segments of 64 tokens; sequences spanning up to 20 segments, so the
    # folds start far back (preceding_start, following_stop) and restart
    # their chains several times, in both directions
    cu = [0, 5, 1300, 1301, 1990, 2048]
    run_case(1, 2048, 2, 64, 64, torch.bfloat16, nseg=32, cu=cu, seed=12)


def test_gdr_many_segments_generic():
    # the same on the generic kernels (fp32, Dk = 32, Dv = 24): 64 segments of 16
    cu = [0, 300, 301, 700, 1024]
    run_case(1, 1024, 2, 32, 24, torch.float32, nseg=64, cu=cu, seed=13)


def test_gdr_tc_weak_writes():
    # beta ~ 0.05: T = (I + A)^{-1} diag(beta) near 0, dbeta from dZ . X
    run_case(1, 512, 2, 64, 64, torch.bfloat16, nseg=2, seed=10, bshift=-3.0)


def test_gdr_tc_full_size_sampled_heads():
    """gdr8k (T = 8192, 16 heads, 16 segments; 256 CTAs) on the GPU; two
    heads against the oracle (heads are independent)."""
    from state_summary_scan_gb300.workloads import GDR_WORKLOADS, make_gdr_inputs
    w = GDR_WORKLOADS["gdr8k"]
    inp = make_gdr_inputs(w)
    dev = "cuda"
    qd, kd, vd, gd, bd, dOd = (t.to(dev).contiguous() for t in (inp.q, inp.k, inp.v, inp.g, inp.beta, inp.dO))
    plan = api.make_gdr_plan(w.B, w.T, w.H, w.Dk, w.Dv, w.num_segments, w.chunk, w.scale, w.torch_dtype,
                             None, dev)
    o = api.gdr_forward(plan, qd, kd, vd, gd, bd)
    grads = api.gdr_backward(plan, qd, kd, vd, gd, bd, dOd)
    torch.cuda.synchronize()
    heads = [0, 9]
    sl = lambda t: t[:, :, heads].contiguous()
    gpu = {n: sl(t).detach().to("cpu", torch.float64).numpy()
           for n, t in zip(("o", "dq", "dk", "dv", "dg", "dbeta"), (o,) + tuple(grads))}
    for n, t in dict(M=plan.M, dS=plan.dS, S_in=plan.S_in).items():
        gpu[n] = t[:, :, heads].detach().to("cpu", torch.float64).numpy()
    q, k, v, g, beta, dO = (sl(t) for t in (inp.q, inp.k, inp.v, inp.g, inp.beta, inp.dO))
    ref = dict(o=oracle.gdr_forward(q, k, v, g, beta, w.scale))
    ref.update(zip(("dq", "dk", "dv", "dg", "dbeta"), oracle.gdr_backward(q, k, v, g, beta, dO, w.scale)))
    seg = oracle.equal_segments(w.T, w.num_segments)
    ref["M"], ref["dS"] = oracle.gdr_forward_prepare(k, v, g, beta, seg)
    ref["S_in"] = oracle.gdr_compose_prefix(ref["M"], ref["dS"])
    compare(gpu, ref, tol_for(w.torch_dtype), ("o", "dq", "dk", "dv", "dg", "dbeta", "M", "dS", "S_in"))


@pytest.mark.parametrize("seed", range(6))
def test_gdr_tc_random_shapes(seed):
    """Seeded random problems on the tensor-core sweeps: rows, heads, segment
    count and length (multiples of 64), packed sequences (one row) with
    starts anywhere, shared query rows, gate and write-strength shifts."""
    rng = np.random.default_rng(100 + seed)
    nseg = int(rng.choice([1, 2, 4, 8]))
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
    run_case(B, T, H, 64, 64, torch.bfloat16, nseg=nseg, cu=cu, qh=qh, seed=200 + seed,
             gshift=float(rng.uniform(-1.0, 4.0)), bshift=float(rng.uniform(-2.0, 2.0)))


@pytest.mark.parametrize("case", ["tc", "generic_packed"])
def test_gated_delta_rule_autograd_equals_direct_calls(case):
    """torch.autograd through gated_delta_rule gives the direct calls' o and
    gradients bit for bit (same kernels, same order), on the tensor-core
    sweeps and on the generic kernels with packed sequences."""
    if case == "tc":
        B, T, H, Dk, Dv, dtype, nseg, cu = 2, 512, 2, 64, 64, torch.bfloat16, 4, None
    else:
        B, T, H, Dk, Dv, dtype, nseg, cu = 1, 256, 2, 32, 48, torch.float32, 8, [0, 40, 41, 200, 256]
    q, k, v, g, beta, dO = (t.to("cuda").contiguous()
                            for t in gdr_inputs(B, T, H, Dk, Dv, dtype, seed=21))
    scale = 1.0 / math.sqrt(Dk)
    plan = api.make_gdr_plan(B, T, H, Dk, Dv, nseg, 16, scale, dtype, cu, "cuda")
    o_ref = api.gdr_forward(plan, q, k, v, g, beta)
    g_ref = api.gdr_backward(plan, q, k, v, g, beta, dO)
    leaves = [t.clone().requires_grad_(True) for t in (q, k, v, g, beta)]
    o = api.gated_delta_rule(*leaves, nseg, 16, scale, cu)
    o.backward(dO)
    torch.cuda.synchronize()
    assert torch.equal(o.detach(), o_ref)
    for name, leaf, ref in zip(("dq", "dk", "dv", "dg", "dbeta"), leaves, g_ref):
        assert leaf.grad.dtype == leaf.dtype, name
        assert torch.equal(leaf.grad, ref), name


@pytest.mark.parametrize("seed", range(6))
def test_gdr_generic_random_shapes(seed):
    """Seeded random problems on the generic kernels: Dk in {16, 32, 64, 128},
    Dv a multiple of 8 up to 128, fp32 or bf16 storage (bf16 with Dk = Dv =
    64 and 64-token segments would take the tensor cores, so those pick
    16-token segments), segment lengths multiples of 16, packed sequences with
    starts anywhere, shared query rows, gate and write-strength shifts."""
    rng = np.random.default_rng(300 + seed)
    Dk = int(rng.choice([16, 32, 64, 128]))
    Dv = 8 * int(rng.integers(1, 17))
    dtype = torch.float32 if rng.integers(0, 2) else torch.bfloat16
    nseg = int(rng.choice([1, 2, 4, 8]))
    L = 16 * int(rng.integers(1, 5))
    if L % 64 == 0:
        L += 16
    T = nseg * L
    packed = bool(rng.integers(0, 2))
    B = 1 if packed else int(rng.integers(1, 3))
    H = int(rng.choice([1, 2, 4]))
    qh = int(rng.choice([0, 1])) if H > 1 else 0
    cu = None
    if packed:
        cuts = sorted(set(int(x) for x in rng.integers(1, T, size=int(rng.integers(1, 6)))))
        cu = [0] + cuts + [T]
    run_case(B, T, H, Dk, Dv, dtype, nseg=nseg, cu=cu, qh=qh, seed=400 + seed,
             gshift=float(rng.uniform(-1.0, 4.0)), bshift=float(rng.uniform(-2.0, 2.0)))
