"""GPU parity: the CUDA path, called through the C ABI, against the fp64
oracle on the same seeded inputs.  Outputs, gradients and the segment
summaries (M, delta_S, S_in, gamma, dS_out) are compared element by element:
max|gpu - ref| <= tol * max|ref| per tensor, tol = 1e-4 for fp32 storage and
2e-2 for bf16 storage (fp32 accumulation in both)."""
import math

import numpy as np
import pytest
import torch

from state_summary_scan_gb300 import _capi as C
from state_summary_scan_gb300.workloads import WORKLOADS, make_inputs, random_cu_seqlens

from _parity import (GRAD_KEYS, SUMMARY_KEYS_BWD, SUMMARY_KEYS_FWD, compare, run_gpu,
                     run_oracle, select_heads, tol_for)

pytestmark = pytest.mark.gpu

ALL_KEYS = ("o",) + SUMMARY_KEYS_FWD + GRAD_KEYS + SUMMARY_KEYS_BWD


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    C.load()


def check_workload(name, heads=None, backward=None):
    w = WORKLOADS[name]
    if backward is None:
        backward = w.backward
    inp = make_inputs(w, with_grad=backward)
    gpu = run_gpu(inp.q, inp.k, inp.v, inp.g, inp.dO if backward else None, w.num_segments,
                  w.chunk, w.scale, inp.cu_seqlens)
    ref = run_oracle(inp.q, inp.k, inp.v, inp.g, inp.dO if backward else None, w.num_segments,
                     w.scale, inp.cu_seqlens, heads)
    keys = ALL_KEYS if backward else ("o",) + SUMMARY_KEYS_FWD
    return compare(select_heads(gpu, heads), ref, tol_for(w.torch_dtype), keys)


def test_tiny_fp32_full():
    check_workload("tiny")


def test_fwd4k_bf16_full():
    check_workload("fwd4k")


def test_32k_bf16_sampled_heads():
    check_workload("32k", heads=[0, 15])


def test_packed64k_bf16_sampled_heads():
    check_workload("packed64k", heads=[0, 31])


def test_256k_bf16_sampled_heads():
    check_workload("256k", heads=[7])


# ------------------------------------------------------------------ edge cases

def synth(B, T, H, Dk, Dv, dtype, seed=0, gate_shift=3.0, gate=None):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, T, H, Dk, generator=gen)
    k = torch.randn(B, T, H, Dk, generator=gen)
    k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn(B, T, H, Dv, generator=gen)
    g = torch.nn.functional.logsigmoid(torch.randn(B, T, H, generator=gen) + gate_shift)
    if gate is not None:
        g = torch.full((B, T, H), float(gate))
    dO = torch.randn(B, T, H, Dv, generator=gen)
    return q.to(dtype), k.to(dtype), v.to(dtype), g.contiguous(), dO.to(dtype)


def check_case(B, T, H, Dk, Dv, dtype, nseg, chunk=16, cu=None, use_metadata=True, fused=False, **kw):
    q, k, v, g, dO = synth(B, T, H, Dk, Dv, dtype, **kw)
    scale = 1.0 / math.sqrt(Dk)
    gpu = run_gpu(q, k, v, g, dO, nseg, chunk, scale, cu, use_metadata=use_metadata, fused=fused)
    ref = run_oracle(q, k, v, g, dO, nseg, scale, cu)
    keys = ALL_KEYS if use_metadata else ("o",) + GRAD_KEYS
    return compare(select_heads(gpu, None), ref, tol_for(dtype), keys)


DTYPES = [torch.float32, torch.bfloat16]


@pytest.mark.parametrize("dtype", DTYPES)
def test_single_segment(dtype):
    check_case(1, 256, 2, 64, 64, dtype, nseg=1)


@pytest.mark.parametrize("dtype", DTYPES)
def test_many_short_segments(dtype):
    check_case(2, 512, 2, 32, 48, dtype, nseg=32)


@pytest.mark.parametrize("dtype", DTYPES)
def test_min_and_odd_head_dims(dtype):
    check_case(1, 128, 3, 16, 8, dtype, nseg=2)
    check_case(1, 128, 1, 64, 200, dtype, nseg=4)


@pytest.mark.parametrize("dtype", DTYPES)
def test_max_head_dims(dtype):
    check_case(1, 512, 2, 128, 256, dtype, nseg=4)


@pytest.mark.parametrize("dtype", DTYPES)
def test_packed_ragged_resets(dtype):
    # resets at a segment start (64), at tile positions 1 and 15, length-1
    # sequences, and a sequence spanning three segments
    cu = [0, 1, 2, 17, 31, 64, 65, 200, 255, 256]
    check_case(1, 256, 2, 32, 32, dtype, nseg=4, cu=cu)


@pytest.mark.parametrize("dtype", DTYPES)
def test_packed_without_metadata_ranges(dtype):
    cu = [0, 5, 90, 91, 256]
    check_case(1, 256, 2, 32, 32, dtype, nseg=8, cu=cu, use_metadata=False)


def test_every_token_starts_a_sequence():
    cu = list(range(0, 129))
    check_case(1, 128, 2, 32, 32, torch.float32, nseg=4, cu=cu)


def test_random_packings():
    gen = torch.Generator().manual_seed(99)
    for trial in range(6):
        T = 256
        cu = random_cu_seqlens(gen, T, max_len=int(torch.randint(1, 300, (1,), generator=gen)))
        check_case(1, T, 2, 32, 32, torch.float32, nseg=int([1, 2, 4, 8, 16][trial % 5]),
                   cu=cu.tolist(), seed=trial)


def test_zero_gate():
    check_case(1, 256, 2, 32, 32, torch.float32, nseg=4, gate=0.0)


@pytest.mark.parametrize("dtype", DTYPES)
def test_strong_decay(dtype):
    """alpha = e^-30: M underflows to 0 and dg is ~1e-13, far below the terms
    of the cumsum identity; dg is compared with the oracle's direct form
    alpha_t <S_{t-1}, D_t>, which forms it without cancellation."""
    import oracle
    B, T, H, D = 1, 256, 2, 32
    q, k, v, g, dO = synth(B, T, H, D, D, dtype, gate=-30.0)
    scale = 1.0 / math.sqrt(D)
    gpu = run_gpu(q, k, v, g, dO, 4, 16, scale)
    ref = run_oracle(q, k, v, g, dO, 4, scale)
    compare(select_heads(gpu, None), ref, tol_for(dtype), ("o", "M", "dS", "S_in", "dq", "dk", "dv"))
    ref["dg"] = oracle.backward(q, k, v, g, dO, scale, direct=True)[3]
    compare(select_heads(gpu, None), ref, tol_for(dtype), ("dg",))


def test_deterministic():
    q, k, v, g, dO = synth(1, 512, 4, 128, 128, torch.bfloat16, seed=3)
    a = run_gpu(q, k, v, g, dO, 4, 64, 0.1)
    b = run_gpu(q, k, v, g, dO, 4, 64, 0.1)
    for key in a:
        assert torch.equal(a[key], b[key]), key


# ------------------------------------------------------------------ tensor-core path

def test_workloads_take_the_tensor_core_path():
    from state_summary_scan_gb300 import _capi as C
    for name, expect in (("fwd4k", 1), ("32k", 1), ("packed64k", 1), ("256k", 1), ("tiny", 0)):
        w = WORKLOADS[name]
        s = C.ProblemSpec(w.B, w.T, w.H, w.Dk, w.Dv, w.num_segments, w.chunk, w.scale,
                          w.torch_dtype)
        assert C.rm_cp_path(s) == expect, name


@pytest.mark.parametrize("Dv", [128, 256])
def test_tc_single_and_many_segments(Dv):
    check_case(1, 512, 2, 128, Dv, torch.bfloat16, nseg=1, chunk=64)
    check_case(2, 512, 2, 128, Dv, torch.bfloat16, nseg=8, chunk=64)


@pytest.mark.parametrize("Dv", [128, 256])
def test_tc_packed_ragged_resets(Dv):
    # starts at chunk positions 0, 1, 63, a segment start (256), length-1
    # sequences, and a sequence across three segments
    cu = [0, 1, 2, 63, 64, 65, 129, 256, 257, 300, 511, 512, 700, 1024]
    check_case(1, 1024, 2, 128, Dv, torch.bfloat16, nseg=4, chunk=64, cu=cu)


def test_tc_every_token_starts_a_sequence():
    cu = list(range(0, 257))
    check_case(1, 256, 2, 128, 128, torch.bfloat16, nseg=2, chunk=64, cu=cu)


def test_tc_zero_gate():
    check_case(1, 512, 2, 128, 128, torch.bfloat16, nseg=4, chunk=64, gate=0.0)


def test_tc_strong_decay():
    import oracle
    q, k, v, g, dO = synth(1, 256, 2, 128, 128, torch.bfloat16, gate=-30.0)
    scale = 1.0 / math.sqrt(128)
    gpu = run_gpu(q, k, v, g, dO, 2, 64, scale)
    ref = run_oracle(q, k, v, g, dO, 2, scale)
    compare(select_heads(gpu, None), ref, 2e-2, ("o", "M", "dS", "S_in", "dq", "dk", "dv"))
    ref["dg"] = oracle.backward(q, k, v, g, dO, scale, direct=True)[3]
    compare(select_heads(gpu, None), ref, 2e-2, ("dg",))


# ------------------------------------------------------------------ wide grids
# More CTAs than SMs select the forward sweep that runs two CTAs a SM; these
# cases put 16 x 16 = 256 (segment, head) sweeps on the GPU with the chunk
# kinds that take its general path (sequence starts, strong decay).

def test_tc_wide_grid_packed_resets():
    T = 2048
    cu = [0, 1, 100, 128, 129, 700, 1024, 1025, 1500, 1999, 2048]
    check_case(1, T, 16, 128, 128, torch.bfloat16, nseg=16, chunk=64, cu=cu)


def test_tc_wide_grid_strong_decay():
    import oracle
    q, k, v, g, dO = synth(1, 2048, 16, 128, 128, torch.bfloat16, gate=-30.0)
    scale = 1.0 / math.sqrt(128)
    gpu = run_gpu(q, k, v, g, dO, 16, 64, scale)
    ref = run_oracle(q, k, v, g, dO, 16, scale)
    compare(select_heads(gpu, None), ref, 2e-2, ("o", "M", "dS", "S_in", "dq", "dk", "dv"))
    ref["dg"] = oracle.backward(q, k, v, g, dO, scale, direct=True)[3]
    compare(select_heads(gpu, None), ref, 2e-2, ("dg",))


def test_tc_wide_grid_value_blocks():
    # Dv = 256: two value blocks per (segment, head) -> 512 forward CTAs
    check_case(1, 1024, 16, 128, 256, torch.bfloat16, nseg=16, chunk=64, seed=5)


@pytest.mark.parametrize("seed", range(6))
def test_tc_random_shapes(seed):
    """Seeded random problems on the tensor-core sweeps: rows, heads, Dv in
    {128, 256}, segment count (not only powers of two) and length (multiples
    of 64), packed sequences (one row) with starts anywhere, and gate shifts
    from strong to weak decay (the wide-grid cases above cover more CTAs than
    SMs)."""
    rng = np.random.default_rng(500 + seed)
    nseg = int(rng.choice([1, 2, 3, 4, 8]))
    L = 64 * int(rng.integers(1, 5))
    T = nseg * L
    packed = bool(rng.integers(0, 2))
    B = 1 if packed else int(rng.integers(1, 3))
    H = int(rng.choice([1, 2, 4, 8, 16]))
    Dv = int(rng.choice([128, 256]))
    cu = None
    if packed:
        cuts = sorted(set(int(x) for x in rng.integers(1, T, size=int(rng.integers(1, 7)))))
        cu = [0] + cuts + [T]
    check_case(B, T, H, 128, Dv, torch.bfloat16, nseg=nseg, chunk=64, cu=cu, seed=600 + seed,
               gate_shift=float(rng.uniform(-1.0, 5.0)))


# ------------------------------------------------------------------ from host memory

@pytest.mark.parametrize("backward", [True, False])
def test_step_host_pipeline_matches_device_path(backward):
    """rm_cp_step_host on pinned host buffers, three steps on two alternating
    device sets: every step's host results equal those of the device-buffer
    calls bit for bit (same kernels, same order), and the oracle to tolerance."""
    from state_summary_scan_gb300 import api
    B, T, H, D, nseg = 1, 512, 2, 128, 4
    q, k, v, g, dO = synth(B, T, H, D, D, torch.bfloat16, seed=7)
    scale = 1.0 / math.sqrt(D)
    ref_dev = run_gpu(q, k, v, g, dO if backward else None, nseg, 64, scale)
    host = {n: t.contiguous().pin_memory() for n, t in
            (("q", q), ("k", k), ("v", v), ("g", g)) + ((("dO", dO),) if backward else ())}
    outs = {"o": v} if not backward else {"o": v, "dq": q, "dk": k, "dv": v, "dg": g}
    results = []
    plan = api.make_plan(B, T, H, D, D, nseg, 64, scale, torch.bfloat16, backward=backward)
    outs_host = []
    for _ in range(3):
        outs_host.append({n: torch.full(t.shape, 7.0, dtype=t.dtype).pin_memory()
                          for n, t in outs.items()})
    pipe = api.HostPipeline(plan, dict(host, **outs_host[0]))
    pipe.begin()
    for i in range(3):
        pipe.host = dict(host, **outs_host[i])  # each step into its own host outputs
        pipe.step()
    pipe.join()
    torch.cuda.synchronize()
    pipe.close()
    for i in range(3):
        for n in outs:
            got = outs_host[i][n].to(torch.float64)
            assert torch.equal(got, ref_dev[n]), (i, n)
        results.append({n: outs_host[i][n].to(torch.float64).numpy() for n in outs})
    ref = run_oracle(q, k, v, g, dO if backward else None, nseg, scale)
    compare(results[-1], ref, 2e-2, tuple(outs))


# ------------------------------------------------------------------ shared queries

@pytest.mark.parametrize("dtype,Dk,Dv,chunk", [(torch.bfloat16, 128, 128, 64),
                                               (torch.bfloat16, 128, 256, 64),
                                               (torch.float32, 32, 16, 16)])
def test_shared_queries(dtype, Dk, Dv, chunk):
    """q_heads = 2 of H = 4: heads 0, 1 read query row 0 and heads 2, 3 row 1;
    the oracle sees the same queries repeated per head.  dq stays per head."""
    shared_queries_case(dtype, Dk, Dv, chunk, 1, 512, 4, 2, 4)


@pytest.mark.parametrize("qh,Dv", [(1, 128), (2, 128), (2, 256)])
def test_shared_queries_wide_grid(qh, Dv):
    """16 segments x 16 heads = 256 (segment, head) sweeps (512 forward CTAs at
    Dv = 256), more than the SMs: the forward sweep that runs two CTAs a SM
    reads query row h / (H / q_heads), as a Mamba2 group's heads read C."""
    shared_queries_case(torch.bfloat16, 128, Dv, 64, 1, 2048, 16, qh, 16)


def shared_queries_case(dtype, Dk, Dv, chunk, B, T, H, qh, nseg):
    from state_summary_scan_gb300 import api
    gen = torch.Generator().manual_seed(21)
    q = torch.randn(B, T, qh, Dk, generator=gen)
    k = torch.randn(B, T, H, Dk, generator=gen)
    k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn(B, T, H, Dv, generator=gen)
    g = torch.nn.functional.logsigmoid(torch.randn(B, T, H, generator=gen) + 3.0)
    dO = torch.randn(B, T, H, Dv, generator=gen)
    q, k, v, dO = (t.to(dtype) for t in (q, k, v, dO))
    scale = 1.0 / math.sqrt(Dk)
    dev = "cuda"
    qd, kd, vd, gd, dOd = (t.to(dev).contiguous() for t in (q, k, v, g, dO))
    plan = api.make_plan(B, T, H, Dk, Dv, nseg, chunk, scale, dtype, device=dev, q_heads=qh)
    o = api.forward(plan, qd, kd, vd, gd)
    grads = (torch.empty_like(kd), torch.empty_like(kd), torch.empty_like(vd), torch.empty_like(gd))
    dq, dk, dv, dg = api.backward(plan, qd, kd, vd, gd, dOd, grads=grads)
    torch.cuda.synchronize()
    gpu = dict(o=o, dq=dq, dk=dk, dv=dv, dg=dg, M=plan.M, dS=plan.dS, S_in=plan.S_in,
               gamma=plan.gamma, dS_out=plan.dS_out)
    gpu = {key: val.detach().to("cpu", torch.float64).numpy() for key, val in gpu.items()}
    ref = run_oracle(q.repeat_interleave(H // qh, dim=2), k, v, g, dO, nseg, scale)
    compare(gpu, ref, tol_for(dtype), ALL_KEYS)


# ------------------------------------------------------------------ fused forward

@pytest.mark.parametrize("T,H,Dv,nseg,cu,qh", [
    (2048, 16, 128, 16, None, 0),                                   # 256 CTAs (> SMs), one wave at two a SM
    (2048, 16, 128, 16, [0, 1, 100, 128, 129, 700, 1024, 1025, 1500, 1999, 2048], 0),  # resets
    (8192, 16, 256, 64, None, 0),                                   # 2048 CTAs: look-back across waves
    (8192, 8, 256, 32, [0, 3000, 3001, 8192], 2),                   # Dv = 256 blocks, resets, shared queries
    (512, 2, 128, 1, None, 0),                                      # one segment
])
def test_fused_forward_equals_three_calls(T, H, Dv, nseg, cu, qh):
    """rm_cp_forward_fused (one launch: prepare, the bounded look-back over the
    summaries the launch's other CTAs publish, apply) writes exactly what
    rm_cp_forward_prepare + rm_cp_compose_prefix + rm_cp_forward_apply write:
    the summaries are composed by the same chain of multiply-adds, whatever
    point of the chain a CTA starts from."""
    from state_summary_scan_gb300 import api
    gen = torch.Generator().manual_seed(T + H + Dv + nseg)
    q = torch.randn(1, T, qh or H, 128, generator=gen).to(torch.bfloat16).cuda()
    k = torch.randn(1, T, H, 128, generator=gen)
    k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16).cuda()
    v = torch.randn(1, T, H, Dv, generator=gen).to(torch.bfloat16).cuda()
    g = torch.nn.functional.logsigmoid(torch.randn(1, T, H, generator=gen) + 4).cuda()
    outs = []
    for fused in (True, False):
        plan = api.make_plan(1, T, H, 128, Dv, nseg, 64, 128 ** -0.5, torch.bfloat16, cu,
                             backward=False, q_heads=qh)
        o = api.forward(plan, q, k, v, g, fused=fused)
        torch.cuda.synchronize()
        outs.append(dict(o=o, M=plan.M, dS=plan.dS, S_in=plan.S_in))
    for key in outs[0]:
        assert torch.equal(outs[0][key], outs[1][key]), key


@pytest.mark.parametrize("Dv", [128, 256])
def test_fused_forward_against_the_oracle(Dv):
    """The one-launch forward (and the backward after it) against the fp64
    oracle: packed sequences with starts at chunk positions 0, 1, 63, a
    segment start and across three segments, on a grid wider than the GPU."""
    cu = [0, 1, 2, 63, 64, 65, 129, 256, 257, 300, 511, 512, 700, 1024, 1500, 2048]
    check_case(1, 2048, 16, 128, Dv, torch.bfloat16, nseg=16, chunk=64, cu=cu, fused=True)


def test_fused_forward_generic_path_runs_the_three_calls():
    from state_summary_scan_gb300 import api
    q, k, v, g, _ = synth(1, 256, 2, 32, 32, torch.float32, seed=9)
    q, k, v, g = (t.cuda() for t in (q, k, v, g))
    outs = []
    for fused in (True, False):
        plan = api.make_plan(1, 256, 2, 32, 32, 4, 16, 0.2, torch.float32, backward=False)
        outs.append(api.forward(plan, q, k, v, g, fused=fused).clone())
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
