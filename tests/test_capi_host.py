"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/rm_cp.h declares, validates problems before any
launch, and builds packed-sequence metadata bit-exactly like the oracle's
brute-force definition."""
import ctypes
import json
import os
import re

import numpy as np
import pytest
import torch

import oracle
from state_summary_scan_gb300 import _capi as C
from state_summary_scan_gb300.workloads import WORKLOADS, make_inputs, random_cu_seqlens

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def declared_entry_points():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(rm_(?:cp|ssd|gdr)_\w+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    lib = C.load()
    declared = declared_entry_points()
    assert len(declared) >= 12
    for name in declared:
        assert hasattr(lib, name), name
    assert set(C.EXPORTS) <= set(declared)


def test_status_strings():
    lib = C.load()
    for code, name in C.STATUS_NAMES.items():
        assert lib.rm_cp_status_string(code).decode() == name


def spec(**kw):
    base = dict(B=1, T=256, H=2, Dk=32, Dv=32, num_segments=4, chunk=64, scale=0.17, dtype=0)
    base.update(kw)
    return C.ProblemSpec(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(T=250), 2),                   # T % num_segments
    (dict(chunk=48), 2),                # segment length % chunk
    (dict(B=0), 1), (dict(T=0), 1), (dict(H=-1), 1), (dict(num_segments=0), 1),
    (dict(dtype=7), 1),
    (dict(scale=float("nan")), 1),
    (dict(Dk=48), 4), (dict(Dk=256), 4), (dict(Dv=12), 4), (dict(Dv=264), 4),
    (dict(q_heads=3), 1), (dict(q_heads=-1), 1),
])
def test_validation_rejects_bad_problems(kw, status):
    with pytest.raises(C.RmCpError) as e:
        C.rm_cp_validate(spec(**kw))
    assert e.value.status == status
    assert C.rm_cp_workspace_size(spec(**kw)) == 0
    assert C.rm_cp_path(spec(**kw)) == -1


def test_validation_accepts_every_workload():
    for w in WORKLOADS.values():
        s = spec(B=w.B, T=w.T, H=w.H, Dk=w.Dk, Dv=w.Dv, num_segments=w.num_segments,
                 chunk=w.chunk, scale=w.scale, dtype=0 if w.dtype == "f32" else 1)
        C.rm_cp_validate(s)
        assert C.rm_cp_workspace_size(s) >= w.B * w.T * w.H * 4


def test_compute_calls_reject_null_and_misaligned_pointers_before_launch():
    """These return from host validation; no CUDA call is reached."""
    lib = C.load()
    s = spec()
    rc = lib.rm_cp_forward_prepare(s.ref, None, None, None, None, None, None, None)
    assert rc == 1 and b"k is NULL" in lib.rm_cp_last_error()
    odd = ctypes.c_void_p(0x1008)
    ok = ctypes.c_void_p(0x1000)
    rc = lib.rm_cp_forward_apply(s.ref, ok, ok, ok, ok, ok, odd, None, None)
    assert rc == 3 and b"o is not 16-byte aligned" in lib.rm_cp_last_error()
    rc = lib.rm_cp_backward_prepare(s.ref, ok, ok, ok, ok, ok, ok, ok, ok, None, None)
    assert rc == 1 and b"ws is NULL" in lib.rm_cp_last_error()
    bad = spec(T=100)
    rc = lib.rm_cp_compose_prefix(bad.ref, ok, ok, ok, None)
    assert rc == 2
    assert lib.rm_cp_selftest_wait_timeout(0, None) == 1
    assert lib.rm_cp_selftest_wait_timeout(2000000, None) == 1
    assert lib.rm_cp_device_status(None, 1, None) == 1
    # the host-fed step checks its argument structs before any CUDA call
    rc = lib.rm_cp_step_host(s.ref, None, None, None, None, None, None)
    assert rc == 1 and b"host is NULL" in lib.rm_cp_last_error()
    hio = C.HostIO(*([0x1000] * 10))
    rc = lib.rm_cp_step_host(s.ref, ctypes.byref(hio), None, None, None, None, None)
    assert rc == 1 and b"set is NULL" in lib.rm_cp_last_error()
    dset = C.StepSet(*([0x1000] * 10), 0x1008, None, 0x1018)
    stt = C.StepState(*([0x1000] * 6))
    rc = lib.rm_cp_step_host(s.ref, ctypes.byref(hio), ctypes.byref(dset), ctypes.byref(stt),
                             None, None, None)
    assert rc == 1 and b"set->computed is NULL" in lib.rm_cp_last_error()
    dset = C.StepSet(*([0x1000] * 4), 0x1004, *([0x1000] * 5), 0x1008, 0x1010, 0x1018)
    rc = lib.rm_cp_step_host(s.ref, ctypes.byref(hio), ctypes.byref(dset), ctypes.byref(stt),
                             None, None, None)
    assert rc == 3 and b"set->dO is not 16-byte aligned" in lib.rm_cp_last_error()
    assert lib.rm_cp_event_create(None) == 1
    assert lib.rm_cp_event_destroy(None) == 1
    # the allocation-free backward rejects problems beyond its fixed scratch
    big = spec(B=1, T=2 ** 21, H=4, num_segments=2 ** 10)   # 8M token-heads > 4M
    args = [ok] * 13
    rc = lib.rm_cp_backward_noalloc(big.ref, *args, None)
    assert rc == 2 and b"fixed scratch" in lib.rm_cp_last_error()


def test_metadata_builder_matches_golden():
    for case in json.load(open(os.path.join(GOLDEN, "packed_metadata.json"))):
        md = C.rm_cp_build_packed_metadata(case["cu_seqlens"], case["T"], case["num_segments"])
        assert md["seq_idx"].tolist() == case["seq_idx"]
        off = md["local_cu_offsets"].tolist()
        loc = md["local_cu_seqlens"].tolist()
        assert [loc[off[j]:off[j + 1]] for j in range(case["num_segments"])] == case["local_cu_seqlens"]
        assert md["preceding_start"].tolist() == case["preceding_start"]
        assert md["following_stop"].tolist() == case["following_stop"]


def check_builder_against_oracle(cu, T, nseg):
    md = C.rm_cp_build_packed_metadata(cu, T, nseg)
    ref = oracle.packed_metadata(cu, T, oracle.equal_segments(T, nseg))
    assert np.array_equal(md["seq_idx"].numpy(), ref["seq_idx"])
    off = md["local_cu_offsets"].numpy()
    loc = md["local_cu_seqlens"].numpy()
    for j in range(nseg):
        assert np.array_equal(loc[off[j]:off[j + 1]], ref["local_cu_seqlens"][j])
    assert np.array_equal(md["preceding_start"].numpy(), ref["preceding_start"])
    assert np.array_equal(md["following_stop"].numpy(), ref["following_stop"])


def test_metadata_builder_bit_exact_random():
    gen = torch.Generator().manual_seed(123)
    for trial in range(300):
        nseg = int(torch.randint(1, 9, (1,), generator=gen))
        L = int(torch.randint(1, 12, (1,), generator=gen))
        T = nseg * L
        cu = random_cu_seqlens(gen, T, max_len=int(torch.randint(1, 2 * T + 1, (1,), generator=gen)))
        check_builder_against_oracle(cu.tolist(), T, nseg)


def test_metadata_builder_packed_workload():
    w = WORKLOADS["packed64k"]
    gen = torch.Generator("cpu").manual_seed(w.seed)
    from state_summary_scan_gb300.workloads import draw_lengths, cu_seqlens_from_lengths
    cu = cu_seqlens_from_lengths(draw_lengths(gen, w.T))
    check_builder_against_oracle(cu.tolist(), w.T, w.num_segments)
    # the workload's segments are not aligned to sequences: some boundary falls
    # inside a sequence and some sequence spans at least three segments
    md = oracle.packed_metadata(cu, w.T, oracle.equal_segments(w.T, w.num_segments))
    pre, fol = md["preceding_start"], md["following_stop"]
    assert any(pre[j] < j for j in range(w.num_segments))
    assert any(fol[j] - pre[j] >= 3 for j in range(w.num_segments))


def test_metadata_builder_rejects_bad_cu_seqlens():
    for cu in ([1, 8], [0, 7], [0, 3, 3, 8], [0, 5, 4, 8]):
        with pytest.raises(C.RmCpError) as e:
            C.rm_cp_build_packed_metadata(cu, 8, 2)
        assert e.value.status == 5
    with pytest.raises(C.RmCpError) as e:
        C.rm_cp_build_packed_metadata([0, 9], 9, 2)
    assert e.value.status == 2


def test_workload_recipe_is_deterministic_and_shaped():
    w = WORKLOADS["tiny"]
    a = make_inputs(w)
    b = make_inputs(w)
    for x, y in zip((a.q, a.k, a.v, a.g, a.dO), (b.q, b.k, b.v, b.g, b.dO)):
        assert torch.equal(x, y)
    assert a.q.shape == (1, 256, 2, 32) and a.q.dtype == torch.float32
    assert torch.allclose(a.k.norm(dim=-1), torch.ones(1, 256, 2), atol=1e-5)
    assert (a.g < 0).all()


def test_ssd_calls_validate_before_any_launch():
    """The SSD maps check the problem, G and every pointer on the host."""
    lib = C.load()
    ok = ctypes.c_void_p(0x1000)
    s = spec(T=256, H=4, Dk=32, Dv=16, chunk=16, scale=1.0)
    # G must divide H
    assert lib.rm_ssd_map_inputs(s.ref, 3, ok, ok, ok, ok, ok, ok, ok, None) == 1
    assert b"G must divide H" in lib.rm_cp_last_error()
    # the SSD scan runs the recurrence with scale 1
    bad = spec(T=256, H=4, Dk=32, Dv=16, chunk=16, scale=0.5)
    assert lib.rm_ssd_finish_forward(bad.ref, ok, ok, ok, None) == 1
    assert b"scale = 1" in lib.rm_cp_last_error()
    # rows must split into 16-byte vectors over a power-of-two number of lanes
    odd = spec(T=256, H=4, Dk=32, Dv=24, chunk=16, scale=1.0, dtype=1)
    assert lib.rm_ssd_finish_forward(odd.ref, ok, ok, ok, None) == 4
    # null and misaligned device pointers
    assert lib.rm_ssd_map_inputs(s.ref, 2, None, ok, ok, ok, ok, ok, ok, None) == 1
    assert b"dt is NULL" in lib.rm_cp_last_error()
    mis = ctypes.c_void_p(0x1004)
    args = [ok] * 16  # x, dt, A, Bm, dy, D, dq, dk, dv, dg, ddt, dA, dB, dC, dD, ws
    args[10] = mis  # ddt
    assert lib.rm_ssd_finish_backward(s.ref, 2, *args, None) == 3
    assert b"ddt is not 16-byte aligned" in lib.rm_cp_last_error()
    # without D the forward finish has nothing to do and enqueues nothing
    assert lib.rm_ssd_finish_forward(s.ref, ok, None, ok, None) == 0
    assert lib.rm_ssd_workspace_size(s.ref) == 4 * (256 * 4 + 2 * 1024 * 4)
    assert lib.rm_ssd_workspace_size(spec(T=250).ref) == 0


def test_problem_spec_cache_builds_metadata_once_and_shares_no_buffers():
    """The autograd adapter's problem description is built once per shape and
    packing (metadata computed and copied once); every plan still gets its own
    summary buffers, so layers of one shape never share an S_in."""
    from state_summary_scan_gb300 import api
    cu = [0, 100, 101, 256]
    a = api.cached_spec(1, 256, 2, 32, 32, 4, 16, None, torch.float32, cu, "cpu")
    b = api.cached_spec(1, 256, 2, 32, 32, 4, 16, None, torch.float32, tuple(cu), "cpu")
    assert a is b
    assert torch.equal(a[1]["seq_idx"], torch.as_tensor(oracle.packed_metadata(
        cu, 256, oracle.equal_segments(256, 4))["seq_idx"]))
    c = api.cached_spec(1, 256, 2, 32, 32, 4, 16, None, torch.float32, [0, 99, 256], "cpu")
    assert c is not a
    p1 = api.make_plan(1, 256, 2, 32, 32, 4, 16, None, torch.float32, cu, "cpu", backward=False)
    p2 = api.make_plan(1, 256, 2, 32, 32, 4, 16, None, torch.float32, cu, "cpu", backward=False)
    assert p1.spec is p2.spec
    assert p1.S_in.data_ptr() != p2.S_in.data_ptr() and p1.M.data_ptr() != p2.M.data_ptr()
    assert p1.gamma.numel() == 0
    api.backward_buffers(p1)
    assert tuple(p1.gamma.shape) == (4, 1, 2, 32, 32) and tuple(p1.dS_out.shape) == (4, 1, 2, 32, 32)
    assert p1.ws.numel() >= C.rm_cp_workspace_size(p1.spec)


def test_vector_gates_validation_and_sizes():
    """vector_gates is 0 or 1; vector gates take the tensor-core path for bf16
    with Dk = Dv = 128 and the generic kernels otherwise, the workspace holds
    one value per key dimension, and the SSD calls (one gate per head) refuse
    them."""
    w = WORKLOADS["32k"]
    base = dict(B=w.B, T=w.T, H=w.H, Dk=w.Dk, Dv=w.Dv, num_segments=w.num_segments,
                chunk=w.chunk, scale=w.scale, dtype=1)
    assert C.rm_cp_path(C.ProblemSpec(**base)) == 1
    vg = C.ProblemSpec(**base, vector_gates=1)
    assert C.rm_cp_path(vg) == 1
    assert C.rm_cp_path(C.ProblemSpec(**dict(base, dtype=0), vector_gates=1)) == 0
    assert C.rm_cp_path(C.ProblemSpec(**dict(base, Dv=256), vector_gates=1)) == 0
    assert C.rm_cp_path(C.ProblemSpec(**dict(base, T=w.T - 16 * 32, chunk=32), vector_gates=1)) == 0
    ntok = w.B * w.T * w.H
    assert C.rm_cp_workspace_size(vg) >= ntok * w.Dk * 4
    assert C.rm_cp_workspace_size(vg) < ntok * w.Dk * 4 + 256
    with pytest.raises(C.RmCpError) as e:
        C.rm_cp_validate(C.ProblemSpec(**base, vector_gates=2))
    assert e.value.status == 1
    ssd = C.ProblemSpec(1, 256, 4, 32, 16, 4, 16, 1.0, torch.float32, vector_gates=1)
    ok = ctypes.c_void_p(0x1000)
    lib = C.load()
    assert lib.rm_ssd_finish_forward(ssd.ref, ok, ok, ok, None) == 1
    assert b"vector_gates" in lib.rm_cp_last_error()


def test_gdr_path_and_workspace():
    """The gated delta rule's sweeps take the tensor cores for bf16 with
    Dk = Dv = 64 and segment lengths that are multiples of 64, the generic
    kernels for the other supported shapes; unsupported problems are -1.  The
    workspace (one fp32 state every 16 tokens) also holds the tensor-core
    sweeps' state every 64 tokens."""
    from state_summary_scan_gb300.workloads import GDR_WORKLOADS
    w = GDR_WORKLOADS["gdr8k"]
    base = dict(B=w.B, T=w.T, H=w.H, Dk=w.Dk, Dv=w.Dv, num_segments=w.num_segments,
                chunk=w.chunk, scale=w.scale, dtype=1)
    tc = C.ProblemSpec(**base)
    assert C.rm_gdr_path(tc) == 1
    assert C.rm_gdr_path(C.ProblemSpec(**dict(base, dtype=0))) == 0                   # fp32 storage
    assert C.rm_gdr_path(C.ProblemSpec(**dict(base, Dk=32))) == 0                     # Dk != 64
    assert C.rm_gdr_path(C.ProblemSpec(**dict(base, Dv=48))) == 0                     # Dv != 64
    assert C.rm_gdr_path(C.ProblemSpec(**dict(base, T=w.T - 32 * 16, chunk=16))) == 0  # L % 64 != 0
    assert C.rm_gdr_path(C.ProblemSpec(**dict(base, Dk=128))) == 0                    # generic kernels
    assert C.rm_gdr_path(C.ProblemSpec(**dict(base, Dk=128, Dv=136))) == -1           # Dv > 128
    assert C.rm_gdr_path(C.ProblemSpec(**base, vector_gates=1)) == -1
    ntok = w.B * w.T * w.H
    ws = C.rm_gdr_workspace_size(tc)
    assert ws >= (ntok // 16) * w.Dk * w.Dv * 4 >= (ntok // 64) * w.Dk * w.Dv * 4
    assert C.rm_gdr_workspace_size(C.ProblemSpec(**dict(base, Dk=128, Dv=136))) == 0
