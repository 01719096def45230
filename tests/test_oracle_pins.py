"""Pins for the fp64 oracle: every check here computes its expected value by a
route other than the oracle's own code (closed forms, textbook routines,
finite differences, hand-worked values, invariants), so that a dropped term,
a wrong sign or index, or a transposed operand in oracle.c fails one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_problem(rng, B=1, T=16, H=2, Dk=4, Dv=3, gate=(0.5, 1.0)):
    q = rng.standard_normal((B, T, H, Dk))
    k = rng.standard_normal((B, T, H, Dk))
    v = rng.standard_normal((B, T, H, Dv))
    # gates of both signs so that exp(g) > 1 terms are exercised too
    g = gate[0] * rng.standard_normal((B, T, H)) - gate[1] * 0.3
    dO = rng.standard_normal((B, T, H, Dv))
    return q, k, v, g, dO


def seq_idx_from_cu(cu, T):
    s = np.empty(T, dtype=np.int32)
    for i in range(len(cu) - 1):
        s[cu[i]:cu[i + 1]] = i
    return s


def closed_form(q, k, v, g, scale, seq_idx=None):
    """o_t = scale * sum_{s<=t, same seq} exp(G_t - G_s) (q_t.k_s) v_s, G = cumsum g."""
    B, T, H, Dk = q.shape
    G = np.cumsum(g, axis=1)
    o = np.zeros(v.shape[:3] + (v.shape[3],))
    for b in range(B):
        for h in range(H):
            for t in range(T):
                for s in range(t + 1):
                    if seq_idx is not None and seq_idx[s] != seq_idx[t]:
                        continue
                    w = math.exp(G[b, t, h] - G[b, s, h]) * float(q[b, t, h] @ k[b, s, h])
                    o[b, t, h] += scale * w * v[b, s, h]
    return o


def rel_err(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ------------------------------------------------------------------ forward

@pytest.mark.parametrize("packed", [False, True])
def test_forward_matches_quadratic_closed_form(packed):
    rng = np.random.default_rng(1)
    q, k, v, g, _ = rand_problem(rng, B=2, T=20, H=2, Dk=5, Dv=3)
    si = seq_idx_from_cu([0, 3, 4, 11, 20], 20) if packed else None
    o = oracle.forward(q, k, v, g, 0.37, si)
    ref = closed_form(q, k, v, g, 0.37, si)
    assert rel_err(o, ref) < 1e-12


def test_forward_zero_gate_is_causal_linear_attention():
    rng = np.random.default_rng(2)
    q, k, v, _, _ = rand_problem(rng, B=1, T=24, H=3, Dk=6, Dv=4)
    g = np.zeros(q.shape[:3])
    o = oracle.forward(q, k, v, g, 0.5)
    kv = np.cumsum(np.einsum("bthi,bthj->bthij", k, v), axis=1)
    ref = 0.5 * np.einsum("bthij,bthi->bthj", kv, q)
    assert rel_err(o, ref) < 1e-12


def test_forward_all_resets_is_diagonal():
    rng = np.random.default_rng(3)
    q, k, v, g, _ = rand_problem(rng, B=1, T=10, H=2, Dk=4, Dv=5)
    si = np.arange(10, dtype=np.int32)
    o = oracle.forward(q, k, v, g, 0.25, si)
    ref = 0.25 * np.einsum("bthi,bthi->bth", q, k)[..., None] * v
    assert rel_err(o, ref) < 1e-13


def test_forward_single_token():
    rng = np.random.default_rng(4)
    q, k, v, g, _ = rand_problem(rng, B=3, T=1, H=2, Dk=3, Dv=2)
    o = oracle.forward(q, k, v, g, 1.0)
    ref = np.einsum("bthi,bthi->bth", q, k)[..., None] * v
    assert rel_err(o, ref) < 1e-14


def test_forward_scalar_recurrence_matches_lfilter():
    """Dk = Dv = 1 with a constant gate: s_t = a s_{t-1} + x_t is a first-order
    IIR filter (scipy.signal.lfilter with denominator [1, -a])."""
    signal = pytest.importorskip("scipy.signal")
    rng = np.random.default_rng(5)
    T = 50
    q = rng.standard_normal((1, T, 1, 1))
    k = rng.standard_normal((1, T, 1, 1))
    v = rng.standard_normal((1, T, 1, 1))
    a = 0.8
    g = np.full((1, T, 1), math.log(a))
    o = oracle.forward(q, k, v, g, 1.0)
    x = (k * v)[0, :, 0, 0]
    s = signal.lfilter([1.0], [1.0, -a], x)
    ref = s * q[0, :, 0, 0]
    assert rel_err(o[0, :, 0, 0], ref) < 1e-12


def test_forward_hand_worked_golden():
    with open(os.path.join(GOLDEN, "scalar_recurrence.json")) as f:
        case = json.load(f)
    T = len(case["q"])
    arr = lambda key: np.array(case[key], dtype=np.float64).reshape(1, T, 1, 1)
    g = np.array(case["g"], dtype=np.float64).reshape(1, T, 1)
    si = np.array(case["seq_idx"], dtype=np.int32) if case.get("seq_idx") else None
    o = oracle.forward(arr("q"), arr("k"), arr("v"), g, case["scale"], si)
    assert np.allclose(o.reshape(-1), case["o"], rtol=0, atol=1e-14)
    dq, dk, dv, dg = oracle.backward(arr("q"), arr("k"), arr("v"), g, arr("dO"), case["scale"], si)
    assert np.allclose(dq.reshape(-1), case["dq"], rtol=0, atol=1e-14)
    assert np.allclose(dk.reshape(-1), case["dk"], rtol=0, atol=1e-14)
    assert np.allclose(dv.reshape(-1), case["dv"], rtol=0, atol=1e-14)
    assert np.allclose(dg.reshape(-1), case["dg"], rtol=0, atol=1e-14)


# ------------------------------------------------------------------ backward

def loss(q, k, v, g, dO, scale, si):
    return float(np.sum(oracle.forward(q, k, v, g, scale, si) * dO))


def finite_diff(x, f, h=1e-6):
    out = np.empty_like(x)
    flat = x.reshape(-1)
    of = out.reshape(-1)
    for n in range(flat.size):
        old = flat[n]
        flat[n] = old + h
        lp = f()
        flat[n] = old - h
        lm = f()
        flat[n] = old
        of[n] = (lp - lm) / (2 * h)
    return out


@pytest.mark.parametrize("packed", [False, True])
def test_backward_matches_finite_differences(packed):
    rng = np.random.default_rng(6)
    q, k, v, g, dO = rand_problem(rng, B=1, T=12, H=2, Dk=3, Dv=4)
    si = seq_idx_from_cu([0, 5, 6, 12], 12) if packed else None
    scale = 0.7
    dq, dk, dv, dg = oracle.backward(q, k, v, g, dO, scale, si)
    f = lambda: loss(q, k, v, g, dO, scale, si)
    for x, ana in ((q, dq), (k, dk), (v, dv), (g, dg)):
        num = finite_diff(x, f)
        assert np.max(np.abs(num - ana)) <= 1e-7 * max(1.0, np.max(np.abs(ana)))


def test_gate_gradient_direct_form_equals_identity():
    rng = np.random.default_rng(7)
    q, k, v, g, dO = rand_problem(rng, B=2, T=30, H=2, Dk=4, Dv=5)
    si = seq_idx_from_cu([0, 7, 8, 19, 30], 30)
    for s in (None, si):
        a = oracle.backward(q, k, v, g, dO, 0.3, s)
        d = oracle.backward(q, k, v, g, dO, 0.3, s, direct=True)
        for x, y in zip(a, d):
            assert rel_err(x, y) < 1e-12


def test_gate_gradient_zero_at_sequence_starts():
    rng = np.random.default_rng(8)
    q, k, v, g, dO = rand_problem(rng, B=2, T=40, H=2, Dk=4, Dv=4)
    cu = [0, 9, 10, 33, 40]
    si = seq_idx_from_cu(cu, 40)
    dg = oracle.backward(q, k, v, g, dO, 1.0, si)[3]
    for c in cu[:-1]:
        assert np.all(dg[:, c] == 0.0)
    # and it is what the direct form gives there (alpha = 0)
    dgd = oracle.backward(q, k, v, g, dO, 1.0, si, direct=True)[3]
    assert np.all(dgd[:, cu[:-1]] == 0.0)


# ------------------------------------------------------------------ resets

def test_packed_run_equals_separate_runs_bit_exact():
    rng = np.random.default_rng(9)
    T = 37
    cu = [0, 5, 6, 20, 37]
    q, k, v, g, dO = rand_problem(rng, B=1, T=T, H=3, Dk=4, Dv=3)
    si = seq_idx_from_cu(cu, T)
    o = oracle.forward(q, k, v, g, 0.5, si)
    grads = oracle.backward(q, k, v, g, dO, 0.5, si)
    for a, b in zip(cu[:-1], cu[1:]):
        sl = slice(a, b)
        o1 = oracle.forward(q[:, sl], k[:, sl], v[:, sl], g[:, sl], 0.5)
        assert np.array_equal(o[:, sl], o1)
        g1 = oracle.backward(q[:, sl], k[:, sl], v[:, sl], g[:, sl], dO[:, sl], 0.5)
        for full, part in zip(grads, g1):
            assert np.array_equal(full[:, sl], part)


# ------------------------------------------------------------------ segments

def test_prepare_transition_is_exp_of_gate_sum_or_zero():
    rng = np.random.default_rng(10)
    T, nseg = 24, 4
    q, k, v, g, _ = rand_problem(rng, B=2, T=T, H=2, Dk=3, Dv=2)
    si = seq_idx_from_cu([0, 7, 12, 24], T)   # resets at 0 (seg 0), 7 (seg 1), 12 (seg 2 first token)
    s = oracle.equal_segments(T, nseg)
    M, _ = oracle.forward_prepare(k, v, g, s, si)
    for j in range(nseg):
        ref = np.exp(g[:, s[j]:s[j + 1]].sum(axis=1))
        has_reset = j in (0, 1, 2)
        assert np.allclose(M[j], 0.0 if has_reset else ref, rtol=1e-14, atol=0)


def test_prepare_delta_is_local_state_closed_form():
    rng = np.random.default_rng(11)
    T, nseg = 18, 3
    q, k, v, g, _ = rand_problem(rng, B=1, T=T, H=2, Dk=3, Dv=4)
    si = seq_idx_from_cu([0, 8, 18], T)
    s = oracle.equal_segments(T, nseg)
    _, dS = oracle.forward_prepare(k, v, g, s, si)
    G = np.cumsum(g, axis=1)
    for j in range(nseg):
        e = s[j + 1] - 1
        ref = np.zeros(dS.shape[2:])
        for h in range(2):
            for t in range(s[j], e + 1):
                if si[t] != si[e]:
                    continue
                ref[h] += math.exp(G[0, e, h] - G[0, t, h]) * np.outer(k[0, t, h], v[0, t, h])
        assert rel_err(dS[j, 0], ref) < 1e-13


def test_compose_prefix_matches_product_formula():
    rng = np.random.default_rng(12)
    nseg, B, H, Dk, Dv = 6, 1, 2, 2, 3
    M = rng.uniform(0.1, 1.5, (nseg, B, H))
    dS = rng.standard_normal((nseg, B, H, Dk, Dv))
    pre = np.array([0, 0, 1, 1, 3, 5], dtype=np.int32)
    S_in = oracle.compose_prefix(M, dS, pre)
    for j in range(nseg):
        ref = np.zeros((B, H, Dk, Dv))
        for i in range(pre[j], j):
            prod = np.ones((B, H))
            for l in range(i + 1, j):
                prod = prod * M[l]
            ref += prod[..., None, None] * dS[i]
        assert rel_err(S_in[j], ref) < 1e-13 if np.any(ref) else np.all(S_in[j] == 0)


def test_compose_suffix_matches_product_formula():
    rng = np.random.default_rng(13)
    nseg, B, H, Dk, Dv = 6, 2, 1, 3, 2
    M = rng.uniform(0.1, 1.5, (nseg, B, H))
    gamma = rng.standard_normal((nseg, B, H, Dk, Dv))
    fol = np.array([3, 3, 6, 6, 6, 6], dtype=np.int32)
    dS_out = oracle.compose_suffix(M, gamma, fol)
    for j in range(nseg):
        ref = np.zeros((B, H, Dk, Dv))
        for i in range(j + 1, fol[j]):
            prod = np.ones((B, H))
            for l in range(j + 1, i):
                prod = prod * M[l]
            ref += prod[..., None, None] * gamma[i]
        assert rel_err(dS_out[j], ref) < 1e-13 if np.any(ref) else np.all(dS_out[j] == 0)


@pytest.mark.parametrize("packed", [False, True])
def test_gamma_is_gradient_of_local_loss_wrt_incoming_state(packed):
    """L_local(S_in) = sum_{t in seg} dO_t . o_t is affine in S_in, so
    gamma[i, j] = L_local(E_ij) - L_local(0)."""
    rng = np.random.default_rng(14)
    T, nseg = 16, 2
    q, k, v, g, dO = rand_problem(rng, B=1, T=T, H=1, Dk=3, Dv=2)
    si = seq_idx_from_cu([0, 11, 16], T) if packed else None  # seg 1 holds a reset at 11
    s = oracle.equal_segments(T, nseg)
    gamma = oracle.backward_prepare(q, g, dO, 0.9, s, si)
    zero = np.zeros((nseg, 1, 1, 3, 2))
    base = oracle.forward_apply(q, k, v, g, zero, 0.9, s, si)
    for i in range(3):
        for jj in range(2):
            S_in = zero.copy()
            S_in[:, 0, 0, i, jj] = 1.0
            o = oracle.forward_apply(q, k, v, g, S_in, 0.9, s, si)
            for seg in range(nseg):
                sl = slice(s[seg], s[seg + 1])
                ref = np.sum((o[:, sl] - base[:, sl]) * dO[:, sl])
                assert abs(gamma[seg, 0, 0, i, jj] - ref) < 1e-12


def all_segmentations(T):
    for mask in range(1 << (T - 1)):
        cuts = [0] + [t for t in range(1, T) if mask >> (t - 1) & 1] + [T]
        yield np.array(cuts, dtype=np.int32)


@pytest.mark.parametrize("packed", [False, True])
def test_every_segmentation_equals_monolithic(packed):
    rng = np.random.default_rng(15)
    T = 12
    q, k, v, g, dO = rand_problem(rng, B=1, T=T, H=1, Dk=2, Dv=3)
    cu = [0, 4, 5, 12] if packed else [0, T]
    si = seq_idx_from_cu(cu, T) if packed else None
    o_ref = oracle.forward(q, k, v, g, 0.8, si)
    grads_ref = oracle.backward(q, k, v, g, dO, 0.8, si)
    n = 0
    for s in all_segmentations(T):
        md = oracle.packed_metadata(cu, T, s)
        for pre, fol in ((md["preceding_start"], md["following_stop"]), (None, None)):
            o, mid = oracle.segmented_forward(q, k, v, g, 0.8, s, si, pre)
            assert rel_err(o, o_ref) < 1e-13
            grads, _ = oracle.segmented_backward(q, k, v, g, dO, 0.8, s, si, pre, fol,
                                                 S_in=mid["S_in"], M=mid["M"])
            for x, y in zip(grads, grads_ref):
                assert rel_err(x, y) < 1e-12
        n += 1
    assert n == 2 ** (T - 1)


def test_segmented_intermediates_are_true_states():
    """S_in[j] is the monolithic state just before segment j; dS_out[j] is the
    adjoint arriving at segment j's last state from later tokens."""
    rng = np.random.default_rng(16)
    T, nseg = 24, 4
    q, k, v, g, dO = rand_problem(rng, B=1, T=T, H=2, Dk=3, Dv=2)
    cu = [0, 10, 24]
    si = seq_idx_from_cu(cu, T)
    s = oracle.equal_segments(T, nseg)
    md = oracle.packed_metadata(cu, T, s)
    _, mid = oracle.segmented_forward(q, k, v, g, 1.0, s, si, md["preceding_start"])
    for j in range(nseg):
        a = s[j]
        if a == 0 or si[a] != si[a - 1]:
            assert np.all(mid["S_in"][j] == 0)
        else:
            start = cu[si[a]]
            G = np.cumsum(g, axis=1)
            ref = np.zeros((2, 3, 2))
            for h in range(2):
                for t in range(start, a):
                    ref[h] += math.exp(G[0, a - 1, h] - G[0, t, h]) * np.outer(k[0, t, h], v[0, t, h])
            assert rel_err(mid["S_in"][j, 0], ref) < 1e-13


# ------------------------------------------------------------------ metadata

def test_metadata_hand_worked_golden():
    with open(os.path.join(GOLDEN, "packed_metadata.json")) as f:
        cases = json.load(f)
    for case in cases:
        T, nseg = case["T"], case["num_segments"]
        md = oracle.packed_metadata(case["cu_seqlens"], T, oracle.equal_segments(T, nseg))
        assert md["seq_idx"].tolist() == case["seq_idx"]
        assert [x.tolist() for x in md["local_cu_seqlens"]] == case["local_cu_seqlens"]
        assert md["preceding_start"].tolist() == case["preceding_start"]
        assert md["following_stop"].tolist() == case["following_stop"]


def test_metadata_properties_random():
    rng = np.random.default_rng(17)
    for _ in range(200):
        nseg = int(rng.integers(1, 9))
        L = int(rng.integers(1, 9))
        T = nseg * L
        cuts = sorted(set(rng.integers(1, T, int(rng.integers(0, T))).tolist())) if T > 1 else []
        cu = [0] + cuts + [T]
        s = oracle.equal_segments(T, nseg)
        md = oracle.packed_metadata(cu, T, s)
        si = md["seq_idx"]
        assert si[0] == 0 and np.all(np.diff(si) >= 0) and si[-1] == len(cu) - 2
        for j in range(nseg):
            lc = md["local_cu_seqlens"][j]
            assert lc[0] == 0 and lc[-1] == L and np.all(np.diff(lc) > 0)
            p, f = md["preceding_start"][j], md["following_stop"][j]
            assert 0 <= p <= j < f <= nseg
            a, e = s[j], s[j + 1] - 1
            first = cu[si[a]]          # start token of the sequence holding a
            last = cu[si[e] + 1] - 1   # last token of the sequence holding e
            assert s[p] <= first < s[p + 1]
            assert s[f - 1] <= last < s[f]


def test_metadata_rejects_bad_cu_seqlens():
    s = oracle.equal_segments(8, 2)
    for cu in ([1, 8], [0, 7], [0, 3, 3, 8], [0, 5, 4, 8]):
        with pytest.raises(ValueError):
            oracle.packed_metadata(cu, 8, s)


# ------------------------------------------------------------------ Mamba2 SSD scan
# The oracle's ssd_forward / ssd_backward walk the token recurrence of the
# Mamba2 SSD scan (the "Mamba2 ... exact CP linear scan" of the context-parallel
# pages, restated from the published SSD formulation).  Pins: its quadratic
# ("attention") form, the decay-free cumulative sum, the reset invariant and
# central finite differences of every gradient.

def _ssd_inputs(rng, B, T, H, G, N, P):
    x = rng.standard_normal((B, T, H, P))
    dt = np.abs(rng.standard_normal((B, T, H))) * 0.5 + 0.01
    A = -np.abs(rng.standard_normal(H)) - 0.1
    Bm = rng.standard_normal((B, T, G, N))
    Cm = rng.standard_normal((B, T, G, N))
    D = rng.standard_normal(H)
    return x, dt, A, Bm, Cm, D


def _ssd_quadratic(x, dt, A, Bm, Cm, D, seq_idx=None):
    """y_t = sum_{s <= t, same sequence} exp(A sum_{r in (s, t]} dt_r) (C_t . B_s) dt_s x_s + D x_t."""
    B, T, H, P = x.shape
    G = Bm.shape[2]
    y = np.zeros_like(x)
    sid = np.zeros(T, dtype=np.int64) if seq_idx is None else np.asarray(seq_idx)
    for b in range(B):
        for h in range(H):
            gi = h // (H // G)
            cs = np.cumsum(dt[b, :, h] * A[h])
            for t in range(T):
                for s in range(t + 1):
                    if sid[s] != sid[t]:
                        continue
                    y[b, t, h] += np.exp(cs[t] - cs[s]) * (Cm[b, t, gi] @ Bm[b, s, gi]) * dt[b, s, h] * x[b, s, h]
                y[b, t, h] += D[h] * x[b, t, h]
    return y


def test_ssd_forward_matches_quadratic_form():
    rng = np.random.default_rng(11)
    x, dt, A, Bm, Cm, D = _ssd_inputs(rng, 2, 16, 4, 2, 5, 3)
    np.testing.assert_allclose(oracle.ssd_forward(x, dt, A, Bm, Cm, D), _ssd_quadratic(x, dt, A, Bm, Cm, D),
                               rtol=0, atol=1e-12)
    si = np.array([0] * 5 + [1] * 7 + [2] * 4, dtype=np.int32)
    x, dt, A, Bm, Cm, D = _ssd_inputs(rng, 1, 16, 2, 1, 4, 4)
    np.testing.assert_allclose(oracle.ssd_forward(x, dt, A, Bm, Cm, D, si),
                               _ssd_quadratic(x, dt, A, Bm, Cm, D, si), rtol=0, atol=1e-12)


def test_ssd_without_decay_is_a_cumulative_sum():
    rng = np.random.default_rng(12)
    x, dt, A, Bm, Cm, _ = _ssd_inputs(rng, 1, 20, 2, 1, 3, 4)
    A = np.zeros_like(A)
    y = oracle.ssd_forward(x, dt, A, Bm, Cm)
    for h in range(2):
        hs = np.cumsum(dt[0, :, h, None, None] * Bm[0, :, 0, :, None] * x[0, :, h, None, :], axis=0)
        np.testing.assert_allclose(y[0, :, h], np.einsum("tnp,tn->tp", hs, Cm[0, :, 0]), rtol=1e-12, atol=1e-12)


def test_ssd_packed_equals_separate_runs():
    rng = np.random.default_rng(13)
    x, dt, A, Bm, Cm, D = _ssd_inputs(rng, 1, 18, 2, 1, 3, 2)
    dy = rng.standard_normal(x.shape)
    cut = [0, 7, 8, 18]
    si = np.concatenate([np.full(cut[i + 1] - cut[i], i) for i in range(3)]).astype(np.int32)
    y = oracle.ssd_forward(x, dt, A, Bm, Cm, D, si)
    gr = oracle.ssd_backward(x, dt, A, Bm, Cm, dy, D, si)
    dA = np.zeros(2)
    dD = np.zeros(2)
    for i in range(3):
        sl = slice(cut[i], cut[i + 1])
        ys = oracle.ssd_forward(x[:, sl], dt[:, sl], A, Bm[:, sl], Cm[:, sl], D)
        assert np.array_equal(y[:, sl], ys)
        gs = oracle.ssd_backward(x[:, sl], dt[:, sl], A, Bm[:, sl], Cm[:, sl], dy[:, sl], D)
        for full, part in zip((gr[0], gr[1], gr[3], gr[4]), (gs[0], gs[1], gs[3], gs[4])):
            assert np.array_equal(full[:, sl], part)
        dA += gs[2]
        dD += gs[5]
    np.testing.assert_allclose(gr[2], dA, rtol=1e-12)
    np.testing.assert_allclose(gr[5], dD, rtol=1e-12)


@pytest.mark.parametrize("reset", [False, True])
def test_ssd_gradients_match_finite_differences(reset):
    rng = np.random.default_rng(14)
    x, dt, A, Bm, Cm, D = _ssd_inputs(rng, 2, 10, 4, 2, 3, 2)
    dy = rng.standard_normal(x.shape)
    si = np.array([0, 0, 0, 1, 1, 2, 2, 2, 2, 2], dtype=np.int32) if reset else None
    grads = oracle.ssd_backward(x, dt, A, Bm, Cm, dy, D, si)
    base = dict(x=x, dt=dt, A=A, Bm=Bm, Cm=Cm, D=D)

    def loss(**kw):
        args = dict(base, **kw)
        return float(np.sum(dy * oracle.ssd_forward(seq_idx=si, **args)))

    eps = 1e-6
    for name, gr in zip(("x", "dt", "A", "Bm", "Cm", "D"), grads):
        arr = base[name]
        fd = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            a1, a2 = arr.copy(), arr.copy()
            a1[i] += eps
            a2[i] -= eps
            fd[i] = (loss(**{name: a1}) - loss(**{name: a2})) / (2 * eps)
        assert np.max(np.abs(fd - gr)) <= 1e-7 * np.max(np.abs(fd)), name


# ------------------------------------------------------------------ vector gates
# One gate per key dimension: S_t = diag(exp(g_t)) S_{t-1} + k_t v_t^T (the
# diagonal case of the summary algebra's general transition M).  Pins: the
# quadratic closed form, the reduction to scalar gates, finite differences of
# every gradient, the direct gate gradient, the segmentation invariant and the
# reset invariant.

def _vg_inputs(rng, B, T, H, Dk, Dv):
    q = rng.standard_normal((B, T, H, Dk))
    k = rng.standard_normal((B, T, H, Dk))
    v = rng.standard_normal((B, T, H, Dv))
    g = -np.abs(rng.standard_normal((B, T, H, Dk))) * 0.5
    return q, k, v, g


def test_vg_forward_matches_quadratic_form():
    rng = np.random.default_rng(31)
    q, k, v, g = _vg_inputs(rng, 1, 14, 2, 3, 2)
    si = np.array([0] * 4 + [1] * 6 + [2] * 4, dtype=np.int32)
    for seq in (None, si):
        o = oracle.vg_forward(q, k, v, g, 0.7, seq)
        sid = np.zeros(14, dtype=np.int64) if seq is None else seq
        G = np.cumsum(g, axis=1)
        ref = np.zeros_like(o)
        for h in range(2):
            for t in range(14):
                for s in range(t + 1):
                    if sid[s] == sid[t]:
                        w = np.sum(q[0, t, h] * k[0, s, h] * np.exp(G[0, t, h] - G[0, s, h]))
                        ref[0, t, h] += 0.7 * w * v[0, s, h]
        np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_vg_equal_gates_reduce_to_scalar_gates():
    """g_t[i] = g_t for every i is the scalar gate: same outputs and gradients,
    and the scalar gate's gradient is the sum of the per-dimension ones."""
    rng = np.random.default_rng(32)
    q, k, v, g = _vg_inputs(rng, 2, 12, 2, 4, 3)
    gs = g[..., 0]
    gv = np.repeat(gs[..., None], 4, axis=-1)
    dO = rng.standard_normal(v.shape)
    np.testing.assert_allclose(oracle.vg_forward(q, k, v, gv, 0.5), oracle.forward(q, k, v, gs, 0.5),
                               rtol=1e-12, atol=1e-12)
    a = oracle.vg_backward(q, k, v, gv, dO, 0.5)
    b = oracle.backward(q, k, v, gs, dO, 0.5)
    for x, y in zip(a[:3], b[:3]):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(a[3].sum(axis=-1), b[3], rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("reset", [False, True])
def test_vg_gradients_match_finite_differences(reset):
    rng = np.random.default_rng(33)
    q, k, v, g = _vg_inputs(rng, 1, 10, 2, 3, 2)
    dO = rng.standard_normal(v.shape)
    si = np.array([0, 0, 0, 1, 1, 2, 2, 2, 2, 2], dtype=np.int32) if reset else None
    grads = oracle.vg_backward(q, k, v, g, dO, 0.7, si)
    direct = oracle.vg_backward(q, k, v, g, dO, 0.7, si, direct=True)
    np.testing.assert_allclose(grads[3], direct[3], rtol=1e-10, atol=1e-12)
    base = dict(q=q, k=k, v=v, g=g)
    eps = 1e-6
    for name, gr in zip(("q", "k", "v", "g"), grads):
        arr = base[name]
        fd = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            a1, a2 = arr.copy(), arr.copy()
            a1[i] += eps
            a2[i] -= eps
            fd[i] = (np.sum(dO * oracle.vg_forward(**dict(base, **{name: a1}), scale=0.7, seq_idx=si))
                     - np.sum(dO * oracle.vg_forward(**dict(base, **{name: a2}), scale=0.7, seq_idx=si))) / (2 * eps)
        assert np.max(np.abs(fd - gr)) <= 1e-7 * np.max(np.abs(fd)), name
    if reset:
        assert np.all(grads[3][:, [0, 3, 5]] == 0.0)


def test_vg_segmented_equals_monolithic():
    """Summaries with a diagonal transition: prepare, compose, then each segment
    from its incoming state gives the monolithic outputs."""
    rng = np.random.default_rng(34)
    q, k, v, g = _vg_inputs(rng, 2, 24, 2, 3, 2)
    mono = oracle.vg_forward(q, k, v, g, 0.6)
    for seg in ([0, 24], [0, 8, 16, 24], [0, 1, 7, 20, 24]):
        seg = np.array(seg, dtype=np.int32)
        M, dS = oracle.vg_forward_prepare(k, v, g, seg)
        S_in = oracle.vg_compose_prefix(M, dS)
        out = np.empty_like(mono)
        for j in range(len(seg) - 1):
            sl = slice(seg[j], seg[j + 1])
            out[:, sl] = oracle.vg_forward(q[:, sl], k[:, sl], v[:, sl], g[:, sl], 0.6, S0=S_in[j])
        np.testing.assert_allclose(out, mono, rtol=1e-12, atol=1e-12)
        # M is the product of a segment's per-dimension decays, 0 for the segment
        # holding the row's first token (a sequence start)
        assert np.all(M[0] == 0.0)
        for j in range(1, len(seg) - 1):
            np.testing.assert_allclose(M[j], np.exp(g[:, seg[j]:seg[j + 1]].sum(axis=1)), rtol=1e-12)


def test_vg_packed_equals_separate_runs():
    rng = np.random.default_rng(35)
    q, k, v, g = _vg_inputs(rng, 1, 15, 2, 3, 2)
    dO = rng.standard_normal(v.shape)
    cut = [0, 6, 7, 15]
    si = np.concatenate([np.full(cut[i + 1] - cut[i], i) for i in range(3)]).astype(np.int32)
    o = oracle.vg_forward(q, k, v, g, 0.5, si)
    gr = oracle.vg_backward(q, k, v, g, dO, 0.5, si)
    for i in range(3):
        sl = slice(cut[i], cut[i + 1])
        assert np.array_equal(o[:, sl], oracle.vg_forward(q[:, sl], k[:, sl], v[:, sl], g[:, sl], 0.5))
        gs = oracle.vg_backward(q[:, sl], k[:, sl], v[:, sl], g[:, sl], dO[:, sl], 0.5)
        for a, b in zip(gr, gs):
            assert np.array_equal(a[:, sl], b)


# ------------------------------------------------------------------ gated delta rule
# S_t = exp(g_t)(I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T: the summary
# algebra with matrix transitions.  Pins: reductions to causal linear attention
# (orthonormal keys), to an overwrite (a repeated key), to pure decay (beta = 0),
# finite differences of every gradient and the segmentation invariant with the
# Dk x Dk transitions.

def _gdr_inputs(rng, B, T, H, Dk, Dv):
    q = rng.standard_normal((B, T, H, Dk))
    k = rng.standard_normal((B, T, H, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, Dv))
    g = -np.abs(rng.standard_normal((B, T, H))) * 0.5
    beta = rng.uniform(0.1, 0.9, (B, T, H))
    return q, k, v, g, beta


def test_gdr_orthonormal_keys_is_linear_attention():
    """alpha = beta = 1 with orthonormal keys: each write leaves the others'
    values alone, so o_t = scale sum_{s<=t} (q_t . k_s) v_s."""
    rng = np.random.default_rng(41)
    T, Dk, Dv = 5, 6, 3
    basis, _ = np.linalg.qr(rng.standard_normal((Dk, Dk)))
    k = basis[:T][None, :, None, :]
    q = rng.standard_normal((1, T, 1, Dk))
    v = rng.standard_normal((1, T, 1, Dv))
    o = oracle.gdr_forward(q, k, v, np.zeros((1, T, 1)), np.ones((1, T, 1)), 0.8)
    ref = np.stack([0.8 * sum((q[0, t, 0] @ k[0, s, 0]) * v[0, s, 0] for s in range(t + 1))
                    for t in range(T)])
    np.testing.assert_allclose(o[0, :, 0], ref, rtol=1e-12, atol=1e-12)


def test_gdr_repeated_key_overwrites():
    rng = np.random.default_rng(42)
    kk = rng.standard_normal(4)
    kk /= np.linalg.norm(kk)
    k = np.stack([kk, kk])[None, :, None, :]
    v = rng.standard_normal((1, 2, 1, 3))
    q = rng.standard_normal((1, 2, 1, 4))
    o = oracle.gdr_forward(q, k, v, np.zeros((1, 2, 1)), np.ones((1, 2, 1)), 1.0)
    np.testing.assert_allclose(o[0, 1, 0], (q[0, 1, 0] @ kk) * v[0, 1, 0], rtol=1e-12, atol=1e-12)


def test_gdr_zero_beta_is_pure_decay():
    rng = np.random.default_rng(43)
    q, k, v, g, _ = _gdr_inputs(rng, 1, 6, 2, 3, 2)
    S0 = rng.standard_normal((1, 2, 3, 2))
    o = oracle.gdr_forward(q, k, v, g, np.zeros((1, 6, 2)), 0.5, S0=S0)
    decay = np.exp(np.cumsum(g, axis=1))
    ref = 0.5 * decay[..., None] * np.einsum("bhij,bthi->bthj", S0, q)
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("reset", [False, True])
def test_gdr_gradients_match_finite_differences(reset):
    rng = np.random.default_rng(44)
    q, k, v, g, beta = _gdr_inputs(rng, 1, 8, 2, 3, 2)
    dO = rng.standard_normal(v.shape)
    si = np.array([0, 0, 0, 1, 1, 1, 1, 1], dtype=np.int32) if reset else None
    grads = oracle.gdr_backward(q, k, v, g, beta, dO, 0.7, si)
    base = dict(q=q, k=k, v=v, g=g, beta=beta)
    eps = 1e-6
    for name, gr in zip(("q", "k", "v", "g", "beta"), grads):
        arr = base[name]
        fd = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            a1, a2 = arr.copy(), arr.copy()
            a1[i] += eps
            a2[i] -= eps
            fd[i] = (np.sum(dO * oracle.gdr_forward(**dict(base, **{name: a1}), scale=0.7, seq_idx=si))
                     - np.sum(dO * oracle.gdr_forward(**dict(base, **{name: a2}), scale=0.7, seq_idx=si))) / (2 * eps)
        assert np.max(np.abs(fd - gr)) <= 1e-7 * np.max(np.abs(fd)), name
    if reset:
        assert np.all(grads[3][:, [0, 3]] == 0.0)


def test_gdr_segmented_equals_monolithic():
    rng = np.random.default_rng(45)
    q, k, v, g, beta = _gdr_inputs(rng, 2, 18, 2, 3, 2)
    mono = oracle.gdr_forward(q, k, v, g, beta, 0.6)
    for seg in ([0, 18], [0, 6, 12, 18], [0, 1, 5, 14, 18]):
        seg = np.array(seg, dtype=np.int32)
        M, dS = oracle.gdr_forward_prepare(k, v, g, beta, seg)
        S_in = oracle.gdr_compose_prefix(M, dS)
        out = np.empty_like(mono)
        for j in range(len(seg) - 1):
            sl = slice(seg[j], seg[j + 1])
            out[:, sl] = oracle.gdr_forward(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], 0.6,
                                            S0=S_in[j])
        np.testing.assert_allclose(out, mono, rtol=1e-12, atol=1e-12)
        assert np.all(M[0] == 0.0)  # the segment holding the row's first token
        for j in range(1, len(seg) - 1):  # M_j = A_last ... A_first, built here in numpy
            for b in range(2):
                for h in range(2):
                    P = np.eye(3)
                    for t in range(seg[j], seg[j + 1]):
                        kt = k[b, t, h]
                        P = np.exp(g[b, t, h]) * (np.eye(3) - beta[b, t, h] * np.outer(kt, kt)) @ P
                    np.testing.assert_allclose(M[j, b, h], P, rtol=1e-12, atol=1e-14)
