"""fp64 CPU oracle for chunkwise gated linear attention with segment summaries.

TEST INFRASTRUCTURE ONLY: imported by tests, by the smoke check and by the
benchmark's CPU-baseline leg, never by the library.  It shares no code with
the CUDA path.  The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP
over independent (segment,) row, head tasks); this module only converts
arrays to float64, allocates outputs and calls it through ctypes.

Every function follows the Megatron-Core API docs page
"core.ssm.context_parallel.chunkwise" for the summary algebra
(CPForwardUnpackedSummary: S_out = M S_in + delta_S; CPBackwardUnpackedSummary:
dS_in = M^T dS_out + gamma; LinearAttentionCPBackend prepare/apply;
PackedSequenceCPMetadata) and the gated recurrence
S_t = exp(g_t) S_{t-1} + k_t v_t^T, o_t = scale S_t^T q_t for the local work.

vg_forward / vg_backward / vg_forward_prepare / vg_compose_prefix are the
same recurrence with one gate per key dimension (a diagonal transition M).

gdr_forward / gdr_backward / gdr_forward_prepare / gdr_compose_prefix are the
gated delta rule, whose segment transitions are Dk x Dk matrices.

ssd_forward / ssd_backward are the Mamba2 SSD scan (named by the
context-parallel pages as the other user of exact state passing), written
from the published SSD recurrence.

Parity status: every function here is pinned by tests/test_oracle_pins.py
(closed forms, finite differences, textbook special cases, segmentation and
reset invariants, brute-force metadata); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.c_void_p
_I = ctypes.c_int
_D = ctypes.c_double

_SIGS = {
    "oracle_set_threads": (_I, [_I]),
    "oracle_forward": (None, [_I, _I, _I, _I, _I, _D, _P, _P, _P, _P, _P, _P]),
    "oracle_backward": (None, [_I, _I, _I, _I, _I, _D, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "oracle_backward_direct": (None, [_I, _I, _I, _I, _I, _D, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "oracle_forward_prepare": (None, [_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "oracle_compose_prefix": (None, [_I, _I, _I, _I, _P, _P, _P, _P]),
    "oracle_forward_apply": (None, [_I, _I, _I, _I, _I, _I, _P, _D, _P, _P, _P, _P, _P, _P, _P]),
    "oracle_backward_prepare": (None, [_I, _I, _I, _I, _I, _I, _P, _D, _P, _P, _P, _P, _P]),
    "oracle_compose_suffix": (None, [_I, _I, _I, _I, _P, _P, _P, _P]),
    "oracle_backward_apply": (None, [_I, _I, _I, _I, _I, _I, _P, _D, _P, _P, _P, _P, _P, _P,
                                     _P, _P, _P, _P, _P, _P]),
    "oracle_packed_metadata": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "oracle_ssd_forward": (None, [_I] * 6 + [_P] * 8),
    "oracle_vg_forward": (None, [_I] * 5 + [_D] + [_P] * 7),
    "oracle_vg_backward": (None, [_I] * 5 + [_D] + [_P] * 6 + [_I] + [_P] * 4),
    "oracle_vg_forward_prepare": (None, [_I] * 6 + [_P] * 7),
    "oracle_gdr_forward": (None, [_I] * 5 + [_D] + [_P] * 8),
    "oracle_gdr_backward": (None, [_I] * 5 + [_D] + [_P] * 12),
    "oracle_gdr_forward_prepare": (None, [_I] * 6 + [_P] * 8),
    "oracle_ssd_backward": (None, [_I] * 6 + [_P] * 14),
}


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            so = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(so, name)
                fn.restype = res
                fn.argtypes = args
            _lib = so
    return _lib


def set_threads(n: int = 0) -> int:
    """Set the OpenMP thread count (n <= 0 keeps it); returns the count in use."""
    return int(lib().oracle_set_threads(int(n)))


# ---------------------------------------------------------------- helpers

def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _i32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dims(q, v):
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    return B, T, H, Dk, Dv


def equal_segments(T: int, nseg: int) -> np.ndarray:
    assert T % nseg == 0
    return np.arange(nseg + 1, dtype=np.int32) * (T // nseg)


def _seg(seg_starts, T):
    s = _i32(seg_starts)
    assert s[0] == 0 and s[-1] == T and np.all(np.diff(s) > 0)
    return s


# ---------------------------------------------------------------- monolithic

def forward(q, k, v, g, scale, seq_idx=None):
    """o [B,T,H,Dv] of the token recurrence (fp64)."""
    q, k, v, g, si = _f64(q), _f64(k), _f64(v), _f64(g), _i32(seq_idx)
    B, T, H, Dk, Dv = _dims(q, v)
    o = np.empty((B, T, H, Dv))
    lib().oracle_forward(B, T, H, Dk, Dv, float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                         _ptr(si), _ptr(o))
    return o


def backward(q, k, v, g, dO, scale, seq_idx=None, direct=False):
    """(dq, dk, dv, dg) of L = sum dO . o.  direct=True uses the stored-state
    gate gradient alpha_t <S_{t-1}, D_t> (small inputs only)."""
    q, k, v, g, dO, si = _f64(q), _f64(k), _f64(v), _f64(g), _f64(dO), _i32(seq_idx)
    B, T, H, Dk, Dv = _dims(q, v)
    dq = np.empty((B, T, H, Dk))
    dk = np.empty((B, T, H, Dk))
    dv = np.empty((B, T, H, Dv))
    dg = np.empty((B, T, H))
    fn = lib().oracle_backward_direct if direct else lib().oracle_backward
    fn(B, T, H, Dk, Dv, float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(si), _ptr(dO),
       _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg))
    return dq, dk, dv, dg


# ---------------------------------------------------------------- segmented

def forward_prepare(k, v, g, seg_starts, seq_idx=None):
    """(M [nseg,B,H], dS [nseg,B,H,Dk,Dv]) with zero incoming state."""
    k, v, g, si = _f64(k), _f64(v), _f64(g), _i32(seq_idx)
    B, T, H, Dk, Dv = _dims(k, v)
    s = _seg(seg_starts, T)
    nseg = len(s) - 1
    M = np.empty((nseg, B, H))
    dS = np.empty((nseg, B, H, Dk, Dv))
    lib().oracle_forward_prepare(B, T, H, Dk, Dv, nseg, _ptr(s), _ptr(k), _ptr(v), _ptr(g),
                                 _ptr(si), _ptr(M), _ptr(dS))
    return M, dS


def compose_prefix(M, dS, preceding_start=None):
    M, dS, pre = _f64(M), _f64(dS), _i32(preceding_start)
    nseg, B, H, Dk, Dv = dS.shape
    S_in = np.empty_like(dS)
    lib().oracle_compose_prefix(nseg, B * H, Dk, Dv, _ptr(M), _ptr(dS), _ptr(pre), _ptr(S_in))
    return S_in


def forward_apply(q, k, v, g, S_in, scale, seg_starts, seq_idx=None):
    q, k, v, g, S_in, si = _f64(q), _f64(k), _f64(v), _f64(g), _f64(S_in), _i32(seq_idx)
    B, T, H, Dk, Dv = _dims(q, v)
    s = _seg(seg_starts, T)
    o = np.empty((B, T, H, Dv))
    lib().oracle_forward_apply(B, T, H, Dk, Dv, len(s) - 1, _ptr(s), float(scale), _ptr(q),
                               _ptr(k), _ptr(v), _ptr(g), _ptr(si), _ptr(S_in), _ptr(o))
    return o


def backward_prepare(q, g, dO, scale, seg_starts, seq_idx=None):
    q, g, dO, si = _f64(q), _f64(g), _f64(dO), _i32(seq_idx)
    B, T, H, Dk, Dv = _dims(q, dO)
    s = _seg(seg_starts, T)
    nseg = len(s) - 1
    gamma = np.empty((nseg, B, H, Dk, Dv))
    lib().oracle_backward_prepare(B, T, H, Dk, Dv, nseg, _ptr(s), float(scale), _ptr(q), _ptr(g),
                                  _ptr(si), _ptr(dO), _ptr(gamma))
    return gamma


def compose_suffix(M, gamma, following_stop=None):
    M, gamma, fol = _f64(M), _f64(gamma), _i32(following_stop)
    nseg, B, H, Dk, Dv = gamma.shape
    dS_out = np.empty_like(gamma)
    lib().oracle_compose_suffix(nseg, B * H, Dk, Dv, _ptr(M), _ptr(gamma), _ptr(fol), _ptr(dS_out))
    return dS_out


def backward_apply(q, k, v, g, dO, S_in, dS_out, scale, seg_starts, seq_idx=None):
    q, k, v, g, dO = _f64(q), _f64(k), _f64(v), _f64(g), _f64(dO)
    S_in, dS_out, si = _f64(S_in), _f64(dS_out), _i32(seq_idx)
    B, T, H, Dk, Dv = _dims(q, v)
    s = _seg(seg_starts, T)
    dq = np.empty((B, T, H, Dk))
    dk = np.empty((B, T, H, Dk))
    dv = np.empty((B, T, H, Dv))
    dg = np.empty((B, T, H))
    lib().oracle_backward_apply(B, T, H, Dk, Dv, len(s) - 1, _ptr(s), float(scale), _ptr(q),
                                _ptr(k), _ptr(v), _ptr(g), _ptr(si), _ptr(dO), _ptr(S_in),
                                _ptr(dS_out), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg))
    return dq, dk, dv, dg


def packed_metadata(cu_seqlens, T, seg_starts):
    """Brute-force PackedSequenceCPMetadata for every segment.

    Returns dict(seq_idx [T], local_cu_seqlens (list of int32 arrays, one per
    segment), preceding_start [nseg], following_stop [nseg])."""
    cu = _i32(cu_seqlens)
    s = _seg(seg_starts, T)
    nseg = len(s) - 1
    nseqs = len(cu) - 1
    seq_idx = np.empty(T, dtype=np.int32)
    local_cu = np.empty(nseqs + 2 * nseg, dtype=np.int32)
    local_off = np.empty(nseg + 1, dtype=np.int32)
    pre = np.empty(nseg, dtype=np.int32)
    fol = np.empty(nseg, dtype=np.int32)
    rc = lib().oracle_packed_metadata(_ptr(cu), nseqs, T, nseg, _ptr(s), _ptr(seq_idx),
                                      _ptr(local_cu), _ptr(local_off), _ptr(pre), _ptr(fol))
    if rc != 0:
        raise ValueError("cu_seqlens must satisfy 0 = cu[0] < cu[1] < ... < cu[-1] = T")
    locals_ = [local_cu[local_off[j]:local_off[j + 1]].copy() for j in range(nseg)]
    return dict(seq_idx=seq_idx, local_cu_seqlens=locals_, preceding_start=pre,
                following_stop=fol)


def segmented_forward(q, k, v, g, scale, seg_starts, seq_idx=None, preceding_start=None):
    """prepare -> compose_prefix -> apply; returns (o, dict of intermediates)."""
    M, dS = forward_prepare(k, v, g, seg_starts, seq_idx)
    S_in = compose_prefix(M, dS, preceding_start)
    o = forward_apply(q, k, v, g, S_in, scale, seg_starts, seq_idx)
    return o, dict(M=M, dS=dS, S_in=S_in)


def segmented_backward(q, k, v, g, dO, scale, seg_starts, seq_idx=None,
                       preceding_start=None, following_stop=None, S_in=None, M=None):
    """Mirror of segmented_forward; returns ((dq, dk, dv, dg), intermediates)."""
    if S_in is None or M is None:
        M, dS = forward_prepare(k, v, g, seg_starts, seq_idx)
        S_in = compose_prefix(M, dS, preceding_start)
    gamma = backward_prepare(q, g, dO, scale, seg_starts, seq_idx)
    dS_out = compose_suffix(M, gamma, following_stop)
    grads = backward_apply(q, k, v, g, dO, S_in, dS_out, scale, seg_starts, seq_idx)
    return grads, dict(M=M, S_in=S_in, gamma=gamma, dS_out=dS_out)


# ---------------------------------------------------------------- Mamba2 SSD

def ssd_forward(x, dt, A, Bm, Cm, D=None, seq_idx=None):
    """y [B,T,H,P] of the Mamba2 SSD scan h_t = exp(dt_t A_h) h_{t-1} +
    dt_t B_t x_t^T, y_t = h_t^T C_t + D_h x_t (fp64; B_t, C_t shared by the
    H / G heads of a group)."""
    x, dt, A, Bm, Cm, D, si = (_f64(x), _f64(dt), _f64(A), _f64(Bm), _f64(Cm), _f64(D),
                               _i32(seq_idx))
    B, T, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    assert H % G == 0 and Cm.shape == Bm.shape and dt.shape == (B, T, H) and A.shape == (H,)
    y = np.empty((B, T, H, P))
    lib().oracle_ssd_forward(B, T, H, G, N, P, _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm),
                             _ptr(D), _ptr(si), _ptr(y))
    return y


def ssd_backward(x, dt, A, Bm, Cm, dy, D=None, seq_idx=None):
    """(dx, ddt, dA, dB, dC, dD) of L = sum dy . y for ssd_forward (dD is zeros
    of [H] when D is None)."""
    x, dt, A, Bm, Cm, dy, D, si = (_f64(x), _f64(dt), _f64(A), _f64(Bm), _f64(Cm), _f64(dy),
                                   _f64(D), _i32(seq_idx))
    B, T, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    dx = np.empty((B, T, H, P))
    ddt = np.empty((B, T, H))
    dA = np.empty(H)
    dB = np.empty((B, T, G, N))
    dC = np.empty((B, T, G, N))
    dD = np.empty(H)
    lib().oracle_ssd_backward(B, T, H, G, N, P, _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm),
                              _ptr(D), _ptr(si), _ptr(dy), _ptr(dx), _ptr(ddt), _ptr(dA),
                              _ptr(dB), _ptr(dC), _ptr(dD))
    return dx, ddt, dA, dB, dC, dD


# ---------------------------------------------------------------- vector gates

def vg_forward(q, k, v, g, scale, seq_idx=None, S0=None):
    """o [B,T,H,Dv] of S_t = diag(exp(g_t)) S_{t-1} + k_t v_t^T, o_t = scale S_t^T q_t
    with g [B,T,H,Dk] (fp64).  S0 [B,H,Dk,Dv]: the state before token 0, which then
    continues it (no reset at token 0)."""
    q, k, v, g, si, S0 = _f64(q), _f64(k), _f64(v), _f64(g), _i32(seq_idx), _f64(S0)
    B, T, H, Dk, Dv = _dims(q, v)
    assert g.shape == (B, T, H, Dk)
    o = np.empty((B, T, H, Dv))
    lib().oracle_vg_forward(B, T, H, Dk, Dv, float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                            _ptr(si), _ptr(S0), _ptr(o))
    return o


def vg_backward(q, k, v, g, dO, scale, seq_idx=None, direct=False):
    """(dq, dk, dv, dg [B,T,H,Dk]) of L = sum dO . o for vg_forward (S0 = 0)."""
    q, k, v, g, dO, si = _f64(q), _f64(k), _f64(v), _f64(g), _f64(dO), _i32(seq_idx)
    B, T, H, Dk, Dv = _dims(q, v)
    dq, dk = np.empty((B, T, H, Dk)), np.empty((B, T, H, Dk))
    dv, dg = np.empty((B, T, H, Dv)), np.empty((B, T, H, Dk))
    lib().oracle_vg_backward(B, T, H, Dk, Dv, float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                             _ptr(si), _ptr(dO), int(bool(direct)), _ptr(dq), _ptr(dk), _ptr(dv),
                             _ptr(dg))
    return dq, dk, dv, dg


def vg_forward_prepare(k, v, g, seg_starts, seq_idx=None):
    """(M [nseg,B,H,Dk], dS [nseg,B,H,Dk,Dv]): each segment's diagonal transition
    and its end state from a zero incoming state."""
    k, v, g, si = _f64(k), _f64(v), _f64(g), _i32(seq_idx)
    B, T, H, Dk, Dv = _dims(k, v)
    seg = _seg(seg_starts, T)
    nseg = len(seg) - 1
    M = np.empty((nseg, B, H, Dk))
    dS = np.empty((nseg, B, H, Dk, Dv))
    lib().oracle_vg_forward_prepare(B, T, H, Dk, Dv, nseg, _ptr(seg), _ptr(k), _ptr(v), _ptr(g),
                                    _ptr(si), _ptr(M), _ptr(dS))
    return M, dS


def vg_compose_prefix(M, dS):
    """S_in[j]: segments [0, j) applied in order to a zero state, S <- diag(M_i) S + dS_i."""
    S = np.zeros(dS.shape[1:])
    out = np.empty_like(dS)
    for j in range(dS.shape[0]):
        out[j] = S
        S = M[j][..., None] * S + dS[j]
    return out


# ---------------------------------------------------------------- gated delta rule

def gdr_forward(q, k, v, g, beta, scale, seq_idx=None, S0=None):
    """o of S_t = exp(g_t)(I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
    o_t = scale S_t^T q_t (fp64); g, beta [B,T,H].  S0 [B,H,Dk,Dv]: the state
    before token 0, which then continues it (no reset at token 0)."""
    q, k, v, g, be, si, S0 = (_f64(q), _f64(k), _f64(v), _f64(g), _f64(beta), _i32(seq_idx),
                              _f64(S0))
    B, T, H, Dk, Dv = _dims(q, v)
    o = np.empty((B, T, H, Dv))
    lib().oracle_gdr_forward(B, T, H, Dk, Dv, float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                             _ptr(be), _ptr(si), _ptr(S0), _ptr(o))
    return o


def gdr_backward(q, k, v, g, beta, dO, scale, seq_idx=None):
    """(dq, dk, dv, dg, dbeta) of L = sum dO . o for gdr_forward (small inputs:
    every state is stored)."""
    q, k, v, g, be, dO, si = (_f64(q), _f64(k), _f64(v), _f64(g), _f64(beta), _f64(dO),
                              _i32(seq_idx))
    B, T, H, Dk, Dv = _dims(q, v)
    dq, dk, dv = np.empty((B, T, H, Dk)), np.empty((B, T, H, Dk)), np.empty((B, T, H, Dv))
    dg, db = np.empty((B, T, H)), np.empty((B, T, H))
    lib().oracle_gdr_backward(B, T, H, Dk, Dv, float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                              _ptr(be), _ptr(si), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
                              _ptr(db))
    return dq, dk, dv, dg, db


def gdr_forward_prepare(k, v, g, beta, seg_starts, seq_idx=None):
    """(M [nseg,B,H,Dk,Dk], dS [nseg,B,H,Dk,Dv]): each segment's transition
    (the ordered product of its A_t) and its end state from a zero state."""
    k, v, g, be, si = _f64(k), _f64(v), _f64(g), _f64(beta), _i32(seq_idx)
    B, T, H, Dk, Dv = _dims(k, v)
    seg = _seg(seg_starts, T)
    nseg = len(seg) - 1
    M = np.empty((nseg, B, H, Dk, Dk))
    dS = np.empty((nseg, B, H, Dk, Dv))
    lib().oracle_gdr_forward_prepare(B, T, H, Dk, Dv, nseg, _ptr(seg), _ptr(k), _ptr(v), _ptr(g),
                                     _ptr(be), _ptr(si), _ptr(M), _ptr(dS))
    return M, dS


def gdr_compose_prefix(M, dS):
    """S_in[j]: segments [0, j) applied in order to a zero state, S <- M_i S + dS_i."""
    S = np.zeros(dS.shape[1:])
    out = np.empty_like(dS)
    for j in range(dS.shape[0]):
        out[j] = S
        S = M[j] @ S + dS[j]
    return out
