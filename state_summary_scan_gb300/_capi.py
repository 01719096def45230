"""ctypes binding of the C ABI in include/rm_cp.h (argument marshalling only).

Every function here has the name of the C entry point it calls and takes
torch tensors where the C call takes pointers.  All the arithmetic runs in the
CUDA library; there is no CPU or PyTorch fallback: if the library cannot be
loaded, or a call returns a non-OK status, a RuntimeError is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

RM_F32, RM_BF16 = 0, 1
STATUS_NAMES = {0: "RM_OK", 1: "RM_ERR_INVALID_ARG", 2: "RM_ERR_SHAPE", 3: "RM_ERR_ALIGNMENT",
                4: "RM_ERR_UNSUPPORTED", 5: "RM_ERR_METADATA", 6: "RM_ERR_CUDA",
                7: "RM_ERR_TIMEOUT"}

# every entry point declared in include/rm_cp.h
EXPORTS = (
    "rm_cp_build_packed_metadata", "rm_cp_validate", "rm_cp_workspace_size",
    "rm_cp_forward_prepare", "rm_cp_compose_prefix", "rm_cp_forward_apply", "rm_cp_forward_fused",
    "rm_cp_backward_prepare", "rm_cp_compose_suffix", "rm_cp_backward_apply",
    "rm_cp_status_string", "rm_cp_last_error", "rm_cp_path", "rm_cp_launch_count",
    "rm_cp_device_status", "rm_cp_selftest_wait_timeout", "rm_cp_backward_noalloc",
    "rm_cp_step_host", "rm_cp_event_create", "rm_cp_event_destroy",
    "rm_ssd_workspace_size", "rm_ssd_map_inputs", "rm_ssd_finish_forward", "rm_ssd_finish_backward",
    "rm_gdr_path", "rm_gdr_workspace_size", "rm_gdr_forward_prepare", "rm_gdr_compose_prefix",
    "rm_gdr_forward_apply",
    "rm_gdr_backward_prepare", "rm_gdr_compose_suffix", "rm_gdr_backward_apply",
)


class RmCpError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {detail}")
        self.status = status


class Problem(ctypes.Structure):
    """Mirror of rm_cp_problem."""
    _fields_ = [
        ("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
        ("Dk", ctypes.c_int32), ("Dv", ctypes.c_int32),
        ("num_segments", ctypes.c_int32), ("chunk", ctypes.c_int32),
        ("scale", ctypes.c_float), ("dtype", ctypes.c_int),
        ("seq_idx", ctypes.c_void_p), ("preceding_start", ctypes.c_void_p),
        ("following_stop", ctypes.c_void_p), ("q_heads", ctypes.c_int32),
        ("vector_gates", ctypes.c_int32),
    ]


class HostIO(ctypes.Structure):
    """Mirror of rm_cp_host_io."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "g", "dO", "o", "dq", "dk", "dv", "dg")]


class StepSet(ctypes.Structure):
    """Mirror of rm_cp_step_set."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "g", "dO", "o", "dq", "dk", "dv", "dg",
                                               "loaded", "computed", "drained")]


class StepState(ctypes.Structure):
    """Mirror of rm_cp_step_state."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("M", "dS", "S_in", "gamma", "dS_out", "ws")]


_P = ctypes.c_void_p
_PP = ctypes.POINTER(Problem)
_S = ctypes.c_int
_SIGS = {
    "rm_cp_build_packed_metadata": (_S, [_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                         _P, _P, _P, _P, _P]),
    "rm_cp_validate": (_S, [_PP]),
    "rm_cp_workspace_size": (ctypes.c_size_t, [_PP]),
    "rm_cp_forward_prepare": (_S, [_PP, _P, _P, _P, _P, _P, _P, _P]),
    "rm_cp_compose_prefix": (_S, [_PP, _P, _P, _P, _P]),
    "rm_cp_forward_apply": (_S, [_PP, _P, _P, _P, _P, _P, _P, _P, _P]),
    "rm_cp_forward_fused": (_S, [_PP] + [_P] * 10),
    "rm_cp_backward_prepare": (_S, [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "rm_cp_compose_suffix": (_S, [_PP, _P, _P, _P, _P]),
    "rm_cp_backward_apply": (_S, [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "rm_cp_status_string": (ctypes.c_char_p, [_S]),
    "rm_cp_last_error": (ctypes.c_char_p, []),
    "rm_cp_path": (ctypes.c_int32, [_PP]),
    "rm_cp_launch_count": (ctypes.c_uint64, []),
    "rm_cp_device_status": (_S, [_P, ctypes.c_int32, _P]),
    "rm_cp_selftest_wait_timeout": (_S, [ctypes.c_uint32, _P]),
    "rm_cp_backward_noalloc": (_S, [_PP] + [_P] * 14),
    "rm_cp_step_host": (_S, [_PP, ctypes.POINTER(HostIO), ctypes.POINTER(StepSet),
                             ctypes.POINTER(StepState), _P, _P, _P]),
    "rm_cp_event_create": (_S, [ctypes.POINTER(ctypes.c_void_p)]),
    "rm_cp_event_destroy": (_S, [_P]),
    "rm_ssd_workspace_size": (ctypes.c_size_t, [_PP]),
    "rm_ssd_map_inputs": (_S, [_PP, ctypes.c_int32] + [_P] * 8),
    "rm_ssd_finish_forward": (_S, [_PP, _P, _P, _P, _P]),
    "rm_ssd_finish_backward": (_S, [_PP, ctypes.c_int32] + [_P] * 17),
    "rm_gdr_path": (ctypes.c_int32, [_PP]),
    "rm_gdr_workspace_size": (ctypes.c_size_t, [_PP]),
    "rm_gdr_forward_prepare": (_S, [_PP] + [_P] * 8),
    "rm_gdr_compose_prefix": (_S, [_PP] + [_P] * 4),
    "rm_gdr_forward_apply": (_S, [_PP] + [_P] * 9),
    "rm_gdr_backward_prepare": (_S, [_PP] + [_P] * 11),
    "rm_gdr_compose_suffix": (_S, [_PP] + [_P] * 4),
    "rm_gdr_backward_apply": (_S, [_PP] + [_P] * 13),
}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_needed: bool = True):
    """Load librmcp.so (building it in-tree first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_needed else _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library not built: {path}")
            so = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(so, name)
                fn.restype = res
                fn.argtypes = args
            _lib = so
    return _lib


def _check(status: int):
    if status != 0:
        raise RmCpError(status, load().rm_cp_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the C ABI must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(handle)


class ProblemSpec:
    """An rm_cp_problem plus references to the device metadata it points at."""

    def __init__(self, B, T, H, Dk, Dv, num_segments, chunk, scale, dtype,
                 seq_idx: Optional[torch.Tensor] = None,
                 preceding_start: Optional[torch.Tensor] = None,
                 following_stop: Optional[torch.Tensor] = None, q_heads: int = 0,
                 vector_gates: int = 0):
        if isinstance(dtype, torch.dtype):
            dtype = RM_F32 if dtype == torch.float32 else RM_BF16 if dtype == torch.bfloat16 else -1
        self._keep = (seq_idx, preceding_start, following_stop)
        for t in self._keep:
            if t is not None and (t.dtype != torch.int32 or not t.is_contiguous()):
                raise ValueError("metadata tensors must be contiguous int32")
        self.c = Problem(int(B), int(T), int(H), int(Dk), int(Dv), int(num_segments), int(chunk),
                         float(scale), int(dtype),
                         None if seq_idx is None else seq_idx.data_ptr(),
                         None if preceding_start is None else preceding_start.data_ptr(),
                         None if following_stop is None else following_stop.data_ptr(),
                         int(q_heads), int(vector_gates))

    @property
    def ref(self):
        return ctypes.byref(self.c)

    def __getattr__(self, name):
        return getattr(self.__dict__["c"], name)


# ----------------------------------------------------------------- C calls

def rm_cp_validate(p: ProblemSpec) -> None:
    _check(load().rm_cp_validate(p.ref))


def rm_cp_path(p: ProblemSpec) -> int:
    return int(load().rm_cp_path(p.ref))


def rm_cp_launch_count() -> int:
    return int(load().rm_cp_launch_count())


def rm_cp_device_status(dev_scratch: torch.Tensor, clear: bool = True, stream=None) -> int:
    """Returns the status code (0 = RM_OK, 7 = RM_ERR_TIMEOUT); synchronises the stream."""
    return int(load().rm_cp_device_status(_ptr(dev_scratch), int(clear), _stream(stream)))


def rm_cp_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    _check(load().rm_cp_selftest_wait_timeout(int(limit_us), _stream(stream)))


def rm_cp_workspace_size(p: ProblemSpec) -> int:
    return int(load().rm_cp_workspace_size(p.ref))


def rm_cp_build_packed_metadata(cu_seqlens, T: int, num_segments: int) -> dict:
    """Host metadata builder; returns CPU int32 tensors."""
    cu = torch.as_tensor(cu_seqlens, dtype=torch.int32).contiguous().cpu()
    nseqs = cu.numel() - 1
    seq_idx = torch.empty(T, dtype=torch.int32)
    local_cu = torch.empty(nseqs + 2 * num_segments, dtype=torch.int32)
    local_off = torch.empty(num_segments + 1, dtype=torch.int32)
    pre = torch.empty(num_segments, dtype=torch.int32)
    fol = torch.empty(num_segments, dtype=torch.int32)
    _check(load().rm_cp_build_packed_metadata(_ptr(cu), nseqs, int(T), int(num_segments),
                                              _ptr(seq_idx), _ptr(local_cu), _ptr(local_off),
                                              _ptr(pre), _ptr(fol)))
    n = int(local_off[-1])
    return dict(seq_idx=seq_idx, local_cu_seqlens=local_cu[:n].clone(),
                local_cu_offsets=local_off, preceding_start=pre, following_stop=fol)


def rm_cp_forward_prepare(p, k, v, g, M, dS, ws=None, stream=None):
    _check(load().rm_cp_forward_prepare(p.ref, _ptr(k), _ptr(v), _ptr(g), _ptr(M), _ptr(dS),
                                        _ptr(ws), _stream(stream)))


def rm_cp_compose_prefix(p, M, dS, S_in, stream=None):
    _check(load().rm_cp_compose_prefix(p.ref, _ptr(M), _ptr(dS), _ptr(S_in), _stream(stream)))


def rm_cp_forward_apply(p, q, k, v, g, S_in, o, ws=None, stream=None):
    _check(load().rm_cp_forward_apply(p.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(S_in),
                                      _ptr(o), _ptr(ws), _stream(stream)))


def rm_cp_forward_fused(p, q, k, v, g, M, dS, S_in, o, ws, stream=None):
    """The three forward calls in one (one launch on the tensor-core path)."""
    _check(load().rm_cp_forward_fused(p.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(M), _ptr(dS),
                                      _ptr(S_in), _ptr(o), _ptr(ws), _stream(stream)))


def rm_cp_backward_prepare(p, q, k, v, g, S_in, dO, gamma, dq, ws, stream=None):
    _check(load().rm_cp_backward_prepare(p.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(S_in),
                                         _ptr(dO), _ptr(gamma), _ptr(dq), _ptr(ws),
                                         _stream(stream)))


def rm_cp_compose_suffix(p, M, gamma, dS_out, stream=None):
    _check(load().rm_cp_compose_suffix(p.ref, _ptr(M), _ptr(gamma), _ptr(dS_out),
                                       _stream(stream)))


def rm_cp_backward_apply(p, q, k, v, g, dO, S_in, dS_out, dk, dv, dg, ws, stream=None):
    _check(load().rm_cp_backward_apply(p.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(dO),
                                       _ptr(S_in), _ptr(dS_out), _ptr(dk), _ptr(dv), _ptr(dg),
                                       _ptr(ws), _stream(stream)))


def rm_cp_backward_noalloc(p, q, k, v, g, S_in, M, dO, gamma, dS_out, dq, dk, dv, dg, stream=None):
    """The whole backward with the library's own fixed scratch (no workspace)."""
    _check(load().rm_cp_backward_noalloc(p.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(S_in),
                                         _ptr(M), _ptr(dO), _ptr(gamma), _ptr(dS_out), _ptr(dq),
                                         _ptr(dk), _ptr(dv), _ptr(dg), _stream(stream)))


def rm_cp_event_create() -> int:
    """A timing-free CUDA event on the current device (raw handle)."""
    ev = ctypes.c_void_p()
    _check(load().rm_cp_event_create(ctypes.byref(ev)))
    return int(ev.value)


def rm_cp_event_destroy(event: int) -> None:
    _check(load().rm_cp_event_destroy(ctypes.c_void_p(event)))


def _host_ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the C ABI must be contiguous")
    return t.data_ptr()


def rm_cp_step_host(p, host: dict, dev: dict, events, state: dict, compute=None, h2d=None, d2h=None):
    """One step from host buffers.  host and dev map q, k, v, g, dO (inputs)
    and o, dq, dk, dv, dg (outputs) to pinned host / device tensors (dO and
    the gradients absent for a forward step); events = (loaded, computed,
    drained) handles of this device set; state maps M, dS, S_in, gamma,
    dS_out, ws to device tensors."""
    names = ("q", "k", "v", "g", "dO", "o", "dq", "dk", "dv", "dg")
    h = HostIO(*(_host_ptr(host.get(n)) for n in names))
    d = StepSet(*(_host_ptr(dev.get(n)) for n in names), *(int(e) for e in events))
    st = StepState(*(_host_ptr(state.get(n)) for n in ("M", "dS", "S_in", "gamma", "dS_out", "ws")))
    _check(load().rm_cp_step_host(p.ref, ctypes.byref(h), ctypes.byref(d), ctypes.byref(st),
                                  _stream(compute), _stream(h2d), _stream(d2h)))


def rm_ssd_workspace_size(p: ProblemSpec) -> int:
    return int(load().rm_ssd_workspace_size(p.ref))


def rm_ssd_map_inputs(p, G, dt, A, Bm, Cm, q, k, g, stream=None):
    _check(load().rm_ssd_map_inputs(p.ref, int(G), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(q),
                                    _ptr(k), _ptr(g), _stream(stream)))


def rm_ssd_finish_forward(p, x, D, o, stream=None):
    _check(load().rm_ssd_finish_forward(p.ref, _ptr(x), _ptr(D), _ptr(o), _stream(stream)))


def rm_ssd_finish_backward(p, G, x, dt, A, Bm, dy, D, dq, dk, dv, dg, ddt, dA, dB, dC, dD, ws,
                           stream=None):
    _check(load().rm_ssd_finish_backward(p.ref, int(G), _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm),
                                         _ptr(dy), _ptr(D), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
                                         _ptr(ddt), _ptr(dA), _ptr(dB), _ptr(dC), _ptr(dD),
                                         _ptr(ws), _stream(stream)))


# ----------------------------------------------------------------- gated delta rule

def rm_gdr_path(p: ProblemSpec) -> int:
    return int(load().rm_gdr_path(p.ref))


def rm_gdr_workspace_size(p: ProblemSpec) -> int:
    return int(load().rm_gdr_workspace_size(p.ref))


def rm_gdr_forward_prepare(p, k, v, g, beta, M, dS, ws, stream=None):
    _check(load().rm_gdr_forward_prepare(p.ref, _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(M),
                                         _ptr(dS), _ptr(ws), _stream(stream)))


def rm_gdr_compose_prefix(p, M, dS, S_in, stream=None):
    _check(load().rm_gdr_compose_prefix(p.ref, _ptr(M), _ptr(dS), _ptr(S_in), _stream(stream)))


def rm_gdr_forward_apply(p, q, k, v, g, beta, S_in, o, ws, stream=None):
    _check(load().rm_gdr_forward_apply(p.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                       _ptr(S_in), _ptr(o), _ptr(ws), _stream(stream)))


def rm_gdr_backward_prepare(p, q, k, v, g, beta, S_in, dO, gamma, dq, ws, stream=None):
    _check(load().rm_gdr_backward_prepare(p.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                          _ptr(S_in), _ptr(dO), _ptr(gamma), _ptr(dq), _ptr(ws),
                                          _stream(stream)))


def rm_gdr_compose_suffix(p, M, gamma, dS_out, stream=None):
    _check(load().rm_gdr_compose_suffix(p.ref, _ptr(M), _ptr(gamma), _ptr(dS_out), _stream(stream)))


def rm_gdr_backward_apply(p, q, k, v, g, beta, dO, dS_out, dk, dv, dg, dbeta, ws, stream=None):
    _check(load().rm_gdr_backward_apply(p.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                        _ptr(dO), _ptr(dS_out), _ptr(dk), _ptr(dv), _ptr(dg),
                                        _ptr(dbeta), _ptr(ws), _stream(stream)))
