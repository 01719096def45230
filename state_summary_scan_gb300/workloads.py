"""Seeded synthetic workloads for chunkwise gated linear attention.

This module only draws random inputs; it holds none of the method's
arithmetic.  Both the fp64 oracle (through the tests and the bench's CPU leg)
and the CUDA path are fed from the tensors it returns, so the two sides always
see identical values.

Recipe (one torch CPU generator, seed 0, fixed draw order):
  1. packed workloads only: sequence lengths ~ U{512, ..., 8192}, drawn until
     their sum reaches T, the last one cut so the sum is exactly T;
  2. q ~ N(0, 1)                                   [B, T, H, Dk]
  3. k ~ N(0, 1), L2-normalised per (token, head)  [B, T, H, Dk]
  4. v ~ N(0, 1)                                   [B, T, H, Dv]
  5. g = logsigmoid(N(0, 1) + c), fp32             [B, T, H] ([B, T, H, Dk] with
     vector gates: one draw per key dimension)
  6. dO ~ N(0, 1)                                  [B, T, H, Dv]
All draws are fp32; q, k, v and dO are then rounded to the workload dtype.
The gate shift c is 3 for the tiny case, 4 for the 4k/32k/packed cases and 5
for the 256k case, so a segment's summed gate lies between about -45 and -62.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    Dk: int
    Dv: int
    dtype: str            # "f32" or "bf16": storage type of q, k, v, o, dO, dq, dk, dv
    num_segments: int
    chunk: int
    gate_shift: float
    packed: bool = False
    backward: bool = True
    seed: int = 0
    vector_gates: bool = False  # one gate per key dimension: g [B, T, H, Dk]

    @property
    def seg_len(self) -> int:
        return self.T // self.num_segments

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.Dk)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", B=1, T=256, H=2, Dk=32, Dv=32, dtype="f32",
                     num_segments=4, chunk=64, gate_shift=3.0),
    "fwd4k": Workload("fwd4k", B=2, T=4096, H=8, Dk=128, Dv=128, dtype="bf16",
                      num_segments=8, chunk=64, gate_shift=4.0, backward=False),
    "32k": Workload("32k", B=1, T=32768, H=16, Dk=128, Dv=128, dtype="bf16",
                    num_segments=16, chunk=64, gate_shift=4.0),
    "packed64k": Workload("packed64k", B=1, T=65536, H=32, Dk=128, Dv=128, dtype="bf16",
                          num_segments=32, chunk=64, gate_shift=4.0, packed=True),
    "256k": Workload("256k", B=1, T=262144, H=16, Dk=128, Dv=256, dtype="bf16",
                     num_segments=64, chunk=64, gate_shift=5.0),
    # The pages give no configuration for per-dimension gates; this one is the
    # 32k configuration with g [B, T, H, Dk] drawn the same way per dimension.
    "vg32k": Workload("vg32k", B=1, T=32768, H=16, Dk=128, Dv=128, dtype="bf16",
                      num_segments=16, chunk=64, gate_shift=4.0, vector_gates=True),
}


def draw_lengths(gen: torch.Generator, total: int, lo: int = 512, hi: int = 8192) -> list:
    """Sequence lengths ~ U{lo..hi} until they cover `total`; the last is cut."""
    lengths = []
    acc = 0
    while acc < total:
        n = int(torch.randint(lo, hi + 1, (1,), generator=gen).item())
        n = min(n, total - acc)
        lengths.append(n)
        acc += n
    return lengths


def cu_seqlens_from_lengths(lengths) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


@dataclasses.dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    dO: Optional[torch.Tensor]
    cu_seqlens: Optional[torch.Tensor]   # int32 [N+1] for packed workloads, else None


def make_inputs(w: Workload, with_grad: Optional[bool] = None,
                gate_shift: Optional[float] = None) -> Inputs:
    """Draw the workload's inputs on the CPU (deterministic for a given seed)."""
    if with_grad is None:
        with_grad = w.backward
    c = w.gate_shift if gate_shift is None else gate_shift
    gen = torch.Generator("cpu").manual_seed(w.seed)
    cu = None
    if w.packed:
        cu = cu_seqlens_from_lengths(draw_lengths(gen, w.T))
    dt = w.torch_dtype
    q = torch.randn(w.B, w.T, w.H, w.Dk, generator=gen, dtype=torch.float32)
    k = torch.randn(w.B, w.T, w.H, w.Dk, generator=gen, dtype=torch.float32)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    v = torch.randn(w.B, w.T, w.H, w.Dv, generator=gen, dtype=torch.float32)
    gshape = (w.B, w.T, w.H) + ((w.Dk,) if w.vector_gates else ())
    g = torch.nn.functional.logsigmoid(
        torch.randn(*gshape, generator=gen, dtype=torch.float32) + c)
    dO = None
    if with_grad:
        dO = torch.randn(w.B, w.T, w.H, w.Dv, generator=gen, dtype=torch.float32).to(dt)
    return Inputs(q=q.to(dt), k=k.to(dt), v=v.to(dt), g=g.contiguous(), dO=dO, cu_seqlens=cu)


def random_cu_seqlens(gen: torch.Generator, T: int, max_len: int) -> torch.Tensor:
    """Random packing of T tokens into sequences of length 1..max_len (test helper)."""
    lengths = []
    acc = 0
    while acc < T:
        n = int(torch.randint(1, max_len + 1, (1,), generator=gen).item())
        n = min(n, T - acc)
        lengths.append(n)
        acc += n
    return cu_seqlens_from_lengths(lengths)


# ------------------------------------------------------------------ Mamba2 SSD
# The pages name the Mamba2 SSD scan but give no workload for it; this one
# has the 32k configuration's size and shape on the path (N = Dk = 128,
# P = Dv = 128, 16 heads, 16 segments of 2048 tokens, bf16) with all heads in
# one group.  Recipe (one torch CPU generator, seed 0, this draw order):
#   x ~ N(0, 1) [B,T,H,P];  dt = softplus(N(0, 1) - 2) [B,T,H];
#   A = -(0.2 + 1.8 U(0, 1)) [H];  B, C ~ N(0, 1) / sqrt(N) [B,T,G,N];
#   D ~ N(0, 1) [H];  dy ~ N(0, 1) [B,T,H,P].
# Per-token decays exp(dt A) then average about exp(-0.19), so a 64-token
# chunk's summed gate lies between about -2 and -22.

@dataclasses.dataclass(frozen=True)
class SsdWorkload:
    name: str
    B: int
    T: int
    H: int
    G: int
    N: int
    P: int
    dtype: str
    num_segments: int
    chunk: int = 64
    seed: int = 0

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


SSD_WORKLOADS = {
    "ssd32k": SsdWorkload("ssd32k", B=1, T=32768, H=16, G=1, N=128, P=128, dtype="bf16",
                          num_segments=16),
}


@dataclasses.dataclass
class SsdInputs:
    x: torch.Tensor
    dt: torch.Tensor
    A: torch.Tensor
    Bm: torch.Tensor
    Cm: torch.Tensor
    D: torch.Tensor
    dy: torch.Tensor


def make_ssd_inputs(w: SsdWorkload) -> SsdInputs:
    gen = torch.Generator("cpu").manual_seed(w.seed)
    x = torch.randn(w.B, w.T, w.H, w.P, generator=gen)
    dt = torch.nn.functional.softplus(torch.randn(w.B, w.T, w.H, generator=gen) - 2.0)
    A = -(0.2 + 1.8 * torch.rand(w.H, generator=gen))
    Bm = torch.randn(w.B, w.T, w.G, w.N, generator=gen) / math.sqrt(w.N)
    Cm = torch.randn(w.B, w.T, w.G, w.N, generator=gen) / math.sqrt(w.N)
    D = torch.randn(w.H, generator=gen)
    dy = torch.randn(w.B, w.T, w.H, w.P, generator=gen)
    d = w.torch_dtype
    return SsdInputs(x.to(d), dt.contiguous(), A, Bm.to(d), Cm.to(d), D, dy.to(d))


# ------------------------------------------------------------------ gated delta rule
# The pages name the gated delta rule (its summaries carry a Dk x Dk
# transition) but give no workload for it.  This one has 8192 tokens, 16
# heads, Dk = Dv = 64 (the head size its generic kernels take) and 16
# segments of 512 tokens.  Recipe (one torch CPU generator, seed 0, this draw
# order): q ~ N(0,1); k ~ N(0,1) L2-normalised per (token, head); v ~ N(0,1);
# g = logsigmoid(N(0,1) + 4); beta = sigmoid(N(0,1)); dO ~ N(0,1); q, k, v, dO
# rounded to the dtype.

@dataclasses.dataclass(frozen=True)
class GdrWorkload:
    name: str
    B: int
    T: int
    H: int
    Dk: int
    Dv: int
    dtype: str
    num_segments: int
    chunk: int = 16
    gate_shift: float = 4.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.Dk)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


GDR_WORKLOADS = {
    "gdr8k": GdrWorkload("gdr8k", B=1, T=8192, H=16, Dk=64, Dv=64, dtype="bf16", num_segments=16),
}


@dataclasses.dataclass
class GdrInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    dO: torch.Tensor


def make_gdr_inputs(w: GdrWorkload) -> GdrInputs:
    gen = torch.Generator("cpu").manual_seed(w.seed)
    q = torch.randn(w.B, w.T, w.H, w.Dk, generator=gen)
    k = torch.randn(w.B, w.T, w.H, w.Dk, generator=gen)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    v = torch.randn(w.B, w.T, w.H, w.Dv, generator=gen)
    g = torch.nn.functional.logsigmoid(torch.randn(w.B, w.T, w.H, generator=gen) + w.gate_shift)
    beta = torch.sigmoid(torch.randn(w.B, w.T, w.H, generator=gen))
    dO = torch.randn(w.B, w.T, w.H, w.Dv, generator=gen)
    d = w.torch_dtype
    return GdrInputs(q.to(d), k.to(d), v.to(d), g.contiguous(), beta.contiguous(), dO.to(d))
