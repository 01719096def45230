"""GB300-native chunkwise gated linear attention with per-segment affine
state summaries.

Layers:
  include/rm_cp.h          the C ABI (six compute calls + metadata builder)
  csrc/*.cu                sm_103a kernels behind it (librmcp.so, built in-tree)
  _capi                    ctypes binding, one Python function per C call
  api                      buffer allocation, call sequence, autograd adapter
  workloads                seeded synthetic inputs (no method arithmetic)
"""
from . import _capi  # noqa: F401
from ._capi import RmCpError, ProblemSpec, load  # noqa: F401
from .api import (Plan, make_plan, plan_like, forward, backward,  # noqa: F401
                  chunkwise_gla, ChunkwiseGatedLinearAttention, GdrPlan, make_gdr_plan,
                  gdr_forward, gdr_backward, gated_delta_rule, GatedDeltaRule)
from .build import build as build_library  # noqa: F401

__all__ = ["RmCpError", "ProblemSpec", "load", "Plan", "make_plan", "plan_like", "forward",
           "backward", "chunkwise_gla", "ChunkwiseGatedLinearAttention", "GdrPlan", "make_gdr_plan",
           "gdr_forward", "gdr_backward", "gated_delta_rule", "GatedDeltaRule", "build_library"]
