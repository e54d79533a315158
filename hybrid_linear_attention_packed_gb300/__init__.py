"""Packed linear-attention pass (and the hybrid model's softmax layer over the
same packed rows) for GB300 (sm_103a).

The compute path is ``libspanla.so`` (hand-written CUDA kernels behind the C
ABI in ``include/spanla.h``); :mod:`.spanla` is its thin Python binding,
:mod:`.sharding` the host side of splitting a pass across ranks by request,
and :mod:`.workloads` the seeded synthetic inputs.
"""
from .spanla import (  # noqa: F401
    SpanLAError,
    ViewStateCache,
    load_library,
    span_la_branches_from_state,
    span_la_check,
    span_la_pass,
    span_la_pass_noalloc,
    span_la_plan_prepare,
    span_la_softmax_branches_from_kv,
    span_la_softmax_pass,
)
