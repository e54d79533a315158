"""The no-allocation entry point against the regular one.

``span_la_pass_noalloc`` serves callers that cannot allocate device memory
while a pass runs (a process that gave the GPU's memory to its own pool, or
code where an allocation could block or fail at the wrong moment): it runs the
same pass in a fixed workspace that the library owns.  These tests call it
through the C ABI and compare two calls in a row with ``span_la_pass`` on the
same inputs, within the tolerance of the other parity tests.  This file is
named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from hybrid_linear_attention_packed_gb300 import spanla, workloads

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2


def _i32p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if a.size else None


def _noalloc(lib, w, q, k, v, out, state):
    vcu = np.ascontiguousarray(w.view_cu, dtype=np.int32)
    bcu = np.ascontiguousarray(w.branch_cu, dtype=np.int32)
    par = np.ascontiguousarray(w.branch_parent, dtype=np.int32)
    dims = spanla.Dims(q.shape[0], q.shape[1], 64, spanla.SPAN_LA_BF16)
    st = lib.span_la_pass_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), dims, _i32p(vcu),
                                  len(vcu) - 1, _i32p(bcu), len(bcu) - 1, _i32p(par),
                                  out.data_ptr(), state.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    return st, lib.span_la_last_error_detail().decode()


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).abs().max() / b.abs().max())


def test_noalloc_matches_span_la_pass_on_two_calls_in_a_row(cuda_device):
    lib = spanla.load_library()
    cases = [workloads.single_request(3),
             workloads.make_pass([300, 129, 64], [20, 50, 200, 7], [0, 0, 1, 2], H=4,
                                 dtype="bf16", seed=31)]
    for w in cases:   # two calls in a row, on different passes
        q, k, v = (t.to(cuda_device).contiguous() for t in (w.q, w.k, w.v))
        out = torch.full_like(q, float("nan"))
        state = torch.full((w.V, w.H, 64, 64), float("nan"), dtype=torch.float32, device=cuda_device)
        st, detail = _noalloc(lib, w, q, k, v, out, state)
        assert st == 0, detail
        torch.cuda.synchronize()
        ref_out, ref_state = spanla.span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent,
                                                 out=torch.full_like(q, float("nan")))
        spanla.span_la_check()
        seg = torch.zeros(w.T, dtype=torch.bool)
        for cu in (w.view_cu, w.branch_cu):
            for s in range(len(cu) - 1):
                seg[cu[s]:cu[s + 1]] = True
        seg = seg.to(cuda_device)
        assert not torch.isnan(out[seg]).any()
        assert torch.isnan(out[~seg]).all()
        assert _rel(out[seg], ref_out[seg]) <= TOL_BF16
        assert _rel(state, ref_state) <= TOL_BF16


def test_noalloc_rejects_a_pass_beyond_its_fixed_scratch(cuda_device):
    lib = spanla.load_library()
    w = workloads.sweep(32, 0)   # needs far more than 16 MiB of span states
    # metadata only is needed before the size check; small dummy tensors would
    # fail the row-range checks, so use real-size (uninitialised) buffers
    q = torch.empty((w.T, w.H, 64), dtype=torch.bfloat16, device=cuda_device)
    out = torch.empty_like(q)
    state = torch.empty((w.V, w.H, 64, 64), dtype=torch.float32, device=cuda_device)
    st, detail = _noalloc(lib, w, q, q, q, out, state)
    assert st == 1 and "fixed scratch" in detail


def test_noalloc_rejects_fp32_inputs(cuda_device):
    lib = spanla.load_library()
    w = workloads.tiny_oracle_case(0)
    q = w.q.to(cuda_device)
    dims = spanla.Dims(q.shape[0], q.shape[1], 64, spanla.SPAN_LA_F32)
    vcu = np.ascontiguousarray(w.view_cu, dtype=np.int32)
    st = lib.span_la_pass_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), dims, _i32p(vcu),
                                  len(vcu) - 1, None, 0, None, q.data_ptr(), q.data_ptr(), None)
    assert st == 2
