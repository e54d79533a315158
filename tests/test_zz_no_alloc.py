"""The no-allocation entry point against the regular one.

``span_la_pass_noalloc`` serves callers that cannot allocate device memory
while a pass runs (a process that gave the GPU's memory to its own pool, or
code where an allocation could block or fail at the wrong moment): it runs the
same pass in a fixed workspace that the library owns.  These tests call it
through the C ABI.  It plans and launches exactly what ``span_la_pass`` does,
so two calls in a row must give the same bits as ``span_la_pass`` on the same
inputs; the 7,400-token pass is also checked against the float64 oracle
within the bf16 bound of the other parity tests.  This file is named so that
pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import f64, rel_err, segment_rows
from hybrid_linear_attention_packed_gb300 import spanla, workloads
from oracle import oracle_pass

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2
SCRATCH_BYTES = 16 << 20


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


def _seg(w, dev):
    return torch.from_numpy(segment_rows(w)).to(dev)


def _equal_to_span_la_pass(lib, w, dev):
    q, k, v = (t.to(dev).contiguous() for t in (w.q, w.k, w.v))
    out = torch.full_like(q, float("nan"))
    state = torch.full((w.V, w.H, 64, 64), float("nan"), dtype=torch.float32, device=dev)
    st, detail = _noalloc(lib, w, q, k, v, out, state)
    assert st == 0, detail
    spanla.span_la_check()
    ref_out, ref_state = spanla.span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent,
                                             out=torch.full_like(q, float("nan")))
    spanla.span_la_check()
    seg = _seg(w, dev)
    assert not torch.isnan(out[seg]).any()
    assert torch.isnan(out[~seg]).all()
    # same plan, same kernels: the same bits
    assert torch.equal(out[seg], ref_out[seg])
    assert torch.equal(state, ref_state)
    return out, state


def test_noalloc_matches_span_la_pass_on_two_calls_in_a_row(cuda_device):
    lib = spanla.load_library()
    cases = [workloads.single_request(3),
             workloads.make_pass([300, 129, 64], [20, 50, 200, 7], [0, 0, 1, 2], H=4,
                                 dtype="bf16", seed=31)]
    for w in cases:   # two calls in a row, on different passes
        _equal_to_span_la_pass(lib, w, cuda_device)


def test_noalloc_single_request_against_the_oracle(cuda_device):
    """The 7,400-token pass through the fixed scratch, element by element
    against the float64 oracle (max|o - o_ref| / max|o_ref| <= 1e-2)."""
    lib = spanla.load_library()
    w = workloads.single_request(0)
    out, state = _equal_to_span_la_pass(lib, w, cuda_device)
    ref, ref_state = oracle_pass(f64(w.q), f64(w.k), f64(w.v), w.view_cu, w.branch_cu,
                                 w.branch_parent)
    seg = segment_rows(w)
    assert rel_err(f64(out)[seg], ref[seg]) <= TOL_BF16
    assert rel_err(f64(state), ref_state) <= TOL_BF16


def test_noalloc_timeout_is_reported_by_span_la_check(cuda_device):
    """A bounded wait that runs out on the no-allocation path's error word is
    reported by span_la_check as SPAN_LA_ERR_TIMEOUT, and cleared by it."""
    spanla.span_la_check()
    spanla.span_la_selftest_wait_timeout_noalloc(1000)
    with pytest.raises(spanla.SpanLAError) as exc:
        spanla.span_la_check()
    assert exc.value.status == 5 and "no-allocation path 0x4" in str(exc.value)
    spanla.span_la_check()   # cleared
    # the path still works afterwards
    _equal_to_span_la_pass(spanla.load_library(), workloads.make_pass(
        [200, 70], [9, 30], [0, 1], H=2, dtype="bf16", seed=5), cuda_device)


def _many_views(n_views, H=16, rows=64, seed=7):
    return workloads.make_pass([rows] * n_views, [], [], H=H, dtype="bf16", seed=seed)


def test_noalloc_size_limit(cuda_device):
    """The scratch holds descriptors plus the 16 KiB workspace states.  In the
    three-launch structure every piece-head has one: 60 one-tile views of 16
    heads need 960 (15.7 MB with the descriptors) and fit and match
    span_la_pass; 66 views need 1,056 (17.3 MB): rejected before anything is
    enqueued, with the bytes the pass needs.  The one-launch structure keeps
    states only across run boundaries, so the 66-view pass fits there."""
    lib = spanla.load_library()
    nsm = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    spanla.set_pass_variant(spanla.PASS_THREE_LAUNCHES)
    try:
        st_fit = spanla.plan_stats(_many_views(60).view_cu, [], [], 16, "bf16", num_sms=nsm)
        assert st_fit["state_slots"] * 16384 < SCRATCH_BYTES
        _equal_to_span_la_pass(lib, _many_views(60), cuda_device)

        w = _many_views(66)
        q = w.q.to(cuda_device)
        out = torch.full_like(q, float("nan"))
        state = torch.full((w.V, w.H, 64, 64), float("nan"), dtype=torch.float32, device=cuda_device)
        st, detail = _noalloc(lib, w, q, q, q, out, state)
        assert st == 1 and "fixed scratch" in detail
        need = int(detail.split("needs ")[1].split(" bytes")[0])
        assert need > SCRATCH_BYTES
        torch.cuda.synchronize()
        assert torch.isnan(out).all() and torch.isnan(state).all()   # nothing written
    finally:
        spanla.set_pass_variant(spanla.PASS_ONE_LAUNCH)
    assert spanla.plan_stats(w.view_cu, [], [], 16, "bf16", num_sms=nsm)["state_slots"] < nsm
    _equal_to_span_la_pass(lib, w, cuda_device)


def test_noalloc_rejects_fp32_inputs(cuda_device):
    lib = spanla.load_library()
    w = workloads.tiny_oracle_case(0)
    q = w.q.to(cuda_device)
    dims = spanla.Dims(q.shape[0], q.shape[1], 64, spanla.SPAN_LA_F32)
    vcu = np.ascontiguousarray(w.view_cu, dtype=np.int32)
    st = lib.span_la_pass_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), dims, _i32p(vcu),
                                  len(vcu) - 1, None, 0, None, q.data_ptr(), q.data_ptr(), None)
    assert st == 2
