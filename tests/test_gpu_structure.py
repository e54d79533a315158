"""Structural GPU tests that need no oracle: determinism, sibling independence,
in-pass branches against branches from the cached state, and the bounded-wait
failure path ("Serving 0.88M TPS from Two RTXs and Mac Minis", section "The
Workload": branches attend to the view, not to each other; section "Long
Requests": branch shards reuse the view's cached state)."""
import numpy as np
import pytest
import torch

from helpers import to_device
from hybrid_linear_attention_packed_gb300 import (SpanLAError, span_la_branches_from_state,
                                                  span_la_check, span_la_pass, spanla, workloads)

pytestmark = pytest.mark.gpu


def _run(w, dev):
    q, k, v = to_device(w, dev)
    out, state = span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent,
                              out=torch.full_like(q, float("nan")))
    span_la_check()
    return out, state


def test_run_to_run_bit_identical(cuda_device):
    w = workloads.packed_four(1)
    o1, s1 = _run(w, cuda_device)
    o2, s2 = _run(w, cuda_device)
    seg = torch.zeros(w.T, dtype=torch.bool)
    seg[: w.branch_cu[-1]] = True
    assert torch.equal(o1[seg.to(cuda_device)], o2[seg.to(cuda_device)])
    assert torch.equal(s1, s2)



@pytest.mark.parametrize("variant", ["one_launch", "three_launches"])
def test_repeated_passes_bit_identical(cuda_device, variant):
    """Thirty passes of the 7,400-token request, with the L2 written over, a
    side stream and back-to-back launches between them, all equal to the
    first bit for bit: the hand-offs between the kernel's warps (tensor
    memory, shared-memory operands and staging) leave no timing-dependent
    result, whichever order the roles happen to run in."""
    spanla.set_pass_variant(spanla.PASS_ONE_LAUNCH if variant == "one_launch" else spanla.PASS_THREE_LAUNCHES)
    try:
        w = workloads.single_request(3)
        q, k, v = to_device(w, cuda_device)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=cuda_device)
        side = torch.cuda.Stream(cuda_device)
        ref, ref_state = span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent)
        span_la_check()
        outs = []
        for rep in range(30):
            if rep % 3 == 0:
                flush.fill_(rep & 0xFF)      # L2 full of dirty lines
            if rep % 3 == 1:
                side.wait_stream(torch.cuda.current_stream(cuda_device))
                with torch.cuda.stream(side):
                    o, s = span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent, stream=side)
                torch.cuda.current_stream(cuda_device).wait_stream(side)
            else:
                o, s = span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent)
            outs.append((o, s))
        torch.cuda.synchronize(cuda_device)
        span_la_check()
        span_la_check(side)
        seg = torch.zeros(w.T, dtype=torch.bool)
        seg[: w.branch_cu[-1]] = True
        seg = seg.to(cuda_device)
        for o, s in outs:
            assert torch.equal(o[seg], ref[seg])
            assert torch.equal(s, ref_state)
    finally:
        spanla.set_pass_variant(spanla.PASS_ONE_LAUNCH)


def test_repeated_softmax_passes_bit_identical(cuda_device):
    """The softmax layer: twenty calls over the 7,400-token request, the L2
    written over between some of them, all equal to the first bit for bit
    (the two softmax warps of a row quarter hand the running maximum to each
    other, so their relative timing must not change a result)."""
    w = workloads.single_request(4)
    q, k, v = to_device(w, cuda_device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=cuda_device)
    lse0 = torch.empty((w.T, w.H), dtype=torch.float32, device=cuda_device)
    ref = spanla.span_la_softmax_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent, lse=lse0)
    span_la_check()
    seg = torch.zeros(w.T, dtype=torch.bool)
    seg[: w.branch_cu[-1]] = True
    seg = seg.to(cuda_device)
    for rep in range(20):
        if rep % 2 == 0:
            flush.fill_(rep & 0xFF)
        lse = torch.empty_like(lse0)
        o = spanla.span_la_softmax_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent, lse=lse)
        span_la_check()
        assert torch.equal(o[seg], ref[seg])
        assert torch.equal(lse[seg], lse0[seg])

def _pack(view_len, branches, H, seed):
    """A view plus the given list of (name, rows) branches, each row drawn from
    the same per-branch seeded stream so a branch is identical wherever it sits."""
    rng = np.random.default_rng([seed, 7])
    view = rng.standard_normal((3, view_len, H, 64), dtype=np.float32)
    parts = [view]
    for name, rows in branches:
        r = np.random.default_rng([seed, 100 + name])
        parts.append(r.standard_normal((3, rows, H, 64), dtype=np.float32))
    x = np.concatenate(parts, axis=1)
    x[0] *= 0.125
    x[1] *= 0.125
    t = torch.from_numpy(x).to(torch.bfloat16)
    lens = [rows for _, rows in branches]
    bcu = np.concatenate([[view_len], view_len + np.cumsum(lens)]).astype(np.int32)
    return t[0].contiguous(), t[1].contiguous(), t[2].contiguous(), bcu


def _branch_outputs(view_len, branches, H, seed, dev):
    q, k, v = (t.to(dev) for t in _pack(view_len, branches, H, seed)[:3])
    bcu = _pack(view_len, branches, H, seed)[3]
    out, _ = span_la_pass(q, k, v, [0, view_len], bcu, [0] * len(branches))
    span_la_check()
    res = {}
    for i, (name, rows) in enumerate(branches):
        res[name] = out[bcu[i]:bcu[i + 1]].clone()
    return res


def test_siblings_do_not_change_a_branch(cuda_device):
    H, view_len, seed = 2, 300, 41
    base = [(0, 30), (1, 45), (2, 20), (3, 90)]
    ref = _branch_outputs(view_len, base, H, seed, cuda_device)
    # removing or adding siblings after a branch leaves its tile position as it
    # was: bit-identical
    fewer = _branch_outputs(view_len, base[:2], H, seed, cuda_device)
    more = _branch_outputs(view_len, base + [(4, 17), (5, 64)], H, seed, cuda_device)
    for name in (0, 1):
        assert torch.equal(fewer[name], ref[name])
    for name in range(4):
        assert torch.equal(more[name], ref[name])
    # permuting moves branches inside the packed tiles: the tensor cores then
    # sum the same products in another grouping, so equal to fp32 rounding
    perm = _branch_outputs(view_len, [base[3], base[1], base[0], base[2]], H, seed, cuda_device)
    for name in range(4):
        a, b = perm[name].double(), ref[name].double()
        assert float((a - b).abs().max()) <= 1e-5 * float(b.abs().max()) + 2 ** -8


def test_in_pass_branches_equal_branches_from_the_cached_state(cuda_device):
    w = workloads.make_pass([700, 129], [30, 60, 100, 5, 128], [0, 0, 1, 1, 0], H=3,
                            dtype="bf16", seed=42)
    q, k, v = to_device(w, cuda_device)
    out, state = span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent)
    out2 = span_la_branches_from_state(state.clone(), q, k, v, w.branch_cu, w.branch_parent,
                                       out=torch.full_like(q, float("nan")))
    span_la_check()
    br = slice(int(w.branch_cu[0]), int(w.branch_cu[-1]))
    assert torch.equal(out[br], out2[br])
    assert torch.isnan(out2[: int(w.view_cu[-1])]).all()


def test_bounded_wait_times_out_without_trapping(cuda_device):
    """A kernel waits on an mbarrier that nothing completes, with a 1 ms limit:
    it records the timeout and returns; span_la_check reports it; the context
    stays usable."""
    spanla.span_la_check()
    spanla.span_la_selftest_wait_timeout(1000)
    with pytest.raises(SpanLAError) as exc:
        span_la_check()
    assert exc.value.status == 5
    span_la_check()   # the error word was cleared
    w = workloads.make_pass([100], [10], [0], H=1, dtype="bf16", seed=43)
    out, _ = _run(w, cuda_device)
    assert not torch.isnan(out[: w.rows]).any()


def test_injected_allocation_failure_enqueues_nothing(cuda_device):
    """A workspace allocation that fails (host-side injection) makes the call
    return SPAN_LA_ERR_NOMEM with nothing enqueued and nothing written; the
    next call runs normally."""
    w = workloads.make_pass([300, 70], [20, 9], [0, 1], H=2, dtype="bf16", seed=44)
    q, k, v = to_device(w, cuda_device)
    out = torch.full_like(q, float("nan"))
    state = torch.full((w.V, w.H, 64, 64), float("nan"), dtype=torch.float32, device=cuda_device)
    spanla.profile_reset()
    spanla.fault_inject(spanla.FAULT_ALLOC, 1)
    try:
        with pytest.raises(SpanLAError) as exc:
            span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent, out=out,
                         view_state_out=state)
    finally:
        spanla.fault_inject(spanla.FAULT_ALLOC, 0)
    assert exc.value.status == 4 and "injected" in str(exc.value)
    span_la_check()
    assert torch.isnan(out).all() and torch.isnan(state).all()
    assert all(p["launches"] == 0 for p in spanla.profile_read().values())
    span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent, out=out, view_state_out=state)
    span_la_check()
    assert not torch.isnan(out[: w.rows]).any() and not torch.isnan(state).any()


@pytest.mark.parametrize("variant", ["one_launch", "three_launches"])
def test_profiler_counts_and_times_every_launch(cuda_device, variant):
    """Three passes launch three span-output kernels, and, in the three-launch
    structure, three span-state and three scan kernels too; each is timed."""
    w = workloads.single_request(0)
    q, k, v = to_device(w, cuda_device)
    one = variant == "one_launch"
    spanla.set_pass_variant(spanla.PASS_ONE_LAUNCH if one else spanla.PASS_THREE_LAUNCHES)
    try:
        spanla.profile_reset()
        spanla.profile_enable(True)
        for _ in range(3):
            span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent)
        span_la_check()
        spanla.profile_enable(False)
        prof = spanla.profile_read()
    finally:
        spanla.profile_enable(False)
        spanla.set_pass_variant(spanla.PASS_ONE_LAUNCH)
    launched = ("span_output",) if one else ("span_state", "segmented_scan", "span_output")
    for name in ("span_state", "segmented_scan", "span_output"):
        n = 3 if name in launched else 0
        assert prof[name]["launches"] == n and prof[name]["timed"] == n
        assert (prof[name]["ms"] > 0) == (n > 0)
    assert prof["chunk_state"]["launches"] == 0


def test_plan_reused_across_calls_and_streams(cuda_device):
    """Passes with the same metadata reuse one uploaded descriptor block (the
    plan depends on the metadata only): new inputs on the same and on another
    stream still give the oracle's results."""
    from helpers import TOL, f64, rel_err, segment_rows
    from oracle import oracle_pass
    base = workloads.make_pass([700, 129], [30, 60, 100, 5], [0, 0, 1, 1], H=3, dtype="bf16", seed=50)
    side = torch.cuda.Stream(device=cuda_device)
    for i, stream in enumerate([torch.cuda.current_stream(cuda_device), side, side]):
        w = workloads.make_pass([700, 129], [30, 60, 100, 5], [0, 0, 1, 1], H=3, dtype="bf16", seed=51 + i)
        assert np.array_equal(w.view_cu, base.view_cu) and np.array_equal(w.branch_cu, base.branch_cu)
        with torch.cuda.stream(stream):
            q, k, v = to_device(w, cuda_device)
            out, state = span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent,
                                      out=torch.full_like(q, float("nan")))
        stream.synchronize()
        span_la_check()
        ref, ref_state = oracle_pass(f64(w.q), f64(w.k), f64(w.v), w.view_cu, w.branch_cu, w.branch_parent)
        seg = segment_rows(w)
        assert rel_err(f64(out)[seg], ref[seg]) <= TOL["bf16"]
        assert rel_err(f64(state), ref_state) <= TOL["bf16"]


def test_prepared_plan_is_used_by_the_pass(cuda_device):
    """span_la_plan_prepare puts a pass's plan in the cache before the pass:
    preparing it again allocates nothing (a pending forced allocation failure
    is not reached), and the pass that follows on another stream gives the
    bits of a pass that builds its own plan (the no-allocation entry point
    plans every call) and the oracle's results.  A capturing stream is
    refused."""
    from helpers import TOL, f64, rel_err, segment_rows
    from oracle import oracle_pass
    w = workloads.make_pass([1300, 250], [40, 90, 33, 200, 7], [0, 0, 1, 1, 1], H=4, dtype="bf16",
                            seed=60)
    side = torch.cuda.Stream(device=cuda_device)
    spanla.span_la_plan_prepare(w.view_cu, w.branch_cu, w.branch_parent, w.T, w.H, stream=side)
    spanla.fault_inject(spanla.FAULT_ALLOC, 1)
    try:
        spanla.span_la_plan_prepare(w.view_cu, w.branch_cu, w.branch_parent, w.T, w.H, stream=side)
    finally:
        spanla.fault_inject(spanla.FAULT_ALLOC, 0)
    q, k, v = to_device(w, cuda_device)
    out, state = span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent,
                              out=torch.full_like(q, float("nan")))
    out_own, state_own = spanla.span_la_pass_noalloc(q, k, v, w.view_cu, w.branch_cu, w.branch_parent,
                                                     out=torch.full_like(q, float("nan")))
    torch.cuda.synchronize()
    span_la_check()
    seg = segment_rows(w)
    segt = torch.from_numpy(seg)
    assert torch.equal(out.cpu()[segt], out_own.cpu()[segt]) and torch.equal(state, state_own)
    ref, ref_state = oracle_pass(f64(w.q), f64(w.k), f64(w.v), w.view_cu, w.branch_cu, w.branch_parent)
    assert rel_err(f64(out)[seg], ref[seg]) <= TOL["bf16"]
    assert rel_err(f64(state), ref_state) <= TOL["bf16"]
    g = torch.cuda.CUDAGraph()
    with pytest.raises(SpanLAError) as exc:
        with torch.cuda.graph(g):
            spanla.span_la_plan_prepare(w.view_cu, w.branch_cu, w.branch_parent, w.T, w.H)
    assert exc.value.status == 2


def test_plan_cache_eviction_is_stream_ordered(cuda_device):
    """More distinct layouts than the plan cache keeps per device (16): each
    further one evicts the least recently used descriptor block, freed in
    stream order behind its last reads.  The evicting call returns while its
    stream is still busy (no host synchronisation); results on the current
    and a second stream, and of a layout evicted earlier and planned again,
    match the oracle."""
    import time
    from helpers import TOL, f64, rel_err, segment_rows
    from oracle import oracle_pass

    ws = [workloads.make_pass([300 + 7 * i, 129], [30, 60], [0, 1], H=2, dtype="bf16", seed=100 + i)
          for i in range(24)]
    ins = [to_device(w, cuda_device) for w in ws]

    def call(i):
        w, (q, k, v) = ws[i], ins[i]
        return span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent,
                            out=torch.full_like(q, float("nan")))

    def check(i, res):
        w = ws[i]
        ref, ref_state = oracle_pass(f64(w.q), f64(w.k), f64(w.v), w.view_cu, w.branch_cu, w.branch_parent)
        seg = segment_rows(w)
        assert rel_err(f64(res[0])[seg], ref[seg]) <= TOL["bf16"]
        assert rel_err(f64(res[1]), ref_state) <= TOL["bf16"]

    results = {i: call(i) for i in range(17)}     # the 17th layout at the latest evicts
    torch.cuda.synchronize()
    span_la_check()
    torch.cuda._sleep(400_000_000)                # ~200 ms of device work ahead of the call
    t0 = time.perf_counter()
    results[17] = call(17)                        # a miss that evicts
    host_ms = (time.perf_counter() - t0) * 1e3
    torch.cuda.synchronize()
    span_la_check()
    assert host_ms < 50.0, "an evicting call waited for the device (%.1f ms)" % host_ms
    side = torch.cuda.Stream(device=cuda_device)
    for i in range(18, 24):
        with torch.cuda.stream(side if i % 2 else torch.cuda.current_stream(cuda_device)):
            torch.cuda._sleep(2_000_000)
            results[i] = call(i)
    results[0] = call(0)                          # evicted above, planned again
    torch.cuda.synchronize()
    span_la_check()
    for i, res in results.items():
        check(i, res)


def test_prepared_plans_across_evictions_and_streams(cuda_device):
    """Forty layouts, each prepared on a side stream held back by device work
    and then passed on the current stream without a host synchronisation:
    every pass waits for its plan's upload, evictions (more layouts than the
    cache's 16) hand their events on to later plans, and every result matches
    the oracle."""
    from helpers import TOL, f64, rel_err, segment_rows
    from oracle import oracle_pass

    ws = [workloads.make_pass([200 + 13 * i, 140], [25, 70, 9], [0, 1, 1], H=2, dtype="bf16", seed=300 + i)
          for i in range(40)]
    ins = [to_device(w, cuda_device) for w in ws]
    side = torch.cuda.Stream(device=cuda_device)
    torch.cuda.synchronize()
    results = []
    for i, w in enumerate(ws):
        with torch.cuda.stream(side):
            torch.cuda._sleep(1_000_000)          # the upload lands after the pass is enqueued
        spanla.span_la_plan_prepare(w.view_cu, w.branch_cu, w.branch_parent, w.T, w.H, stream=side)
        q, k, v = ins[i]
        results.append(span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent,
                                    out=torch.full_like(q, float("nan"))))
    torch.cuda.synchronize()
    span_la_check()
    for w, (out, state) in zip(ws, results):
        ref, ref_state = oracle_pass(f64(w.q), f64(w.k), f64(w.v), w.view_cu, w.branch_cu, w.branch_parent)
        seg = segment_rows(w)
        assert rel_err(f64(out)[seg], ref[seg]) <= TOL["bf16"]
        assert rel_err(f64(state), ref_state) <= TOL["bf16"]


def _graph_replay_equals_eager(dev, record, w_a, w_b):
    """Record `record(q, k, v, outs)` into a CUDA graph on inputs A, replay it
    after copying inputs B into the same buffers, and compare with an eager
    call on B, bit for bit."""
    qa, ka, va = to_device(w_a, dev)
    qb, kb, vb = to_device(w_b, dev)
    eager = record(qb, kb, vb)
    span_la_check()
    q, k, v = qa.clone(), ka.clone(), va.clone()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = record(q, k, v)
    for _ in range(2):
        q.copy_(qb)
        k.copy_(kb)
        v.copy_(vb)
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        span_la_check()
        for got, want in zip(outs, eager):
            assert torch.equal(got, want)


def test_cuda_graph_replays_the_pass(cuda_device):
    shape = dict(view_lens=[700, 129], branch_lens=[40, 9, 100], parent=[0, 0, 1])
    w_a, w_b = (workloads.make_pass(shape["view_lens"], shape["branch_lens"], shape["parent"], H=4,
                                    dtype="bf16", seed=s) for s in (50, 51))

    def record(q, k, v):
        out = torch.zeros_like(q)
        state = torch.zeros((w_a.V, w_a.H, 64, 64), dtype=torch.float32, device=q.device)
        span_la_pass(q, k, v, w_a.view_cu, w_a.branch_cu, w_a.branch_parent, out=out,
                     view_state_out=state)
        return out, state
    _graph_replay_equals_eager(cuda_device, record, w_a, w_b)


def test_cuda_graph_replays_the_noalloc_pass(cuda_device):
    w_a, w_b = (workloads.make_pass([300, 64], [20, 70], [1, 0], H=2, dtype="bf16", seed=s)
                for s in (52, 53))

    def record(q, k, v):
        out = torch.zeros_like(q)
        state = torch.zeros((w_a.V, w_a.H, 64, 64), dtype=torch.float32, device=q.device)
        spanla.span_la_pass_noalloc(q, k, v, w_a.view_cu, w_a.branch_cu, w_a.branch_parent,
                                    out=out, view_state_out=state)
        return out, state
    _graph_replay_equals_eager(cuda_device, record, w_a, w_b)


def test_cuda_graph_replays_the_softmax_layer(cuda_device):
    from hybrid_linear_attention_packed_gb300 import span_la_softmax_pass
    w_a, w_b = (workloads.make_pass([500, 130], [33, 7, 128], [0, 1, 1], H=2, dtype="bf16", seed=s,
                                    q_scale=1.0, k_scale=1.0) for s in (54, 55))

    def record(q, k, v):
        out = torch.zeros_like(q)
        span_la_softmax_pass(q, k, v, w_a.view_cu, w_a.branch_cu, w_a.branch_parent, out=out)
        return (out,)
    _graph_replay_equals_eager(cuda_device, record, w_a, w_b)


def test_cache_calls_refuse_graph_capture(cuda_device):
    from hybrid_linear_attention_packed_gb300 import ViewStateCache
    state = torch.zeros((1, 2, 64, 64), dtype=torch.float32, device=cuda_device)
    with ViewStateCache(2, capacity=2) as cache:
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with pytest.raises(SpanLAError) as exc:
            with torch.cuda.graph(g):
                cache.put([1], state)
        assert exc.value.status == 2
        torch.cuda.synchronize()
        cache.put([1], state)
        span_la_check()
        assert cache.contains([1]).tolist() == [True]
