"""GPU parity of the softmax-attention layer (``span_la_softmax_pass``, through
the C ABI) against the float64 softmax oracle on the same seeded inputs.

Tolerance (bf16 inputs, written here and applied per call):
max|o_gpu - o_ref| / max|o_ref| <= 1e-2 over the rows compared, and
|lse_gpu - lse_ref| <= 1e-2 * max(1, |lse_ref|) elementwise.
"""
import numpy as np
import pytest
import torch

from helpers import f64, rel_err, segment_rows, to_device
from hybrid_linear_attention_packed_gb300 import (SpanLAError, span_la_check, span_la_softmax_pass,
                                                  workloads)
from oracle import oracle_softmax_pass, oracle_softmax_rows

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _run(w, dev, scale=0.0, with_lse=True):
    q, k, v = to_device(w, dev)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.T, w.H), float("nan"), dtype=torch.float32, device=dev) if with_lse else None
    span_la_softmax_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent, scale=scale, out=out, lse=lse)
    span_la_check()
    return out, lse


def _check_full(w, dev, scale=0.0):
    out, lse = _run(w, dev, scale)
    ref, ref_lse = oracle_softmax_pass(f64(w.q), f64(w.k), f64(w.v), w.view_cu, w.branch_cu,
                                       w.branch_parent, scale=scale if scale else None)
    got, got_lse = f64(out), f64(lse)
    seg = segment_rows(w)
    assert not np.any(np.isnan(got[seg])), "a segment row was not written"
    assert np.all(np.isnan(got[~seg])), "a row outside every segment was written"
    assert np.all(np.isnan(got_lse[~seg]))
    e = rel_err(got[seg], ref[seg])
    el = float(np.max(np.abs(got_lse[seg] - ref_lse[seg]) / np.maximum(1.0, np.abs(ref_lse[seg]))))
    print("%s: out %.2e lse %.2e" % (w.name, e, el))
    assert e <= TOL and el <= TOL
    return out


def _check_sampled(w, dev, n_rows=96, seed=0):
    out, lse = _run(w, dev)
    seg = segment_rows(w)
    got, got_lse = f64(out), f64(lse)
    assert not np.any(np.isnan(got[seg]))
    assert np.all(np.isnan(got[~seg]))
    rng = np.random.default_rng(seed)
    segrows = np.flatnonzero(seg)
    # random rows plus the first and last rows of every tile of the first view
    rows = set(rng.choice(segrows, size=min(n_rows, segrows.size), replace=False).tolist())
    a, e = int(w.view_cu[0]), int(w.view_cu[1])
    for r0 in range(a, e, 128):
        rows.update({r0, min(r0 + 127, e - 1)})
    for b in range(min(w.B, 4)):
        rows.update({int(w.branch_cu[b]), int(w.branch_cu[b + 1]) - 1})
    rows = sorted(r for r in rows if seg[r])
    ref, ref_lse = oracle_softmax_rows(f64(w.q), f64(w.k), f64(w.v), w.view_cu, w.branch_cu,
                                       w.branch_parent, rows)
    e_o = rel_err(got[rows], ref)
    e_l = float(np.max(np.abs(got_lse[rows] - ref_lse) / np.maximum(1.0, np.abs(ref_lse))))
    print("%s (%d sampled rows): out %.2e lse %.2e" % (w.name, len(rows), e_o, e_l))
    assert e_o <= TOL and e_l <= TOL


def test_tiny_case(cuda_device):
    w = workloads.make_pass([130, 77], [9, 14, 20, 9, 14, 20], [0, 0, 0, 1, 1, 1], H=2,
                            dtype="bf16", seed=0, q_scale=1.0, k_scale=1.0)
    _check_full(w, cuda_device)


@pytest.mark.parametrize("seed", [0, 1])
def test_single_request_7400_sampled(cuda_device, seed):
    _check_sampled(workloads.single_request(seed), cuda_device, seed=seed)


def test_packed_four_requests_sampled(cuda_device):
    _check_sampled(workloads.packed_four(0), cuda_device)


@pytest.mark.parametrize("n_views", [4, 16])
def test_sweep_sampled(cuda_device, n_views):
    """Full-size sweep passes (views log-U[500,18000], log-U[1,300] branches each)."""
    _check_sampled(workloads.sweep(n_views, 0), cuda_device, n_rows=128, seed=n_views)


EDGE = [0, 1, 63, 64, 65, 127, 128, 129, 255, 256, 257]


def test_edge_lengths(cuda_device):
    views = EDGE
    branches = EDGE + [300, 2, 3] + [1] * 20 + [5, 16, 7]
    parent = [i % len(views) for i in range(len(branches))]
    w = workloads.make_pass(views, branches, parent, H=3, dtype="bf16", seed=21, q_scale=1.0,
                            k_scale=1.0, lead_rows=5, mid_rows=70, tail_rows=130)
    _check_full(w, cuda_device)


def test_many_short_siblings_packed(cuda_device):
    """Runs of short branches of one parent share tiles; each sees only itself."""
    lens = [1, 2, 3, 16, 7, 30, 1, 64, 9, 128, 4, 4, 4, 4, 120, 8]
    parent = [0] * 8 + [1] * 8
    w = workloads.make_pass([200, 90], lens, parent, H=2, dtype="bf16", seed=25, q_scale=1.0,
                            k_scale=1.0)
    _check_full(w, cuda_device)


@pytest.mark.parametrize("scale", [0.03, 0.5])
def test_other_scales(cuda_device, scale):
    w = workloads.make_pass([300, 129], [40, 100, 5], [0, 1, 0], H=2, dtype="bf16", seed=26,
                            q_scale=1.0, k_scale=1.0)
    _check_full(w, cuda_device, scale=scale)


def test_gap_rows_with_nan_inputs_do_not_leak(cuda_device):
    w = workloads.make_pass([100, 64, 1], [20, 44, 7, 200], [0, 0, 1, 2], H=2, dtype="bf16",
                            seed=22, q_scale=1.0, k_scale=1.0, lead_rows=3, mid_rows=9, tail_rows=64)
    seg = segment_rows(w)
    for t in (w.q, w.k, w.v):
        t[torch.from_numpy(~seg)] = float("nan")
    _check_full(w, cuda_device)


def test_sibling_order_does_not_matter(cuda_device):
    base = workloads.make_pass([260], [30, 50, 20, 90], [0, 0, 0, 0], H=2, dtype="bf16", seed=27,
                               q_scale=1.0, k_scale=1.0)
    out = f64(_run(base, cuda_device)[0])
    perm = [3, 1, 0, 2]
    nv = int(base.view_lens.sum())
    rows = np.concatenate([np.arange(nv)] + [np.arange(base.branch_cu[b], base.branch_cu[b + 1])
                                             for b in perm])
    w = workloads.make_pass([260], [base.branch_lens[b] for b in perm], [0] * 4, H=2, dtype="bf16",
                            seed=27)
    w.q, w.k, w.v = base.q[rows].contiguous(), base.k[rows].contiguous(), base.v[rows].contiguous()
    out2 = f64(_run(w, cuda_device)[0])
    assert np.array_equal(out2[:nv], out[:nv])
    assert rel_err(out2, out[rows]) <= TOL


@pytest.mark.parametrize("growth", [0.02, 0.1])
def test_rising_scores_take_the_rescale_path(cuda_device, growth):
    """Key norms grow along each segment, so a later key block's maximum keeps
    exceeding the reference maximum by more than the 2^8 margin: O and the
    partial row sums are rescaled many times (by both warps of a row) and the
    result must still match the oracle; lse too."""
    w = workloads.make_pass([1000, 300], [60, 200, 9], [0, 0, 1], H=2, dtype="bf16", seed=33,
                            q_scale=1.0, k_scale=1.0)
    ramp = torch.ones(w.T)
    for cu in (w.view_cu, w.branch_cu):
        for s in range(len(cu) - 1):
            n = int(cu[s + 1] - cu[s])
            ramp[int(cu[s]):int(cu[s + 1])] = 1.0 + growth * torch.arange(n, dtype=torch.float32)
    w.k = (w.k.float() * ramp[:, None, None]).to(torch.bfloat16)
    _check_full(w, cuda_device)


def test_rejections_and_empty_pass(cuda_device):
    dev = cuda_device
    q = torch.zeros((10, 2, 64), dtype=torch.float32, device=dev)
    with pytest.raises(SpanLAError, match="bf16"):
        span_la_softmax_pass(q, q, q, [0, 10], None, None)
    qb = q.to(torch.bfloat16)
    with pytest.raises(SpanLAError, match="scale"):
        span_la_softmax_pass(qb, qb, qb, [0, 10], None, None, scale=-1.0)
    out = torch.full_like(qb, 3.0)
    span_la_softmax_pass(qb, qb, qb, [0], None, None, out=out)
    span_la_check()
    assert torch.all(out == 3.0)


def test_branches_from_kept_view_kv_equal_in_pass_branches(cuda_device):
    """The long-request procedure for the softmax layer: the view's K and V are
    kept (copied away) from the pass that ran it; the 256 branches then run over
    them, as one call and as 4 shard calls, from a buffer of branch rows only."""
    from hybrid_linear_attention_packed_gb300 import span_la_softmax_branches_from_kv
    w = workloads.cached_long(0)
    q, k, v = to_device(w, cuda_device)
    whole = torch.full_like(q, float("nan"))
    span_la_softmax_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent, out=whole)
    nv = int(w.view_cu[-1])
    view_k, view_v = k[:nv].clone(), v[:nv].clone()
    qb, kb, vb = q[nv:].contiguous(), k[nv:].contiguous(), v[nv:].contiguous()
    bcu = (w.branch_cu - nv).astype(np.int32)
    one = torch.full_like(qb, float("nan"))
    lse = torch.full((qb.shape[0], w.H), float("nan"), dtype=torch.float32, device=cuda_device)
    span_la_softmax_branches_from_kv(view_k, view_v, w.view_cu, qb, kb, vb, bcu, w.branch_parent,
                                     out=one, lse=lse)
    shards = torch.full_like(qb, float("nan"))
    for cu in workloads.shards(w, 4):
        cu = (cu - nv).astype(np.int32)
        span_la_softmax_branches_from_kv(view_k, view_v, w.view_cu, qb, kb, vb, cu,
                                         np.zeros(len(cu) - 1, np.int32), out=shards)
    span_la_check()
    # same tiles, same keys: bit for bit the branch rows of the whole pass
    assert torch.equal(one, whole[nv:])
    assert not torch.isnan(shards).any()
    rows = np.random.default_rng(3).choice(qb.shape[0], size=64, replace=False)
    rows = sorted(set(rows.tolist()) | {0, qb.shape[0] - 1})
    ref, ref_lse = oracle_softmax_rows(f64(w.q), f64(w.k), f64(w.v), w.view_cu, w.branch_cu,
                                       w.branch_parent, [nv + r for r in rows])
    e1 = rel_err(f64(one)[rows], ref)
    e4 = rel_err(f64(shards)[rows], ref)
    el = float(np.max(np.abs(f64(lse)[rows] - ref_lse) / np.maximum(1.0, np.abs(ref_lse))))
    print("branches from kept K/V: one call %.2e, 4 shards %.2e, lse %.2e" % (e1, e4, el))
    assert max(e1, e4, el) <= TOL


def test_branches_from_kv_several_views_and_rejections(cuda_device):
    from hybrid_linear_attention_packed_gb300 import span_la_softmax_branches_from_kv
    w = workloads.make_pass([129, 0, 300], [5, 130, 64, 1], [2, 0, 1, 2], H=2, dtype="bf16", seed=31,
                            q_scale=1.0, k_scale=1.0)
    q, k, v = to_device(w, cuda_device)
    whole = torch.full_like(q, float("nan"))
    span_la_softmax_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent, out=whole)
    nv = int(w.view_cu[-1])
    out = torch.full_like(q, float("nan"))
    # the pass's own arrays as the kept K/V: branch rows in place
    span_la_softmax_branches_from_kv(k[:nv].clone(), v[:nv].clone(), w.view_cu, q, k, v, w.branch_cu,
                                     w.branch_parent, out=out)
    span_la_check()
    assert torch.equal(out[nv:], whole[nv:])
    assert torch.isnan(out[:nv]).all()
    with pytest.raises(SpanLAError):
        span_la_softmax_branches_from_kv(k[:nv], v[:nv], [0, nv + 1], q, k, v, w.branch_cu[:2], [0],
                                         out=out)
    with pytest.raises(SpanLAError, match="branch_parent"):
        span_la_softmax_branches_from_kv(k[:nv], v[:nv], w.view_cu, q, k, v, w.branch_cu[:2], [3],
                                         out=out)
