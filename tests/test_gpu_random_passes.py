"""Randomised packed passes (fixed seeds) through the CUDA path against the
float64 oracles, element by element: view and branch lengths drawn from a
wide range (empty segments, single rows, multi-tile views and branches), 1 to
3 heads, both input types for the linear pass, several scales for the softmax
layer, rows of no segment between the segments; and 16-head passes of up to
8 requests in both structures of the bf16 pass (one launch, three launches).

Tolerances as in the other parity tests: max|o_gpu - o_ref| / max|o_ref| <=
1e-3 (fp32 inputs) or 1e-2 (bf16 inputs); the view states likewise; lse
within 1e-2 * max(1, |lse_ref|).
"""
import numpy as np
import pytest
import torch

from helpers import TOL, f64, rel_err, segment_rows, to_device
from hybrid_linear_attention_packed_gb300 import (span_la_check, span_la_pass, span_la_softmax_pass,
                                                  spanla, workloads)
from oracle import oracle_pass, oracle_softmax_pass

pytestmark = pytest.mark.gpu


def _random_pass(seed, dtype, q_scale=1.0 / 8, k_scale=1.0 / 8):
    rng = np.random.default_rng([seed, 77])
    V = int(rng.integers(1, 6))
    view_lens = [int(x) for x in rng.choice([0, 1, 63, 64, 129, 300, 640, 1000], size=V)]
    view_lens = [int(rng.integers(0, 1200)) if rng.random() < 0.5 else L for L in view_lens]
    lens, parents = [], []
    for v in range(V):
        for _ in range(int(rng.integers(0, 7))):
            lens.append(int(rng.choice([0, 1, 5, 31, 64, 100, 128, 129, 250, 400])))
            parents.append(v)
    H = int(rng.integers(1, 4))
    return workloads.make_pass(view_lens, lens, parents, H=H, dtype=dtype, seed=seed,
                               q_scale=q_scale, k_scale=k_scale,
                               lead_rows=int(rng.integers(0, 20)), mid_rows=int(rng.integers(0, 20)),
                               tail_rows=int(rng.integers(0, 20)))


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_random_linear_passes(cuda_device, seed, dtype):
    _check_random_linear(cuda_device, _random_pass(seed, dtype), seed, dtype)


def _random_wide_pass(seed):
    """16 heads and up to 8 requests of up to 3,000-row views with up to 40
    branches each: the plan cuts every head's tiles into several runs, so
    pieces, workspace states, carried final states and branch tiles in other
    runs all occur."""
    rng = np.random.default_rng([seed, 91])
    V = int(rng.integers(1, 9))
    view_lens = [int(rng.integers(0, 3000)) for _ in range(V)]
    lens, parents = [], []
    for v in range(V):
        for _ in range(int(rng.integers(0, 41))):
            lens.append(int(rng.choice([1, 16, 40, 96, 128, 129, 300])))
            parents.append(v)
    return workloads.make_pass(view_lens, lens, parents, H=16, dtype="bf16", seed=1000 + seed,
                               lead_rows=int(rng.integers(0, 20)), mid_rows=int(rng.integers(0, 20)),
                               tail_rows=int(rng.integers(0, 20)))


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("structure", ["one_launch", "three_launches"])
def test_random_wide_passes_both_structures(cuda_device, seed, structure):
    spanla.set_pass_variant(spanla.PASS_ONE_LAUNCH if structure == "one_launch" else spanla.PASS_THREE_LAUNCHES)
    try:
        _check_random_linear(cuda_device, _random_wide_pass(seed), seed, "bf16")
    finally:
        spanla.set_pass_variant(spanla.PASS_ONE_LAUNCH)


def _check_random_linear(cuda_device, w, seed, dtype):
    q, k, v = to_device(w, cuda_device)
    out = torch.full_like(q, float("nan"))
    out, state = span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent, out=out)
    span_la_check()
    ref, ref_state = oracle_pass(f64(w.q), f64(w.k), f64(w.v), w.view_cu, w.branch_cu,
                                 w.branch_parent)
    got = f64(out)
    seg = segment_rows(w)
    assert not np.any(np.isnan(got[seg])) and np.all(np.isnan(got[~seg]))
    e = rel_err(got[seg], ref[seg]) if seg.any() else 0.0
    es = rel_err(f64(state), ref_state) if w.V else 0.0
    print("seed %d %s: V=%d B=%d H=%d rows=%d out %.2e state %.2e"
          % (seed, dtype, w.V, w.B, w.H, w.rows, e, es))
    assert e <= TOL[dtype] and es <= TOL[dtype]


@pytest.mark.parametrize("seed", range(8))
def test_random_softmax_passes(cuda_device, seed):
    w = _random_pass(seed, "bf16", q_scale=1.0, k_scale=1.0)
    scale = [0.0, 0.05, 0.125, 0.4][seed % 4]
    q, k, v = to_device(w, cuda_device)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.T, w.H), float("nan"), dtype=torch.float32, device=cuda_device)
    span_la_softmax_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent, scale=scale, out=out,
                         lse=lse)
    span_la_check()
    ref, ref_lse = oracle_softmax_pass(f64(w.q), f64(w.k), f64(w.v), w.view_cu, w.branch_cu,
                                       w.branch_parent, scale=scale if scale else None)
    got, got_lse = f64(out), f64(lse)
    seg = segment_rows(w)
    assert not np.any(np.isnan(got[seg])) and np.all(np.isnan(got[~seg]))
    if seg.any():
        e = rel_err(got[seg], ref[seg])
        el = float(np.max(np.abs(got_lse[seg] - ref_lse[seg]) / np.maximum(1.0, np.abs(ref_lse[seg]))))
    else:
        e = el = 0.0
    print("seed %d scale %g: V=%d B=%d H=%d rows=%d out %.2e lse %.2e"
          % (seed, scale, w.V, w.B, w.H, w.rows, e, el))
    assert e <= TOL["bf16"] and el <= TOL["bf16"]


def test_many_heads_both_layers(cuda_device):
    """48 heads: the head index runs through TMA coordinates, the schedules and
    the state layout [n][H][64][64]."""
    w = workloads.make_pass([300, 129], [40, 1, 130], [0, 1, 1], H=48, dtype="bf16", seed=91,
                            q_scale=1.0, k_scale=1.0)
    q, k, v = to_device(w, cuda_device)
    out, state = span_la_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent,
                              out=torch.full_like(q, float("nan")))
    sm = span_la_softmax_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent,
                              out=torch.full_like(q, float("nan")))
    span_la_check()
    ref, ref_state = oracle_pass(f64(w.q), f64(w.k), f64(w.v), w.view_cu, w.branch_cu,
                                 w.branch_parent)
    sref, _ = oracle_softmax_pass(f64(w.q), f64(w.k), f64(w.v), w.view_cu, w.branch_cu,
                                  w.branch_parent)
    seg = segment_rows(w)
    e = rel_err(f64(out)[seg], ref[seg])
    es = rel_err(f64(state), ref_state)
    e_sm = rel_err(f64(sm)[seg], sref[seg])
    print("48 heads: linear out %.2e state %.2e; softmax out %.2e" % (e, es, e_sm))
    assert e <= TOL["bf16"] and es <= TOL["bf16"] and e_sm <= TOL["bf16"]
