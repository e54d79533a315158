"""The largest passes: element offsets past 2^31 in q, k, v and out.

70 views of 30,000 rows and 4 branches per view (U[32,160] rows, some longer
than one 128-row tile) at 16 heads: 2.13 M rows, 2.18e9 elements per tensor.
The last view straddles element 2^31 (row 2,097,152) and every branch lies
past it, so 32-bit row or element arithmetic anywhere on the path would
misplace them.  Inputs are drawn on the device (bf16 standard normals; q and k
scaled by 1/8); the oracles check the first, a middle and the last request
(each view with all its branches) for the linear pass, and sampled rows of the
same requests for the softmax layer.  Every row of the pass is a segment row,
so no output may stay NaN.

Tolerance (bf16 inputs): max|o_gpu - o_ref| / max|o_ref| <= 1e-2, the view
states likewise; lse within 1e-2 * max(1, |lse_ref|).
"""
import numpy as np
import pytest
import torch

from helpers import TOL, rel_err
from hybrid_linear_attention_packed_gb300 import (span_la_check, span_la_pass, span_la_softmax_pass,
                                                  workloads)
from oracle import oracle_pass, oracle_softmax_rows

pytestmark = pytest.mark.gpu

H = 16
N_VIEWS, VIEW_ROWS, PER_VIEW = 70, 30000, 4
SAMPLE = [0, 35, N_VIEWS - 1]


@pytest.fixture(scope="module")
def big_pass(cuda_device):
    rng = np.random.default_rng([2031, 0])
    branch_lens = rng.integers(32, 161, size=N_VIEWS * PER_VIEW)
    parent = np.repeat(np.arange(N_VIEWS, dtype=np.int32), PER_VIEW)
    view_cu, branch_cu = workloads.pass_layout([VIEW_ROWS] * N_VIEWS, branch_lens)
    T = int(branch_cu[-1])
    assert T * H * 64 > 2 ** 31 and int(view_cu[-2]) * H * 64 < 2 ** 31
    q, k, v = workloads.draw_qkv_device(2031, T, H, cuda_device)
    yield view_cu, branch_cu, parent, q, k, v
    del q, k, v
    torch.cuda.empty_cache()


def _sub_pass(view_cu, branch_cu, parent, views):
    rows, vlens, blens, par = [], [], [], []
    for s in views:
        rows.append(np.arange(view_cu[s], view_cu[s + 1]))
        vlens.append(int(view_cu[s + 1] - view_cu[s]))
    for b in range(len(parent)):
        if int(parent[b]) in views:
            rows.append(np.arange(branch_cu[b], branch_cu[b + 1]))
            blens.append(int(branch_cu[b + 1] - branch_cu[b]))
            par.append(views.index(int(parent[b])))
    idx = np.concatenate(rows)
    vcu = np.concatenate([[0], np.cumsum(vlens)]).astype(np.int32)
    bcu = (np.concatenate([[0], np.cumsum(blens)]) + vcu[-1]).astype(np.int32)
    return idx, vcu, bcu, np.asarray(par, dtype=np.int32)


def _rows64(t, idx):
    return t[torch.from_numpy(idx).to(t.device)].double().cpu().numpy()


def test_linear_pass_past_2_31_elements(big_pass):
    view_cu, branch_cu, parent, q, k, v = big_pass
    out = torch.full_like(q, float("nan"))
    out, state = span_la_pass(q, k, v, view_cu, branch_cu, parent, out=out)
    span_la_check()
    assert not bool(torch.isnan(out).any()), "a row of the pass was not written"
    idx, vcu, bcu, par = _sub_pass(view_cu, branch_cu, parent, SAMPLE)
    ref, ref_state = oracle_pass(_rows64(q, idx), _rows64(k, idx), _rows64(v, idx), vcu, bcu, par)
    got = _rows64(out, idx)
    got_state = state[SAMPLE].double().cpu().numpy()
    e, es = rel_err(got, ref), rel_err(got_state, ref_state)
    print("2^31+ elements, requests %s: out %.2e state %.2e" % (SAMPLE, e, es))
    assert e <= TOL["bf16"] and es <= TOL["bf16"]


def test_softmax_layer_past_2_31_elements(big_pass):
    view_cu, branch_cu, parent, q, k, v = big_pass
    scale = 1.0   # q.k has standard deviation 1/8 here
    out = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[0], H), float("nan"), dtype=torch.float32, device=q.device)
    span_la_softmax_pass(q, k, v, view_cu, branch_cu, parent, scale=scale, out=out, lse=lse)
    span_la_check()
    assert not bool(torch.isnan(out).any()) and not bool(torch.isnan(lse).any())
    idx, vcu, bcu, par = _sub_pass(view_cu, branch_cu, parent, SAMPLE)
    # sampled rows of the sub-pass: the first and last row of every request's
    # view tiles past row 29,000, of every branch, and 64 random rows
    rng = np.random.default_rng(7)
    rows = set(rng.choice(idx.size, size=64, replace=False).tolist())
    for s in range(len(SAMPLE)):
        for r in range(int(vcu[s]) + 29000, int(vcu[s + 1]), 128):
            rows.update({r, min(r + 127, int(vcu[s + 1]) - 1)})
    for b in range(len(par)):
        rows.update({int(bcu[b]), int(bcu[b + 1]) - 1})
    rows = sorted(rows)
    ref, ref_lse = oracle_softmax_rows(_rows64(q, idx), _rows64(k, idx), _rows64(v, idx), vcu, bcu,
                                       par, rows, scale=scale)
    grow = idx[rows]
    got = _rows64(out, grow)
    got_lse = lse[torch.from_numpy(grow).to(lse.device)].double().cpu().numpy()
    e = rel_err(got, ref)
    el = float(np.max(np.abs(got_lse - ref_lse) / np.maximum(1.0, np.abs(ref_lse))))
    print("2^31+ elements, softmax, %d sampled rows: out %.2e lse %.2e" % (len(rows), e, el))
    assert e <= TOL["bf16"] and el <= TOL["bf16"]
