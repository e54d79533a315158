"""Pins for the float64 softmax-layer oracle (``oracle/softmax_oracle.py``)
against facts other than itself.

The layer ("Serving 0.88M TPS from Two RTXs and Mac Minis", sections "The
Workload" and "Long Requests"): per head, a view row attends causally to its
own view; a branch row attends to all of its parent view and causally to its
own branch, never to a sibling.  Checked here:

* the library attention routine (``torch.nn.functional.scaled_dot_product_attention``,
  float64 on the CPU) with ``is_causal`` for views and an explicit visibility
  mask for branches;
* closed forms: q = 0 gives the running mean of the visible values and
  lse = log(count); a first view row returns its own value; a huge scale with
  distinct scores gives hard attention (the value at the argmax, found by
  brute force);
* invariants: a branch equals the tail of view ++ branch run as one view;
  siblings added, removed or permuted leave a branch unchanged; a packed pass
  equals per-view runs; scores shifted by the same amount for every key of a
  row leave the output unchanged and shift lse; the sampled-rows form equals
  the whole-pass form.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle_softmax_pass, oracle_softmax_rows


def _cu(lens, start=0):
    return np.concatenate([[start], start + np.cumsum(lens)]).astype(np.int32)


def _rand(rng, T, H, D, s=1.0):
    return rng.standard_normal((T, H, D)) * s


def _sdpa(q, k, v, mask=None, causal=False, scale=None):
    """q [n,H,D], k/v [m,H,D] float64 -> [n,H,D] via the library routine."""
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x.transpose(1, 0, 2))) for x in (q, k, v))
    m = None if mask is None else torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=m, is_causal=causal,
                                                         scale=scale)
    return o.numpy().transpose(1, 0, 2)


@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 129, 300])
def test_view_equals_library_causal_attention(L):
    rng = np.random.default_rng(L)
    H, D = 3, 64
    q, k, v = _rand(rng, L, H, D), _rand(rng, L, H, D), _rand(rng, L, H, D)
    out, _ = oracle_softmax_pass(q, k, v, [0, L], None, None)
    ref = _sdpa(q, k, v, causal=True)
    assert np.max(np.abs(out - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


@pytest.mark.parametrize("scale", [None, 0.3])
def test_branches_equal_library_attention_with_visibility_mask(scale):
    rng = np.random.default_rng(7)
    H, D = 2, 16
    vl, bl = [40, 70], [5, 17, 1, 30]
    par = [1, 0, 1, 1]
    vcu = _cu(vl)
    bcu = _cu(bl, vcu[-1])
    T = int(bcu[-1])
    q, k, v = _rand(rng, T, H, D), _rand(rng, T, H, D), _rand(rng, T, H, D)
    out, _ = oracle_softmax_pass(q, k, v, vcu, bcu, par, scale=scale)
    for b in range(len(bl)):
        a, e = bcu[b], bcu[b + 1]
        pa, pe = vcu[par[b]], vcu[par[b] + 1]
        # visibility over ALL rows of the pass, written from the rule
        mask = np.zeros((e - a, T), dtype=bool)
        for i, t in enumerate(range(a, e)):
            mask[i, pa:pe] = True
            mask[i, a:t + 1] = True
        ref = _sdpa(q[a:e], k, v, mask=mask, scale=scale)
        assert np.max(np.abs(out[a:e] - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_zero_queries_give_running_means():
    rng = np.random.default_rng(3)
    H, D = 2, 8
    vl, bl, par = [9, 4], [3, 6], [0, 1]
    vcu = _cu(vl)
    bcu = _cu(bl, vcu[-1])
    T = int(bcu[-1])
    q = np.zeros((T, H, D))
    k, v = _rand(rng, T, H, D), _rand(rng, T, H, D)
    out, lse = oracle_softmax_pass(q, k, v, vcu, bcu, par)
    for s in range(2):
        a, e = vcu[s], vcu[s + 1]
        n = np.arange(1, e - a + 1)[:, None, None]
        assert np.allclose(out[a:e], np.cumsum(v[a:e], axis=0) / n, rtol=0, atol=1e-13)
        assert np.allclose(lse[a:e], np.log(n[:, :, 0]).repeat(H, 1), rtol=0, atol=1e-13)
    for b in range(2):
        a, e = bcu[b], bcu[b + 1]
        pa, pe = vcu[par[b]], vcu[par[b] + 1]
        n = (pe - pa) + np.arange(1, e - a + 1)[:, None, None]
        want = (v[pa:pe].sum(axis=0)[None] + np.cumsum(v[a:e], axis=0)) / n
        assert np.allclose(out[a:e], want, rtol=0, atol=1e-13)
        assert np.allclose(lse[a:e], np.log(n[:, :, 0]).repeat(H, 1), rtol=0, atol=1e-13)


def test_first_view_row_returns_its_value_and_score():
    rng = np.random.default_rng(4)
    H, D = 4, 64
    q, k, v = _rand(rng, 5, H, D), _rand(rng, 5, H, D), _rand(rng, 5, H, D)
    out, lse = oracle_softmax_pass(q, k, v, [0, 2, 5], None, None)
    for r in (0, 2):
        assert np.array_equal(out[r], v[r])
        assert np.allclose(lse[r], (q[r] * k[r]).sum(-1) / 8.0, rtol=1e-14, atol=0)


def test_huge_scale_is_hard_attention():
    rng = np.random.default_rng(5)
    H, D = 2, 8
    vl, bl, par = [12], [6, 5], [0, 0]
    vcu = _cu(vl)
    bcu = _cu(bl, vcu[-1])
    T = int(bcu[-1])
    q, k, v = _rand(rng, T, H, D), _rand(rng, T, H, D), _rand(rng, T, H, D)
    out, _ = oracle_softmax_pass(q, k, v, vcu, bcu, par, scale=1e6)
    for t in range(T):
        if t < vcu[-1]:
            keys = list(range(0, t + 1))
        else:
            b = 0 if t < bcu[1] else 1
            keys = list(range(0, 12)) + list(range(bcu[b], t + 1))
        for h in range(H):
            best = max(keys, key=lambda j: float(np.dot(q[t, h], k[j, h])))
            assert np.allclose(out[t, h], v[best, h], rtol=0, atol=1e-12)


def test_branch_equals_tail_of_view_plus_branch():
    rng = np.random.default_rng(6)
    H, D = 2, 64
    L, n = 150, 37
    q, k, v = _rand(rng, L + n, H, D), _rand(rng, L + n, H, D), _rand(rng, L + n, H, D)
    pass_out, pass_lse = oracle_softmax_pass(q, k, v, [0, L], [L, L + n], [0])
    whole, whole_lse = oracle_softmax_pass(q, k, v, [0, L + n], None, None)
    # a branch sees all of the view and its own prefix: exactly a causal row of the
    # concatenation
    assert np.max(np.abs(pass_out[L:] - whole[L:])) <= 1e-12 * np.max(np.abs(whole[L:]))
    assert np.max(np.abs(pass_lse[L:] - whole_lse[L:])) <= 1e-12 * np.max(np.abs(whole_lse[L:]))


def test_siblings_do_not_change_a_branch_and_packing_equals_separate_runs():
    rng = np.random.default_rng(8)
    H, D = 2, 16
    vl = [20, 33]
    bl = [7, 9, 4]
    par = [0, 1, 0]
    vcu = _cu(vl)
    bcu = _cu(bl, vcu[-1])
    T = int(bcu[-1])
    q, k, v = _rand(rng, T, H, D), _rand(rng, T, H, D), _rand(rng, T, H, D)
    out, _ = oracle_softmax_pass(q, k, v, vcu, bcu, par)
    # branch 2 alone with its view: rows of view 0 then branch 2
    idx = np.r_[vcu[0]:vcu[1], bcu[2]:bcu[3]]
    solo, _ = oracle_softmax_pass(q[idx], k[idx], v[idx], [0, vl[0]], [vl[0], vl[0] + bl[2]], [0])
    assert np.array_equal(solo[vl[0]:], out[bcu[2]:bcu[3]])
    # permuting the branches permutes the rows of the result
    perm = [2, 0, 1]
    rows = np.r_[0:vcu[-1], np.concatenate([np.arange(bcu[b], bcu[b + 1]) for b in perm])]
    bcu2 = _cu([bl[b] for b in perm], vcu[-1])
    out2, _ = oracle_softmax_pass(q[rows], k[rows], v[rows], vcu, bcu2, [par[b] for b in perm])
    assert np.array_equal(out2, out[rows])
    # view 1 run alone equals its rows of the packed pass
    a, e = vcu[1], vcu[2]
    alone, _ = oracle_softmax_pass(q[a:e], k[a:e], v[a:e], [0, e - a], None, None)
    assert np.array_equal(alone, out[a:e])


def test_a_common_score_shift_leaves_output_and_shifts_lse():
    rng = np.random.default_rng(9)
    H, D = 2, 64
    vl, bl, par = [50], [20], [0]
    vcu = _cu(vl)
    bcu = _cu(bl, vcu[-1])
    T = int(bcu[-1])
    q, k, v = _rand(rng, T, H, D), _rand(rng, T, H, D), _rand(rng, T, H, D)
    k[:, :, 0] = 2.0                     # every key has the same first component
    out, lse = oracle_softmax_pass(q, k, v, vcu, bcu, par)
    q2 = q.copy()
    dq = rng.standard_normal((T, H))
    q2[:, :, 0] += dq                    # shifts every score of row t, head h by 2*dq/8
    out2, lse2 = oracle_softmax_pass(q2, k, v, vcu, bcu, par)
    assert np.max(np.abs(out2 - out)) <= 1e-12
    assert np.max(np.abs(lse2 - lse - 2.0 * dq / 8.0)) <= 1e-12


def test_sampled_rows_equal_whole_pass():
    rng = np.random.default_rng(10)
    H, D = 2, 64
    vl, bl, par = [70, 0, 130], [3, 64, 65], [2, 0, 2]
    vcu = _cu(vl)
    bcu = _cu(bl, vcu[-1])
    T = int(bcu[-1])
    q, k, v = _rand(rng, T, H, D), _rand(rng, T, H, D), _rand(rng, T, H, D)
    out, lse = oracle_softmax_pass(q, k, v, vcu, bcu, par)
    rows = [0, 69, 70, 199, 200, 202, 203, 266, 267, T - 1]
    o2, l2 = oracle_softmax_rows(q, k, v, vcu, bcu, par, rows)
    assert np.max(np.abs(o2 - out[rows])) <= 1e-12 * np.max(np.abs(out))
    assert np.max(np.abs(l2 - lse[rows])) <= 1e-12 * np.max(np.abs(lse))


def test_bad_metadata_is_rejected():
    q = np.zeros((10, 1, 4))
    with pytest.raises(ValueError):
        oracle_softmax_pass(q, q, q, [0, 11], None, None)
    with pytest.raises(ValueError):
        oracle_softmax_pass(q, q, q, [0, 5], [5, 3], [0])
    with pytest.raises(ValueError):
        oracle_softmax_pass(q, q, q, [0, 5], [5, 8], [1])


@pytest.mark.parametrize("seed", range(4))
def test_random_packed_passes_equal_library_attention(seed):
    """Whole random packed passes (views, branches, rows in no segment) against
    the library routine with the visibility of every row over the whole buffer
    written out from the rule."""
    rng = np.random.default_rng([seed, 5])
    V = int(rng.integers(1, 4))
    vl = [int(x) for x in rng.integers(0, 90, size=V)]
    bl, par = [], []
    for v in range(V):
        for _ in range(int(rng.integers(0, 4))):
            bl.append(int(rng.integers(0, 40)))
            par.append(v)
    lead = int(rng.integers(0, 5))
    vcu = _cu(vl, lead)
    bcu = _cu(bl, int(vcu[-1]) + int(rng.integers(0, 5)))
    T = int(bcu[-1]) + int(rng.integers(0, 5))
    H, D = 2, 16
    q, k, v = _rand(rng, T, H, D), _rand(rng, T, H, D), _rand(rng, T, H, D)
    scale = float(rng.choice([0.1, 0.25, 0.6]))
    out, _ = oracle_softmax_pass(q, k, v, vcu, bcu, par, scale=scale, fill=7.0)
    mask = np.zeros((T, T), dtype=bool)
    seg = np.zeros(T, dtype=bool)
    for s in range(V):
        for t in range(vcu[s], vcu[s + 1]):
            mask[t, vcu[s]:t + 1] = True
            seg[t] = True
    for b in range(len(bl)):
        p = par[b]
        for t in range(bcu[b], bcu[b + 1]):
            mask[t, vcu[p]:vcu[p + 1]] = True
            mask[t, bcu[b]:t + 1] = True
            seg[t] = True
    rows = np.flatnonzero(seg)
    if rows.size:
        ref = _sdpa(q[rows], k, v, mask=mask[rows], scale=scale)
        assert np.max(np.abs(out[rows] - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))
    assert np.all(out[~seg] == 7.0)
