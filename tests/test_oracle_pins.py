"""Pins for the float64 oracle against things other than itself.

Each test checks the C recurrence in ``oracle/`` against a fact that the
definition of unnormalised causal linear attention (per head,
``S_t = S_{t-1} + k_t v_t^T``, ``o_t = S_t^T q_t``) or the page's workload
statements fix ("Serving 0.88M TPS from Two RTXs and Mac Minis", sections
"The Workload", "Kernels", "Long Requests"):

* a hand-worked example (``tests/golden/hand_d2.txt``);
* the masked quadratic form ``tril(Q K^T) V + Q S0`` (plain matmuls);
* closed forms: final state ``K^T V``; ``d = 1`` reduces to a cumulative sum;
  one-hot inputs give integer counts found by brute-force counting;
* invariants: branch == tail of (view ++ branch); siblings added, removed or
  permuted leave a branch bit-identical; a packed pass equals per-view runs;
  branches from the cached final state equal the in-pass branches; linearity.
"""
import os

import numpy as np
import pytest

from oracle import (oracle_branches_from_state, oracle_pass, segment_chunked,
                    segment_quadratic)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, T, H, D, scale=1.0):
    return rng.standard_normal((T, H, D)) * scale


def _rel(a, b):
    den = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / (den if den > 0 else 1.0))


def _cu(lens, start=0):
    return np.concatenate([[start], start + np.cumsum(lens)]).astype(np.int32)


# ---------------------------------------------------------------- hand example
def _load_golden():
    meta, rows, final = {}, [], None
    with open(os.path.join(GOLDEN, "hand_d2.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "row":
                rows.append([float(x) for x in vals])
            elif key == "final":
                final = np.array([float(x) for x in vals]).reshape(2, 2)
            else:
                meta[key] = np.array([int(x) for x in vals], dtype=np.int32)
    rows = np.array(rows)
    k = rows[:, 0:2][:, None, :]
    v = rows[:, 2:4][:, None, :]
    q = rows[:, 4:6][:, None, :]
    o = rows[:, 6:8][:, None, :]
    return meta, q, k, v, o, final


def test_hand_worked_example():
    meta, q, k, v, o, final = _load_golden()
    out, state = oracle_pass(q, k, v, meta["view_cu"], meta["branch_cu"],
                             meta["branch_parent"])
    assert np.array_equal(out, o)
    assert np.array_equal(state[0, 0], final)


# ---------------------------------------------------------------- quadratic and chunked forms
EDGE_LENS = [0, 1, 63, 64, 65, 127, 128, 129]


@pytest.mark.parametrize("L", EDGE_LENS)
def test_recurrent_equals_quadratic_and_chunked(L):
    rng = np.random.default_rng(100 + L)
    H, D = 2, 64
    branch_lens = [1, 5, 64, 70]
    T = L + sum(branch_lens)
    q, k, v = (_rand(rng, T, H, D, s) for s in (0.125, 0.125, 1.0))
    vcu = _cu([L])
    bcu = _cu(branch_lens, L)
    par = np.zeros(len(branch_lens), np.int32)
    out, state = oracle_pass(q, k, v, vcu, bcu, par)

    ref_v, S_v = segment_quadratic(q[:L], k[:L], v[:L])
    chk_v, S_c = segment_chunked(q[:L], k[:L], v[:L])
    assert _rel(out[:L], ref_v) <= 1e-12 if L else True
    assert _rel(out[:L], chk_v) <= 1e-12 if L else True
    assert _rel(state[0], S_v) <= 1e-12 if L else np.all(state == 0)
    assert _rel(S_c, S_v) <= 1e-12 if L else True
    for b in range(len(branch_lens)):
        r0, r1 = bcu[b], bcu[b + 1]
        ref_b, _ = segment_quadratic(q[r0:r1], k[r0:r1], v[r0:r1], S_v)
        chk_b, _ = segment_chunked(q[r0:r1], k[r0:r1], v[r0:r1], S_v)
        assert _rel(out[r0:r1], ref_b) <= 1e-12
        assert _rel(out[r0:r1], chk_b) <= 1e-12


def test_tiny_workload_matches_quadratic_form():
    from hybrid_linear_attention_packed_gb300 import workloads
    w = workloads.tiny_oracle_case(0)
    q, k, v = (t.double().numpy() for t in (w.q, w.k, w.v))
    out, state = oracle_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent)
    finals = []
    for s in range(w.V):
        r0, r1 = w.view_cu[s], w.view_cu[s + 1]
        ref, S = segment_quadratic(q[r0:r1], k[r0:r1], v[r0:r1])
        finals.append(S)
        assert _rel(out[r0:r1], ref) <= 1e-12
        assert _rel(state[s], S) <= 1e-12
    for b in range(w.B):
        r0, r1 = w.branch_cu[b], w.branch_cu[b + 1]
        ref, _ = segment_quadratic(q[r0:r1], k[r0:r1], v[r0:r1], finals[w.branch_parent[b]])
        assert _rel(out[r0:r1], ref) <= 1e-12


# ---------------------------------------------------------------- closed forms
def test_final_state_is_kt_v():
    rng = np.random.default_rng(7)
    lens = [300, 1, 64]
    T, H, D = sum(lens), 3, 64
    q, k, v = (_rand(rng, T, H, D) for _ in range(3))
    vcu = _cu(lens)
    _, state = oracle_pass(q, k, v, vcu, [0], [])
    for s in range(len(lens)):
        r0, r1 = vcu[s], vcu[s + 1]
        for h in range(H):
            ref = k[r0:r1, h, :].T @ v[r0:r1, h, :]
            assert _rel(state[s, h], ref) <= 1e-12


def test_d1_is_a_cumulative_sum():
    rng = np.random.default_rng(8)
    T, H = 257, 2
    q, k, v = (_rand(rng, T, H, 1) for _ in range(3))
    out, _ = oracle_pass(q, k, v, [0, T], [T], [])
    for h in range(H):
        ref = q[:, h, 0] * np.cumsum(k[:, h, 0] * v[:, h, 0])
        assert _rel(out[:, h, 0], ref) <= 1e-12


def test_one_hot_inputs_give_exact_counts():
    # k_t = e_a, v_t = e_b, q_t = e_c: o_t[j] counts the rows s <= t of the
    # same segment (plus, for branches, all parent-view rows) with a_s = c_t
    # and b_s = j.  Counted here by brute force, with no matrix products.
    rng = np.random.default_rng(9)
    D, H = 8, 2
    view_lens, branch_lens, par = [40, 17], [5, 9, 12], [0, 1, 0]
    vcu = _cu(view_lens)
    bcu = _cu(branch_lens, int(vcu[-1]))
    T = int(bcu[-1])
    a, b, c = (rng.integers(0, D, size=(T, H)) for _ in range(3))
    eye = np.eye(D)
    k, v, q = eye[a], eye[b], eye[c]
    out, _ = oracle_pass(q, k, v, vcu, bcu, par)

    def rows_before(seg_rows_prefix, t_rows):
        return list(seg_rows_prefix) + list(t_rows)

    for h in range(H):
        for s in range(len(view_lens)):
            r0, r1 = vcu[s], vcu[s + 1]
            for t in range(r0, r1):
                for j in range(D):
                    n = sum(1 for u in range(r0, t + 1) if a[u, h] == c[t, h] and b[u, h] == j)
                    assert out[t, h, j] == n
        for bi in range(len(branch_lens)):
            p = par[bi]
            v0, v1 = vcu[p], vcu[p + 1]
            r0, r1 = bcu[bi], bcu[bi + 1]
            for t in range(r0, r1):
                src = rows_before(range(v0, v1), range(r0, t + 1))
                for j in range(D):
                    n = sum(1 for u in src if a[u, h] == c[t, h] and b[u, h] == j)
                    assert out[t, h, j] == n


# ---------------------------------------------------------------- invariants
def _random_pass(seed, view_lens, branch_lens, par, H=2, D=64):
    rng = np.random.default_rng(seed)
    vcu = _cu(view_lens)
    bcu = _cu(branch_lens, int(vcu[-1]))
    T = int(bcu[-1])
    q, k, v = (_rand(rng, T, H, D, s) for s in (0.125, 0.125, 1.0))
    return q, k, v, vcu, bcu, np.asarray(par, np.int32)


def test_branch_equals_tail_of_view_plus_branch():
    q, k, v, vcu, bcu, par = _random_pass(11, [150, 90], [20, 33, 7], [1, 0, 1])
    out, _ = oracle_pass(q, k, v, vcu, bcu, par)
    for b in range(3):
        p = par[b]
        rows = np.r_[vcu[p]:vcu[p + 1], bcu[b]:bcu[b + 1]]
        n = len(rows)
        o1, _ = oracle_pass(q[rows], k[rows], v[rows], [0, n], [n], [])
        nb = bcu[b + 1] - bcu[b]
        assert np.array_equal(o1[n - nb:], out[bcu[b]:bcu[b + 1]])


def test_siblings_do_not_change_a_branch():
    q, k, v, vcu, bcu, par = _random_pass(12, [130], [9, 14, 20, 31], [0, 0, 0, 0])
    out, _ = oracle_pass(q, k, v, vcu, bcu, par)
    # permute: branches in reverse order, repacked
    order = [3, 2, 1, 0]
    vrows = np.r_[vcu[0]:vcu[1]]
    rows = [vrows] + [np.r_[bcu[b]:bcu[b + 1]] for b in order]
    idx = np.concatenate(rows)
    lens = [bcu[b + 1] - bcu[b] for b in order]
    out2, _ = oracle_pass(q[idx], k[idx], v[idx], [0, len(vrows)],
                          _cu(lens, len(vrows)), [0] * 4)
    pos = len(vrows)
    for b, L in zip(order, lens):
        assert np.array_equal(out2[pos:pos + L], out[bcu[b]:bcu[b] + L])
        pos += L
    # remove all siblings but one, and add a new one
    for keep in range(4):
        extra = 17
        rng = np.random.default_rng(99)
        idx = np.concatenate([vrows, np.r_[bcu[keep]:bcu[keep + 1]]])
        qq = np.concatenate([q[idx], rng.standard_normal((extra,) + q.shape[1:])])
        kk = np.concatenate([k[idx], rng.standard_normal((extra,) + q.shape[1:])])
        vv = np.concatenate([v[idx], rng.standard_normal((extra,) + q.shape[1:])])
        L = bcu[keep + 1] - bcu[keep]
        out3, _ = oracle_pass(qq, kk, vv, [0, len(vrows)],
                              [len(vrows), len(vrows) + L, len(vrows) + L + extra], [0, 0])
        assert np.array_equal(out3[len(vrows):len(vrows) + L], out[bcu[keep]:bcu[keep + 1]])


def test_packed_pass_equals_per_view_runs():
    view_lens, branch_lens, par = [70, 200, 1, 64], [5, 6, 7, 8, 9], [0, 1, 3, 1, 2]
    q, k, v, vcu, bcu, par = _random_pass(13, view_lens, branch_lens, par)
    out, state = oracle_pass(q, k, v, vcu, bcu, par)
    for s in range(len(view_lens)):
        bs = [b for b in range(len(branch_lens)) if par[b] == s]
        idx = np.concatenate([np.r_[vcu[s]:vcu[s + 1]]] + [np.r_[bcu[b]:bcu[b + 1]] for b in bs])
        n_v = vcu[s + 1] - vcu[s]
        lens = [bcu[b + 1] - bcu[b] for b in bs]
        o1, st1 = oracle_pass(q[idx], k[idx], v[idx], [0, n_v], _cu(lens, n_v),
                              [0] * len(bs))
        assert np.array_equal(st1[0], state[s])
        assert np.array_equal(o1[:n_v], out[vcu[s]:vcu[s + 1]])
        pos = n_v
        for b, L in zip(bs, lens):
            assert np.array_equal(o1[pos:pos + L], out[bcu[b]:bcu[b + 1]])
            pos += L


def test_branches_from_cached_state_equal_in_pass_branches():
    q, k, v, vcu, bcu, par = _random_pass(14, [100, 129], [3, 64, 65, 1], [1, 1, 0, 0])
    out, state = oracle_pass(q, k, v, vcu, bcu, par)
    out2 = oracle_branches_from_state(state, q, k, v, bcu, par, fill=np.nan)
    for b in range(4):
        assert np.array_equal(out2[bcu[b]:bcu[b + 1]], out[bcu[b]:bcu[b + 1]])
    assert np.all(np.isnan(out2[:vcu[-1]]))   # view rows untouched


def test_linear_in_v_and_in_q():
    q, k, v, vcu, bcu, par = _random_pass(15, [77], [12], [0])
    rng = np.random.default_rng(16)
    v2 = rng.standard_normal(v.shape)
    q2 = rng.standard_normal(q.shape)
    o, _ = oracle_pass(q, k, v, vcu, bcu, par)
    o_v2, _ = oracle_pass(q, k, v2, vcu, bcu, par)
    o_sum, _ = oracle_pass(q, k, 2.0 * v - 3.0 * v2, vcu, bcu, par)
    assert _rel(o_sum, 2.0 * o - 3.0 * o_v2) <= 1e-12
    o_q2, _ = oracle_pass(q2, k, v, vcu, bcu, par)
    o_qs, _ = oracle_pass(q + q2, k, v, vcu, bcu, par)
    assert _rel(o_qs, o + o_q2) <= 1e-12


def test_heads_are_independent_and_threads_do_not_matter():
    q, k, v, vcu, bcu, par = _random_pass(17, [200, 33], [40, 2], [0, 1], H=4)
    o1, s1 = oracle_pass(q, k, v, vcu, bcu, par, nthreads=1)
    o4, s4 = oracle_pass(q, k, v, vcu, bcu, par, nthreads=4)
    assert np.array_equal(o1, o4) and np.array_equal(s1, s4)
    oh, sh = oracle_pass(q[:, 2:3], k[:, 2:3], v[:, 2:3], vcu, bcu, par)
    assert np.array_equal(oh[:, 0], o1[:, 2]) and np.array_equal(sh[:, 0], s1[:, 2])


def test_rows_outside_segments_untouched_and_bad_metadata_rejected():
    q, k, v, _, _, _ = _random_pass(18, [10], [5], [0])
    T = q.shape[0]
    out, _ = oracle_pass(q, k, v, [2, 8], [9, 12], [0], fill=np.nan)
    assert np.all(np.isnan(out[:2])) and np.all(np.isnan(out[8:9])) and np.all(np.isnan(out[12:]))
    assert not np.any(np.isnan(out[2:8])) and not np.any(np.isnan(out[9:12]))
    with pytest.raises(ValueError):
        oracle_pass(q, k, v, [0, T + 1], [T + 1], [])
    with pytest.raises(ValueError):
        oracle_pass(q, k, v, [5, 2], [5], [])
    with pytest.raises(ValueError):
        oracle_pass(q, k, v, [0, 5], [5, 8], [1])


@pytest.mark.parametrize("seed", range(4))
def test_random_packed_passes_equal_quadratic_forms(seed):
    """Whole random packed passes through the C recurrence against the masked
    quadratic form per segment, each branch started from its parent's final
    state written in closed form (K_p^T V_p by einsum), rows of no segment
    untouched."""
    rng = np.random.default_rng([seed, 9])
    V = int(rng.integers(1, 4))
    vl = [int(x) for x in rng.integers(0, 150, size=V)]
    bl, par = [], []
    for v in range(V):
        for _ in range(int(rng.integers(0, 4))):
            bl.append(int(rng.integers(0, 80)))
            par.append(v)
    vcu = _cu(vl, int(rng.integers(0, 5)))
    bcu = _cu(bl, int(vcu[-1]) + int(rng.integers(0, 5)))
    T = int(bcu[-1]) + int(rng.integers(0, 5))
    H, D = 2, 8
    q, k, v = _rand(rng, T, H, D), _rand(rng, T, H, D), _rand(rng, T, H, D)
    out, state = oracle_pass(q, k, v, vcu, bcu, par, fill=5.0)
    seg = np.zeros(T, dtype=bool)
    for s in range(V):
        a, e = vcu[s], vcu[s + 1]
        seg[a:e] = True
        final = np.einsum("thi,thj->hij", k[a:e], v[a:e])
        assert np.max(np.abs(state[s] - final)) <= 1e-12 * max(1.0, np.max(np.abs(final)))
        if e > a:
            ref, _ = segment_quadratic(q[a:e], k[a:e], v[a:e])
            assert _rel(out[a:e], ref) <= 1e-12
    for b in range(len(bl)):
        a, e = bcu[b], bcu[b + 1]
        seg[a:e] = True
        pa, pe = vcu[par[b]], vcu[par[b] + 1]
        S0 = np.einsum("thi,thj->hij", k[pa:pe], v[pa:pe])
        if e > a:
            ref, _ = segment_quadratic(q[a:e], k[a:e], v[a:e], S0)
            assert _rel(out[a:e], ref) <= 1e-12
    assert np.all(out[~seg] == 5.0)
