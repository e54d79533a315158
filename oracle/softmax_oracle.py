"""Float64 oracle of the softmax-attention layers over the packed layout.

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the CPU
baseline of the benchmark, never by the product path.

The hybrid model has a few softmax-attention layers between its linear
layers ("Serving 0.88M TPS from Two RTXs and Mac Minis", section "The
Workload": a branch attends to its view but not to its siblings; section
"Long Requests": the view cache holds the softmax layers' K/V beside the
linear layers' state).  Over the same packed rows as the linear pass, per head:

* view row t of a view starting at row s attends to the rows s..t of its view;
* branch row t of a branch starting at row b, forking from view [s, e),
  attends to every row of that view and to the rows b..t of its branch;

    o_t = sum_j softmax_j(scale * q_t . k_j) v_j        over the visible j,
    lse_t = log sum_j exp(scale * q_t . k_j)           (natural log),

with scale = 1/sqrt(d) unless given.  Everything is computed in float64 from
the inputs widened exactly; rows in no segment hold ``fill``.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Tuple

import numpy as np


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().to(dtype=__import__("torch").float64).cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    if a is None:
        return np.zeros(0, dtype=np.int32)
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.asarray(a, dtype=np.int64).reshape(-1)


def _check(T, vcu, bcu, par):
    for name, cu in (("view_cu_seqlens", vcu), ("branch_cu_seqlens", bcu)):
        if cu.size == 1 and not (0 <= cu[0] <= T):
            raise ValueError("%s out of range" % name)
        if cu.size > 1 and (np.any(np.diff(cu) < 0) or cu[0] < 0 or cu[-1] > T):
            raise ValueError("%s must be non-decreasing within [0, T]" % name)
    V = max(vcu.size - 1, 0)
    B = max(bcu.size - 1, 0)
    if par.size != B:
        raise ValueError("one parent per branch")
    if B and (np.any(par < 0) or np.any(par >= V)):
        raise ValueError("branch parent out of range")


def softmax_rows(scores: np.ndarray, values: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Softmax over the last axis of ``scores`` (rows of visible scores, -inf
    where a key is hidden) applied to ``values``; returns (out, lse).  The row
    maximum is subtracted before exponentiating (the result is unchanged)."""
    m = np.max(scores, axis=-1, keepdims=True)
    p = np.exp(scores - m)
    l = np.sum(p, axis=-1, keepdims=True)
    return (p @ values) / l, (m + np.log(l))[..., 0]


def _segment(qs, ks, vs, kp, vp, scale):
    """One segment, all heads: queries qs [n,H,D] with own keys/values ks, vs
    [n,H,D] (causal, inclusive) after prefix keys/values kp, vp [m,H,D] that
    every query sees.  Returns out [n,H,D], lse [n,H]."""
    n, H, D = qs.shape
    m = kp.shape[0]
    out = np.empty((n, H, D))
    lse = np.empty((n, H))
    causal = np.tril(np.ones((n, n), dtype=bool))
    for h in range(H):
        kk = np.concatenate([kp[:, h], ks[:, h]], axis=0)      # [m+n, D]
        vv = np.concatenate([vp[:, h], vs[:, h]], axis=0)
        s = scale * (qs[:, h] @ kk.T)                         # [n, m+n]
        s[:, m:][~causal] = -np.inf
        out[:, h], lse[:, h] = softmax_rows(s, vv)
    return out, lse


def oracle_softmax_pass(q, k, v, view_cu_seqlens, branch_cu_seqlens, branch_parent,
                        scale: Optional[float] = None, fill: float = 0.0):
    """Float64 packed softmax-attention layer.  q, k, v: [T, H, D].
    Returns ``(out [T,H,D], lse [T,H])``; rows in no segment hold ``fill``."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, D = q.shape
    vcu, bcu, par = _i32(view_cu_seqlens), _i32(branch_cu_seqlens), _i32(branch_parent)
    _check(T, vcu, bcu, par)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.full((T, H, D), fill)
    lse = np.full((T, H), fill)
    empty = np.zeros((0, H, D))
    for s in range(max(vcu.size - 1, 0)):
        a, b = int(vcu[s]), int(vcu[s + 1])
        if b > a:
            out[a:b], lse[a:b] = _segment(q[a:b], k[a:b], v[a:b], empty, empty, scale)
    for br in range(max(bcu.size - 1, 0)):
        a, b = int(bcu[br]), int(bcu[br + 1])
        pa, pb = int(vcu[par[br]]), int(vcu[par[br] + 1])
        if b > a:
            out[a:b], lse[a:b] = _segment(q[a:b], k[a:b], v[a:b], k[pa:pb], v[pa:pb], scale)
    return out, lse


def oracle_softmax_rows(q, k, v, view_cu_seqlens, branch_cu_seqlens, branch_parent,
                        rows: Iterable[int], scale: Optional[float] = None):
    """The same layer for a sample of rows only (each row needs only its own
    visible keys), for checking passes too large to run whole.  Returns
    ``(out [len(rows),H,D], lse [len(rows),H])``; every row must lie in a
    segment."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, D = q.shape
    vcu, bcu, par = _i32(view_cu_seqlens), _i32(branch_cu_seqlens), _i32(branch_parent)
    _check(T, vcu, bcu, par)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rows = [int(r) for r in rows]
    out = np.empty((len(rows), H, D))
    lse = np.empty((len(rows), H))
    for n, t in enumerate(rows):
        sv = np.searchsorted(vcu, t, side="right") - 1
        sb = np.searchsorted(bcu, t, side="right") - 1
        if 0 <= sv < vcu.size - 1 and vcu[sv] <= t < vcu[sv + 1]:
            keys = np.arange(vcu[sv], t + 1)
        elif 0 <= sb < bcu.size - 1 and bcu[sb] <= t < bcu[sb + 1]:
            p = par[sb]
            keys = np.concatenate([np.arange(vcu[p], vcu[p + 1]), np.arange(bcu[sb], t + 1)])
        else:
            raise ValueError("row %d is in no segment" % t)
        for h in range(H):
            s = scale * (k[keys, h] @ q[t, h])
            o, l = softmax_rows(s[None, :], v[keys, h])
            out[n, h], lse[n, h] = o[0], l[0]
    return out, lse
