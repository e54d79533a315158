"""Shared helpers of the GPU tests: run the CUDA path and the oracle on the same
seeded inputs and compare them."""
from __future__ import annotations

import numpy as np
import torch

TOL = {"f32": 1e-3, "bf16": 1e-2}


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    diff = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    return diff / den if den > 0 else diff


def segment_rows(w) -> np.ndarray:
    """Boolean mask of the rows that belong to a segment."""
    m = np.zeros(w.T, dtype=bool)
    for cu in (w.view_cu, w.branch_cu):
        for s in range(len(cu) - 1):
            m[cu[s]:cu[s + 1]] = True
    return m


def to_device(w, dev):
    return tuple(t.to(dev).contiguous() for t in (w.q, w.k, w.v))


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def sub_pass(w, views):
    """The rows, metadata and row map of the sub-pass made of the given views and
    their branches (segments are independent, so the oracle can check a sample
    of a large pass one request at a time)."""
    views = list(views)
    rows, vlens, blens, par = [], [], [], []
    for nv, s in enumerate(views):
        rows.append(np.arange(w.view_cu[s], w.view_cu[s + 1]))
        vlens.append(w.view_cu[s + 1] - w.view_cu[s])
    for b in range(w.B):
        p = int(w.branch_parent[b])
        if p in views:
            rows.append(np.arange(w.branch_cu[b], w.branch_cu[b + 1]))
            blens.append(w.branch_cu[b + 1] - w.branch_cu[b])
            par.append(views.index(p))
    idx = np.concatenate(rows) if rows else np.zeros(0, dtype=np.int64)
    vcu = np.concatenate([[0], np.cumsum(vlens)]).astype(np.int32)
    bcu = (np.concatenate([[0], np.cumsum(blens)]) + vcu[-1]).astype(np.int32)
    return idx, vcu, bcu, np.asarray(par, dtype=np.int32)
