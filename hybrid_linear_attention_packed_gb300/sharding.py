"""Data-parallel split of a packed pass across ranks (one GPU per rank).

Requests -- a view with all of its branches -- are independent ("Serving
0.88M TPS from Two RTXs and Mac Minis", section "The Workload": a branch sees
only its own view), so a pass shards by request with no exchange between
ranks: each rank runs its own requests as its own pass.  This module holds the
host side of that split; it computes nothing of the attention itself.
"""
from __future__ import annotations

import heapq
from typing import List, Sequence, Tuple

import numpy as np


def request_rows(view_lens: Sequence[int], branch_lens: Sequence[int],
                 branch_parent: Sequence[int]) -> np.ndarray:
    """Rows of each request (its view plus its branches)."""
    rows = np.asarray(view_lens, dtype=np.int64).copy()
    np.add.at(rows, np.asarray(branch_parent, dtype=np.int64),
              np.asarray(branch_lens, dtype=np.int64))
    return rows


def split_requests(view_lens: Sequence[int], branch_lens: Sequence[int],
                   branch_parent: Sequence[int], world: int) -> List[List[int]]:
    """Deal the requests to `world` ranks, largest first, each to the rank with
    the fewest rows so far; every rank's list is in request order."""
    if world < 1:
        raise ValueError("world must be >= 1")
    rows = request_rows(view_lens, branch_lens, branch_parent)
    heap = [(0, r) for r in range(world)]
    out: List[List[int]] = [[] for _ in range(world)]
    for v in sorted(range(len(rows)), key=lambda i: (-rows[i], i)):
        load, r = heapq.heappop(heap)
        out[r].append(v)
        heapq.heappush(heap, (load + int(rows[v]), r))
    return [sorted(x) for x in out]


def request_sub_pass(view_cu: Sequence[int], branch_cu: Sequence[int],
                     branch_parent: Sequence[int],
                     requests: Sequence[int]) -> Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """The rows and metadata of the pass made of the given requests: returns
    (row index into the full pass, view_cu, branch_cu, branch_parent), views
    first in the given order, then each view's branches in their order."""
    view_cu = np.asarray(view_cu, dtype=np.int64)
    branch_cu = np.asarray(branch_cu, dtype=np.int64)
    parent = np.asarray(branch_parent, dtype=np.int64)
    requests = [int(v) for v in requests]
    pos = {v: n for n, v in enumerate(requests)}
    rows, vlens, blens, par = [], [], [], []
    for v in requests:
        rows.append(np.arange(view_cu[v], view_cu[v + 1]))
        vlens.append(view_cu[v + 1] - view_cu[v])
    for b in range(len(parent)):
        if int(parent[b]) in pos:
            rows.append(np.arange(branch_cu[b], branch_cu[b + 1]))
            blens.append(branch_cu[b + 1] - branch_cu[b])
            par.append(pos[int(parent[b])])
    idx = np.concatenate(rows) if rows else np.zeros(0, dtype=np.int64)
    vcu = np.concatenate([[0], np.cumsum(vlens, dtype=np.int64)]).astype(np.int32)
    bcu = (np.concatenate([[0], np.cumsum(blens, dtype=np.int64)]) + vcu[-1]).astype(np.int32)
    return idx, vcu, bcu, np.asarray(par, dtype=np.int32)


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest `value` over the ranks of the default process group (the
    step time a weak-scaling job reports), or `value` itself without one."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
