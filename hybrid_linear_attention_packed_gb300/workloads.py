"""Seeded synthetic packed passes (inputs only -- no attention arithmetic here).

The pages measure on real spans and real requests that are not available; the
generators below stand in for them with the shapes the pages give ("Serving
0.88M TPS from Two RTXs and Mac Minis": views of 500 to 18,000 tokens with one
to hundreds of branches, section "Cost Model"; 8 behaviours, section
"Kernels"; 4-request passes, section "Kernels"; 4 shards, section "Long
Requests"; 7,400 tokens, section "Kernels").

Recipe (shared by the CUDA path and the oracle, which both read the same bytes):

* structure stream ``numpy.random.default_rng([seed, 0])``, data stream
  ``numpy.random.default_rng([seed, 1])`` (PCG64);
* "uniform in [a, b]" is ``integers(a, b + 1)``; "log-uniform in [a, b]" is
  ``round(exp(uniform(ln a, ln b)))`` clipped to ``[a, b]``;
* q, k, v are drawn in that order as float32 ``standard_normal((T, H, D))``,
  multiplied by their scale (powers of two, so exact), then rounded to
  nearest-even bf16 where the workload is bf16;
* packed row order: all views in order, then all branches grouped by parent
  view in view order (each branch's parent is its own view).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch

HEAD_DIM = 64


@dataclasses.dataclass
class Workload:
    name: str
    H: int
    D: int
    dtype: str                      # "bf16" or "f32"
    view_lens: np.ndarray           # int64 [V]
    branch_lens: np.ndarray         # int64 [B]
    branch_parent: np.ndarray       # int32 [B]
    view_cu: np.ndarray             # int32 [V+1]
    branch_cu: np.ndarray           # int32 [B+1]
    q: torch.Tensor                 # CPU [T, H, D]
    k: torch.Tensor
    v: torch.Tensor

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    @property
    def V(self) -> int:
        return int(len(self.view_lens))

    @property
    def B(self) -> int:
        return int(len(self.branch_lens))

    @property
    def rows(self) -> int:
        """Rows that belong to a segment (view rows plus branch rows)."""
        return int(self.view_lens.sum() + self.branch_lens.sum())

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


def _uniform_int(rng, a: int, b: int, n: int) -> np.ndarray:
    return rng.integers(a, b + 1, size=n).astype(np.int64)


def _log_uniform_int(rng, a: int, b: int, n: int) -> np.ndarray:
    x = np.exp(rng.uniform(math.log(a), math.log(b), size=n))
    return np.clip(np.round(x), a, b).astype(np.int64)


def _cu(lens: np.ndarray, start: int) -> np.ndarray:
    cu = np.zeros(len(lens) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lens)
    cu += start
    if cu[-1] > np.iinfo(np.int32).max:
        raise ValueError("packed pass too large for int32 row offsets")
    return cu.astype(np.int32)


def _cast(x: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(x)
    return t.to(torch.bfloat16) if dtype == "bf16" else t.to(torch.float32)


def draw_qkv(seed: int, T: int, H: int, D: int, dtype: str,
             q_scale: float, k_scale: float, v_scale: float):
    """Draw q, k, v [T, H, D] from the data stream of ``seed`` (see module doc)."""
    rng = np.random.default_rng([seed, 1])
    out = []
    for scale in (q_scale, k_scale, v_scale):
        x = rng.standard_normal((T, H, D), dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        out.append(_cast(x, dtype))
    return tuple(out)


def make_pass(view_lens: Sequence[int], branch_lens: Sequence[int],
              branch_parent: Sequence[int], *, H: int, dtype: str, seed: int,
              q_scale: float = 1.0 / 8, k_scale: float = 1.0 / 8,
              v_scale: float = 1.0, D: int = HEAD_DIM, name: str = "custom",
              lead_rows: int = 0, mid_rows: int = 0, tail_rows: int = 0) -> Workload:
    """Pack explicit view and branch lengths into one buffer.

    Rows that belong to no segment can be placed before the first view
    (``lead_rows``), between the last view and the first branch
    (``mid_rows``) and after the last branch (``tail_rows``); they are drawn
    like every other row.
    """
    view_lens = np.asarray(view_lens, dtype=np.int64).reshape(-1)
    branch_lens = np.asarray(branch_lens, dtype=np.int64).reshape(-1)
    branch_parent = np.asarray(branch_parent, dtype=np.int32).reshape(-1)
    if len(branch_parent) != len(branch_lens):
        raise ValueError("one parent per branch")
    view_cu = _cu(view_lens, lead_rows)
    branch_cu = _cu(branch_lens, int(view_cu[-1]) + mid_rows)
    T = int(branch_cu[-1]) + tail_rows
    q, k, v = draw_qkv(seed, T, H, D, dtype, q_scale, k_scale, v_scale)
    return Workload(name, H, D, dtype, view_lens, branch_lens, branch_parent,
                    view_cu, branch_cu, q, k, v)


def pass_layout(view_lens: Sequence[int], branch_lens: Sequence[int]):
    """int32 (view_cu, branch_cu) of a pass packed with no gaps (views, then
    branches), for passes whose inputs are drawn on the device."""
    view_cu = _cu(np.asarray(view_lens, dtype=np.int64).reshape(-1), 0)
    branch_cu = _cu(np.asarray(branch_lens, dtype=np.int64).reshape(-1), int(view_cu[-1]))
    return view_cu, branch_cu


def draw_qkv_device(seed: int, T: int, H: int, device, q_scale: float = 1.0 / 8,
                    k_scale: float = 1.0 / 8, v_scale: float = 1.0, D: int = HEAD_DIM):
    """q, k, v [T, H, D] bf16 drawn on ``device`` by torch's generator for that
    device, seeded with ``seed`` (q, k, v in that order, each a standard normal
    times its scale): passes of billions of elements that host generation
    would take minutes to draw and copy.  Tests read back only the rows they
    check."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = []
    for scale in (q_scale, k_scale, v_scale):
        x = torch.randn((T, H, D), generator=g, device=device, dtype=torch.bfloat16)
        if scale != 1.0:
            x.mul_(scale)
        out.append(x)
    return tuple(out)


def tiny_oracle_case(seed: int = 0) -> Workload:
    """1 head, d=64, fp32, q,k,v ~ N(0,1)/8; views of 130 and 77 tokens; three
    branches of 9, 14 and 20 tokens per view, each forking from its view."""
    view_lens = [130, 77]
    branch_lens = [9, 14, 20, 9, 14, 20]
    parent = [0, 0, 0, 1, 1, 1]
    return make_pass(view_lens, branch_lens, parent, H=1, dtype="f32", seed=seed,
                     q_scale=1 / 8, k_scale=1 / 8, v_scale=1 / 8,
                     name="tiny: 1 head, fp32, views 130+77, 3 branches each")


def single_request(seed: int = 0) -> Workload:
    """16 heads, bf16; one 7,400-token view plus 8 branches of U[32,96] rows."""
    rng = np.random.default_rng([seed, 0])
    branch_lens = _uniform_int(rng, 32, 96, 8)
    return make_pass([7400], branch_lens, [0] * 8, H=16, dtype="bf16", seed=seed,
                     name="single request: 16 heads, bf16, 7400-token view + 8 branches")


def packed_four(seed: int = 0) -> Workload:
    """16 heads, bf16; 4 views of U[500,18000] tokens, 8 branches each of U[32,96]."""
    rng = np.random.default_rng([seed, 0])
    view_lens = _uniform_int(rng, 500, 18000, 4)
    branch_lens = _uniform_int(rng, 32, 96, 32)
    parent = np.repeat(np.arange(4), 8)
    return make_pass(view_lens, branch_lens, parent, H=16, dtype="bf16", seed=seed,
                     name="packed pass of 4 requests: 16 heads, bf16, 8 branches each")


def cached_long(seed: int = 0) -> Workload:
    """16 heads, bf16; one 18,000-token view plus 256 branches of U[24,128] rows.

    The view is run once without branches to get its final state; the branches
    then run from that cached state in 4 shards of 64 (``shards()``).
    """
    rng = np.random.default_rng([seed, 0])
    branch_lens = _uniform_int(rng, 24, 128, 256)
    return make_pass([18000], branch_lens, [0] * 256, H=16, dtype="bf16", seed=seed,
                     name="long request from cached state: 18000-token view, 256 branches")


def shards(w: Workload, n_shards: int) -> List[np.ndarray]:
    """Split a workload's branches into ``n_shards`` runs of consecutive branches;
    each entry is the int32 branch_cu slice (absolute row offsets)."""
    B = w.B
    per = (B + n_shards - 1) // n_shards
    out = []
    for s in range(n_shards):
        b0, b1 = s * per, min(B, (s + 1) * per)
        out.append(np.ascontiguousarray(w.branch_cu[b0:b1 + 1]))
    return out


def sweep(n_views: int, seed: int = 0) -> Workload:
    """16 heads, bf16; ``n_views`` views of log-U[500,18000] tokens, log-U[1,300]
    branches per view, branch lengths U[16,128]."""
    rng = np.random.default_rng([seed, 0])
    view_lens = _log_uniform_int(rng, 500, 18000, n_views)
    counts = _log_uniform_int(rng, 1, 300, n_views)
    branch_lens = _uniform_int(rng, 16, 128, int(counts.sum()))
    parent = np.repeat(np.arange(n_views), counts)
    return make_pass(view_lens, branch_lens, parent, H=16, dtype="bf16", seed=seed,
                     name="throughput sweep: %d views" % n_views)


def by_name(name: str, seed: int = 0) -> Workload:
    if name == "tiny":
        return tiny_oracle_case(seed)
    if name == "single":
        return single_request(seed)
    if name == "packed4":
        return packed_four(seed)
    if name == "cached_long":
        return cached_long(seed)
    if name.startswith("sweep"):
        return sweep(int(name[5:]), seed)
    raise KeyError(name)


def one_hot_pass(view_lens, branch_lens, branch_parent, *, H: int, D: int,
                 dtype: str, seed: int, q_scale: float = 1.0) -> Workload:
    """Inputs whose rows are one-hot vectors e_a (k), e_b (v), q_scale * e_c (q)
    with a, b, c uniform over [0, D) from the data stream of ``seed``."""
    w = make_pass(view_lens, branch_lens, branch_parent, H=1, D=1, dtype="f32",
                  seed=seed)
    T = w.T
    rng = np.random.default_rng([seed, 1])
    mats = []
    for scale in (q_scale, 1.0, 1.0):
        idx = rng.integers(0, D, size=(T, H))
        x = np.zeros((T, H, D), dtype=np.float32)
        np.put_along_axis(x, idx[..., None], np.float32(scale), axis=2)
        mats.append(_cast(x, dtype))
    w.q, w.k, w.v = mats
    w.H, w.D, w.dtype = H, D, dtype
    return w
