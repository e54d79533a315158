"""GPU tests of the view-state cache (``span_la_cache_*``): branches forked from
cached states by key equal branches forked from the same states passed
directly, match the oracle, and the cache evicts least recently used keys.

The long-request procedure these follow ("Serving 0.88M TPS from Two RTXs and
Mac Minis", section "Long Requests"): the view's final state is computed
once and cached, and the request's branches run as shards from it.
"""
import numpy as np
import pytest
import torch

from helpers import TOL, f64, rel_err, to_device
from hybrid_linear_attention_packed_gb300 import (SpanLAError, ViewStateCache,
                                                  span_la_branches_from_state, span_la_check,
                                                  span_la_pass, workloads)
from oracle import oracle_pass

pytestmark = pytest.mark.gpu

KEY0 = 0x9E3779B97F4A7C15   # arbitrary 64-bit keys, above 2**63 on purpose


def _branch_rows(w):
    m = np.zeros(w.T, bool)
    m[w.branch_cu[0]:w.branch_cu[-1]] = True
    return m


def test_cache_branches_equal_direct_and_oracle(cuda_device):
    """Four requests: views in one pass, their states put under keys, then all
    branches from the cache by key."""
    w = workloads.packed_four(0)
    q, k, v = to_device(w, cuda_device)
    _, state = span_la_pass(q, k, v, w.view_cu, None, None)
    keys = np.array([KEY0 + 7 * i for i in range(w.V)], dtype=np.uint64)
    with ViewStateCache(w.q.shape[1], capacity=8) as cache:
        cache.put(keys, state)
        out = cache.branches(keys[w.branch_parent], q, k, v, w.branch_cu,
                             out=torch.full_like(q, float("nan")))
        direct = span_la_branches_from_state(state, q, k, v, w.branch_cu, w.branch_parent,
                                             out=torch.full_like(q, float("nan")))
        span_la_check()
        br = _branch_rows(w)
        assert torch.equal(out[torch.from_numpy(br).to(cuda_device)],
                           direct[torch.from_numpy(br).to(cuda_device)])
        assert torch.isnan(out[torch.from_numpy(~br).to(cuda_device)]).all()
        ref, _ = oracle_pass(f64(w.q), f64(w.k), f64(w.v), w.view_cu, w.branch_cu,
                             w.branch_parent)
        e = rel_err(f64(out)[br], ref[br])
        print("cache branches vs oracle: %.2e" % e)
        assert e <= TOL[w.dtype]
        st = cache.stats()
        assert st["entries"] == w.V and st["puts"] == w.V and st["hits"] == w.B
        assert st["misses"] == 0 and st["evictions"] == 0


def test_cache_long_request_shards(cuda_device):
    """18,000-token view cached once; 256 branches as 4 shard calls by key equal
    one direct call over all branches, bit for bit."""
    w = workloads.cached_long(0)
    q, k, v = to_device(w, cuda_device)
    _, state = span_la_pass(q, k, v, w.view_cu, None, None)
    with ViewStateCache(w.q.shape[1], capacity=4) as cache:
        cache.put([KEY0], state)
        out = torch.full_like(q, float("nan"))
        for cu in workloads.shards(w, 4):
            cache.branches(np.full(len(cu) - 1, KEY0, np.uint64), q, k, v, cu, out=out)
        direct = span_la_branches_from_state(state, q, k, v, w.branch_cu, w.branch_parent)
        span_la_check()
        br = torch.from_numpy(_branch_rows(w)).to(cuda_device)
        assert torch.equal(out[br], direct[br])
        assert cache.stats()["hits"] == w.B


def test_cache_evicts_least_recently_used(cuda_device):
    w = workloads.packed_four(1)
    q, k, v = to_device(w, cuda_device)
    _, state = span_la_pass(q, k, v, w.view_cu, None, None)
    A, B, C = KEY0, KEY0 + 1, KEY0 + 2
    with ViewStateCache(w.q.shape[1], capacity=2) as cache:
        cache.put([A], state[0:1])
        cache.put([B], state[1:2])
        assert cache.contains([A]).tolist() == [True]          # A is now the most recent
        cache.put([C], state[2:3])                              # evicts B
        assert cache.contains([A, B, C]).tolist() == [True, False, True]
        st = cache.stats()
        assert st["entries"] == 2 and st["evictions"] == 1 and st["misses"] == 1
        # a branch call naming an evicted key is rejected and enqueues nothing
        b0, b1 = int(w.branch_cu[0]), int(w.branch_cu[1])
        out = torch.full_like(q, float("nan"))
        with pytest.raises(SpanLAError, match="not cached"):
            cache.branches([B], q, k, v, [b0, b1], out=out)
        span_la_check()
        assert torch.isnan(out).all()
        # C holds view 2's state: a branch from C equals the direct fork from view 2
        cache.branches([C], q, k, v, [b0, b1], out=out)
        direct = span_la_branches_from_state(state, q, k, v, [b0, b1], [2])
        span_la_check()
        assert torch.equal(out[b0:b1], direct[b0:b1])
        # a put of n keys never evicts one of its own keys; more than capacity is refused
        cache.put([A, B], state[0:2])
        assert cache.contains([A, B, C]).tolist() == [True, True, False]
        with pytest.raises(SpanLAError):
            cache.put([A, B, C], state[0:3])
        with pytest.raises(SpanLAError, match="distinct"):
            cache.put([A, A], state[0:2])


def test_cache_orders_puts_and_reads_across_streams(cuda_device):
    """A branch call on one stream reads the state put on another; a later put
    into the same slot on the first stream waits for that read."""
    w = workloads.cached_long(1)
    q, k, v = to_device(w, cuda_device)
    _, state = span_la_pass(q, k, v, w.view_cu, None, None)
    zeros = torch.zeros_like(state)
    out = torch.full_like(q, float("nan"))
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with ViewStateCache(w.q.shape[1], capacity=1) as cache:
        cache.put([KEY0], state, stream=s1)
        cache.branches(np.full(w.B, KEY0, np.uint64), q, k, v, w.branch_cu, out=out, stream=s2)
        cache.put([KEY0], zeros, stream=s1)      # overwrites the slot the branches read
        torch.cuda.synchronize()
        direct = span_la_branches_from_state(state, q, k, v, w.branch_cu, w.branch_parent)
        span_la_check()
        br = torch.from_numpy(_branch_rows(w)).to(cuda_device)
        assert torch.equal(out[br], direct[br])


def test_cache_rejects_mismatched_heads(cuda_device):
    w = workloads.tiny_oracle_case(0)
    q, k, v = to_device(w, cuda_device)
    with ViewStateCache(w.q.shape[1] + 1, capacity=2) as cache:
        with pytest.raises(ValueError):
            cache.put([1], torch.zeros(1, w.q.shape[1], 64, 64, device=cuda_device))
        with pytest.raises(SpanLAError, match="num_heads"):
            cache.branches([], q, k, v, [int(w.branch_cu[0])])
