"""The data-parallel split on CPU: world size 2 over gloo (127.0.0.1), no GPU.

Each rank takes its share of the requests of a packed pass
(``sharding.split_requests``), builds its own sub-pass
(``sharding.request_sub_pass``) and runs the float64 oracle on it; rank 0
gathers the pieces.  Requests are independent ("Serving 0.88M TPS from Two
RTXs and Mac Minis", section "The Workload"), so the reassembled outputs and
view states equal the whole pass's bit for bit.  The step time reduction of a
weak-scaling job (``sharding.max_over_ranks``) is checked on the same group.
"""
import datetime
import os
import socket
import time

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from hybrid_linear_attention_packed_gb300 import sharding, workloads

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload():
    return workloads.make_pass([300, 70, 129, 1, 500], [9, 40, 128, 3, 200, 17, 5, 66],
                               [0, 0, 1, 2, 2, 3, 4, 4], H=2, dtype="f32", seed=11)


def _rank_main(rank, port, result_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        from oracle import oracle_pass
        w = _workload()
        parts = sharding.split_requests(w.view_lens, w.branch_lens, w.branch_parent, WORLD)
        mine = parts[rank]
        idx, vcu, bcu, par = sharding.request_sub_pass(w.view_cu, w.branch_cu, w.branch_parent, mine)
        q, k, v = (t.double().numpy()[idx] for t in (w.q, w.k, w.v))
        out, state = oracle_pass(q, k, v, vcu, bcu, par, nthreads=1)
        gathered = [None] * WORLD
        dist.all_gather_object(gathered, (rank, mine, idx, out, state))
        # each rank times a different amount; the job reports the slowest
        t_max = sharding.max_over_ranks(1.5 + rank, dist)
        if rank == 0:
            np.savez(result_path, t_max=t_max,
                     **{"r%d_%s" % (r, n): a for r, m, i, o, s in gathered
                        for n, a in (("req", np.asarray(m)), ("idx", i), ("out", o), ("state", s))})
    finally:
        dist.destroy_process_group()


def test_split_covers_every_request_once_and_balances():
    w = workloads.sweep(16, 0)
    parts = sharding.split_requests(w.view_lens, w.branch_lens, w.branch_parent, 4)
    assert sorted(v for p in parts for v in p) == list(range(w.V))
    rows = sharding.request_rows(w.view_lens, w.branch_lens, w.branch_parent)
    loads = [int(rows[p].sum()) for p in parts]
    assert max(loads) - min(loads) <= int(rows.max())     # greedy largest-first bound
    assert sharding.split_requests([5], [], [], 3) == [[0], [], []]
    with pytest.raises(ValueError):
        sharding.split_requests([5], [], [], 0)


def test_two_ranks_reassemble_the_whole_pass(tmp_path):
    from oracle import build_oracle, oracle_pass
    build_oracle()
    path = str(tmp_path / "ranks.npz")
    mp.start_processes(_rank_main, args=(_free_port(), path), nprocs=WORLD, start_method="spawn")
    res = np.load(path)
    assert float(res["t_max"]) == 2.5
    w = _workload()
    ref, ref_state = oracle_pass(w.q.double().numpy(), w.k.double().numpy(), w.v.double().numpy(),
                                 w.view_cu, w.branch_cu, w.branch_parent, nthreads=1)
    got = np.zeros_like(ref)
    got_state = np.zeros_like(ref_state)
    seen = []
    for r in range(WORLD):
        req, idx = res["r%d_req" % r], res["r%d_idx" % r]
        got[idx] = res["r%d_out" % r]
        got_state[req] = res["r%d_state" % r]
        seen.extend(req.tolist())
    assert sorted(seen) == list(range(w.V))
    assert np.array_equal(got, ref)
    assert np.array_equal(got_state, ref_state)


def _leaver_main(rank, port, result_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD, timeout=datetime.timedelta(seconds=5))
    if rank == 1:
        return      # leaves between steps: never joins the next collective
    t0 = time.monotonic()
    try:
        sharding.max_over_ranks(1.0, dist)
        outcome = "completed"
    except RuntimeError as exc:     # the peer's connection closed, or the timeout ran out
        outcome = "error: %s" % str(exc).splitlines()[0]
    with open(result_path, "w") as f:
        f.write("%s\n%.3f\n" % (outcome, time.monotonic() - t0))
    dist.destroy_process_group()


def test_a_rank_that_leaves_ends_the_others_step_with_an_error(tmp_path):
    """Failure detection on the host: a rank that leaves between steps makes
    the next step-time reduction of the others fail within the process
    group's short timeout instead of waiting for ever."""
    path = str(tmp_path / "leaver.txt")
    mp.start_processes(_leaver_main, args=(_free_port(), path), nprocs=WORLD, start_method="spawn")
    outcome, elapsed = open(path).read().splitlines()[:2]
    print(outcome, elapsed)
    assert outcome.startswith("error"), outcome
    assert float(elapsed) < 30.0
