"""The benchmark's reference arm on the CPU: `bench.py --impl reference` times
the float64 oracle and prints one JSON line with the keys the timing contract
names (no GPU needed)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True,
                       text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


@pytest.mark.parametrize("layer", ["linear", "softmax"])
def test_reference_arm_prints_one_contract_line(layer):
    d = _run("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1",
             "--layer", layer)
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"].startswith("tiny")


def test_error_measure_of_the_cpu_baseline_leg():
    """The leg that compares the benchmarked output with the oracle uses the
    parity tests' measure over the rows of segments only."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    from hybrid_linear_attention_packed_gb300 import workloads
    w = workloads.make_pass([5, 3], [2], [1], H=1, dtype="f32", seed=0, lead_rows=1, mid_rows=2,
                            tail_rows=1)
    m = bench.segment_mask(w)
    assert m.tolist() == [False] + [True] * 8 + [False, False] + [True] * 2 + [False]
    ref = np.array([[1.0, -4.0], [2.0, 0.5]])
    assert bench.max_rel_err(ref + np.array([[0.0, 0.4], [0.0, 0.0]]), ref) == pytest.approx(0.1)
    assert bench.max_rel_err(np.zeros((0, 2)), np.zeros((0, 2))) == 0.0


def test_reference_arm_config_matches_the_gpu_arm_keys():
    """Both arms name the workload with the same config keys (the GPU arm adds
    no key the reference arm lacks)."""
    d = _run("--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "1")
    assert d["config"]["parallelism"] == "dp1"


def test_branch_variants_for_the_cold_plan_leg():
    """The cold-plan leg's metadata variants cover the same rows with the same
    parents and views, and cut the branches differently (fresh plans)."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    from hybrid_linear_attention_packed_gb300 import workloads
    w = workloads.single_request(0)
    vs = bench.branch_variants(w, 24)
    seen = set()
    for cu, par in vs:
        assert cu[0] == w.branch_cu[0] and cu[-1] == w.branch_cu[-1]
        assert np.array_equal(par, w.branch_parent)
        assert sorted(np.diff(cu).tolist()) == sorted(w.branch_lens.tolist())
        seen.add(tuple(cu.tolist()))
    assert len(seen) > 16   # more distinct plans than the plan cache holds
