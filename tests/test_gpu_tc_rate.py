"""The tensor-core rate probe (``tests/probes/tc_rate.cu``) runs its modes
cleanly and gives self-consistent rates: the tile's 28 MMAs take no less than
its slowest part and no more than its parts one after another, and no mode
runs faster than the part's nominal dense bf16 rate (2.25 PFLOP/s over the SM
count at the sampled clock against 2,070 MHz) -- faster would mean the
instructions did not execute."""
import pytest
import torch

from probes import tc_rate

pytestmark = pytest.mark.gpu

NOMINAL_BF16_TFLOPS = 2250.0
MAX_SM_MHZ = 2070.0


def test_tc_rate_modes_are_consistent(cuda_device):
    nsm = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    res = {m: tc_rate.run(m, 0, 256) for m in tc_rate.MODES}
    for m, r in res.items():
        assert r["err"] == 0, m
        assert r["grid"] == nsm
        assert r["ns_per_group"] > 0
    parts = [res[m]["ns_per_group"] for m in ("qk", "kv", "pv", "qs")]
    assert max(parts) * 0.9 <= res["tile"]["ns_per_group"] <= sum(parts) * 1.1
    for m in ("qk", "kv", "pv", "qs"):
        cap = NOMINAL_BF16_TFLOPS / nsm * res[m]["mhz"] / MAX_SM_MHZ
        assert res[m]["tflops_per_sm"] <= cap * 1.05, (m, res[m])
