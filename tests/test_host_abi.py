"""CPU-side checks of the C ABI: the library builds, loads and exports every
symbol ``include/spanla.h`` declares; host-side validation rejects bad
metadata before any CUDA call; the binding fails loudly when the library is
missing.  No compute call runs here (there is no GPU on this side)."""
import ctypes
import os
import re

import numpy as np
import pytest

from hybrid_linear_attention_packed_gb300 import build as spanla_build
from hybrid_linear_attention_packed_gb300 import spanla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = spanla_build.build()
    return spanla.load_library(path)


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "spanla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(span_la_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_symbols()
    assert set(declared) >= {"span_la_pass", "span_la_branches_from_state", "span_la_check"}
    for name in declared:
        assert hasattr(lib, name), "missing export %s" % name
    assert set(declared) == set(spanla.EXPORTED)


def test_version_and_status_strings(lib):
    assert lib.span_la_version() == 20000
    for code in range(6):
        assert lib.span_la_status_string(code)


def _dims(T=100, H=2, D=64, dtype=0):
    return spanla.Dims(T, H, D, dtype)


def _arr(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


FAKE = 1 << 20   # a 16-byte-aligned non-NULL address; never dereferenced on the host


def _pass(lib, vcu, bcu, par, dims=None, q=FAKE, out=FAKE, state=FAKE):
    dims = dims or _dims()
    (va, vp), (ba, bp), (pa, pp) = _arr(vcu), _arr(bcu), _arr(par)
    V, B = max(len(va) - 1, 0), max(len(ba) - 1, 0)
    st = lib.span_la_pass(q, q, q, dims, vp if V else None, V, bp if B else None, B,
                          pp if B else None, out, state, None)
    return st, lib.span_la_last_error_detail().decode()


@pytest.mark.parametrize("vcu,bcu,par,what", [
    ([0, 50, 40], [], [], "non-decreasing"),
    ([0, 101], [], [], "non-decreasing"),
    ([-1, 10], [], [], "non-decreasing"),
    ([0, 50], [40, 60], [0], "overlap"),
    ([0, 50], [50, 60], [1], "branch_parent"),
    ([0, 50], [50, 60], [-1], "branch_parent"),
])
def test_bad_metadata_is_rejected_before_any_launch(lib, vcu, bcu, par, what):
    st, detail = _pass(lib, vcu, bcu, par)
    assert st == 1 and what in detail


def _prepare(lib, vcu, bcu, par, dims=None):
    dims = dims or _dims()
    (va, vp), (ba, bp), (pa, pp) = _arr(vcu), _arr(bcu), _arr(par)
    V, B = max(len(va) - 1, 0), max(len(ba) - 1, 0)
    st = lib.span_la_plan_prepare(dims, vp if V else None, V, bp if B else None, B,
                                  pp if B else None, None)
    return st, lib.span_la_last_error_detail().decode()


@pytest.mark.parametrize("vcu,bcu,par,what", [
    ([0, 50, 40], [], [], "non-decreasing"),
    ([0, 101], [], [], "non-decreasing"),
    ([0, 50], [40, 60], [0], "overlap"),
    ([0, 50], [50, 60], [1], "branch_parent"),
])
def test_plan_prepare_rejects_what_the_pass_rejects(lib, vcu, bcu, par, what):
    """span_la_plan_prepare runs the pass's metadata checks before any device
    work: the same metadata gets the same status and detail."""
    st, detail = _prepare(lib, vcu, bcu, par)
    assert st == 1 and what in detail
    assert (st, detail) == _pass(lib, vcu, bcu, par)
    st, detail = _prepare(lib, [0, 10], [], [], dims=_dims(D=128))
    assert st == 2 and "head_dim" in detail
    assert _prepare(lib, [0], [], [])[0] == 0   # nothing to plan: no device work


def test_unsupported_shapes_and_pointers(lib):
    st, detail = _pass(lib, [0, 10], [], [], dims=_dims(D=128))
    assert st == 2 and "head_dim" in detail
    st, detail = _pass(lib, [0, 10], [], [], dims=_dims(dtype=7))
    assert st == 2
    st, detail = _pass(lib, [0, 10], [], [], dims=_dims(H=0))
    assert st == 1
    st, detail = _pass(lib, [0, 10], [], [], q=FAKE + 8)
    assert st == 1 and "aligned" in detail
    st, detail = _pass(lib, [0, 10], [], [], state=0)
    assert st == 1 and "view_state_out" in detail
    st, detail = _pass(lib, [0, 10], [], [], q=0)
    assert st == 1


def test_from_state_validation(lib):
    (ba, bp), (pa, pp) = _arr([0, 10, 20]), _arr([0, 1])
    st = lib.span_la_branches_from_state(FAKE, 1, FAKE, FAKE, FAKE, _dims(), bp, 2, pp, FAKE, None)
    assert st == 1 and "branch_parent" in lib.span_la_last_error_detail().decode()
    st = lib.span_la_branches_from_state(0, 2, FAKE, FAKE, FAKE, _dims(), bp, 2, pp, FAKE, None)
    assert st == 1 and "cached_state" in lib.span_la_last_error_detail().decode()


def test_empty_call_is_a_no_op(lib):
    st, _ = _pass(lib, [0], [], [], q=0, out=0, state=0)
    assert st == 0


def test_metadata_addresses(lib):
    """The binding passes int32 metadata by address: writable arrays through a
    ctypes view of their buffer, read-only ones through numpy's helper, empty
    ones as NULL; the address is the array's own data either way, and
    non-int32 or strided input is first copied to a contiguous int32 array."""
    a = np.arange(7, dtype=np.int32)
    b = np.arange(7, dtype=np.int32)
    b.flags.writeable = False
    assert spanla._iptr(a) == a.__array_interface__["data"][0]
    assert spanla._iptr(b) == b.__array_interface__["data"][0]
    assert spanla._iptr(np.zeros(0, dtype=np.int32)) is None
    c = spanla._i32(np.arange(14, dtype=np.int64)[::2])
    assert c.dtype == np.int32 and c.flags.c_contiguous and list(c) == list(range(0, 14, 2))
    assert spanla._i32(a) is a


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not found"):
        spanla.load_library(str(tmp_path / "nope.so"))


@pytest.mark.parametrize("variant", [spanla.PASS_ONE_LAUNCH, spanla.PASS_THREE_LAUNCHES])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("name", ["tiny", "single", "packed4", "cached_long", "sweep4"])
def test_plan_covers_every_row_once(lib, dtype, name, variant):
    """The planner's output tiles cover every segment row of every head and it
    writes one final state per view-head.  With three launches the state
    slots cover exactly the rows of views (and of long branches cut into
    pieces) and the scan runs once per view-head; the one-launch pass publishes
    only the pieces another CTA reads, and has no scan.  Counts are summed
    over heads."""
    from hybrid_linear_attention_packed_gb300 import workloads
    w = workloads.by_name(name)
    H = w.H
    spanla.set_pass_variant(variant)
    try:
        st = spanla.plan_stats(w.view_cu, w.branch_cu, w.branch_parent, H, dtype, num_sms=152)
    finally:
        spanla.set_pass_variant(spanla.PASS_ONE_LAUNCH)
    assert st["tile_rows"] == w.rows * H
    view_rows = int(w.view_lens.sum())
    long_rows = int(sum(L for L in w.branch_lens if L > 128))
    assert st["final_states"] == w.V * H
    if dtype == "f32":
        assert st["run_tiles"] == 1
        assert st["state_rows"] == (view_rows + long_rows) * H
        assert st["scan_segments"] == (w.V + sum(1 for L in w.branch_lens if L > 128)) * H
        assert st["state_slots"] == H * sum(-(-int(L) // 64) for L in list(w.view_lens)
                                            + [L for L in w.branch_lens if L > 128])
        return
    # runs of equal length over at least 85 % of the SMs
    assert st["run_tiles"] <= -(-st["tiles"] // int(0.85 * min(152, st["tiles"])))
    n_seg = w.V + sum(1 for L in w.branch_lens if L > 128)
    assert st["state_slots"] <= n_seg * H + 152
    if variant == spanla.PASS_THREE_LAUNCHES:
        assert view_rows * H <= st["state_rows"] <= (view_rows + long_rows) * H
        assert st["scan_segments"] >= w.V * H
    else:
        assert 0 <= st["state_rows"] <= (view_rows + long_rows) * H
        assert st["scan_segments"] == 0


@pytest.mark.parametrize("variant", [spanla.PASS_ONE_LAUNCH, spanla.PASS_THREE_LAUNCHES])
@pytest.mark.parametrize("H,sms", [(16, 152), (8, 152), (3, 152), (48, 152), (4, 20)])
def test_head_aligned_plan_is_heads_times_one_head(lib, variant, H, sms):
    """When the runs line up with the heads (R = SMs // H runs per head), the
    planner plans one head and copies it to the others; every count summed
    over heads must then be H times that of the one-head plan on R SMs,
    which the planner builds directly."""
    from hybrid_linear_attention_packed_gb300 import workloads
    R = sms // H
    assert R * H * 100 >= sms * 85   # the aligned case
    spanla.set_pass_variant(variant)
    try:
        for w in (workloads.single_request(0), workloads.packed_four(2)):
            many = spanla.plan_stats(w.view_cu, w.branch_cu, w.branch_parent, H, num_sms=sms)
            one = spanla.plan_stats(w.view_cu, w.branch_cu, w.branch_parent, 1, num_sms=R)
            for f in ("state_slots", "state_rows", "scan_segments", "final_states", "tiles",
                      "tile_rows", "start_state_reads", "out_items"):
                assert many[f] == H * one[f], (f, many[f], one[f])
            assert many["run_tiles"] == one["run_tiles"]
    finally:
        spanla.set_pass_variant(spanla.PASS_ONE_LAUNCH)


def test_one_launch_plan_of_a_pass_that_fits_one_run_per_request(lib):
    """Requests small next to a run: in the one-launch pass a view whose
    branches all lie in the run that holds its last tile publishes nothing
    (its CTA computes the final state and starts the branches from it), so
    passes of many small requests read K and V once."""
    from hybrid_linear_attention_packed_gb300 import workloads
    w = workloads.make_pass([130] * 40, [20] * 80, np.repeat(np.arange(40), 2), H=2, dtype="bf16", seed=1)
    st = spanla.plan_stats(w.view_cu, w.branch_cu, w.branch_parent, w.H, "bf16", num_sms=8)
    assert st["tile_rows"] == w.rows * w.H and st["final_states"] == w.V * w.H
    assert st["scan_segments"] == 0
    # at most the view-heads cut by a run boundary publish their pieces
    assert st["state_slots"] <= 2 * 8


@pytest.mark.parametrize("name", ["single", "packed4", "sweep4"])
def test_span_plan_runs_are_balanced(lib, name):
    """The bf16 planner cuts the output work into runs of equal length (+-1
    tile) over at least 85 % of the SMs, whatever the SM count; on the
    7,400-token pass with 16 heads and 148 or 152 SMs every run is 7 tiles."""
    from hybrid_linear_attention_packed_gb300 import workloads
    w = workloads.by_name(name)
    for nsm in (1, 7, 64, 148, 152, 1000):
        st = spanla.plan_stats(w.view_cu, w.branch_cu, w.branch_parent, w.H, "bf16", num_sms=nsm)
        assert st["run_tiles"] <= -(-st["tiles"] // max(1, int(0.85 * min(nsm, st["tiles"]))))
        assert st["tile_rows"] == w.rows * w.H
        if name == "single" and nsm in (148, 152):
            assert st["run_tiles"] == 7


def test_view_cache_validation_without_a_device(lib):
    """Argument checks of the view-state cache run before any CUDA call; with no
    device, create reports the CUDA error instead of returning a handle."""
    handle = ctypes.c_void_p(123)
    st = lib.span_la_cache_create(0, 4, ctypes.byref(handle))
    assert st == 1 and "num_heads" in lib.span_la_last_error_detail().decode()
    assert handle.value is None
    st = lib.span_la_cache_create(2, 0, ctypes.byref(handle))
    assert st == 1 and "capacity" in lib.span_la_last_error_detail().decode()
    st = lib.span_la_cache_create(2, 4, None)
    assert st == 1
    assert lib.span_la_cache_destroy(None) == 0
    st = lib.span_la_cache_put(None, None, 1, FAKE, None)
    assert st == 1 and "NULL" in lib.span_la_last_error_detail().decode()
    stats = (ctypes.c_int64 * 6)()
    assert lib.span_la_cache_stats(None, stats) == 1
    st = lib.span_la_cache_create(2, 4, ctypes.byref(handle))
    if st == 0:   # a device is visible after all: release it
        assert lib.span_la_cache_destroy(handle) == 0
    else:
        assert st == 3 and handle.value is None


def _softmax(lib, vcu, bcu, par, dims=None, scale=0.0, lse=None, q=FAKE):
    dims = dims or _dims()
    (va, vp), (ba, bp), (pa, pp) = _arr(vcu), _arr(bcu), _arr(par)
    V, B = max(len(va) - 1, 0), max(len(ba) - 1, 0)
    st = lib.span_la_softmax_pass(q, q, q, dims, vp if V else None, V, bp if B else None, B,
                                  pp if B else None, scale, q, lse, None)
    return st, lib.span_la_last_error_detail().decode()


def test_softmax_layer_validation(lib):
    """The softmax layer checks its arguments on the host before any CUDA call."""
    st, detail = _softmax(lib, [0, 10], [], [], dims=_dims(dtype=1))
    assert st == 2 and "bf16" in detail
    st, detail = _softmax(lib, [0, 10], [], [], scale=-0.5)
    assert st == 1 and "scale" in detail
    st, detail = _softmax(lib, [0, 10], [], [], scale=float("nan"))
    assert st == 1 and "scale" in detail
    st, detail = _softmax(lib, [0, 10], [], [], lse=FAKE + 2)
    assert st == 1 and "lse_out" in detail
    st, detail = _softmax(lib, [0, 50], [40, 60], [0])
    assert st == 1 and "overlap" in detail
    st, detail = _softmax(lib, [0, 50], [50, 60], [1])
    assert st == 1 and "branch_parent" in detail
    st, detail = _softmax(lib, [0, 10], [], [], q=FAKE + 8)
    assert st == 1 and "aligned" in detail
    st, detail = _softmax(lib, [0], [], [], q=0)
    assert st == 0     # nothing to do: no CUDA call


def test_softmax_branches_from_kv_validation(lib):
    (va, vp), (ba, bp), (pa, pp) = _arr([0, 30]), _arr([0, 10, 20]), _arr([0, 1])
    st = lib.span_la_softmax_branches_from_kv(FAKE, FAKE, 30, vp, 1, FAKE, FAKE, FAKE, _dims(), bp, 2,
                                              pp, 0.0, FAKE, None, None)
    assert st == 1 and "branch_parent" in lib.span_la_last_error_detail().decode()
    (va, vp) = _arr([0, 31])
    (pa, pp) = _arr([0, 0])
    st = lib.span_la_softmax_branches_from_kv(FAKE, FAKE, 30, vp, 1, FAKE, FAKE, FAKE, _dims(), bp, 2,
                                              pp, 0.0, FAKE, None, None)
    assert st == 1 and "view_cu_seqlens" in lib.span_la_last_error_detail().decode()
    (va, vp) = _arr([0, 30])
    st = lib.span_la_softmax_branches_from_kv(0, FAKE, 30, vp, 1, FAKE, FAKE, FAKE, _dims(), bp, 2,
                                              pp, 0.0, FAKE, None, None)
    assert st == 1 and "view_k" in lib.span_la_last_error_detail().decode()


def test_fault_injection_knob(lib):
    assert lib.span_la_fault_inject(7, 1) == 1
    assert lib.span_la_fault_inject(spanla.FAULT_ALLOC, -1) == 1
    assert lib.span_la_fault_inject(spanla.FAULT_ALLOC, 2) == 0
    assert lib.span_la_fault_inject(spanla.FAULT_ALLOC, 0) == 0


def test_c_client_builds_against_the_header(lib, tmp_path):
    """The plain C client compiles and links against include/spanla.h and
    libspanla.so (it runs in the GPU tests)."""
    import shutil
    import subprocess
    cuda = next((c for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda")
                 if c and os.path.exists(os.path.join(c, "include", "cuda_runtime_api.h"))), None)
    if cuda is None or shutil.which("gcc") is None:
        pytest.skip("no CUDA headers or gcc")
    lib_path = spanla_build.build()
    exe = str(tmp_path / "spanla_client")
    r = subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-Werror", "-o", exe,
                        os.path.join(ROOT, "tests", "c_client", "spanla_client.c"),
                        "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                        "-L", os.path.dirname(lib_path), "-lspanla", "-L", os.path.join(cuda, "lib64"),
                        "-lcudart"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_softmax_plan_covers_every_segment_row_once(lib):
    """Host-only plan of the softmax layer: the items cover every segment row of
    every head once; a view tile j of a view sees j + 1 key blocks, a branch
    tile its parent's blocks plus its own."""
    from hybrid_linear_attention_packed_gb300 import workloads
    w = workloads.make_pass([300, 129, 0], [40, 9, 130, 1], [0, 0, 1, 2], H=3, dtype="bf16", seed=1)
    st = spanla.softmax_plan_stats(w.view_cu, w.branch_cu, w.branch_parent, w.H, num_sms=152)
    assert st["rows"] == w.rows * w.H
    # views: 300 rows -> tiles with 1, 2, 3 blocks; 129 -> 1, 2.  Branches of view 0 (40 + 9 rows,
    # one packed tile): 3 prefix blocks + 1; branch 130 of view 1: two tiles, 2 prefix blocks + 1 or
    # 2 own; branch 1 of the empty view 2: 1 block.
    per_head = (1 + 2 + 3) + (1 + 2) + (3 + 1) + (2 + 1) + (2 + 2) + 1
    assert st["key_blocks"] == per_head * w.H
    assert st["items"] == (3 + 2 + 1 + 2 + 1) * w.H
    assert st["grid"] == min(152, st["items"])
    assert lib.span_la_softmax_plan_stats(None, 1, None, 0, None, 1, 152, None) == 1


@pytest.mark.parametrize("seed", range(6))
def test_random_metadata_plans_cover_every_row(lib, seed):
    """Random packed-pass metadata (host only): both planners cover every segment
    row of every head exactly once, the softmax plan needs at least one key
    block per query tile, and a branch naming a view that does not exist is
    rejected by both."""
    rng = np.random.default_rng([seed, 3])
    V = int(rng.integers(1, 8))
    vl = rng.integers(0, 3000, size=V)
    counts = rng.integers(0, 12, size=V)
    bl = rng.integers(0, 300, size=int(counts.sum()))
    par = np.repeat(np.arange(V), counts).astype(np.int32)
    vcu = np.concatenate([[0], np.cumsum(vl)]).astype(np.int32)
    bcu = (np.concatenate([[0], np.cumsum(bl)]) + vcu[-1]).astype(np.int32)
    H = int(rng.integers(1, 17))
    rows = int(vl.sum() + bl.sum())
    for dtype in ("bf16", "f32"):
        st = spanla.plan_stats(vcu, bcu, par, H, dtype, num_sms=152)
        assert st["tile_rows"] == rows * H
        assert st["final_states"] == V * H
    sa = spanla.softmax_plan_stats(vcu, bcu, par, H, num_sms=152)
    assert sa["rows"] == rows * H
    assert sa["key_blocks"] >= sa["items"]
    assert sa["grid"] == (min(152, sa["items"]) if sa["items"] else 0)
    if len(par):
        bad = par.copy()
        bad[-1] = V
        with pytest.raises(spanla.SpanLAError):
            spanla.plan_stats(vcu, bcu, bad, H)
        with pytest.raises(spanla.SpanLAError):
            spanla.softmax_plan_stats(vcu, bcu, bad, H)
