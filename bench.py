#!/usr/bin/env python
"""Benchmark of the packed linear-attention pass (one layer) on one GB300.

A step is one ``span_la_pass`` call over the whole pass (chunk state, segmented
scan, tile output with the branch fork) on inputs already resident in HBM.
The default workload is the single request of the pages' 7,400-token figure
("Serving 0.88M TPS from Two RTXs and Mac Minis", section "Kernels"): 16 heads,
d = 64, bf16 inputs with fp32 state, one 7,400-token view plus 8 branches of
U[32, 96] rows, synthetic and seeded.

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle on the host cores instead (the only other place this script runs it).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "packed-pass tokens/s per layer"
UNIT = "tokens/s"
STATE_BYTES = 64 * 64 * 4
# ms per layer the page reports for one scan per pass at 7,400 tokens (section
# "Kernels"), measured on an older RTX GPU: context for vs_baseline only.
PAGE_MS_PER_LAYER_7400 = 1.50
PAGE_TOKENS_7400 = 7400


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="single",
                    help="single | packed4 | cached_long | sweepN (N views) | tiny")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cache", action="store_true",
                    help="cached_long: run the shards through the view-state cache API "
                         "(span_la_cache_branches by key) instead of span_la_branches_from_state")
    ap.add_argument("--per-request", action="store_true",
                    help="run each request of the workload (a view and its branches) as its own "
                         "pass instead of one shared pass (the page's shared-branch-pass lever)")
    ap.add_argument("--pass-variant", choices=["one", "three"], default="one",
                    help="bf16 pass structure: one cooperative launch (default) or span state -> "
                         "scan -> output in three launches")
    ap.add_argument("--layer", choices=["linear", "softmax"], default="linear",
                    help="linear: the packed linear-attention pass (default); softmax: the "
                         "hybrid model's softmax-attention layer over the same packed rows")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while running (SM clock, throttle reasons)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "utilization.gpu")

    def __init__(self, gpu_id: str):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append(parts)
        return rows


def summarize_clocks(rows, t0: float, t1: float):
    """Median SM clock and the throttle reasons seen between wall times t0 and t1."""
    import datetime
    sel = []
    for r in rows:
        try:
            ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            ts = None
        if ts is None or (t0 - 0.25) <= ts <= (t1 + 0.25):
            sel.append(r)
    if not sel:
        sel = rows[-3:]
    if not sel:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                "samples": 0}
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = set()
    for r in sel:
        for n, val in zip(names, r[6:10]):
            if val.strip().lower() in ("active", "0x1", "1"):
                reasons.add(n)

    def num(x):
        try:
            return float(x)
        except ValueError:
            return None
    sm = [num(r[2]) for r in sel if num(r[2]) is not None]
    mx = [num(r[3]) for r in sel if num(r[3]) is not None]
    pw = [num(r[4]) for r in sel if num(r[4]) is not None]
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(mx) if mx else None,
            "power_w_max": max(pw) if pw else None,
            "reasons": sorted(reasons), "samples": len(sel)}


def summarize_busy_clocks(rows, min_util: float = 1.0):
    """Median SM clock and the throttle reasons over every sample of the run in
    which the GPU ran kernels (utilization >= min_util % over nvidia-smi's
    sample period): a longer record than the timed region alone, which lasts
    milliseconds."""
    busy = []
    for r in rows:
        try:
            if len(r) > 10 and float(r[10]) >= min_util:
                busy.append(r)
        except ValueError:
            pass
    if not busy:
        return {"sm_mhz": None, "samples": 0, "reasons": []}
    out = summarize_clocks(busy, -1e18, 1e18)
    out["min_utilization_pct"] = min_util
    return out


def gpu_id_for_smi(torch, dev_index: int) -> str:
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[dev_index]
    return str(dev_index)


# ---------------------------------------------------------------- algorithmic bytes
def algorithmic_bytes(plan: dict, H: int, esize: int, T: int) -> dict:
    """Bytes each kernel must move at least once per launch, from the library's
    own plan (counts summed over heads): operand rows read, states
    written/read, outputs written."""
    row = 64 * esize
    state_k = plan["state_rows"] * 2 * row + plan["state_slots"] * STATE_BYTES
    out_k = plan["tile_rows"] * 4 * row + plan["start_state_reads"] * STATE_BYTES
    return {
        "chunk_state": state_k, "span_state": state_k,
        "segmented_scan": (2 * plan["state_slots"] + plan["final_states"]) * STATE_BYTES,
        "tile_output": out_k, "span_output": out_k,
        "split_f32": T * H * 64 * (3 * 4 + 6 * 2),
    }


def io_bytes(w, esize: int) -> int:
    """Bytes of the call's inputs and outputs alone: q, k, v read and o written
    once per segment row, view states written once."""
    return w.rows * w.H * 64 * esize * 4 + w.V * w.H * STATE_BYTES


def chunked_method_bytes(w, esize: int) -> int:
    """Bytes of the chunked three-launch method as the pages lay it out, one
    fp32 64x64 state per 64-token chunk: q, k, v read and o written (4 rows),
    k and v read again by the state kernel (2 rows), and each chunk state
    written, read and written by the scan and read by the output kernel
    (4 x 16 KiB per 64 rows) -- per view token-head; branch rows count q, k,
    v, o only."""
    row = 64 * esize
    view_rows = int(w.view_lens.sum())
    per_view_row = 6 * row + 4 * STATE_BYTES // 64
    return (view_rows * per_view_row + (w.rows - view_rows) * 4 * row) * w.H


def kernel_sha(name: str) -> str:
    files = {"tile_output": "k_tile_output.cu", "chunk_state": "k_chunk_state.cu",
             "segmented_scan": "k_scan.cu", "split_f32": "k_misc.cu",
             "span_state": "k_span_state.cu", "span_output": "k_span_output.cu",
             "softmax_attn": "k_softmax_attn.cu"}
    p = os.path.join(ROOT, "hybrid_linear_attention_packed_gb300", "csrc", files[name])
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    when there is none or the kernel source changed since it was captured."""
    p = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(p):
        return None
    pat = re.compile(r"^\|\s*%s\s*\|\s*%s\s*\|\s*([0-9a-f]+)\s*\|\s*([0-9.eE+]+)\s*\|"
                     % (re.escape(kernel), re.escape(workload)))
    with open(p) as f:
        for line in f:
            m = pat.match(line.strip())
            if m and m.group(1) == kernel_sha(kernel):
                return float(m.group(2))
    return None


def event_floor_us(torch, stream, flush, reps: int = 60) -> float:
    """Median elapsed time of an empty CUDA-event pair on `stream` right after an
    L2 flush: the floor every event-timed kernel duration includes."""
    ts = []
    for _ in range(reps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    return statistics.median(ts[5:])


def branch_variants(w, n: int, seed: int = 12345):
    """n variants of a workload's branch metadata over the same rows: within each
    parent's run of branches the lengths are permuted, so every variant packs
    the same rows and views but cuts its branches differently (a fresh plan for
    the library's plan cache).  Returns (branch_cu, branch_parent) pairs."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(w.branch_lens, dtype=np.int64)
    par = np.asarray(w.branch_parent, dtype=np.int32)
    out = []
    for _ in range(n):
        perm = np.arange(len(lens))
        b = 0
        while b < len(lens):
            e = b
            while e < len(lens) and par[e] == par[b]:
                e += 1
            perm[b:e] = b + rng.permutation(e - b)
            b = e
        cu = np.concatenate([[int(w.branch_cu[0])], int(w.branch_cu[0]) + np.cumsum(lens[perm])])
        out.append((np.ascontiguousarray(cu, dtype=np.int32), par.copy()))
    return out


# ---------------------------------------------------------------- CPU oracle
def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return "unknown"

def oracle_time(w, budget_s: float = 8.0, max_reps: int = 50, nthreads: int = 0):
    """Time the float64 oracle on the whole workload, repeated within ~budget_s
    (nthreads = 0: every host core); also returns its last result."""
    from oracle import oracle_max_threads, oracle_pass
    q, k, v = (t.double().numpy() for t in (w.q, w.k, w.v))
    times = []
    result = None
    t_all = time.perf_counter()
    while len(times) < max_reps and (time.perf_counter() - t_all) < budget_s:
        t0 = time.perf_counter()
        result = oracle_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent, nthreads=nthreads)
        times.append(time.perf_counter() - t0)
    return statistics.median(times), len(times), (nthreads or oracle_max_threads()), result


def segment_mask(w):
    m = np.zeros(w.T, dtype=bool)
    for cu in (w.view_cu, w.branch_cu):
        for s_ in range(len(cu) - 1):
            m[int(cu[s_]):int(cu[s_ + 1])] = True
    return m


def max_rel_err(got, ref):
    """max |got - ref| / max |ref| (the parity tests' measure)."""
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    diff = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    return diff / den if den > 0 else diff


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from hybrid_linear_attention_packed_gb300 import workloads
    from oracle import oracle_max_threads, oracle_pass
    w = workloads.by_name(args.workload, args.seed)
    q, k, v = (t.double().numpy() for t in (w.q, w.k, w.v))
    for _ in range(max(0, min(args.warmup, 3))):
        oracle_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent)
    # bounded: at most ~60 s of timed oracle work whatever --steps asks for
    times = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all > 60.0:
            break
    ms = statistics.mean(times) * 1e3
    value = w.rows / (ms / 1e3)
    cores = oracle_max_threads()
    sample = ("the whole workload (%d rows x %d heads) per step, %d timed steps"
              % (w.rows, w.H, len(times)))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": len(times), "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_config(w, args.workload), parallelism="dp1"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def workload_config(w, name: str) -> dict:
    cfg = {"workload": w.name, "key": name, "heads": w.H, "head_dim": w.D, "views": w.V,
           "branches": w.B, "rows": w.rows, "view_rows": int(w.view_lens.sum()),
           "branch_rows": int(w.branch_lens.sum()),
           "l2": "flushed before every timed step (512 MiB write)"}
    if name == "cached_long":
        cfg["step"] = ("span_la_branches_from_state over the view's cached final state, 4 shards "
                       "of 64 branches; tokens/s counts branch rows")
    return cfg


def pass_structure(args) -> str:
    """The bf16 pass structure this run used (a top-level key of the line, not
    part of `config`: the workload is the same whichever structure runs it)."""
    return "three launches" if getattr(args, "pass_variant", "one") == "three" else "one launch"


def add_mode(cfg: dict, args) -> dict:
    if getattr(args, "cache", False) and args.workload == "cached_long":
        cfg = dict(cfg, step="span_la_cache_branches by key over the view-state cache, 4 shards of "
                             "64 branches; tokens/s counts branch rows")
    if getattr(args, "per_request", False):
        cfg = dict(cfg, step="one span_la_pass per request (view + its branches) over the same "
                             "buffers, instead of one shared pass")
    return cfg


# ---------------------------------------------------------------- softmax layer
SOFTMAX_METRIC = "packed softmax-layer tokens/s"


def visible_pairs(w) -> int:
    """(query, key) pairs the softmax layer scores, per head: a view row sees its
    view up to itself, a branch row its parent view and its branch up to itself."""
    vl = w.view_lens.astype(np.int64) if hasattr(w.view_lens, "astype") else w.view_lens
    n = int(sum(int(L) * (int(L) + 1) // 2 for L in vl))
    for b in range(w.B):
        nb = int(w.branch_lens[b])
        n += nb * int(w.view_lens[int(w.branch_parent[b])]) + nb * (nb + 1) // 2
    return n


def softmax_oracle_time(w, budget_s: float = 20.0, max_reps: int = 3):
    from oracle import oracle_softmax_pass
    q, k, v = (t.double().numpy() for t in (w.q, w.k, w.v))
    times = []
    result = None
    t_all = time.perf_counter()
    while len(times) < max_reps and (time.perf_counter() - t_all) < budget_s:
        t0 = time.perf_counter()
        result = oracle_softmax_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent)
        times.append(time.perf_counter() - t0)
    return statistics.median(times), len(times), result


def softmax_cpu_line(w, value, reps, args):
    cores = os.cpu_count() or 1
    return {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "the whole workload (%d rows x %d heads), median of %d passes; numpy "
                      "float64 (matmuls on the BLAS threads, the rest on one thread)"
                      % (w.rows, w.H, reps),
            "cpu_model": cpu_model()}


def run_softmax_reference(args):
    rank, _, _ = dist_env()
    if rank != 0:
        return 0
    from hybrid_linear_attention_packed_gb300 import workloads
    w = workloads.by_name(args.workload, args.seed)
    med, reps, _ = softmax_oracle_time(w, budget_s=60.0, max_reps=max(1, min(args.steps, 10)))
    value = w.rows / med
    cpu = softmax_cpu_line(w, value, reps, args)
    line = {"impl": "reference", "metric": SOFTMAX_METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": reps, "warmup": 0, "ms_per_step": med * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": dict(workload_config(w, args.workload), layer="softmax",
                                                parallelism="dp1"),
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main_softmax(args):
    """The softmax-attention layer over a packed pass: one span_la_softmax_pass
    call per step on resident inputs, L2 flushed before every step."""
    rank, world, local = dist_env()
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    from hybrid_linear_attention_packed_gb300 import build as libbuild
    if rank == 0:
        libbuild.build()
    if pg:
        pg.barrier()
    from hybrid_linear_attention_packed_gb300 import sharding, spanla, workloads
    w = workloads.by_name(args.workload, args.seed + rank)
    if w.dtype != "bf16":
        raise SystemExit("the softmax layer takes bf16 inputs; workload %s is %s" % (args.workload, w.dtype))
    q, k, v = (t.to(dev).contiguous() for t in (w.q, w.k, w.v))
    out = torch.zeros_like(q)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def run_on(qq, kk, vv, oo, strm=None):
        spanla.span_la_softmax_pass(qq, kk, vv, w.view_cu, w.branch_cu, w.branch_parent, out=oo,
                                    stream=strm)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        run_on(q, k, v, out)
    spanla.span_la_check()
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(gpu_id_for_smi(torch, local))
    time.sleep(0.5)
    spanla.profile_reset()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(K):
        flush.zero_()
        starts[i].record(stream)
        run_on(q, k, v, out)
        ends[i].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if pg:
        pg.barrier()
    launches = spanla.profile_read()
    spanla.span_la_check()
    clock_rows = sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms = sharding.max_over_ranks(statistics.mean(step_ms), pg, dev)
    value = w.rows * world / (ms / 1e3)

    # Kernel time from events around each launch, on the call's stream.
    spanla.profile_reset()
    spanla.profile_enable(True)
    for _ in range(min(K, 300)):
        flush.zero_()
        run_on(q, k, v, out)
    torch.cuda.synchronize()
    spanla.profile_enable(False)
    prof = spanla.profile_read()["softmax_attn"]
    kern_us = prof["ms"] / max(prof["timed"], 1) * 1e3
    pairs = visible_pairs(w)
    flops = 4 * 64 * pairs * w.H
    peaks = {}
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        with open(pk) as f:
            peaks = json.load(f)
    peak = peaks.get("bf16_tflops")
    peak_src = "measured (burst)" if peak else "fallback"
    peak = peak or 1900.0
    achieved = flops / (kern_us / 1e6) / 1e12
    # The tensor work the kernel issues: one 128x128x64 Q K^T and one 128x64x128
    # P V per (query tile, key block), masked or not.
    sa_plan = spanla.softmax_plan_stats(w.view_cu, w.branch_cu, w.branch_parent, w.H,
                                        torch.cuda.get_device_properties(dev).multi_processor_count)
    mma_flops = sa_plan["key_blocks"] * 2 * (2 * 128 * 128 * 64)
    roofline_mma = {"issued_flops_per_launch": mma_flops,
                    "issued_tflops": mma_flops / (kern_us / 1e6) / 1e12,
                    "issued_frac": mma_flops / (kern_us / 1e6) / 1e12 / peak,
                    "plan": sa_plan}
    roofline = {"bound": "tensor", "kernel": "softmax_attn", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": recorded_traffic("softmax_attn", args.workload),
                "peak_source": peak_src, "alg_flops_per_launch": flops,
                "visible_pairs_per_head": pairs,
                "exp_per_s": pairs * w.H / (kern_us / 1e6),
                "tensor_issued": roofline_mma}

    # End to end with host buffers: every step copies its q, k, v in from
    # pinned memory, runs the call and reads out back, pipelined over two
    # device buffer sets and three streams (copies in, the call, copies out)
    # as for the linear pass; the value is the steps' rows over the time from
    # the first copy-in to the last read-back.
    hq, hk, hv = (t.pin_memory() for t in (w.q, w.k, w.v))
    hout = torch.empty_like(hq).pin_memory()
    sets = [(q, k, v, out), (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                             torch.empty_like(out))]
    s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))

    def e2e_run(n_steps):
        ready, ran, read = [None, None], [None, None], [None, None]
        for i in range(n_steps):
            b = i & 1
            dq, dk, dv, dout = sets[b]
            with torch.cuda.stream(s_in):
                if ran[b] is not None:
                    s_in.wait_event(ran[b])
                dq.copy_(hq, non_blocking=True)
                dk.copy_(hk, non_blocking=True)
                dv.copy_(hv, non_blocking=True)
                ready[b] = torch.cuda.Event()
                ready[b].record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(ready[b])
                if read[b] is not None:
                    s_run.wait_event(read[b])
                run_on(dq, dk, dv, dout, s_run)
                ran[b] = torch.cuda.Event()
                ran[b].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ran[b])
                hout.copy_(dout, non_blocking=True)
                read[b] = torch.cuda.Event()
                read[b].record(s_out)

    e2e_run(4)
    torch.cuda.synchronize()
    KE = max(2, args.e2e_steps)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    e2e_run(KE)
    s_in.wait_stream(s_out)
    e1.record(s_in)
    torch.cuda.synchronize()
    spanla.span_la_check()
    e2e_ms = sharding.max_over_ranks(e0.elapsed_time(e1) / KE, pg, dev)
    esize = 2
    h2d = 3 * w.T * w.H * 64 * esize
    d2h = w.T * w.H * 64 * esize

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        med, reps, (ref, _) = softmax_oracle_time(w)
        cpu = softmax_cpu_line(w, w.rows / med, reps, args)
        # The benchmarked output against the oracle's (the parity tests' measure).
        seg = segment_mask(w)
        got = out.detach().double().cpu().numpy()
        cpu["max_rel_err_vs_gpu"] = max_rel_err(got[seg], ref[seg])
    if rank == 0:
        line = {"metric": SOFTMAX_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": dict(workload_config(w, args.workload), layer="softmax",
                               parallelism="dp%d" % world),
                "roofline": roofline,
                "kernels": {"softmax_attn": {"avg_us": kern_us, "launches": prof["launches"]}},
                "cpu_baseline": cpu,
                "e2e": {"value": w.rows * world / (e2e_ms / 1e3), "unit": UNIT, "ms_per_step": e2e_ms,
                        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": KE,
                        "mode": "pinned host buffers; copies of step i+1 overlap the call and "
                                "read-back of step i (two device buffer sets, three streams)"},
                "gpu_launches": int(sum(p["launches"] for p in launches.values())),
                "clocks": summarize_clocks(clock_rows, t0, t1),
                "step_ms_p50": statistics.median(step_ms), "step_ms_min": min(step_ms)}
        print(json.dumps(line))
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    return 0


# ---------------------------------------------------------------- GPU arm
def main():
    args = parse_args()
    if args.layer == "softmax":
        return run_softmax_reference(args) if args.impl == "reference" else main_softmax(args)
    if args.impl == "reference":
        return run_reference(args)

    rank, world, local = dist_env()
    import numpy as np
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    from hybrid_linear_attention_packed_gb300 import build as libbuild
    if rank == 0:
        libbuild.build()
    if pg:
        pg.barrier()
    from hybrid_linear_attention_packed_gb300 import sharding, spanla, workloads
    spanla.set_pass_variant(spanla.PASS_THREE_LAUNCHES if args.pass_variant == "three"
                            else spanla.PASS_ONE_LAUNCH)

    # Weak scaling: every rank runs its own pass (independent requests).
    w = workloads.by_name(args.workload, args.seed + rank)
    esize = 2 if w.dtype == "bf16" else 4
    q, k, v = (t.to(dev).contiguous() for t in (w.q, w.k, w.v))
    out = torch.zeros_like(q)
    state = torch.zeros((w.V, w.H, 64, 64), dtype=torch.float32, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # The call a step makes.  cached_long follows its configuration: the
    # view's final state is computed once (untimed) and cached, and every step
    # runs the 256 branches from it in 4 shards of 64 branches.
    shards_mode = args.workload == "cached_long"
    if shards_mode:
        _, cached = spanla.span_la_pass(q, k, v, w.view_cu, [], [])
        cached = cached.clone()
        shard_cu = workloads.shards(w, 4)
        shard_par = [np.zeros(len(c) - 1, dtype=np.int32) for c in shard_cu]
        rows_per_step = int(w.branch_lens.sum())
        row_lo = int(w.branch_cu[0])     # rows a step reads and writes: [row_lo, T)

        if args.cache:
            view_cache = spanla.ViewStateCache(w.H, capacity=4)
            view_cache.put([0x5EED], cached)
            shard_keys = [np.full(len(c) - 1, 0x5EED, dtype=np.uint64) for c in shard_cu]

            def run_on(qq, kk, vv, oo, ss, strm=None):
                for cu, keys in zip(shard_cu, shard_keys):
                    view_cache.branches(keys, qq, kk, vv, cu, out=oo, stream=strm)
        else:
            def run_on(qq, kk, vv, oo, ss, strm=None):
                for cu, par in zip(shard_cu, shard_par):
                    spanla.span_la_branches_from_state(cached, qq, kk, vv, cu, par, out=oo, stream=strm)
    elif args.per_request:
        # One pass per request over the same buffers: view v and its branches
        # (contiguous in the branch list, grouped by parent).
        rows_per_step = w.rows
        row_lo = 0
        req_calls = []
        for vi in range(w.V):
            bsel = np.flatnonzero(w.branch_parent == vi)
            if bsel.size and bsel[-1] - bsel[0] + 1 != bsel.size:
                raise SystemExit("--per-request needs each view's branches listed together")
            bcu_r = (np.ascontiguousarray(w.branch_cu[bsel[0]:bsel[-1] + 2], dtype=np.int32)
                     if bsel.size else np.zeros(0, np.int32))
            req_calls.append((np.ascontiguousarray(w.view_cu[vi:vi + 2], dtype=np.int32), bcu_r,
                              np.zeros(bsel.size, np.int32), vi))

        def run_on(qq, kk, vv, oo, ss, strm=None):
            for vcu_r, bcu_r, par_r, vi in req_calls:
                spanla.span_la_pass(qq, kk, vv, vcu_r, bcu_r, par_r, out=oo,
                                    view_state_out=ss[vi:vi + 1], stream=strm)
    else:
        rows_per_step = w.rows
        row_lo = 0

        def run_on(qq, kk, vv, oo, ss, strm=None):
            spanla.span_la_pass(qq, kk, vv, w.view_cu, w.branch_cu, w.branch_parent, out=oo,
                                view_state_out=ss, stream=strm)

    def step():
        run_on(q, k, v, out, state)

    run_sampler = ClockSampler(gpu_id_for_smi(torch, local))   # the whole GPU part of the run
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    spanla.span_la_check()

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(gpu_id_for_smi(torch, local))
    time.sleep(0.5)
    spanla.profile_reset()        # launch counters only; no per-kernel events here
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(K):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if pg:
        pg.barrier()
    launches = spanla.profile_read()
    spanla.span_la_check()
    clock_rows = sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = statistics.mean(step_ms)
    ms_max = sharding.max_over_ranks(ms, pg, dev)
    rows_total = rows_per_step * world
    value = rows_total / (ms_max / 1e3)

    # Per-kernel durations: the same steps again with CUDA events recorded
    # around every launch on the call's stream (the events keep consecutive
    # kernels from overlapping, so these add up to more than a step).
    KP = min(K, 500)
    spanla.profile_reset()
    spanla.profile_enable(True)
    for i in range(KP):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    spanla.profile_enable(False)
    prof = spanla.profile_read()
    spanla.span_la_check()

    # Roofline of the dominant kernel, from live event timings.
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    if shards_mode:
        plan = None
        for cu, par in zip(shard_cu, shard_par):
            st_ = spanla.plan_stats([], cu, par, w.H, w.dtype, num_parents=1, from_state=True,
                                    num_sms=nsm)
            plan = st_ if plan is None else {key: plan[key] + st_[key] for key in plan}
    elif args.per_request:
        plan = None
        for vcu_r, bcu_r, par_r, _ in req_calls:
            st_ = spanla.plan_stats(vcu_r, bcu_r, par_r, w.H, w.dtype, num_sms=nsm)
            plan = st_ if plan is None else {key: plan[key] + st_[key] for key in plan}
    else:
        plan = spanla.plan_stats(w.view_cu, w.branch_cu, w.branch_parent, w.H, w.dtype, num_sms=nsm)
    # the plan above covers every call of a step; bytes per launch divide it by
    # the calls a step makes (each call launches each kernel once)
    calls_per_step = len(shard_cu) if shards_mode else (len(req_calls) if args.per_request else 1)
    alg = {name: b / calls_per_step for name, b in algorithmic_bytes(plan, w.H, esize, w.T).items()}
    peaks = {}
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        with open(pk) as f:
            peaks = json.load(f)
    hbm_peak = peaks.get("hbm_gbs")
    peak_src = "measured" if hbm_peak else "fallback"
    hbm_peak = hbm_peak or 6800.0
    kernels = {}
    for name, p in prof.items():
        if p["timed"]:
            avg_ms = p["ms"] / p["timed"]
            kernels[name] = {"avg_us": avg_ms * 1e3, "launches": p["launches"],
                             "share": None, "alg_bytes": alg.get(name, 0),
                             "gbs": alg.get(name, 0) / (avg_ms / 1e3) / 1e9 if avg_ms > 0 else None}
    tot = sum(kk["avg_us"] for kk in kernels.values()) or 1.0
    profiled_step_us = tot
    for kk in kernels.values():
        kk["share"] = kk["avg_us"] / tot
    dom = max(kernels, key=lambda n: kernels[n]["avg_us"])
    dk = kernels[dom]
    traffic = recorded_traffic(dom, args.workload + ("/three" if args.pass_variant == "three" else ""))
    roofline = {"bound": "hbm", "kernel": dom, "achieved": dk["gbs"], "peak": hbm_peak,
                "unit": "GB/s", "frac": dk["gbs"] / hbm_peak, "traffic": traffic,
                "peak_source": peak_src,
                "alg_bytes_per_launch": dk["alg_bytes"]}
    step_bytes = sum(alg[n] for n in kernels) * calls_per_step
    chunked = chunked_method_bytes(w, esize) if not shards_mode else rows_per_step * w.H * 4 * 64 * esize
    iob = io_bytes(w, esize) if not shards_mode else rows_per_step * w.H * 4 * 64 * esize
    pass_roofline = {"method_bytes": step_bytes,
                     "method_frac": step_bytes / (ms / 1e3) / 1e9 / hbm_peak,
                     "io_bytes": iob,
                     "io_frac": iob / (ms / 1e3) / 1e9 / hbm_peak,
                     "chunked_method_bytes": chunked,
                     "chunked_method_frac": chunked / (ms / 1e3) / 1e9 / hbm_peak,
                     "chunked_method_note": "bytes of the pages' layout (one fp32 state per 64-token "
                                            "chunk through the scan), which this design does not move: "
                                            "context only; method_frac and io_frac are this design's"}

    # The floor of an event-timed duration on this stream (an empty event pair
    # after an L2 flush): reported beside the roofline, whose kernel time
    # includes it.
    floor_us = event_floor_us(torch, stream, flush)
    roofline["event_floor_us"] = floor_us
    if dk["avg_us"] > floor_us:
        roofline["frac_above_event_floor"] = dk["alg_bytes"] / ((dk["avg_us"] - floor_us) / 1e6) / 1e9 / hbm_peak

    # Fresh metadata every step: 24 variants of the branch layout over the same
    # rows, cycled, so that every call misses the library's 16-entry plan cache
    # and builds, uploads and launches a new plan (the host plan build and the
    # descriptor upload fall inside each step).
    cold = None
    if w.B > 1 and not args.per_request:
        NV = 24
        variants = branch_variants(w, NV)
        if shards_mode:
            def cold_call(j):
                bcu_j, par_j = variants[j]
                per = (w.B + 3) // 4
                for s_ in range(4):
                    b0, b1 = s_ * per, min(w.B, (s_ + 1) * per)
                    spanla.span_la_branches_from_state(cached, q, k, v, bcu_j[b0:b1 + 1],
                                                       np.zeros(b1 - b0, np.int32), out=out)
        else:
            def cold_call(j):
                bcu_j, par_j = variants[j]
                spanla.span_la_pass(q, k, v, w.view_cu, bcu_j, par_j, out=out, view_state_out=state)
        for j in range(NV):
            cold_call(j)
        torch.cuda.synchronize()
        KC = min(K, 240)
        cs = [torch.cuda.Event(enable_timing=True) for _ in range(KC)]
        ce = [torch.cuda.Event(enable_timing=True) for _ in range(KC)]
        for i in range(KC):
            flush.zero_()
            cs[i].record(stream)
            cold_call(i % NV)
            ce[i].record(stream)
        torch.cuda.synchronize()
        spanla.span_la_check()
        cms = statistics.mean(a.elapsed_time(b) for a, b in zip(cs, ce))
        # The same fresh plans, each prepared on a side stream while the L2
        # flush before its step runs (a server preparing the next pass while
        # the device is busy): the pass waits for the upload through an event.
        cms_p = None
        if not shards_mode:
            side = torch.cuda.Stream(device=dev)
            dt_p = torch.bfloat16 if w.dtype == "bf16" else torch.float32
            for i in range(KC):
                bcu_j, par_j = variants[i % NV]
                spanla.span_la_plan_prepare(w.view_cu, bcu_j, par_j, q.shape[0], q.shape[1], dtype=dt_p,
                                            stream=side)
                flush.zero_()
                cs[i].record(stream)
                cold_call(i % NV)
                ce[i].record(stream)
            torch.cuda.synchronize()
            spanla.span_la_check()
            cms_p = statistics.mean(a.elapsed_time(b) for a, b in zip(cs, ce))
        # Host time of one call that builds a new plan, with the device busy
        # on earlier work (as in a serving loop) but no backlog of calls
        # ahead of it: the loop above runs ahead of the device, so its host
        # times would measure the device's pace, not the host's cost.
        cbusy = torch.empty(256 << 20, dtype=torch.float32, device=dev)
        chost = []
        for i in range(2 * NV):
            torch.cuda.synchronize()
            cbusy.zero_()
            t_h = time.perf_counter()
            cold_call((i + 1) % NV)
            chost.append((time.perf_counter() - t_h) * 1e6)
        torch.cuda.synchronize()
        spanla.span_la_check()
        # The same through the C entry point with prepared arguments (the
        # library's own cost of a new plan, without the Python binding).
        chost_c = None
        if not shards_mode:
            lib_c = spanla.load_library()
            dims_c = spanla.Dims(q.shape[0], q.shape[1], 64,
                                 spanla.SPAN_LA_BF16 if w.dtype == "bf16" else spanla.SPAN_LA_F32)
            vcu_c = np.ascontiguousarray(w.view_cu, dtype=np.int32)
            prep = [(np.ascontiguousarray(b_, dtype=np.int32), np.ascontiguousarray(p_, dtype=np.int32))
                    for b_, p_ in variants]
            raw_c = [(q.data_ptr(), k.data_ptr(), v.data_ptr(), dims_c, vcu_c.ctypes.data, len(vcu_c) - 1,
                      b_.ctypes.data, len(b_) - 1, p_.ctypes.data, out.data_ptr(), state.data_ptr(),
                      stream.cuda_stream) for b_, p_ in prep]
            chost_c = []
            for i in range(2 * NV):
                torch.cuda.synchronize()
                cbusy.zero_()
                t_h = time.perf_counter()
                st_c = lib_c.span_la_pass(*raw_c[(i + 1) % NV])
                chost_c.append((time.perf_counter() - t_h) * 1e6)
                assert st_c == 0
            torch.cuda.synchronize()
            spanla.span_la_check()
        # The same new plans built ahead by span_la_plan_prepare (as a server
        # would while the pass's inputs are copied in): the host time of the
        # prepare call, and of the pass that then finds its plan cached.
        prep_host, chost_p = None, None
        if not shards_mode:
            prep_host, chost_p = [], []
            dt_c = torch.bfloat16 if w.dtype == "bf16" else torch.float32
            for i in range(2 * NV):
                bcu_j, par_j = variants[(i + 1) % NV]
                torch.cuda.synchronize()
                cbusy.zero_()
                t_h = time.perf_counter()
                spanla.span_la_plan_prepare(w.view_cu, bcu_j, par_j, q.shape[0], q.shape[1], dtype=dt_c)
                prep_host.append((time.perf_counter() - t_h) * 1e6)
                t_h = time.perf_counter()
                st_c = lib_c.span_la_pass(*raw_c[(i + 1) % NV])
                chost_p.append((time.perf_counter() - t_h) * 1e6)
                assert st_c == 0
            torch.cuda.synchronize()
            spanla.span_la_check()
        del cbusy
        cold = {"cold_plan_ms_per_step": cms, "cold_plan_host_us": statistics.median(chost),
                "cold_plan_host_us_c_abi": statistics.median(chost_c) if chost_c else None,
                "prepared_ms_per_step": cms_p,
                "prepare_host_us": statistics.median(prep_host) if prep_host else None,
                "prepared_pass_host_us_c_abi": statistics.median(chost_p) if chost_p else None,
                "cold_plan_value": rows_per_step / (cms / 1e3), "variants": NV, "steps": KC,
                "mode": "branch lengths permuted within each parent's run of branches: a new "
                        "plan (host build + descriptor upload) in every step"}

    # Long request: the view pass alone, and the 4 shards run concurrently on
    # 4 streams, or as one call over all branches, beside the serial shards.
    long_req = None
    if shards_mode:
        def timed(fn, reps):
            a_ = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
            b_ = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
            for i in range(reps):
                flush.zero_()
                a_[i].record(stream)
                fn()
                b_[i].record(stream)
            torch.cuda.synchronize()
            spanla.span_la_check()
            return statistics.mean(x.elapsed_time(y) for x, y in zip(a_, b_)) * 1e3
        vstate = torch.empty((1, w.H, 64, 64), dtype=torch.float32, device=dev)
        side = [torch.cuda.Stream(device=dev) for _ in range(4)]

        def shards_4_streams():
            go = torch.cuda.Event()
            go.record(stream)
            done = []
            for strm, cu, par in zip(side, shard_cu, shard_par):
                strm.wait_event(go)
                spanla.span_la_branches_from_state(cached, q, k, v, cu, par, out=out, stream=strm)
                ev = torch.cuda.Event()
                ev.record(strm)
                done.append(ev)
            for ev in done:
                stream.wait_event(ev)

        all_par = np.zeros(w.B, np.int32)
        reps = min(K, 200)
        for fn in (shards_4_streams,):
            fn()
        long_req = {
            "view_pass_us": timed(lambda: spanla.span_la_pass(q, k, v, w.view_cu, [], [], out=out,
                                                              view_state_out=vstate), reps),
            "shards_serial_us": ms * 1e3,
            "shards_4_streams_us": timed(shards_4_streams, reps),
            "one_call_256_branches_us": timed(lambda: spanla.span_la_branches_from_state(
                cached, q, k, v, w.branch_cu, all_par, out=out), reps),
            "view_rows": int(w.view_lens.sum()), "branch_rows": rows_per_step}

    # End to end through the public API with host buffers: every step copies
    # its q, k, v from pinned host memory, runs the call and reads out and the
    # view states back to pinned host memory.  Steps are pipelined over two
    # device buffer sets and three streams (host-to-device copies, the call,
    # device-to-host copies), so that the copies of step i+1 overlap the call
    # and the read-back of step i; the value is the steps' rows over the time
    # from the first copy-in to the last read-back.
    hq, hk, hv = (t[row_lo:].pin_memory() for t in (w.q, w.k, w.v))
    hout = torch.empty_like(hq).pin_memory()
    hstate = torch.empty((w.V, w.H, 64, 64), dtype=torch.float32).pin_memory()
    sets = [(q, k, v, out, state)] + [
        (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(out),
         torch.empty_like(state))]
    s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))

    def e2e_run(n):
        ev = lambda: torch.cuda.Event()   # noqa: E731
        ready = [None, None]      # inputs of a set copied in
        ran = [None, None]        # call on a set done
        read = [None, None]       # outputs of a set read back
        for i in range(n):
            b = i & 1
            dq, dk, dv, dout, dstate = sets[b]
            with torch.cuda.stream(s_in):
                if ran[b] is not None:
                    s_in.wait_event(ran[b])       # the set's inputs are no longer read
                dq[row_lo:].copy_(hq, non_blocking=True)
                dk[row_lo:].copy_(hk, non_blocking=True)
                dv[row_lo:].copy_(hv, non_blocking=True)
                ready[b] = ev()
                ready[b].record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(ready[b])
                if read[b] is not None:
                    s_run.wait_event(read[b])     # the set's outputs were read back
                run_on(dq, dk, dv, dout, dstate, s_run)
                ran[b] = ev()
                ran[b].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ran[b])
                hout.copy_(dout[row_lo:], non_blocking=True)
                if not shards_mode:
                    hstate.copy_(dstate, non_blocking=True)
                read[b] = ev()
                read[b].record(s_out)

    e2e_run(4)
    torch.cuda.synchronize()
    KE = max(2, args.e2e_steps)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(s_in)
    e2e_run(KE)
    s_in.wait_stream(s_out)
    e_end.record(s_in)
    torch.cuda.synchronize()
    spanla.span_la_check()
    e2e_ms = sharding.max_over_ranks(e_start.elapsed_time(e_end) / KE, pg, dev)
    # Host time to enqueue one call (the device kept busy so that no launch
    # waits on it), and the device time per call with the L2 warm: calls
    # enqueued back to back with no flush between them.
    busy = torch.empty(256 << 20, dtype=torch.float32, device=dev)
    host_us = []
    for _ in range(50):
        busy.zero_()
        t_h = time.perf_counter()
        step()
        host_us.append((time.perf_counter() - t_h) * 1e6)
    torch.cuda.synchronize()
    del busy
    # Back to back through the C entry points with prepared arguments, so that
    # the host (about 14 us per call) stays ahead of the device.
    lib = spanla.load_library()
    dims = spanla.Dims(q.shape[0], q.shape[1], 64, spanla.SPAN_LA_BF16 if w.dtype == "bf16" else spanla.SPAN_LA_F32)
    sh = stream.cuda_stream
    if shards_mode and args.cache:
        raw = [(view_cache._handle, keys.ctypes.data, q.data_ptr(), k.data_ptr(), v.data_ptr(), dims,
                cu.ctypes.data, len(cu) - 1, out.data_ptr(), sh) for cu, keys in zip(shard_cu, shard_keys)]
        fn = lib.span_la_cache_branches
    elif shards_mode:
        raw = [(cached.data_ptr(), 1, q.data_ptr(), k.data_ptr(), v.data_ptr(), dims, cu.ctypes.data,
                len(cu) - 1, par.ctypes.data, out.data_ptr(), sh) for cu, par in zip(shard_cu, shard_par)]
        fn = lib.span_la_branches_from_state
    elif args.per_request:
        raw = [(q.data_ptr(), k.data_ptr(), v.data_ptr(), dims, vcu_r.ctypes.data, 1,
                bcu_r.ctypes.data if len(bcu_r) else None, max(len(bcu_r) - 1, 0),
                par_r.ctypes.data if len(par_r) else None, out.data_ptr(),
                state[vi:vi + 1].data_ptr(), sh) for vcu_r, bcu_r, par_r, vi in req_calls]
        fn = lib.span_la_pass
    else:
        vcu, bcu, par = (np.ascontiguousarray(a, dtype=np.int32) for a in (w.view_cu, w.branch_cu, w.branch_parent))
        raw = [(q.data_ptr(), k.data_ptr(), v.data_ptr(), dims, vcu.ctypes.data, len(vcu) - 1,
                bcu.ctypes.data if len(bcu) else None, max(len(bcu) - 1, 0),
                par.ctypes.data if len(par) else None, out.data_ptr(), state.data_ptr(), sh)]
        fn = lib.span_la_pass

    def raw_step():
        for a in raw:
            fn(*a)

    # Host time of one warm call through the C entry point (prepared
    # arguments, device kept busy), beside host_enqueue_us through Python.
    busy = torch.empty(256 << 20, dtype=torch.float32, device=dev)
    host_c = []
    for _ in range(50):
        busy.zero_()
        t_h = time.perf_counter()
        raw_step()
        host_c.append((time.perf_counter() - t_h) * 1e6)
    torch.cuda.synchronize()
    spanla.span_la_check()
    del busy

    NW = 200
    w_start = torch.cuda.Event(enable_timing=True)
    w_end = torch.cuda.Event(enable_timing=True)
    for _ in range(5):
        raw_step()
    w_start.record(stream)
    for _ in range(NW):
        raw_step()
    w_end.record(stream)
    torch.cuda.synchronize()
    spanla.span_la_check()
    warm_us = w_start.elapsed_time(w_end) * 1e3 / NW

    # The same step recorded once into a CUDA graph and replayed (L2 flushed
    # before each replay, outside the graph).
    graph_us = None
    try:
        gstream = torch.cuda.Stream(device=dev)
        gstream.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gstream):
            run_on(q, k, v, out, state)
        torch.cuda.synchronize()
        for _ in range(3):
            flush.zero_()
            g.replay()
        torch.cuda.synchronize()
        gs = [torch.cuda.Event(enable_timing=True) for _ in range(50)]
        ge = [torch.cuda.Event(enable_timing=True) for _ in range(50)]
        for i in range(50):
            flush.zero_()
            gs[i].record(stream)
            g.replay()
            ge[i].record(stream)
        torch.cuda.synchronize()
        spanla.span_la_check()
        graph_us = statistics.mean(a.elapsed_time(b) for a, b in zip(gs, ge)) * 1e3
        del g
    except (RuntimeError, spanla.SpanLAError) as exc:   # report, do not fail the bench
        graph_us = "unavailable: %s" % exc

    h2d = 3 * (w.T - row_lo) * w.H * 64 * esize
    d2h = (w.T - row_lo) * w.H * 64 * esize + (0 if shards_mode else w.V * w.H * STATE_BYTES)
    clocks_busy = summarize_busy_clocks(run_sampler.stop())

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not shards_mode:
        med, reps, cores, (ref, ref_state) = oracle_time(w)
        med1, reps1, _, _ = oracle_time(w, budget_s=6.0, max_reps=3, nthreads=1)
        cpu = {"value": w.rows / med, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "the whole workload (%d rows x %d heads), median of %d passes"
                         % (w.rows, w.H, reps),
               "one_thread": {"value": w.rows / med1, "unit": UNIT, "cores": 1,
                              "sample": "median of %d passes" % reps1},
               "cpu_model": cpu_model()}
        # The benchmarked pass's output and view states against the oracle's
        # (the parity tests' measure).
        seg = segment_mask(w)
        got = out.detach().double().cpu().numpy()
        cpu["max_rel_err_vs_gpu"] = {
            "out": max_rel_err(got[seg], ref[seg]),
            "view_states": max_rel_err(state.detach().double().cpu().numpy(), ref_state)}

    vs = None
    if args.workload == "single":
        vs = value / (PAGE_TOKENS_7400 / (PAGE_MS_PER_LAYER_7400 / 1e3))

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": vs, "dtype": w.dtype, "data": "synthetic",
                "config": dict(add_mode(workload_config(w, args.workload), args), parallelism="dp%d" % world),
                "pass_structure": pass_structure(args),
                "roofline": roofline, "pass_roofline": pass_roofline,
                "kernels": kernels, "plan": plan,
                "cpu_baseline": cpu,
                "e2e": {"value": rows_total / (e2e_ms / 1e3), "unit": UNIT,
                        "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "steps": KE,
                        "mode": "pinned host buffers; copies of step i+1 overlap the call and "
                                "read-back of step i (two device buffer sets, three streams)"},
                "gpu_launches": int(sum(p["launches"] for p in launches.values())),
                "clocks": summarize_clocks(clock_rows, t0, t1),
                "step_ms_p50": statistics.median(step_ms),
                "profiled_kernel_us_sum": profiled_step_us,
                "step_ms_min": min(step_ms),
                "host_enqueue_us": statistics.median(host_us),
                "host_enqueue_us_c_abi": statistics.median(host_c),
                "clocks_busy": clocks_busy,
                "graph_us_per_step": graph_us,
                "warm_l2_us_per_step": warm_us,
                "cold_plan": cold,
                "long_request": long_req}
        print(json.dumps(line))
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
