"""Build and run the tensor-core rate probe (``tc_rate.cu``).

``python tests/probes/tc_rate.py`` builds the probe for sm_103a (into
``tests/probes/_build``) and runs every mode on one CTA per SM, printing one
line per mode: mode, grid, groups, ns per group, SM MHz, TFLOP/s per SM and in
all, and the error word.  ``--mode tile`` runs one mode (the form used under
ncu).  Measurement infrastructure: nothing in the library depends on it.
"""
import argparse
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
CSRC = os.path.join(ROOT, "hybrid_linear_attention_packed_gb300", "csrc")
BUILD = os.path.join(HERE, "_build")
BIN = os.path.join(BUILD, "tc_rate")
MODES = ["qk", "kv", "pv", "qs", "tile"]


def build() -> str:
    src = os.path.join(HERE, "tc_rate.cu")
    hdr = os.path.join(CSRC, "tc_ptx.cuh")
    if os.path.exists(BIN) and os.path.getmtime(BIN) >= max(os.path.getmtime(src), os.path.getmtime(hdr)):
        return BIN
    os.makedirs(BUILD, exist_ok=True)
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo",
                           "-I", CSRC, src, "-o", BIN])
    return BIN


def run(mode: str, grid: int = 0, iters: int = 256) -> dict:
    args = [build(), mode, str(grid), str(iters)]
    line = subprocess.check_output(args).decode().split()
    keys = ["mode", "grid", "iters", "ns_per_group", "mhz", "tflops_per_sm", "tflops", "err"]
    vals = [line[0]] + [int(line[1]), int(line[2])] + [float(x) for x in line[3:7]] + [int(line[7])]
    return dict(zip(keys, vals))


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--mode", choices=MODES)
    ap.add_argument("--grid", type=int, default=0, help="CTAs (default: one per SM)")
    ap.add_argument("--iters", type=int, default=256)
    a = ap.parse_args()
    for m in ([a.mode] if a.mode else MODES):
        r = run(m, a.grid, a.iters)
        print(" ".join(str(r[k]) for k in r))
        sys.stdout.flush()
    return 0


if __name__ == "__main__":
    sys.exit(main())
