"""The C ABI without Python: a plain C program (``tests/c_client/spanla_client.c``,
built here with gcc against ``include/spanla.h`` and ``libspanla.so``) runs a
packed pass, the softmax layer and branches from the pass's view states; the
results are compared with the float64 oracles."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from helpers import TOL, rel_err, segment_rows
from hybrid_linear_attention_packed_gb300 import build as spanla_build
from hybrid_linear_attention_packed_gb300 import workloads
from oracle import oracle_pass, oracle_softmax_pass

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            return cand
    nvcc = shutil.which("nvcc")
    return os.path.dirname(os.path.dirname(nvcc)) if nvcc else None


def _bf16_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _from_bf16_bits(a):
    return torch.from_numpy(a.astype(np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


def test_c_client_matches_the_oracles(tmp_path, cuda_device):
    lib = spanla_build.build()
    cuda = _cuda_home()
    assert cuda, "CUDA toolkit headers not found"
    exe = str(tmp_path / "spanla_client")
    lib_dir = os.path.dirname(lib)
    cmd = ["gcc", "-O2", "-std=c11", "-o", exe, os.path.join(HERE, "c_client", "spanla_client.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           "-L", lib_dir, "-lspanla", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           "-Wl,-rpath," + lib_dir + ":" + os.path.join(cuda, "lib64")]
    subprocess.run(cmd, check=True)

    w = workloads.make_pass([300, 129, 0], [40, 9, 130, 1], [0, 0, 1, 2], H=3, dtype="bf16", seed=61,
                            q_scale=1.0, k_scale=1.0)
    T, H = w.T, w.H
    with open(tmp_path / "in.bin", "wb") as f:
        f.write(np.array([T, H, w.V, w.B], dtype=np.int32).tobytes())
        f.write(w.view_cu.astype(np.int32).tobytes())
        f.write(w.branch_cu.astype(np.int32).tobytes())
        f.write(w.branch_parent.astype(np.int32).tobytes())
        for t in (w.q, w.k, w.v):
            f.write(_bf16_bits(t).tobytes())
    r = subprocess.run([exe, str(tmp_path / "in.bin"), str(tmp_path / "out.bin")], capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    print(r.stdout.strip())

    n = T * H * 64
    raw = np.fromfile(tmp_path / "out.bin", dtype=np.uint8)
    off = 0
    out = _from_bf16_bits(raw[off:off + 2 * n].view(np.uint16)).reshape(T, H, 64); off += 2 * n
    state = raw[off:off + 4 * w.V * H * 4096].view(np.float32).reshape(w.V, H, 64, 64); off += 4 * w.V * H * 4096
    out_sm = _from_bf16_bits(raw[off:off + 2 * n].view(np.uint16)).reshape(T, H, 64); off += 2 * n
    out_fs = _from_bf16_bits(raw[off:off + 2 * n].view(np.uint16)).reshape(T, H, 64); off += 2 * n
    assert off == raw.size

    q, k, v = (t.double().numpy() for t in (w.q, w.k, w.v))
    ref, ref_state = oracle_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent)
    sref, _ = oracle_softmax_pass(q, k, v, w.view_cu, w.branch_cu, w.branch_parent)
    seg = segment_rows(w)
    br = np.zeros(T, bool)
    br[w.branch_cu[0]:w.branch_cu[-1]] = True
    e = rel_err(out[seg], ref[seg])
    es = rel_err(state.astype(np.float64), ref_state)
    e_sm = rel_err(out_sm[seg], sref[seg])
    assert np.array_equal(out_fs[br & seg], out[br & seg])   # same kernels, same start states
    print("C client: pass %.2e state %.2e softmax %.2e" % (e, es, e_sm))
    assert max(e, es, e_sm) <= TOL["bf16"]
