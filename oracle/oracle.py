"""Python side of the float64 oracle.

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the CPU
baseline of the benchmark, never by the product path.

The oracle proper is the C recurrence in ``spanla_oracle.c`` (the plain
definition of unnormalised causal linear attention, per head:
``S_t = S_{t-1} + k_t v_t^T``, ``o_t = S_t^T q_t``, views from ``S = 0`` and
branches from their parent view's final state -- "Serving 0.88M TPS from Two
RTXs and Mac Minis", sections "The Workload", "Kernels" and "Long Requests").

Two further numpy forms live here for cross-checking the C recurrence only:

* :func:`segment_quadratic` -- the masked quadratic form
  ``O = tril(Q K^T) V + Q S0`` (textbook matmuls, no recurrence at all);
* :func:`segment_chunked` -- the 64-token chunked form the page's "Kernels"
  section describes (each chunk: an intra-chunk masked product plus the
  inter-chunk state term, then the state update).

All three agree in exact arithmetic; the pins in ``tests/`` hold them to
float64 rounding.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spanla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source with gcc and OpenMP."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O3", "-fPIC", "-shared", "-fopenmp", "-std=c11",
           "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind_library(path: str):
    """Load a build of ``spanla_oracle.c`` from ``path`` and declare its entry
    points (the tests also bind copies built with planted mistakes)."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int32)
    lib.oracle_pass.argtypes = [dp, dp, dp, ctypes.c_int64, ctypes.c_int64,
                                ctypes.c_int64, ip, ctypes.c_int32, ip,
                                ctypes.c_int32, ip, dp, dp, ctypes.c_int]
    lib.oracle_pass.restype = ctypes.c_int
    lib.oracle_branches_from_state.argtypes = [
        dp, ctypes.c_int32, dp, dp, dp, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int64, ip, ctypes.c_int32, ip, dp, ctypes.c_int]
    lib.oracle_branches_from_state.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind_library(build_oracle())
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32).reshape(-1))


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _iptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def oracle_max_threads() -> int:
    return int(_load().oracle_max_threads())


def oracle_pass(q, k, v, view_cu_seqlens, branch_cu_seqlens, branch_parent,
                nthreads: int = 0, fill: float = 0.0):
    """Float64 packed pass.

    q, k, v: [T, H, D] (any float dtype; widened exactly to float64).
    Returns ``(out [T,H,D] float64, view_state [V,H,D,D] float64)``.  Rows in
    no segment hold ``fill``.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, D = q.shape
    vcu, bcu, par = _i32(view_cu_seqlens), _i32(branch_cu_seqlens), _i32(branch_parent)
    V = max(len(vcu) - 1, 0)
    B = max(len(bcu) - 1, 0)
    out = np.full((T, H, D), fill, dtype=np.float64)
    state = np.zeros((max(V, 0), H, D, D), dtype=np.float64)
    rc = _load().oracle_pass(_dptr(q), _dptr(k), _dptr(v), T, H, D,
                             _iptr(vcu), V, _iptr(bcu), B, _iptr(par),
                             _dptr(out), _dptr(state), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_pass rejected its input (code %d)" % rc)
    return out, state


def oracle_branches_from_state(states, q, k, v, branch_cu_seqlens, branch_parent,
                               nthreads: int = 0, fill: float = 0.0):
    """Float64 branches from cached per-view states ``states [P,H,D,D]``."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    st = _f64(states)
    T, H, D = q.shape
    P = st.shape[0]
    bcu, par = _i32(branch_cu_seqlens), _i32(branch_parent)
    B = max(len(bcu) - 1, 0)
    out = np.full((T, H, D), fill, dtype=np.float64)
    rc = _load().oracle_branches_from_state(_dptr(st), P, _dptr(q), _dptr(k), _dptr(v),
                                            T, H, D, _iptr(bcu), B, _iptr(par),
                                            _dptr(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_branches_from_state rejected its input (code %d)" % rc)
    return out


def segment_quadratic(q, k, v, S0=None):
    """Masked quadratic form for one segment, all heads.

    q, k, v: [L, H, D].  S0: [H, D, D] start state (zero if None).
    Per head: ``O = tril(Q K^T) V + Q S0`` -- the inclusive causal mask is the
    lower triangle with its diagonal.  Returns ``(O [L,H,D], S_end [H,D,D])``
    with ``S_end = S0 + K^T V``.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    L, H, D = q.shape
    S0 = np.zeros((H, D, D)) if S0 is None else _f64(S0)
    out = np.zeros((L, H, D))
    S_end = np.zeros((H, D, D))
    for h in range(H):
        Q, K, Vv = q[:, h, :], k[:, h, :], v[:, h, :]
        A = np.tril(Q @ K.T)
        out[:, h, :] = A @ Vv + Q @ S0[h]
        S_end[h] = S0[h] + K.T @ Vv
    return out, S_end


def segment_chunked(q, k, v, S0=None, C: int = 64):
    """Chunked form for one segment, all heads (chunks aligned to the segment start).

    For each chunk c: ``O_c = tril(Q_c K_c^T) V_c + Q_c S``, then
    ``S <- S + K_c^T V_c``.  The last chunk may be shorter than C.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    L, H, D = q.shape
    S = np.zeros((H, D, D)) if S0 is None else _f64(S0).copy()
    out = np.zeros((L, H, D))
    for c0 in range(0, L, C):
        c1 = min(c0 + C, L)
        for h in range(H):
            Q, K, Vv = q[c0:c1, h, :], k[c0:c1, h, :], v[c0:c1, h, :]
            out[c0:c1, h, :] = np.tril(Q @ K.T) @ Vv + Q @ S[h]
            S[h] = S[h] + K.T @ Vv
    return out, S
