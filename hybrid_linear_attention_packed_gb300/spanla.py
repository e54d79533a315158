"""Thin Python binding of ``libspanla.so`` (argument marshalling only).

Every step of the pass runs in the library's CUDA kernels; this module only
checks tensor dtypes, shapes, devices and contiguity, converts host metadata to
int32 arrays and passes raw pointers and the current CUDA stream through the C
ABI declared in ``include/spanla.h``.  PyTorch is used for device memory and
streams only.  There is no fallback: if the library is missing or cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence, Tuple

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("SPANLA_LIB", os.path.join(_PKG, "libspanla.so"))

SPAN_LA_BF16 = 0
SPAN_LA_F32 = 1

STATUS = {0: "SPAN_LA_OK", 1: "SPAN_LA_ERR_INVALID", 2: "SPAN_LA_ERR_UNSUPPORTED",
          3: "SPAN_LA_ERR_CUDA", 4: "SPAN_LA_ERR_NOMEM", 5: "SPAN_LA_ERR_TIMEOUT"}

EXPORTED = ("span_la_pass", "span_la_branches_from_state", "span_la_check",
            "span_la_status_string", "span_la_last_error_detail", "span_la_version",
            "span_la_selftest_wait_timeout", "span_la_profile_enable", "span_la_profile_read",
            "span_la_profile_reset", "span_la_kernel_name", "span_la_plan_stats",
            "span_la_pass_noalloc", "span_la_cache_create", "span_la_cache_destroy",
            "span_la_cache_put", "span_la_cache_contains", "span_la_cache_branches",
            "span_la_cache_stats", "span_la_softmax_pass", "span_la_softmax_branches_from_kv",
            "span_la_fault_inject", "span_la_softmax_plan_stats",
            "span_la_selftest_wait_timeout_noalloc", "span_la_pass_variant",
            "span_la_plan_prepare")
NUM_KERNELS = 7


class SpanLAError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__("%s: %s (%s)" % (where, STATUS.get(status, status), detail))


class Dims(ctypes.Structure):
    _fields_ = [("total_rows", ctypes.c_int64), ("num_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load_library(path: Optional[str] = None):
    """Load the CUDA library (raises if it is missing: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError("libspanla.so not found at %s: build it with "
                               "hybrid_linear_attention_packed_gb300.build.build()" % p)
        lib = ctypes.CDLL(p)
        # int32 arrays go in as addresses (c_void_p also takes ctypes pointers)
        vp = ctypes.c_void_p
        i32p = vp
        lib.span_la_pass.argtypes = [vp, vp, vp, Dims, i32p, ctypes.c_int32, i32p,
                                     ctypes.c_int32, i32p, vp, vp, vp]
        lib.span_la_pass.restype = ctypes.c_int
        lib.span_la_pass_noalloc.argtypes = [vp, vp, vp, Dims, i32p, ctypes.c_int32, i32p,
                                             ctypes.c_int32, i32p, vp, vp, vp]
        lib.span_la_pass_noalloc.restype = ctypes.c_int
        lib.span_la_branches_from_state.argtypes = [vp, ctypes.c_int32, vp, vp, vp, Dims, i32p,
                                                    ctypes.c_int32, i32p, vp, vp]
        lib.span_la_branches_from_state.restype = ctypes.c_int
        lib.span_la_check.argtypes = [vp]
        lib.span_la_check.restype = ctypes.c_int
        lib.span_la_status_string.argtypes = [ctypes.c_int]
        lib.span_la_status_string.restype = ctypes.c_char_p
        lib.span_la_last_error_detail.argtypes = []
        lib.span_la_last_error_detail.restype = ctypes.c_char_p
        lib.span_la_version.argtypes = []
        lib.span_la_version.restype = ctypes.c_int32
        lib.span_la_selftest_wait_timeout.argtypes = [ctypes.c_int32, vp]
        lib.span_la_selftest_wait_timeout.restype = ctypes.c_int
        lib.span_la_selftest_wait_timeout_noalloc.argtypes = [ctypes.c_int32, vp]
        lib.span_la_selftest_wait_timeout_noalloc.restype = ctypes.c_int
        lib.span_la_profile_enable.argtypes = [ctypes.c_int32]
        lib.span_la_profile_enable.restype = ctypes.c_int
        lib.span_la_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double),
                                             ctypes.POINTER(ctypes.c_int64),
                                             ctypes.POINTER(ctypes.c_int64), ctypes.c_int32]
        lib.span_la_profile_read.restype = ctypes.c_int
        lib.span_la_profile_reset.argtypes = []
        lib.span_la_profile_reset.restype = ctypes.c_int
        lib.span_la_kernel_name.argtypes = [ctypes.c_int32]
        lib.span_la_kernel_name.restype = ctypes.c_char_p
        lib.span_la_plan_stats.argtypes = [i32p, ctypes.c_int32, i32p, ctypes.c_int32, i32p,
                                           ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_int32,
                                           ctypes.POINTER(ctypes.c_int64)]
        lib.span_la_plan_stats.restype = ctypes.c_int
        lib.span_la_softmax_pass.argtypes = [vp, vp, vp, Dims, i32p, ctypes.c_int32, i32p,
                                             ctypes.c_int32, i32p, ctypes.c_float, vp, vp, vp]
        lib.span_la_softmax_pass.restype = ctypes.c_int
        lib.span_la_softmax_plan_stats.argtypes = [i32p, ctypes.c_int32, i32p, ctypes.c_int32, i32p,
                                                   ctypes.c_int32, ctypes.c_int32,
                                                   ctypes.POINTER(ctypes.c_int64)]
        lib.span_la_softmax_plan_stats.restype = ctypes.c_int
        lib.span_la_pass_variant.argtypes = [ctypes.c_int32]
        lib.span_la_pass_variant.restype = ctypes.c_int
        lib.span_la_plan_prepare.argtypes = [Dims, i32p, ctypes.c_int32, i32p, ctypes.c_int32, i32p, vp]
        lib.span_la_plan_prepare.restype = ctypes.c_int
        lib.span_la_fault_inject.argtypes = [ctypes.c_int32, ctypes.c_int32]
        lib.span_la_fault_inject.restype = ctypes.c_int
        lib.span_la_softmax_branches_from_kv.argtypes = [vp, vp, ctypes.c_int64, i32p, ctypes.c_int32,
                                                         vp, vp, vp, Dims, i32p, ctypes.c_int32, i32p,
                                                         ctypes.c_float, vp, vp, vp]
        lib.span_la_softmax_branches_from_kv.restype = ctypes.c_int
        lib.span_la_cache_create.argtypes = [ctypes.c_int32, ctypes.c_int32,
                                             ctypes.POINTER(ctypes.c_void_p)]
        lib.span_la_cache_create.restype = ctypes.c_int
        lib.span_la_cache_destroy.argtypes = [vp]
        lib.span_la_cache_destroy.restype = ctypes.c_int
        lib.span_la_cache_put.argtypes = [vp, vp, ctypes.c_int32, vp, vp]
        lib.span_la_cache_put.restype = ctypes.c_int
        lib.span_la_cache_contains.argtypes = [vp, vp, ctypes.c_int32, vp]
        lib.span_la_cache_contains.restype = ctypes.c_int
        lib.span_la_cache_branches.argtypes = [vp, vp, vp, vp, vp, Dims, i32p, ctypes.c_int32,
                                               vp, vp]
        lib.span_la_cache_branches.restype = ctypes.c_int
        lib.span_la_cache_stats.argtypes = [vp, ctypes.POINTER(ctypes.c_int64)]
        lib.span_la_cache_stats.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _raise(lib, status: int, where: str):
    if status != 0:
        raise SpanLAError(status, where, lib.span_la_last_error_detail().decode())


def _i32(a) -> np.ndarray:
    if a is None:
        return np.zeros(0, dtype=np.int32)
    if isinstance(a, np.ndarray) and a.dtype == np.int32 and a.ndim == 1 and a.flags.c_contiguous:
        return a
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64).reshape(-1).astype(np.int32))


def _iptr(a: np.ndarray):
    """Address of an int32 array for a ``const int32_t*`` argument (None when empty)."""
    if a.size == 0:
        return None
    if a.flags.writeable:   # (cheaper than numpy's .ctypes helper object)
        return ctypes.addressof(ctypes.c_int32.from_buffer(a))
    return a.ctypes.data


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_raw_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream_handle(stream) -> int:
    """The CUDA stream handle for a call: ``stream``'s, or the current device's
    current stream."""
    if stream is None:
        if _raw_stream is not None and _raw_device is not None:
            return int(_raw_stream(_raw_device()))
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _dims_of(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> Dims:
    # The usual case in one expression; anything else goes through the
    # checks below, which name the problem.
    sh, dt = q.shape, q.dtype
    if (len(sh) == 3 and sh[2] == 64 and k.shape == sh and v.shape == sh and k.dtype == dt
            and v.dtype == dt and (dt == torch.bfloat16 or dt == torch.float32)
            and q.is_cuda and k.is_cuda and v.is_cuda
            and q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        return Dims(sh[0], sh[1], 64, SPAN_LA_BF16 if dt == torch.bfloat16 else SPAN_LA_F32)
    return _dims_checked(q, k, v)


def _dims_checked(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> Dims:
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % name)
        if t.dim() != 3 or t.shape[2] != 64:
            raise ValueError("%s must be [T, H, 64], got %s" % (name, tuple(t.shape)))
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    if q.shape != k.shape or q.shape != v.shape or q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError("q, k and v must share shape and dtype")
    if q.dtype == torch.bfloat16:
        dt = SPAN_LA_BF16
    elif q.dtype == torch.float32:
        dt = SPAN_LA_F32
    else:
        raise ValueError("dtype %s not supported (bf16 or fp32)" % q.dtype)
    return Dims(q.shape[0], q.shape[1], q.shape[2], dt)


def span_la_pass(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                 view_cu_seqlens: Sequence[int], branch_cu_seqlens: Optional[Sequence[int]],
                 branch_parent: Optional[Sequence[int]],
                 out: Optional[torch.Tensor] = None,
                 view_state_out: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None,
                 _entry: str = "span_la_pass") -> Tuple[torch.Tensor, torch.Tensor]:
    """One packed pass (see ``span_la_pass`` in ``include/spanla.h``).

    Returns ``(out [T,H,64], view_state_out [V,H,64,64] fp32)``.  ``out`` is
    allocated with ``torch.empty`` when not given: rows in no segment then
    hold whatever the allocator returned.
    """
    lib = load_library()
    dims = _dims_of(q, k, v)
    vcu, bcu, par = _i32(view_cu_seqlens), _i32(branch_cu_seqlens), _i32(branch_parent)
    V = max(len(vcu) - 1, 0)
    B = max(len(bcu) - 1, 0)
    H = q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if view_state_out is None:
        view_state_out = torch.empty((V, H, 64, 64), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA tensor like q")
    if (view_state_out.dtype != torch.float32 or not view_state_out.is_contiguous()
            or not view_state_out.is_cuda or view_state_out.numel() < V * H * 4096):
        raise ValueError("view_state_out must be a contiguous fp32 CUDA tensor [V, H, 64, 64]")
    st = getattr(lib, _entry)(q.data_ptr(), k.data_ptr(), v.data_ptr(), dims,
                              _iptr(vcu), V, _iptr(bcu), B, _iptr(par),
                              out.data_ptr(), view_state_out.data_ptr(), _stream_handle(stream))
    _raise(lib, st, _entry)
    return out, view_state_out


def span_la_plan_prepare(view_cu_seqlens: Sequence[int], branch_cu_seqlens: Optional[Sequence[int]],
                         branch_parent: Optional[Sequence[int]], total_rows: int, num_heads: int,
                         dtype: torch.dtype = torch.bfloat16,
                         stream: Optional[torch.cuda.Stream] = None) -> None:
    """Build and upload the plan of a later :func:`span_la_pass` with this
    metadata on the current device (``span_la_plan_prepare`` in
    ``include/spanla.h``), so that the pass finds it in the plan cache."""
    lib = load_library()
    if dtype == torch.bfloat16:
        dt = SPAN_LA_BF16
    elif dtype == torch.float32:
        dt = SPAN_LA_F32
    else:
        raise ValueError("dtype %s not supported (bf16 or fp32)" % dtype)
    vcu, bcu, par = _i32(view_cu_seqlens), _i32(branch_cu_seqlens), _i32(branch_parent)
    V = max(len(vcu) - 1, 0)
    B = max(len(bcu) - 1, 0)
    st = lib.span_la_plan_prepare(Dims(int(total_rows), int(num_heads), 64, dt), _iptr(vcu), V,
                                  _iptr(bcu), B, _iptr(par), _stream_handle(stream))
    _raise(lib, st, "span_la_plan_prepare")


def span_la_pass_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                         view_cu_seqlens: Sequence[int], branch_cu_seqlens: Optional[Sequence[int]],
                         branch_parent: Optional[Sequence[int]],
                         out: Optional[torch.Tensor] = None,
                         view_state_out: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """As :func:`span_la_pass`, with the workspace in the library's fixed
    scratch instead of a per-call allocation (``span_la_pass_noalloc``)."""
    return span_la_pass(q, k, v, view_cu_seqlens, branch_cu_seqlens, branch_parent, out=out,
                        view_state_out=view_state_out, stream=stream, _entry="span_la_pass_noalloc")


def span_la_branches_from_state(cached_state: torch.Tensor, q: torch.Tensor, k: torch.Tensor,
                                v: torch.Tensor, branch_cu_seqlens: Sequence[int],
                                branch_parent: Sequence[int],
                                out: Optional[torch.Tensor] = None,
                                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Branches forking from cached view states (``span_la_branches_from_state``)."""
    lib = load_library()
    dims = _dims_of(q, k, v)
    bcu, par = _i32(branch_cu_seqlens), _i32(branch_parent)
    B = max(len(bcu) - 1, 0)
    if (cached_state.dtype != torch.float32 or not cached_state.is_contiguous()
            or not cached_state.is_cuda or cached_state.dim() != 4
            or tuple(cached_state.shape[1:]) != (q.shape[1], 64, 64)):
        raise ValueError("cached_state must be contiguous fp32 CUDA [P, H, 64, 64]")
    if out is None:
        out = torch.empty_like(q)
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA tensor like q")
    st = lib.span_la_branches_from_state(cached_state.data_ptr(), cached_state.shape[0],
                                         q.data_ptr(), k.data_ptr(), v.data_ptr(), dims,
                                         _iptr(bcu), B, _iptr(par), out.data_ptr(),
                                         _stream_handle(stream))
    _raise(lib, st, "span_la_branches_from_state")
    return out


def span_la_softmax_pass(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                         view_cu_seqlens: Sequence[int], branch_cu_seqlens: Sequence[int],
                         branch_parent: Sequence[int], scale: float = 0.0,
                         out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """One softmax-attention layer over the packed rows (``span_la_softmax_pass``):
    views causal, branches over their parent view plus their own causal prefix.
    ``lse`` (fp32 [T, H], optional) receives the natural-log normaliser."""
    lib = load_library()
    dims = _dims_of(q, k, v)
    vcu, bcu, par = _i32(view_cu_seqlens), _i32(branch_cu_seqlens), _i32(branch_parent)
    V = max(len(vcu) - 1, 0)
    B = max(len(bcu) - 1, 0)
    if out is None:
        out = torch.empty_like(q)
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA tensor like q")
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous() or not lse.is_cuda
                            or tuple(lse.shape) != (q.shape[0], q.shape[1])):
        raise ValueError("lse must be contiguous fp32 CUDA [T, H]")
    st = lib.span_la_softmax_pass(q.data_ptr(), k.data_ptr(), v.data_ptr(), dims, _iptr(vcu), V,
                                  _iptr(bcu), B, _iptr(par), float(scale), out.data_ptr(),
                                  lse.data_ptr() if lse is not None else None,
                                  _stream_handle(stream))
    _raise(lib, st, "span_la_softmax_pass")
    return out


def span_la_softmax_branches_from_kv(view_k: torch.Tensor, view_v: torch.Tensor,
                                     view_cu_seqlens: Sequence[int], q: torch.Tensor, k: torch.Tensor,
                                     v: torch.Tensor, branch_cu_seqlens: Sequence[int],
                                     branch_parent: Sequence[int], scale: float = 0.0,
                                     out: Optional[torch.Tensor] = None,
                                     lse: Optional[torch.Tensor] = None,
                                     stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Softmax-layer branches over their parent views' K and V kept from an
    earlier pass (``span_la_softmax_branches_from_kv``)."""
    lib = load_library()
    dims = _dims_of(q, k, v)
    for name, t in (("view_k", view_k), ("view_v", view_v)):
        if (not t.is_cuda or t.dtype != q.dtype or not t.is_contiguous() or t.dim() != 3
                or tuple(t.shape[1:]) != tuple(q.shape[1:])):
            raise ValueError("%s must be a contiguous CUDA tensor [rows, H, 64] like q" % name)
    if view_k.shape != view_v.shape:
        raise ValueError("view_k and view_v must share shape")
    vcu, bcu, par = _i32(view_cu_seqlens), _i32(branch_cu_seqlens), _i32(branch_parent)
    V = max(len(vcu) - 1, 0)
    B = max(len(bcu) - 1, 0)
    if out is None:
        out = torch.empty_like(q)
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA tensor like q")
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous() or not lse.is_cuda
                            or tuple(lse.shape) != (q.shape[0], q.shape[1])):
        raise ValueError("lse must be contiguous fp32 CUDA [T, H]")
    st = lib.span_la_softmax_branches_from_kv(
        view_k.data_ptr(), view_v.data_ptr(), view_k.shape[0], _iptr(vcu), V, q.data_ptr(),
        k.data_ptr(), v.data_ptr(), dims, _iptr(bcu), B, _iptr(par), float(scale), out.data_ptr(),
        lse.data_ptr() if lse is not None else None, _stream_handle(stream))
    _raise(lib, st, "span_la_softmax_branches_from_kv")
    return out


def _keys(keys) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(keys, dtype=np.uint64).reshape(-1))
    return a


CACHE_FIELDS = ("entries", "capacity", "hits", "misses", "evictions", "puts")


class ViewStateCache:
    """Keyed least-recently-used cache of view final states in device memory
    (``span_la_cache_*``): put a pass's ``view_state_out`` rows under keys,
    then run branches (or shards of them) from the cached states by key."""

    def __init__(self, num_heads: int, capacity: int):
        self._lib = load_library()
        handle = ctypes.c_void_p()
        _raise(self._lib, self._lib.span_la_cache_create(int(num_heads), int(capacity),
                                                         ctypes.byref(handle)),
               "span_la_cache_create")
        self._handle = handle.value
        self.num_heads = int(num_heads)
        self.capacity = int(capacity)

    def close(self) -> None:
        if self._handle:
            handle, self._handle = self._handle, None
            _raise(self._lib, self._lib.span_la_cache_destroy(handle), "span_la_cache_destroy")

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _live(self):
        if not self._handle:
            raise ValueError("the cache is closed")
        return self._handle

    def put(self, keys, states: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> None:
        """Store states[i] (fp32 CUDA [n, H, 64, 64], contiguous) under keys[i]."""
        ks = _keys(keys)
        if (states.dtype != torch.float32 or not states.is_contiguous() or not states.is_cuda
                or states.dim() != 4 or tuple(states.shape[1:]) != (self.num_heads, 64, 64)
                or states.shape[0] != ks.size):
            raise ValueError("states must be contiguous fp32 CUDA [len(keys), H, 64, 64]")
        _raise(self._lib, self._lib.span_la_cache_put(self._live(), ks.ctypes.data, ks.size,
                                                      states.data_ptr(), _stream_handle(stream)),
               "span_la_cache_put")

    def contains(self, keys) -> np.ndarray:
        ks = _keys(keys)
        present = np.zeros(ks.size, dtype=np.int32)
        _raise(self._lib, self._lib.span_la_cache_contains(
            self._live(), ks.ctypes.data if ks.size else None, ks.size,
            present.ctypes.data if ks.size else None), "span_la_cache_contains")
        return present.astype(bool)

    def branches(self, parent_keys, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                 branch_cu_seqlens: Sequence[int], out: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """Branch b forks from the state cached under parent_keys[b]."""
        dims = _dims_of(q, k, v)
        bcu = _i32(branch_cu_seqlens)
        B = max(len(bcu) - 1, 0)
        ks = _keys(parent_keys)
        if ks.size != B:
            raise ValueError("one parent key per branch")
        if out is None:
            out = torch.empty_like(q)
        if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or not out.is_cuda:
            raise ValueError("out must be a contiguous CUDA tensor like q")
        _raise(self._lib, self._lib.span_la_cache_branches(
            self._live(), ks.ctypes.data if ks.size else None, q.data_ptr(), k.data_ptr(),
            v.data_ptr(), dims, _iptr(bcu), B, out.data_ptr(), _stream_handle(stream)),
            "span_la_cache_branches")
        return out

    def stats(self) -> dict:
        st = (ctypes.c_int64 * len(CACHE_FIELDS))()
        _raise(self._lib, self._lib.span_la_cache_stats(self._live(), st), "span_la_cache_stats")
        return dict(zip(CACHE_FIELDS, (int(x) for x in st)))


def span_la_check(stream: Optional[torch.cuda.Stream] = None) -> None:
    """Synchronise the stream and raise on a CUDA error or a device wait timeout."""
    lib = load_library()
    _raise(lib, lib.span_la_check(_stream_handle(stream)), "span_la_check")


FAULT_ALLOC = 1


def fault_inject(kind: int, count: int) -> None:
    """Make the library's next `count` device allocations fail (kind FAULT_ALLOC)."""
    lib = load_library()
    _raise(lib, lib.span_la_fault_inject(int(kind), int(count)), "span_la_fault_inject")


def span_la_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    lib = load_library()
    _raise(lib, lib.span_la_selftest_wait_timeout(int(limit_us), _stream_handle(stream)),
           "span_la_selftest_wait_timeout")


PASS_ONE_LAUNCH = 0
PASS_THREE_LAUNCHES = 1


def set_pass_variant(variant: int) -> None:
    """Process-wide structure of the bf16 pass (``span_la_pass_variant``):
    ``PASS_ONE_LAUNCH`` (default) or ``PASS_THREE_LAUNCHES``."""
    lib = load_library()
    _raise(lib, lib.span_la_pass_variant(int(variant)), "span_la_pass_variant")


def span_la_selftest_wait_timeout_noalloc(limit_us: int, stream=None) -> None:
    lib = load_library()
    _raise(lib, lib.span_la_selftest_wait_timeout_noalloc(int(limit_us), _stream_handle(stream)),
           "span_la_selftest_wait_timeout_noalloc")


PLAN_FIELDS = ("state_slots", "state_rows", "scan_segments", "final_states", "tiles",
               "tile_rows", "start_state_reads", "out_items", "run_tiles")


def plan_stats(view_cu_seqlens, branch_cu_seqlens, branch_parent, num_heads: int,
               dtype: str = "bf16", num_parents: int = 0, from_state: bool = False,
               num_sms: int = 152) -> dict:
    """Work units the library would launch for this metadata on a GPU with
    ``num_sms`` SMs (host only; every count summed over heads)."""
    lib = load_library()
    vcu, bcu, par = _i32(view_cu_seqlens), _i32(branch_cu_seqlens), _i32(branch_parent)
    V = max(len(vcu) - 1, 0)
    B = max(len(bcu) - 1, 0)
    stats = (ctypes.c_int64 * len(PLAN_FIELDS))()
    dt = SPAN_LA_BF16 if dtype == "bf16" else SPAN_LA_F32
    _raise(lib, lib.span_la_plan_stats(_iptr(vcu), V, _iptr(bcu), B, _iptr(par), int(num_parents),
                                       1 if from_state else 0, int(num_heads), dt, int(num_sms),
                                       stats),
           "span_la_plan_stats")
    return dict(zip(PLAN_FIELDS, (int(x) for x in stats)))


SOFTMAX_PLAN_FIELDS = ("items", "rows", "key_blocks", "grid")


def softmax_plan_stats(view_cu_seqlens, branch_cu_seqlens, branch_parent, num_heads: int,
                       num_sms: int = 152) -> dict:
    """Work units of the softmax layer for this metadata (host only)."""
    lib = load_library()
    vcu, bcu, par = _i32(view_cu_seqlens), _i32(branch_cu_seqlens), _i32(branch_parent)
    V = max(len(vcu) - 1, 0)
    B = max(len(bcu) - 1, 0)
    stats = (ctypes.c_int64 * len(SOFTMAX_PLAN_FIELDS))()
    _raise(lib, lib.span_la_softmax_plan_stats(_iptr(vcu), V, _iptr(bcu), B, _iptr(par), int(num_heads),
                                               int(num_sms), stats), "span_la_softmax_plan_stats")
    return dict(zip(SOFTMAX_PLAN_FIELDS, (int(x) for x in stats)))


def profile_enable(on: bool = True) -> None:
    """Time every kernel launch with CUDA events on its stream (tracing hook)."""
    lib = load_library()
    _raise(lib, lib.span_la_profile_enable(1 if on else 0), "span_la_profile_enable")


def profile_reset() -> None:
    lib = load_library()
    _raise(lib, lib.span_la_profile_reset(), "span_la_profile_reset")


def profile_read() -> dict:
    """Per kernel name: {"ms": summed event time, "timed": launches timed,
    "launches": launches counted} since the last reset."""
    lib = load_library()
    ms = (ctypes.c_double * NUM_KERNELS)()
    timed = (ctypes.c_int64 * NUM_KERNELS)()
    launches = (ctypes.c_int64 * NUM_KERNELS)()
    _raise(lib, lib.span_la_profile_read(ms, timed, launches, NUM_KERNELS), "span_la_profile_read")
    return {lib.span_la_kernel_name(k).decode(): {"ms": ms[k], "timed": timed[k],
                                                  "launches": launches[k]}
            for k in range(NUM_KERNELS)}


def version() -> int:
    return int(load_library().span_la_version())
