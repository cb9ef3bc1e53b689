"""Python binding of libsplitkv (include/splitkv.h): argument marshalling only.

Every entry point of the C ABI is exposed under the same name and takes the
same arguments (ctypes pointers/ints; torch tensors are accepted wherever the
C function takes a device pointer). All arithmetic runs in the library's
CUDA kernels; there is no CPU path. If the shared library is missing this
module raises at import time.

The ``SplitKV`` helper bundles a problem, its two workspaces and the three
passes for callers that hold their tensors in torch.

With the environment variable ``SPLITKV_DEBUG=1`` set at import, the module
loads the debug build (``libsplitkv_debug.so``, ``build.py --debug``), whose
kernels check their indices and report failures through
``splitkv_plan_stats`` (``debug_violations``); it is never the default.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Dict, Optional

HERE = os.path.dirname(os.path.abspath(__file__))
DEBUG_BUILD = os.environ.get("SPLITKV_DEBUG", "") == "1"
LIB_PATH = os.path.join(HERE, "libsplitkv_debug.so" if DEBUG_BUILD else "libsplitkv.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "splitkv.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python block_sparse_cross_gb300/build.py"
        f"{' --debug' if DEBUG_BUILD else ''}` "
        "(no CPU fallback exists)")

_lib = ctypes.CDLL(LIB_PATH)

# ---- constants (mirrors include/splitkv.h) ---------------------------------
SPLITKV_OK = 0
SPLITKV_EINVAL = 1
SPLITKV_EUNSUPPORTED = 2
SPLITKV_EWORKSPACE = 3
SPLITKV_ECUDA = 4
SPLITKV_EDEVICE = 5
SPLITKV_ETIMEOUT = 6
SPLITKV_EPLAN = 7
SPLITKV_EMETA = 8
SPLITKV_ECAPACITY = 9
SPLITKV_BF16 = 0
SPLITKV_FP32 = 1
SPLITKV_FLAG_CUDA_CORE = 1
SPLITKV_FLAG_CONTIGUOUS = 2
SPLITKV_FLAG_MASK_INCLUSIVE = 4
SPLITKV_FLAG_MASK_CAUSAL_BLOCK = 8
SPLITKV_FLAG_MASK_CONTEXT_OFFSET = 16
SPLITKV_BUILD_DEBUG = 1
SPLITKV_NUM_KERNELS = 9
SPLITKV_NOALLOC_SCRATCH_BYTES = 64 << 20
(SPLITKV_K_PLAN, SPLITKV_K_FWD_ATTN, SPLITKV_K_MERGE, SPLITKV_K_BWD_DRAFT, SPLITKV_K_BWD_DQ,
 SPLITKV_K_BWD_DKDV, SPLITKV_K_DQ_REDUCE, SPLITKV_K_ZERO, SPLITKV_K_PROJ) = range(9)


class splitkv_problem(ctypes.Structure):
    _fields_ = [
        ("num_samples", ctypes.c_int32),
        ("cu_ctx", ctypes.c_void_p),
        ("cu_anchor", ctypes.c_void_p),
        ("anchors", ctypes.c_void_p),
        ("total_ctx", ctypes.c_int64),
        ("total_anchors", ctypes.c_int64),
        ("max_ctx", ctypes.c_int32),
        ("B", ctypes.c_int32),
        ("Hq", ctypes.c_int32),
        ("Hkv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("chunk", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("dtype", ctypes.c_int32),
        ("num_workers", ctypes.c_int32),
        ("flags", ctypes.c_int32),
        ("ctx_lo", ctypes.c_void_p),
    ]


class splitkv_stats(ctypes.Structure):
    _fields_ = [
        ("device_status", ctypes.c_int32),
        ("workers", ctypes.c_int32),
        ("fwd_items", ctypes.c_int64),
        ("bwd_items", ctypes.c_int64),
        ("fwd_slots", ctypes.c_int64),
        ("fwd_total_cost", ctypes.c_int64),
        ("bwd_total_cost", ctypes.c_int64),
        ("fwd_lpt_max_load", ctypes.c_int64),
        ("fwd_contig_max_load", ctypes.c_int64),
        ("bwd_lpt_max_load", ctypes.c_int64),
        ("bwd_contig_max_load", ctypes.c_int64),
        ("fwd_lpt_imbalance", ctypes.c_double),
        ("fwd_contig_imbalance", ctypes.c_double),
        ("bwd_lpt_imbalance", ctypes.c_double),
        ("bwd_contig_imbalance", ctypes.c_double),
        ("fwd_tiles", ctypes.c_int64),
        ("dense_tiles", ctypes.c_int64),
        ("work_bytes_used", ctypes.c_size_t),
        ("debug_violations", ctypes.c_int64),
        ("debug_site", ctypes.c_int32),
        ("pad0", ctypes.c_int32),
        ("debug_index", ctypes.c_int64),
    ]

    def as_dict(self) -> Dict[str, object]:
        return {k: getattr(self, k) for k, _ in self._fields_}


_P = ctypes.POINTER(splitkv_problem)
_vp = ctypes.c_void_p
_sz = ctypes.c_size_t

_SIGS = {
    "splitkv_workspace_size": ([_P, ctypes.POINTER(_sz), ctypes.POINTER(_sz)], ctypes.c_int),
    "splitkv_plan": ([_P, _vp, _sz, _vp], ctypes.c_int),
    "splitkv_fwd": ([_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], ctypes.c_int),
    "splitkv_bwd": ([_P, _vp] + [_vp] * 14 + [_sz, _vp], ctypes.c_int),
    "splitkv_plan_stats": ([_P, _vp, ctypes.POINTER(splitkv_stats), _vp], ctypes.c_int),
    "splitkv_plan_export": ([_P, _vp, ctypes.c_int, _vp, _vp, _vp, _vp, ctypes.c_int64,
                             ctypes.POINTER(ctypes.c_int64), _vp], ctypes.c_int),
    "splitkv_device_status": ([_P, _vp, ctypes.POINTER(ctypes.c_int), _vp], ctypes.c_int),
    "splitkv_resolve_workers": ([_P, ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
    "splitkv_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "splitkv_fwd_noalloc": ([_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp], ctypes.c_int),
    "splitkv_profile_enable": ([ctypes.c_int], ctypes.c_int),
    "splitkv_profile_read": ([_vp, _vp, ctypes.c_int], ctypes.c_int),
    "splitkv_kernel_name": ([ctypes.c_int], ctypes.c_char_p),
    "splitkv_busy_read": ([_P, _vp, ctypes.c_int, _vp, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                           _vp], ctypes.c_int),
    "splitkv_proj_in_fwd": ([_P, ctypes.c_int] + [_vp] * 8 + [_vp], ctypes.c_int),
    "splitkv_proj_in_bwd": ([_P, ctypes.c_int] + [_vp] * 11 + [_vp], ctypes.c_int),
    "splitkv_proj_out_fwd": ([_P, ctypes.c_int, _vp, _vp, _vp, _vp], ctypes.c_int),
    "splitkv_proj_out_bwd": ([_P, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp], ctypes.c_int),
    "splitkv_proj_status": ([ctypes.POINTER(ctypes.c_int), ctypes.c_int, _vp], ctypes.c_int),
    "splitkv_selftest_wait_timeout": ([ctypes.POINTER(ctypes.c_int), _vp], ctypes.c_int),
    "splitkv_build_flags": ([], ctypes.c_int),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


def header_functions() -> list:
    """Names of every function declared in include/splitkv.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^(?:int|const char\*)\s+(splitkv_\w+)\(", text, re.M)))


def _ptr(x) -> Optional[int]:
    """Device pointer of a torch tensor, or an int / None passed through."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class SplitKVError(RuntimeError):
    def __init__(self, where: str, status: int):
        super().__init__(f"{where}: {splitkv_status_string(status)} ({status})")
        self.status = status


def _check(where: str, st: int) -> None:
    if st != SPLITKV_OK:
        raise SplitKVError(where, st)


# ---- same-name wrappers ----------------------------------------------------
def splitkv_status_string(status: int) -> str:
    return _lib.splitkv_status_string(int(status)).decode()


def splitkv_build_flags() -> int:
    """SPLITKV_BUILD_DEBUG when the loaded library checks its indices."""
    return _lib.splitkv_build_flags()


def splitkv_kernel_name(kernel_id: int) -> str:
    return _lib.splitkv_kernel_name(int(kernel_id)).decode()


def splitkv_profile_enable(on: bool) -> int:
    return _lib.splitkv_profile_enable(1 if on else 0)


def splitkv_profile_read():
    """Returns (status, {kernel name: (launches, total_ms)})."""
    import numpy as np
    n = SPLITKV_NUM_KERNELS
    launches = np.zeros(n, np.int32)
    ms = np.zeros(n, np.float64)
    st = _lib.splitkv_profile_read(launches.ctypes.data, ms.ctypes.data, n)
    return st, {splitkv_kernel_name(i): (int(launches[i]), float(ms[i])) for i in range(n)}


def splitkv_workspace_size(prob: splitkv_problem):
    """Returns (status, plan_bytes, work_bytes)."""
    pb, wb = _sz(0), _sz(0)
    st = _lib.splitkv_workspace_size(ctypes.byref(prob), ctypes.byref(pb), ctypes.byref(wb))
    return st, pb.value, wb.value


def splitkv_resolve_workers(prob: splitkv_problem):
    w = ctypes.c_int(0)
    st = _lib.splitkv_resolve_workers(ctypes.byref(prob), ctypes.byref(w))
    return st, w.value


def splitkv_plan(prob, plan_ws, plan_bytes: int, stream=None) -> int:
    return _lib.splitkv_plan(ctypes.byref(prob), _ptr(plan_ws), plan_bytes, _stream(stream))


def splitkv_fwd(prob, plan_ws, Q, Kc, Vc, Kd, Vd, O, LSE, work, work_bytes: int,
                stream=None) -> int:
    return _lib.splitkv_fwd(ctypes.byref(prob), _ptr(plan_ws), _ptr(Q), _ptr(Kc), _ptr(Vc),
                            _ptr(Kd), _ptr(Vd), _ptr(O), _ptr(LSE), _ptr(work), work_bytes,
                            _stream(stream))


def splitkv_fwd_noalloc(prob, Q, Kc, Vc, Kd, Vd, O, LSE, stream=None) -> int:
    """Forward without caller workspaces (fixed per-device scratch array)."""
    return _lib.splitkv_fwd_noalloc(ctypes.byref(prob), _ptr(Q), _ptr(Kc), _ptr(Vc), _ptr(Kd),
                                    _ptr(Vd), _ptr(O), _ptr(LSE), _stream(stream))


def splitkv_bwd(prob, plan_ws, Q, Kc, Vc, Kd, Vd, O, LSE, dO, dQ, dKc, dVc, dKd, dVd, work,
                work_bytes: int, stream=None) -> int:
    return _lib.splitkv_bwd(ctypes.byref(prob), _ptr(plan_ws), _ptr(Q), _ptr(Kc), _ptr(Vc),
                            _ptr(Kd), _ptr(Vd), _ptr(O), _ptr(LSE), _ptr(dO), _ptr(dQ),
                            _ptr(dKc), _ptr(dVc), _ptr(dKd), _ptr(dVd), _ptr(work),
                            work_bytes, _stream(stream))


def splitkv_plan_stats(prob, plan_ws, stream=None):
    out = splitkv_stats()
    st = _lib.splitkv_plan_stats(ctypes.byref(prob), _ptr(plan_ws), ctypes.byref(out),
                                 _stream(stream))
    return st, out


def splitkv_busy_read(prob, plan_ws, kernel_id, ns, stream=None):
    """ns: host uint64 numpy array of length >= 2 * workers. Returns (status, workers)."""
    w = ctypes.c_int(0)
    st = _lib.splitkv_busy_read(ctypes.byref(prob), _ptr(plan_ws), int(kernel_id),
                                ns.ctypes.data_as(ctypes.c_void_p), int(ns.size), ctypes.byref(w),
                                _stream(stream))
    return st, w.value


def splitkv_device_status(prob, plan_ws, stream=None):
    s = ctypes.c_int(0)
    st = _lib.splitkv_device_status(ctypes.byref(prob), _ptr(plan_ws), ctypes.byref(s),
                                    _stream(stream))
    return st, s.value


def splitkv_plan_export(prob, plan_ws, kind: int, capacity: int, stream=None):
    """Returns (status, ids, costs, worker, pos) as numpy arrays."""
    import numpy as np
    ids = np.zeros(max(capacity, 1), np.int64)
    costs = np.zeros(max(capacity, 1), np.int64)
    worker = np.zeros(max(capacity, 1), np.int32)
    pos = np.zeros(max(capacity, 1), np.int32)
    count = ctypes.c_int64(0)
    st = _lib.splitkv_plan_export(ctypes.byref(prob), _ptr(plan_ws), int(kind),
                                  ids.ctypes.data, costs.ctypes.data, worker.ctypes.data,
                                  pos.ctypes.data, capacity, ctypes.byref(count),
                                  _stream(stream))
    n = min(count.value, capacity)
    return st, ids[:n], costs[:n], worker[:n], pos[:n]


def splitkv_proj_in_fwd(prob, hidden: int, Xd, Xc, Wqkv, Q, Kc, Vc, Kd, Vd, stream=None) -> int:
    return _lib.splitkv_proj_in_fwd(ctypes.byref(prob), int(hidden), _ptr(Xd), _ptr(Xc),
                                    _ptr(Wqkv), _ptr(Q), _ptr(Kc), _ptr(Vc), _ptr(Kd), _ptr(Vd),
                                    _stream(stream))


def splitkv_proj_in_bwd(prob, hidden: int, Xd, Xc, Wqkv, dQ, dKc, dVc, dKd, dVd, dXd, dXc,
                        dWqkv, stream=None) -> int:
    return _lib.splitkv_proj_in_bwd(ctypes.byref(prob), int(hidden), _ptr(Xd), _ptr(Xc),
                                    _ptr(Wqkv), _ptr(dQ), _ptr(dKc), _ptr(dVc), _ptr(dKd),
                                    _ptr(dVd), _ptr(dXd), _ptr(dXc), _ptr(dWqkv),
                                    _stream(stream))


def splitkv_proj_out_fwd(prob, hidden: int, O, Wo, Y, stream=None) -> int:
    return _lib.splitkv_proj_out_fwd(ctypes.byref(prob), int(hidden), _ptr(O), _ptr(Wo), _ptr(Y),
                                     _stream(stream))


def splitkv_proj_out_bwd(prob, hidden: int, O, Wo, dY, dO, dWo, stream=None) -> int:
    return _lib.splitkv_proj_out_bwd(ctypes.byref(prob), int(hidden), _ptr(O), _ptr(Wo),
                                     _ptr(dY), _ptr(dO), _ptr(dWo), _stream(stream))


def splitkv_proj_status(clear: bool = False, stream=None):
    """Returns (status, device status of the projection kernels)."""
    s = ctypes.c_int(0)
    st = _lib.splitkv_proj_status(ctypes.byref(s), 1 if clear else 0, _stream(stream))
    return st, s.value


def splitkv_selftest_wait_timeout(stream=None):
    """Returns (status, what the probe kernel reported): SPLITKV_ETIMEOUT
    when its unsatisfiable bounded wait gave up as designed."""
    s = ctypes.c_int(-1)
    st = _lib.splitkv_selftest_wait_timeout(ctypes.byref(s), _stream(stream))
    return st, s.value


# ---- convenience wrapper over torch tensors --------------------------------
class SplitKV:
    """One problem (metadata resident on the device) plus its workspaces.

    cu_ctx / cu_anchor / anchors (and ctx_lo, the per-block context offsets,
    which select SPLITKV_FLAG_MASK_CONTEXT_OFFSET): int32 CUDA tensors; the
    host scalars are taken from the caller (no device read). Allocates the two workspaces with
    torch once; ``plan()``, ``forward()`` and ``backward()`` then only enqueue
    kernels on the current torch stream.
    """

    def __init__(self, cu_ctx, cu_anchor, anchors, total_ctx: int, total_anchors: int,
                 max_ctx: int, B: int, Hq: int, Hkv: int, d: int, chunk: int,
                 scale: float, dtype: int = SPLITKV_BF16, num_workers: int = 0,
                 flags: int = 0, ctx_lo=None):
        import torch
        self._keep = (cu_ctx, cu_anchor, anchors, ctx_lo)
        if ctx_lo is not None:
            flags |= SPLITKV_FLAG_MASK_CONTEXT_OFFSET
        self.prob = splitkv_problem(
            num_samples=int(cu_ctx.numel() - 1), cu_ctx=_ptr(cu_ctx), cu_anchor=_ptr(cu_anchor),
            anchors=_ptr(anchors) if anchors.numel() else None, total_ctx=int(total_ctx),
            total_anchors=int(total_anchors), max_ctx=int(max_ctx), B=B, Hq=Hq, Hkv=Hkv, d=d,
            chunk=chunk, scale=float(scale), dtype=dtype, num_workers=num_workers, flags=flags,
            ctx_lo=_ptr(ctx_lo) if ctx_lo is not None and ctx_lo.numel() else None)
        st, self.plan_bytes, self.work_bytes = splitkv_workspace_size(self.prob)
        _check("splitkv_workspace_size", st)
        dev = cu_ctx.device
        self.plan_ws = torch.empty(self.plan_bytes, dtype=torch.uint8, device=dev)
        self.work = torch.empty(self.work_bytes, dtype=torch.uint8, device=dev)

    def _stream(self):
        import torch
        return torch.cuda.current_stream().cuda_stream

    def plan(self) -> None:
        _check("splitkv_plan", splitkv_plan(self.prob, self.plan_ws, self.plan_bytes,
                                            self._stream()))

    def forward(self, Q, Kc, Vc, Kd, Vd, O, LSE) -> None:
        _check("splitkv_fwd", splitkv_fwd(self.prob, self.plan_ws, Q, Kc, Vc, Kd, Vd, O, LSE,
                                          self.work, self.work_bytes, self._stream()))

    def backward(self, Q, Kc, Vc, Kd, Vd, O, LSE, dO, dQ, dKc, dVc, dKd, dVd) -> None:
        _check("splitkv_bwd", splitkv_bwd(self.prob, self.plan_ws, Q, Kc, Vc, Kd, Vd, O, LSE,
                                          dO, dQ, dKc, dVc, dKd, dVd, self.work,
                                          self.work_bytes, self._stream()))

    def stats(self) -> splitkv_stats:
        st, out = splitkv_plan_stats(self.prob, self.plan_ws, self._stream())
        _check("splitkv_plan_stats", st)
        return out

    def busy_ns(self, kernel_id: int):
        """[workers][2] start / end %globaltimer stamps (ns) of the latest launch of
        an attention kernel (SPLITKV_K_FWD_ATTN, _BWD_DQ or _BWD_DKDV)."""
        import numpy as np
        ns = np.zeros(2 * 4096, np.uint64)
        st, w = splitkv_busy_read(self.prob, self.plan_ws, kernel_id, ns, self._stream())
        _check("splitkv_busy_read", st)
        return ns[:2 * w].reshape(w, 2)

    # ---- projections of the drafter layer (splitkv_proj_*) ----
    def proj_in_forward(self, hidden: int, Xd, Xc, Wqkv, Q, Kc, Vc, Kd, Vd) -> None:
        _check("splitkv_proj_in_fwd", splitkv_proj_in_fwd(self.prob, hidden, Xd, Xc, Wqkv, Q, Kc,
                                                          Vc, Kd, Vd, self._stream()))

    def proj_in_backward(self, hidden: int, Xd, Xc, Wqkv, dQ, dKc, dVc, dKd, dVd, dXd, dXc,
                         dWqkv) -> None:
        _check("splitkv_proj_in_bwd", splitkv_proj_in_bwd(self.prob, hidden, Xd, Xc, Wqkv, dQ, dKc,
                                                          dVc, dKd, dVd, dXd, dXc, dWqkv,
                                                          self._stream()))

    def proj_out_forward(self, hidden: int, O, Wo, Y) -> None:
        _check("splitkv_proj_out_fwd", splitkv_proj_out_fwd(self.prob, hidden, O, Wo, Y,
                                                            self._stream()))

    def proj_out_backward(self, hidden: int, O, Wo, dY, dO, dWo) -> None:
        _check("splitkv_proj_out_bwd", splitkv_proj_out_bwd(self.prob, hidden, O, Wo, dY, dO, dWo,
                                                            self._stream()))

    def device_status(self) -> int:
        st, s = splitkv_device_status(self.prob, self.plan_ws, self._stream())
        _check("splitkv_device_status", st)
        return s
