"""The C ABI: the library loads, exports every declared symbol, and its
host-only entry points validate arguments without touching a GPU."""
import ctypes
import math

import pytest

import block_sparse_cross_gb300 as S


def make_problem(**kw):
    p = dict(num_samples=1, cu_ctx=16, cu_anchor=16, anchors=16, total_ctx=16384,
             total_anchors=64, max_ctx=16384, B=16, Hq=32, Hkv=8, d=128, chunk=1024,
             scale=1 / math.sqrt(128), dtype=S.SPLITKV_BF16, num_workers=0, flags=0)
    p.update(kw)
    return S.splitkv_problem(**p)


def test_every_header_function_is_exported():
    names = S.header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(S._lib, n), n
    assert set(S._SIGS) == set(names)


def test_workspace_size_is_host_only_and_positive():
    st, pb, wb = S.splitkv_workspace_size(make_problem())
    assert st == S.SPLITKV_OK and pb > 0 and wb > 0
    # the work bound covers every (chunk, slab, kv head) partial of 128 rows
    slabs = 64 // 2
    chunks = 16384 // 1024
    assert wb >= slabs * chunks * 8 * 128 * 128 * 4


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), S.SPLITKV_EUNSUPPORTED),
    (dict(B=48), S.SPLITKV_EUNSUPPORTED),            # B*group does not divide 128
    (dict(Hq=30), S.SPLITKV_EUNSUPPORTED),           # Hq % Hkv != 0
    (dict(chunk=1000), S.SPLITKV_EUNSUPPORTED),      # chunk not a multiple of 128
    (dict(dtype=7), S.SPLITKV_EUNSUPPORTED),
    (dict(num_workers=12), S.SPLITKV_EUNSUPPORTED),  # not a multiple of Hkv
    (dict(cu_ctx=None), S.SPLITKV_EINVAL),
    (dict(num_samples=0), S.SPLITKV_EINVAL),
    (dict(scale=0.0), S.SPLITKV_EINVAL),
    (dict(scale=float("nan")), S.SPLITKV_EINVAL),
    (dict(flags=64), S.SPLITKV_EINVAL),
    (dict(total_anchors=-1), S.SPLITKV_EINVAL),
])
def test_workspace_size_rejects_bad_problems(kw, code):
    st, _, _ = S.splitkv_workspace_size(make_problem(**kw))
    assert st == code


def test_null_problem_and_outputs():
    pb = ctypes.c_size_t(0)
    assert S._lib.splitkv_workspace_size(None, ctypes.byref(pb), ctypes.byref(pb)) == S.SPLITKV_EINVAL
    p = make_problem()
    assert S._lib.splitkv_workspace_size(ctypes.byref(p), None, None) == S.SPLITKV_EINVAL


def test_status_strings():
    for code in range(10):
        assert S.splitkv_status_string(code) != "unknown status"
    assert S.splitkv_status_string(1234) == "unknown status"


def test_busy_read_validates_on_the_host():
    # explicit worker count: nothing below touches a device
    import numpy as np
    p = make_problem(num_workers=16)
    dummy = ctypes.c_void_p(1 << 20)  # never dereferenced before the checks
    ns = np.zeros(64, np.uint64)
    w = ctypes.c_int(-1)
    buf = ns.ctypes.data_as(ctypes.c_void_p)
    # only the three attention kernel families have stamps
    for kid in (S.SPLITKV_K_PLAN, S.SPLITKV_K_MERGE, S.SPLITKV_K_DQ_REDUCE, 99, -1):
        assert S._lib.splitkv_busy_read(ctypes.byref(p), dummy, kid, buf, 64, ctypes.byref(w),
                                        None) == S.SPLITKV_EINVAL
    # capacity below 2 * workers: EINVAL, but the worker count is reported
    assert S._lib.splitkv_busy_read(ctypes.byref(p), dummy, S.SPLITKV_K_FWD_ATTN, buf, 31,
                                    ctypes.byref(w), None) == S.SPLITKV_EINVAL
    assert w.value == 16
    assert S._lib.splitkv_busy_read(ctypes.byref(p), None, S.SPLITKV_K_FWD_ATTN, buf, 64,
                                    ctypes.byref(w), None) == S.SPLITKV_EINVAL
    assert S._lib.splitkv_busy_read(ctypes.byref(make_problem(d=96, num_workers=16)), dummy,
                                    S.SPLITKV_K_FWD_ATTN, buf, 64, ctypes.byref(w),
                                    None) == S.SPLITKV_EUNSUPPORTED


def test_projection_entry_points_validate_on_the_host():
    # every call below returns before any CUDA runtime call
    p = make_problem()
    dummy = 1 << 20           # 16-byte aligned, never dereferenced
    odd = (1 << 20) + 8
    u, inval = S.SPLITKV_EUNSUPPORTED, S.SPLITKV_EINVAL
    assert S.splitkv_proj_out_fwd(p, 100, dummy, dummy, dummy) == u       # hidden % 64
    assert S.splitkv_proj_out_fwd(p, 0, dummy, dummy, dummy) == inval     # hidden <= 0
    assert S.splitkv_proj_out_fwd(make_problem(dtype=S.SPLITKV_FP32), 128, dummy, dummy,
                                  dummy) == u
    assert S.splitkv_proj_out_fwd(p, 128, odd, dummy, dummy) == inval      # misaligned
    assert S.splitkv_proj_out_fwd(p, 128, None, dummy, dummy) == inval
    assert S.splitkv_proj_out_bwd(p, 128, dummy, dummy, dummy, dummy, None) == inval
    assert S.splitkv_proj_in_fwd(p, 128, dummy, dummy, None, dummy, dummy, dummy, dummy,
                                 dummy) == inval                           # no weight
    assert S.splitkv_proj_in_fwd(p, 128, dummy, dummy, dummy, dummy, None, dummy, dummy,
                                 dummy) == inval                           # Xc given, no Kc
    assert S.splitkv_proj_in_bwd(p, 128, dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                                 dummy, dummy, dummy, None) == inval       # no dWqkv
    assert S.splitkv_proj_in_bwd(make_problem(d=96), 128, *([dummy] * 11)) == u
    assert S._lib.splitkv_proj_status(None, 0, None) == inval
    assert S.splitkv_kernel_name(S.SPLITKV_K_PROJ) == "projection"


def test_selftest_validates_on_the_host():
    assert S._lib.splitkv_selftest_wait_timeout(None, None) == S.SPLITKV_EINVAL
