"""Error paths: every one is raised on the host or latched in the plan's
status word; none faults, traps or hangs the device."""
import math

import numpy as np
import pytest
import torch

import block_sparse_cross_gb300 as S
import oracle.attention as OA
import workloads as W
from gpu_case import TOL, Case, rel_l2

pytestmark = pytest.mark.gpu


def meta(cu_ctx, cu_anchor, anchors):
    t = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")
    return t(cu_ctx), t(cu_anchor), t(anchors)


@pytest.mark.parametrize("anchors,code", [
    ([5, 3, 9], S.SPLITKV_EMETA),       # not sorted
    ([5, 9, 1000], S.SPLITKV_EMETA),    # beyond L - B
    ([-1, 3, 9], S.SPLITKV_EMETA),      # negative
])
def test_invalid_anchors_latch_status(anchors, code):
    c, a, an = meta([0, 512], [0, 3], anchors)
    kv = S.SplitKV(c, a, an, 512, 3, 512, 16, 8, 2, 64, 256, 0.125)
    kv.plan()
    assert kv.device_status() == code
    # forward / backward on an invalid plan skip their work and keep the status
    nq = 48
    Q = torch.zeros(nq, 8, 64, dtype=torch.bfloat16, device="cuda")
    K = torch.zeros(512, 2, 64, dtype=torch.bfloat16, device="cuda")
    Kd = torch.zeros(nq, 2, 64, dtype=torch.bfloat16, device="cuda")
    O = torch.zeros_like(Q)
    LSE = torch.zeros(8, nq, device="cuda")
    kv.forward(Q, K, K, Kd, Kd, O, LSE)
    assert kv.device_status() == code


def test_inconsistent_totals_latch_status():
    c, a, an = meta([0, 512], [0, 3], [5, 9, 20])
    kv = S.SplitKV(c, a, an, 600, 3, 600, 16, 8, 2, 64, 256, 0.125)  # total_ctx wrong
    kv.plan()
    assert kv.device_status() == S.SPLITKV_EMETA


def test_plan_from_other_problem_is_rejected():
    w = W.config(0)
    case = Case(w).plan()
    other = S.splitkv_problem.from_buffer_copy(case.kv.prob)
    other.chunk = 512
    d = case.dev
    st = S.splitkv_fwd(other, case.kv.plan_ws, d["Q"], d["Kc"], d["Vc"], d["Kd"], d["Vd"],
                       case.O, case.LSE, case.kv.work, case.kv.work_bytes,
                       torch.cuda.current_stream().cuda_stream)
    assert st == S.SPLITKV_OK           # asynchronous: detected on the device
    s, status = S.splitkv_device_status(case.kv.prob, case.kv.plan_ws)
    assert s == S.SPLITKV_OK and status == S.SPLITKV_EPLAN


def test_workspace_too_small_and_null_pointers():
    case = Case(W.config(0)).plan()
    d = case.dev
    kv = case.kv
    assert S.splitkv_fwd(kv.prob, kv.plan_ws, d["Q"], d["Kc"], d["Vc"], d["Kd"], d["Vd"], case.O,
                         case.LSE, kv.work, kv.work_bytes - 1) == S.SPLITKV_EWORKSPACE
    assert S.splitkv_plan(kv.prob, kv.plan_ws, kv.plan_bytes - 1) == S.SPLITKV_EWORKSPACE
    assert S.splitkv_fwd(kv.prob, kv.plan_ws, None, d["Kc"], d["Vc"], d["Kd"], d["Vd"], case.O,
                         case.LSE, kv.work, kv.work_bytes) == S.SPLITKV_EINVAL
    assert S.splitkv_fwd(kv.prob, kv.plan_ws, d["Q"].data_ptr() + 2, d["Kc"], d["Vc"], d["Kd"],
                         d["Vd"], case.O, case.LSE, kv.work, kv.work_bytes) == S.SPLITKV_EINVAL


@pytest.mark.gpu
def test_bounded_wait_times_out_and_the_context_survives():
    """A wait that nothing satisfies gives up after its limit and reports
    SPLITKV_ETIMEOUT (no trap, no hang); the same process then runs the
    whole path correctly."""
    import time
    t0 = time.perf_counter()
    st, s = S.splitkv_selftest_wait_timeout()
    dt = time.perf_counter() - t0
    assert st == S.SPLITKV_OK
    assert s == S.SPLITKV_ETIMEOUT
    assert 0.5 < dt < 30.0
    c = Case(W.config(0)).plan().forward()
    torch.cuda.synchronize()
    assert c.kv.device_status() == S.SPLITKV_OK
    O, LSE = OA.forward(c.w, c.host["Q"], c.host["Kc"], c.host["Vc"], c.host["Kd"], c.host["Vd"])
    assert rel_l2(c.O.float().cpu().numpy(), O) < TOL["O_rel"]
