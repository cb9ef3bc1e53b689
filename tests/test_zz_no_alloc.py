"""splitkv_fwd_noalloc against splitkv_fwd, through the C ABI.

splitkv_fwd_noalloc serves callers that may not allocate device memory
where they run attention (framework hooks that own all device memory,
services that freeze allocation after start-up): it keeps the plan and the
forward partials in a fixed per-device array instead of caller workspaces.
This file is collected last so that a failure here leaves every other test
already run.
"""
import numpy as np
import pytest
import torch

import block_sparse_cross_gb300 as S
import oracle.attention as OA
import workloads as W
from gpu_case import TOL, Case, rel_l2

pytestmark = pytest.mark.gpu


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("which", ["tiny", "ragged"])
def test_noalloc_forward_matches_workspace_forward_twice(which):
    if which == "tiny":
        w = W.config(0)
    else:
        w = W.custom(77, [700, 300], [100, 0], [9, 4], B=16, Hq=8, Hkv=2, d=128, chunk=256)
    case = Case(w).plan().forward()
    ref = case.numpy()
    # the workspace forward itself against the float64 oracle
    h = case.host
    O_or, LSE_or = OA.forward(w, h["Q"], h["Kc"], h["Vc"], h["Kd"], h["Vd"])
    assert rel_l2(ref["O"], O_or) <= TOL["O_rel"]
    assert np.abs(ref["O"] - O_or).max() <= TOL["O_abs"]
    assert np.abs(ref["LSE"] - LSE_or).max() <= TOL["LSE_abs"]
    st, pb, wb = S.splitkv_workspace_size(case.kv.prob)
    assert st == S.SPLITKV_OK
    assert (pb + 255) // 256 * 256 + wb <= S.SPLITKV_NOALLOC_SCRATCH_BYTES
    d = case.dev
    for call in range(2):                       # two calls in a row share the array
        O = torch.full_like(case.O, float("nan"))
        LSE = torch.full_like(case.LSE, float("nan"))
        st = S.splitkv_fwd_noalloc(case.kv.prob, d["Q"], d["Kc"], d["Vc"], d["Kd"], d["Vd"],
                                   O, LSE, _stream())
        assert st == S.SPLITKV_OK, S.splitkv_status_string(st)
        torch.cuda.synchronize()
        # the same plan and the same kernels: bit-identical to the workspace call
        assert torch.equal(O, case.O), call
        assert torch.equal(LSE, case.LSE), call
        o = O.float().cpu().numpy()
        assert rel_l2(o, O_or) <= TOL["O_rel"], call
        assert np.abs(LSE.cpu().numpy() - LSE_or).max() <= TOL["LSE_abs"], call


def test_noalloc_rejects_problems_beyond_the_fixed_array():
    w = W.config(0)
    case = Case(w)
    big = S.splitkv_problem.from_buffer_copy(case.kv.prob)
    big.max_ctx = 1 << 28                       # inflates the host-side size bound only
    st, pb, wb = S.splitkv_workspace_size(big)
    assert st == S.SPLITKV_OK and pb + wb > S.SPLITKV_NOALLOC_SCRATCH_BYTES
    d = case.dev
    O = torch.zeros_like(case.O)
    LSE = torch.zeros_like(case.LSE)
    st = S.splitkv_fwd_noalloc(big, d["Q"], d["Kc"], d["Vc"], d["Kd"], d["Vd"], O, LSE, _stream())
    assert st == S.SPLITKV_EWORKSPACE
    torch.cuda.synchronize()
    assert float(O.float().abs().max()) == 0.0  # nothing was launched
