"""Mask variants (inclusive context, causal draft block) on the GPU against
the float64 oracle, and the planner's inclusive costs against the CPU LPT."""
import pytest

import block_sparse_cross_gb300 as S
import workloads as W
from gpu_case import Case
from test_gpu_parity import FUZZ, compare_full
from test_gpu_plan import check_plan

pytestmark = pytest.mark.gpu
CC = S.SPLITKV_FLAG_CUDA_CORE
MASKS = [(True, False), (False, True), (True, True)]


@pytest.mark.parametrize("inclusive,causal", MASKS)
@pytest.mark.parametrize("dtype,flags", [("fp32", 0), ("bf16", CC), ("bf16", 0)])
def test_tiny_config_mask_variants(inclusive, causal, dtype, flags):
    w = W.config(0).with_mask(inclusive, causal)
    case = Case(w, dtype=dtype, flags=flags).plan().forward().backward()
    compare_full(case, f"cfg0 {w.name} {dtype} flags={flags}")


@pytest.mark.parametrize("inclusive,causal", MASKS)
@pytest.mark.parametrize("spec", [0, 1, 3])
def test_ragged_fuzz_mask_variants(inclusive, causal, spec):
    L, P, A, B, Hq, Hkv, d, chunk = FUZZ[spec]
    w = W.custom(500 + spec, L, P, A, B=B, Hq=Hq, Hkv=Hkv, d=d, chunk=chunk).with_mask(
        inclusive, causal)
    case = Case(w).plan().forward().backward()
    compare_full(case, f"fuzz{spec} {w.name}")


def test_config1_inclusive_causal():
    w = W.config(1).with_mask(True, True)
    case = Case(w).plan().forward().backward()
    compare_full(case, f"cfg1 {w.name}")


@pytest.mark.parametrize("cfg,workers", [(1, 152), (3, 152), (0, 4)])
def test_inclusive_plan_bit_exact(cfg, workers):
    w = W.config(cfg).with_mask(True, False)
    check_plan(w, workers, flags=S.SPLITKV_FLAG_MASK_INCLUSIVE)


def test_anchor_at_the_last_key_is_valid_when_inclusive():
    # a = L - B (the largest anchor) sees keys [0, L - B]: still inside the sample
    import numpy as np
    w = W.custom(77, [300], [0], [2], B=8, Hq=4, Hkv=2, d=64, chunk=128)
    w2 = W.Workload(w.name, w.cu_ctx, w.cu_anchor, np.array([5, 292], np.int32), w.B, w.Hq,
                    w.Hkv, w.d, w.chunk, w.seed).with_mask(True, True)
    case = Case(w2).plan().forward().backward()
    compare_full(case, "last-anchor inclusive causal")
