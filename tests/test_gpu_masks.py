"""Mask variants (inclusive context, causal draft block, per-block context
offsets) on the GPU against the float64 oracle, and the planner's costs and
queues for them against the CPU LPT."""
import pytest

import block_sparse_cross_gb300 as S
import workloads as W
from gpu_case import Case
from test_gpu_parity import FUZZ, compare_full, compare_subset
from test_gpu_plan import check_plan, check_queues

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


# ---- per-block context offsets ([o_j, a_j) instead of [0, a_j)) -------------
def with_offsets(w, seed, window=None):
    return w.with_ctx_offsets(W.context_offsets(w, seed, window),
                              "_off" if window is None else f"_win{window}")


@pytest.mark.parametrize("inclusive,causal", [(False, False)] + MASKS)
@pytest.mark.parametrize("dtype,flags", [("fp32", 0), ("bf16", CC), ("bf16", 0)])
def test_tiny_config_context_offsets(inclusive, causal, dtype, flags):
    w = with_offsets(W.config(0).with_mask(inclusive, causal), 900)
    case = Case(w, dtype=dtype, flags=flags).plan().forward().backward()
    compare_full(case, f"cfg0 {w.name} {dtype} flags={flags}")


@pytest.mark.parametrize("window", [None, 300])
@pytest.mark.parametrize("spec", [0, 1, 2, 3, 4, 5, 6])
@pytest.mark.parametrize("flags", [CC, 0])
def test_ragged_fuzz_context_offsets(spec, window, flags):
    L, P, A, B, Hq, Hkv, d, chunk = FUZZ[spec]
    w = with_offsets(W.custom(500 + spec, L, P, A, B=B, Hq=Hq, Hkv=Hkv, d=d, chunk=chunk),
                     910 + spec, window)
    case = Case(w, flags=flags).plan().forward().backward()
    compare_full(case, f"fuzz{spec} {w.name} flags={flags}")


@pytest.mark.parametrize("window", [None, 4096])
def test_config1_context_offsets(window):
    w = with_offsets(W.config(1).with_mask(True, True), 920, window)
    case = Case(w).plan().forward().backward()
    compare_full(case, f"cfg1 {w.name}")


@pytest.mark.parametrize("idx,sweep,nh,na,window", [(3, 0, 4, 32, 2048), (2, 0, 4, 32, None),
                                                    (4, 0, 2, 16, 8192)])
def test_large_configs_context_offsets_subset(idx, sweep, nh, na, window):
    w = with_offsets(W.config(idx, sweep), 930 + idx, window)
    heads, blocks = W.subset(w, nh, na, seed=w.seed + 7)
    case = Case(w).plan().forward().backward()
    compare_subset(case, heads, blocks, f"{w.name} subset")


@pytest.mark.parametrize("cfg,workers,window", [(1, 152, None), (3, 152, 2048), (0, 4, None),
                                                (4, 152, 8192)])
def test_context_offset_plan_and_queues_bit_exact(cfg, workers, window):
    w = with_offsets(W.config(cfg), 940 + cfg, window)
    check_plan(w, workers, flags=S.SPLITKV_FLAG_MASK_CONTEXT_OFFSET)
    check_queues(w, workers, S.SPLITKV_FLAG_MASK_CONTEXT_OFFSET)
    check_queues(w, workers, S.SPLITKV_FLAG_MASK_CONTEXT_OFFSET | S.SPLITKV_FLAG_CONTIGUOUS)


def test_context_offsets_leave_interior_tiles_unseen():
    """Blocks whose ranges leave whole 128-key tiles in the middle of the
    sample unseen: those tiles get exact zero gradients (tile-wise zeroing),
    the partial slots the offsets skip are never read (the outputs start
    poisoned), and an empty context (o_j = a_j) leaves the draft keys only."""
    import numpy as np
    w0 = W.custom(95, [2000], [0], [4], B=16, Hq=8, Hkv=2, d=128, chunk=256)
    anchors = np.array([300, 1200, 1500, 1900], np.int32)
    lo = np.array([100, 1000, 1500, 1700], np.int32)   # keys 300..999 unseen; block 2 empty
    w = W.Workload("interior", w0.cu_ctx, w0.cu_anchor, anchors, 16, 8, 2, 128, 256,
                   w0.seed).with_ctx_offsets(lo)
    for flags in (0, CC):
        case = Case(w, flags=flags).plan().forward().backward()
        compare_full(case, f"interior flags={flags}")
        out = case.numpy()
        for k in ("dKc", "dVc"):
            assert np.all(out[k][384:896] == 0.0), k   # whole tiles inside the gap
            assert np.all(out[k][:100] == 0.0), k      # before every range
            assert np.abs(out[k][100:300]).max() > 0, k
