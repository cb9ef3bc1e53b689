"""CUDA path vs the float64 oracle, element by element, through the C ABI.

Tolerances (bf16 inputs, fp32 accumulation): O rel-L2 <= 5e-3 and max-abs
<= 2e-2, |dLSE| <= 1e-3, dQ/dK/dV rel-L2 <= 1e-2. The fp32 problem is held to
the same bounds and its achieved error is printed.
"""
import numpy as np
import pytest
import torch

import block_sparse_cross_gb300 as S
import oracle.attention as OA
import workloads as W
from gpu_case import TOL, Case, rel_l2

pytestmark = pytest.mark.gpu
CC = S.SPLITKV_FLAG_CUDA_CORE


def compare_full(case, tag=""):
    w, h = case.w, case.host
    out = case.numpy()
    assert case.status() == S.SPLITKV_OK
    O, LSE = OA.forward(w, h["Q"], h["Kc"], h["Vc"], h["Kd"], h["Vd"])
    g = OA.backward(w, h["Q"], h["Kc"], h["Vc"], h["Kd"], h["Vd"], h["dO"])
    errs = {"O_rel": rel_l2(out["O"], O), "O_abs": float(np.abs(out["O"] - O).max()),
            "LSE_abs": float(np.abs(out["LSE"] - LSE).max())}
    for k in ("dQ", "dKc", "dVc", "dKd", "dVd"):
        errs[k] = rel_l2(out[k], g[k])
    print(tag, {k: f"{v:.2e}" for k, v in errs.items()})
    assert errs["O_rel"] <= TOL["O_rel"], errs
    assert errs["O_abs"] <= TOL["O_abs"], errs
    assert errs["LSE_abs"] <= TOL["LSE_abs"], errs
    for k in ("dQ", "dKc", "dVc", "dKd", "dVd"):
        assert errs[k] <= TOL["grad_rel"], (k, errs)
    return errs


@pytest.mark.parametrize("dtype,flags", [("fp32", 0), ("bf16", CC), ("bf16", 0)])
def test_tiny_config_full(dtype, flags):
    case = Case(W.config(0), dtype=dtype, flags=flags).plan().forward().backward()
    compare_full(case, f"cfg0 {dtype} flags={flags}")


FUZZ = [
    # lengths, prompts, counts, B, Hq, Hkv, d, chunk
    ([300, 1000, 129], [0, 100, 10], [3, 9, 2], 16, 8, 2, 128, 256),
    ([777, 64, 2000], [5, 0, 1500], [7, 0, 30], 4, 8, 8, 64, 128),
    ([1500], [200], [33], 1, 4, 1, 128, 384),
    ([513, 900], [0, 0], [5, 17], 8, 4, 2, 64, 512),
    ([4096, 130], [1000, 0], [21, 3], 16, 32, 8, 128, 1024),
    # one draft block per 128-row slab (B * group = 128), B up to 128
    ([2500, 700], [100, 0], [11, 4], 32, 8, 2, 128, 512),
    ([3000], [500], [6], 128, 2, 2, 64, 1024),
]


@pytest.mark.parametrize("spec", range(len(FUZZ)))
@pytest.mark.parametrize("flags", [CC, 0])
def test_ragged_fuzz_full(spec, flags):
    L, P, A, B, Hq, Hkv, d, chunk = FUZZ[spec]
    w = W.custom(500 + spec, L, P, A, B=B, Hq=Hq, Hkv=Hkv, d=d, chunk=chunk)
    case = Case(w, flags=flags).plan().forward().backward()
    compare_full(case, f"fuzz{spec} flags={flags}")


@pytest.mark.parametrize("flags", [0, CC])
def test_config1_full(flags):
    case = Case(W.config(1), flags=flags).plan().forward().backward()
    compare_full(case, f"cfg1 flags={flags}")


def compare_subset(case, heads, blocks, tag):
    """Rows of (blocks x heads) exactly; dK/dV via a second backward whose dO
    is zero outside the subset (the oracle's restricted loss)."""
    w, h = case.w, case.host
    out = case.numpy()
    O, LSE = OA.forward(w, h["Q"], h["Kc"], h["Vc"], h["Kd"], h["Vd"], blocks=blocks, heads=heads)
    g = OA.backward(w, h["Q"], h["Kc"], h["Vc"], h["Kd"], h["Vd"], h["dO"], blocks=blocks,
                    heads=heads)
    rows = np.concatenate([np.arange(j * w.B, (j + 1) * w.B) for j in blocks])
    sel = np.ix_(rows, heads)
    errs = {"O_rel": rel_l2(out["O"][sel], O[sel]),
            "O_abs": float(np.abs(out["O"][sel] - O[sel]).max()),
            "LSE_abs": float(np.abs(out["LSE"][np.ix_(heads, rows)] - LSE[np.ix_(heads, rows)]).max()),
            "dQ": rel_l2(out["dQ"][sel], g["dQ"][sel])}
    # restricted backward on the device
    mask = torch.zeros(w.n_q, w.Hq, 1, dtype=case.dev["dO"].dtype, device="cuda")
    mask[torch.from_numpy(rows).cuda()[:, None], torch.from_numpy(np.asarray(heads)).cuda()[None, :]] = 1
    case.backward(dO=(case.dev["dO"] * mask).contiguous())
    out2 = case.numpy()
    kvh = sorted(set(int(x) // (w.Hq // w.Hkv) for x in heads))
    for k in ("dKc", "dVc", "dKd", "dVd"):
        errs[k] = rel_l2(out2[k][:, kvh], g[k][:, kvh])
        other = [x for x in range(w.Hkv) if x not in kvh]
        if other:
            assert np.abs(out2[k][:, other]).max() == 0.0, k
    print(tag, {k: f"{v:.2e}" for k, v in errs.items()})
    assert errs["O_rel"] <= TOL["O_rel"] and errs["O_abs"] <= TOL["O_abs"], errs
    assert errs["LSE_abs"] <= TOL["LSE_abs"], errs
    for k in ("dQ", "dKc", "dVc", "dKd", "dVd"):
        assert errs[k] <= TOL["grad_rel"], (k, errs)


@pytest.mark.parametrize("idx,sweep,nh,na", [
    (2, 0, 4, 32), (3, 0, 4, 32), (4, 0, 2, 16), (4, 1, 2, 16), (4, 2, 2, 16), (4, 3, 2, 16),
    (4, 4, 2, 16),
])
def test_large_configs_seeded_subset(idx, sweep, nh, na):
    w = W.config(idx, sweep)
    heads, blocks = W.subset(w, nh, na, seed=w.seed + 7)
    case = Case(w).plan().forward().backward()
    compare_subset(case, heads, blocks, f"{w.name} subset")


def test_deterministic_bitwise():
    w = W.config(1)
    a = Case(w).plan().forward().backward().numpy()
    b = Case(w).plan().forward().backward().numpy()
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_tensor_core_matches_cuda_core_partials():
    """Two independent GPU implementations of the same items agree."""
    w = W.config(1)
    tc = Case(w).plan().forward().numpy()
    cc = Case(w, flags=CC).plan().forward().numpy()
    assert rel_l2(tc["O"], cc["O"]) < 5e-3
    assert np.abs(tc["LSE"] - cc["LSE"]).max() < 1e-3


CONTIG = S.SPLITKV_FLAG_CONTIGUOUS


@pytest.mark.parametrize("which", ["cfg0", "fuzz0", "fuzz4", "fuzz6", "cfg1"])
def test_contiguous_plan_full(which):
    """The same kernels walking the naive contiguous queues give the same
    results as the LPT queues: every item is run exactly once either way."""
    if which == "cfg0":
        w = W.config(0)
    elif which == "cfg1":
        w = W.config(1)
    else:
        spec = int(which[4:])
        L, P, A, B, Hq, Hkv, d, chunk = FUZZ[spec]
        w = W.custom(500 + spec, L, P, A, B=B, Hq=Hq, Hkv=Hkv, d=d, chunk=chunk)
    case = Case(w, flags=CONTIG).plan().forward().backward()
    compare_full(case, f"{which} contiguous")


@pytest.mark.parametrize("idx,sweep,nh,na", [(3, 0, 4, 32), (3, 1, 4, 32), (3, 2, 4, 32),
                                             (4, 0, 2, 16), (4, 2, 2, 16)])
def test_contiguous_plan_large_configs_subset(idx, sweep, nh, na):
    w = W.config(idx, sweep)
    heads, blocks = W.subset(w, nh, na, seed=w.seed + 7)
    case = Case(w, flags=CONTIG).plan().forward().backward()
    compare_subset(case, heads, blocks, f"{w.name} contiguous subset")


def test_config3_full():
    """The packed variable-length batch (8 samples, 4096 queries, 109k keys)
    against the float64 oracle on every row, head and gradient."""
    case = Case(W.config(3)).plan().forward().backward()
    compare_full(case, "cfg3 full")


def test_unseen_keys_get_zero_gradients():
    """Keys past a sample's last anchor (and every key of a sample without
    anchors) are seen by no block: their dK, dV must be written as exact
    zeros, not left as they were (the outputs start poisoned)."""
    B, Hq, Hkv, d = 16, 8, 2, 128
    w0 = W.custom(91, [2000, 640, 1500], [0, 0, 0], [2, 0, 3], B=B, Hq=Hq, Hkv=Hkv, d=d,
                  chunk=256)
    anchors = np.array([100, 300, 20, 700, 900], np.int32)  # sample 0 covers keys < 384 only
    w = W.Workload("unseen", w0.cu_ctx, w0.cu_anchor, anchors, B, Hq, Hkv, d, 256, w0.seed)
    case = Case(w).plan().forward().backward()
    compare_full(case, "unseen keys")
    out = case.numpy()
    for k in ("dKc", "dVc"):
        g = out[k]
        assert np.all(g[384:2000] == 0.0), k          # sample 0 past its last anchor's tile
        assert np.all(g[2000:2640] == 0.0), k         # sample 1 has no anchors
        assert np.all(g[2640 + 1024:] == 0.0), k      # sample 2 past its last anchor's tile
        assert np.abs(g[:300]).max() > 0, k
