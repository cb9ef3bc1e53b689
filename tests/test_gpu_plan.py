"""Device planner vs the CPU oracle: costs, LPT assignment and queue order
bit-exact; imbalance statistics equal."""
import numpy as np
import pytest
import torch

import block_sparse_cross_gb300 as S
import oracle.plan as OP
import workloads as W
from gpu_case import assert_no_debug_violations

pytestmark = pytest.mark.gpu


def planned(w, workers, flags=0):
    cu_ctx = torch.from_numpy(w.cu_ctx.astype(np.int32)).cuda()
    cu_anchor = torch.from_numpy(w.cu_anchor.astype(np.int32)).cuda()
    anchors = torch.from_numpy(w.anchors.astype(np.int32)).cuda()
    ctx_lo = None if w.ctx_lo is None else torch.from_numpy(w.ctx_lo.astype(np.int32)).cuda()
    kv = S.SplitKV(cu_ctx, cu_anchor, anchors, w.total_ctx, w.total_anchors, w.max_ctx, w.B,
                   w.Hq, w.Hkv, w.d, w.chunk, w.scale, num_workers=workers, flags=flags,
                   ctx_lo=ctx_lo)
    kv.plan()
    torch.cuda.synchronize()
    assert_no_debug_violations(kv)
    return kv


def cpu_lpt_order(items, m):
    ids = [it[0] for it in items]
    costs = [it[-1] for it in items]
    worker_of, queues, loads = OP.lpt(ids, costs, m)
    pos = {}
    for wk, q in enumerate(queues):
        for p, i in enumerate(q):
            pos[i] = p
    order = sorted(range(len(items)), key=lambda i: (-costs[i], ids[i]))
    return (np.array([ids[i] for i in order], np.int64), np.array([costs[i] for i in order], np.int64),
            np.array([worker_of[i] for i in order], np.int32),
            np.array([pos[i] for i in order], np.int32), loads)


def check_plan(w, workers, flags=0):
    kv = planned(w, workers, flags)
    st = kv.stats()
    assert st.device_status == S.SPLITKV_OK
    assert st.workers == workers
    for kind, items in ((0, OP.fwd_items(w)), (1, OP.bwd_items(w))):
        ids, costs, worker, pos, loads = cpu_lpt_order(items, workers)
        s, gi, gc, gw, gp = S.splitkv_plan_export(kv.prob, kv.plan_ws, kind, len(items) + 5)
        assert s == S.SPLITKV_OK
        assert np.array_equal(gi, ids), kind
        assert np.array_equal(gc, costs), kind
        assert np.array_equal(gw, worker), kind
        assert np.array_equal(gp, pos), kind
        imb = OP.imbalance(loads)
        contig = OP.imbalance(OP.contiguous([it[-1] for it in items], workers))
        if kind == 0:
            assert st.fwd_items == len(items) and st.fwd_total_cost == sum(costs)
            assert abs(st.fwd_lpt_imbalance - imb) < 1e-12
            assert abs(st.fwd_contig_imbalance - contig) < 1e-12
        else:
            assert st.bwd_items == len(items) and st.bwd_total_cost == sum(costs)
            assert abs(st.bwd_lpt_imbalance - imb) < 1e-12
            assert abs(st.bwd_contig_imbalance - contig) < 1e-12
    return st


@pytest.mark.parametrize("idx,sweep,workers", [
    (0, 0, 152), (1, 0, 152), (2, 0, 152), (3, 0, 152), (4, 0, 152), (4, 2, 152), (4, 4, 152),
    (1, 0, 64), (3, 0, 8), (0, 0, 5),
])
def test_plan_bit_exact_on_configs(idx, sweep, workers):
    st = check_plan(W.config(idx, sweep), workers)
    if idx >= 1 and workers == 152:
        assert st.fwd_lpt_imbalance < 0.01


@pytest.mark.parametrize("seed", range(8))
def test_plan_bit_exact_fuzz(seed):
    rng = np.random.default_rng(seed)
    S_ = int(rng.integers(1, 6))
    B = int(rng.choice([1, 2, 4, 8, 16]))
    Hkv = int(rng.choice([1, 2, 4]))
    group = int(rng.choice([g for g in (1, 2, 4, 8) if 128 % (B * g) == 0]))
    lengths = rng.integers(1, 3000, size=S_).tolist()
    prompts = [int(rng.integers(0, max(1, L // 2))) for L in lengths]
    counts = [int(rng.integers(0, max(1, min(40, L - B - P + 1)))) if L - B - P + 1 > 0 else 0
              for L, P in zip(lengths, prompts)]
    w = W.custom(seed, lengths, prompts, counts, B=B, Hq=Hkv * group, Hkv=Hkv, d=64,
                 chunk=int(rng.choice([128, 256, 512])))
    workers = Hkv * int(rng.integers(1, 40))
    check_plan(w, workers)


def test_contiguous_mode_loads():
    w = W.config(3)
    kv = planned(w, 152, flags=S.SPLITKV_FLAG_CONTIGUOUS)
    st = kv.stats()
    for kind, items in (("fwd", OP.fwd_items(w)), ("bwd", OP.bwd_items(w))):
        contig = OP.imbalance(OP.contiguous([i[-1] for i in items], 152))
        assert abs(getattr(st, f"{kind}_contig_imbalance") - contig) < 1e-12
        assert getattr(st, f"{kind}_contig_imbalance") > getattr(st, f"{kind}_lpt_imbalance")


def test_skip_accounting():
    w = W.config(2)
    st = planned(w, 152).stats()
    assert 0 < st.fwd_tiles < st.dense_tiles


def expected_queues(w, workers, contiguous):
    """Per-worker queues of (per-head item id, cost) from the CPU oracle:
    LPT queues in assignment order, or the contiguous id ranges."""
    out = []
    for items in (OP.fwd_items(w), OP.bwd_items(w)):
        ids = [it[0] for it in items]
        costs = [it[-1] for it in items]
        if contiguous:
            n = len(items)
            queues = [list(range(wk * n // workers, (wk + 1) * n // workers))
                      for wk in range(workers)]
        else:
            _, queues, _ = OP.lpt(ids, costs, workers)
        q = [(ids[i], costs[i], wk, p) for wk, qq in enumerate(queues) for p, i in enumerate(qq)]
        out.append(np.array(q, np.int64).reshape(-1, 4))
    return out


def check_queues(w, workers, flags=0):
    kv = planned(w, workers, flags)
    assert kv.stats().device_status == S.SPLITKV_OK
    exp = expected_queues(w, workers, bool(flags & S.SPLITKV_FLAG_CONTIGUOUS))
    for kind, e in zip((2, 3), exp):
        s, gi, gc, gw, gp = S.splitkv_plan_export(kv.prob, kv.plan_ws, kind, len(e) + 5)
        assert s == S.SPLITKV_OK
        got = np.stack([gi, gc, gw.astype(np.int64), gp.astype(np.int64)], axis=1)
        assert got.shape == e.shape, (kind, got.shape, e.shape)
        assert np.array_equal(got, e), kind


@pytest.mark.parametrize("contig", [False, True])
@pytest.mark.parametrize("idx,sweep,workers", [
    (0, 0, 152), (1, 0, 152), (3, 0, 152), (3, 1, 152), (3, 2, 152), (4, 0, 152), (4, 4, 152),
    (0, 0, 5),
])
def test_executed_queues_bit_exact(idx, sweep, workers, contig):
    """The queues the kernels walk, LPT or contiguous, match the CPU rule
    entry by entry (item, cost, worker, position)."""
    check_queues(W.config(idx, sweep), workers,
                 S.SPLITKV_FLAG_CONTIGUOUS if contig else 0)


@pytest.mark.parametrize("seed", range(4))
def test_executed_contiguous_queues_fuzz(seed):
    rng = np.random.default_rng(100 + seed)
    S_ = int(rng.integers(1, 6))
    B = int(rng.choice([1, 4, 8, 16]))
    Hkv = int(rng.choice([1, 2, 4]))
    group = int(rng.choice([g for g in (1, 2, 4, 8) if 128 % (B * g) == 0]))
    lengths = rng.integers(1, 3000, size=S_).tolist()
    prompts = [int(rng.integers(0, max(1, L // 2))) for L in lengths]
    counts = [int(rng.integers(0, max(1, min(40, L - B - P + 1)))) if L - B - P + 1 > 0 else 0
              for L, P in zip(lengths, prompts)]
    w = W.custom(100 + seed, lengths, prompts, counts, B=B, Hq=Hkv * group, Hkv=Hkv, d=64,
                 chunk=int(rng.choice([128, 256, 512])))
    workers = Hkv * int(rng.integers(1, 40))
    check_queues(w, workers, S.SPLITKV_FLAG_CONTIGUOUS)
    check_queues(w, workers, 0)
