"""Pins for the CPU cost model and LPT planner (independent of its code).

* chunk cost == brute-force count of mask entries that fall in the chunk
* hand-derived LPT and contiguous assignments (tests/golden)
* Graham's bound LPT <= (4/3 - 1/(3m)) OPT against exhaustive OPT, with the
  textbook tight instances reaching it exactly
* heap LPT == linear-scan LPT; grouping identity used by the device planner
"""
import json
import os

import numpy as np
import pytest

import oracle.plan as OP
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def brute_mask_count(w, s, k0, k1):
    """Count (row, key) pairs of sample s's mask with key in [k0, k1)."""
    B = w.B
    anc = w.anchors[w.cu_anchor[s]:w.cu_anchor[s + 1]]
    los = (np.zeros(len(anc), np.int64) if w.ctx_lo is None
           else w.ctx_lo[w.cu_anchor[s]:w.cu_anchor[s + 1]])
    L = int(w.cu_ctx[s + 1] - w.cu_ctx[s])
    mask = np.zeros((len(anc) * B, L), bool)
    for j, (a, o) in enumerate(zip(anc, los)):
        for k in range(L):  # the set rule, key by key
            if (k < a or (w.mask_inclusive and k == a)) and k >= o:
                mask[j * B:(j + 1) * B, k] = True
    return int(mask[:, k0:k1].sum())


@pytest.mark.parametrize("seed", range(6))
def test_chunk_cost_equals_mask_count(seed):
    rng = np.random.default_rng(seed)
    S = 3
    lengths = rng.integers(40, 400, size=S).tolist()
    prompts = [int(rng.integers(0, L // 2)) for L in lengths]
    B = int(rng.choice([1, 2, 4, 8]))
    counts = [int(rng.integers(0, max(1, min(12, L - B - P + 1)))) for L, P in zip(lengths, prompts)]
    w = W.custom(seed, lengths, prompts, counts, B=B, Hq=2, Hkv=1, d=4,
                 chunk=int(rng.choice([16, 33, 64])))
    for s in range(S):
        anc = w.anchors[w.cu_anchor[s]:w.cu_anchor[s + 1]]
        L = lengths[s]
        for cs in range(0, L, w.chunk):
            cl = min(w.chunk, L - cs)
            assert OP.chunk_cost(anc, cs, cl, B) == brute_mask_count(w, s, cs, cs + cl)


def test_items_partition_the_chunk_costs():
    w = W.custom(5, [700, 260], [100, 30], [9, 4], B=16, Hq=16, Hkv=2, d=8, chunk=128)
    bps = OP.blocks_per_slab(w)
    assert bps == 1
    fwd = OP.fwd_items(w)
    bwd = OP.bwd_items(w)
    total_pairs = sum(brute_mask_count(w, s, 0, int(np.diff(w.cu_ctx)[s])) for s in range(2))
    assert sum(it[-1] for it in fwd) == total_pairs * w.Hkv
    assert sum(it[-1] for it in bwd) == total_pairs * w.Hkv
    ids = [it[0] for it in fwd]
    assert ids == sorted(ids) and len(set(ids)) == len(ids)


def test_lpt_golden_worked_example():
    with open(os.path.join(GOLDEN, "lpt_worked_example.json")) as f:
        gold = json.load(f)
    costs = gold["costs"]
    worker_of, queues, loads = OP.lpt(list(range(len(costs))), costs, gold["m"])
    assert queues == gold["lpt_queues"]
    assert loads == gold["lpt_loads"]
    assert OP.contiguous(costs, gold["m"]) == gold["contiguous_loads"]


@pytest.mark.parametrize("costs,m,lpt_ms,opt_ms", [
    ([3, 3, 2, 2, 2], 2, 7, 6),                  # Graham tight instance, m=2
    ([5, 5, 4, 4, 3, 3, 3], 3, 11, 9),           # Graham tight instance, m=3
    ([4, 4, 4, 4, 4, 4], 3, 8, 8),               # equal jobs: LPT optimal
])
def test_lpt_textbook_instances(costs, m, lpt_ms, opt_ms):
    _, _, loads = OP.lpt(list(range(len(costs))), costs, m)
    assert max(loads) == lpt_ms
    assert OP.optimal_makespan(costs, m) == opt_ms


@pytest.mark.parametrize("seed", range(12))
def test_lpt_within_graham_bound(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(3, 10))
    m = int(rng.integers(2, 5))
    costs = rng.integers(1, 50, size=n).tolist()
    _, _, loads = OP.lpt(list(range(n)), costs, m)
    opt = OP.optimal_makespan(costs, m)
    assert opt <= max(loads)
    assert max(loads) * 3 * m <= (4 * m - 1) * opt      # (4/3 - 1/(3m)) * OPT


@pytest.mark.parametrize("seed", range(5))
def test_heap_and_linear_lpt_agree(seed):
    rng = np.random.default_rng(seed)
    n = 300
    costs = rng.integers(1, 20, size=n).tolist()        # many ties
    ids = rng.permutation(n).tolist()
    a, _, la = OP.lpt(ids, costs, 7)
    b, lb = OP.lpt_linear(ids, costs, 7)
    assert a == b and la == lb


def test_grouped_lpt_identity():
    """Per-head LPT over m = Hkv*m' workers == LPT over base items on m' groups.

    Items of one (sample, chunk, slab) share a cost across kv heads and have
    consecutive ids (kv head fastest); replica g then lands on worker
    Hkv*G + g where G is the base item's group. The device planner relies on it.
    """
    for idx, sweep in ((1, 0), (3, 0), (4, 0)):
        w = W.config(idx, sweep)
        for kind in ("fwd", "bwd"):
            items = OP.fwd_items(w) if kind == "fwd" else OP.bwd_items(w)
            ids = [it[0] for it in items]
            costs = [it[-1] for it in items]
            m_groups = 19
            worker_of, _, _ = OP.lpt(ids, costs, m_groups * w.Hkv)
            base = [(i, it) for i, it in enumerate(items) if it[-2 if kind == "bwd" else 4] == 0]
            bids = [it[0] // w.Hkv for _, it in base]
            bcost = [it[-1] for _, it in base]
            gworker, _, _ = OP.lpt(bids, bcost, m_groups)
            gmap = {bid: gw for bid, gw in zip(bids, gworker)}
            for i, it in enumerate(items):
                g = it[0] % w.Hkv
                assert worker_of[i] == w.Hkv * gmap[it[0] // w.Hkv] + g


def test_imbalance_definition():
    assert OP.imbalance([10, 10, 10]) == 0.0
    assert abs(OP.imbalance([14, 12, 12]) - (14 / (38 / 3) - 1)) < 1e-15


@pytest.mark.parametrize("seed", range(3))
def test_inclusive_items_equal_mask_count(seed):
    """With the inclusive context [0, a_j] the forward items of every chunk and
    the backward items of every key tile still sum to the mask count."""
    rng = np.random.default_rng(50 + seed)
    lengths = rng.integers(60, 400, size=3).tolist()
    prompts = [int(rng.integers(0, L // 2)) for L in lengths]
    counts = [int(rng.integers(1, 8)) for _ in lengths]
    w = W.custom(seed, lengths, prompts, counts, B=4, Hq=8, Hkv=2, d=4,
                 chunk=int(rng.choice([32, 64]))).with_mask(True, False)
    fwd = OP.fwd_items(w)
    bwd = OP.bwd_items(w)
    for s in range(3):
        L = lengths[s]
        for c, cs in enumerate(range(0, L, w.chunk)):
            got = sum(it[-1] for it in fwd if it[1] == s and it[2] == c)
            assert got == brute_mask_count(w, s, cs, min(L, cs + w.chunk)) * w.Hkv
        for kt, ks in enumerate(range(0, L, OP.KEY_TILE)):
            got = sum(it[-1] for it in bwd if it[1] == s and it[2] == kt)
            assert got == brute_mask_count(w, s, ks, min(L, ks + OP.KEY_TILE)) * w.Hkv


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("inclusive", [False, True])
def test_chunk_cost_with_context_offsets_equals_mask_count(seed, inclusive):
    rng = np.random.default_rng(50 + seed)
    S = 3
    lengths = rng.integers(40, 400, size=S).tolist()
    prompts = [int(rng.integers(0, L // 2)) for L in lengths]
    B = int(rng.choice([1, 2, 4, 8]))
    counts = [int(rng.integers(0, max(1, min(12, L - B - P + 1)))) for L, P in zip(lengths, prompts)]
    w0 = W.custom(50 + seed, lengths, prompts, counts, B=B, Hq=2, Hkv=1, d=4,
                  chunk=int(rng.choice([16, 33, 64]))).with_mask(inclusive, False)
    w = w0.with_ctx_offsets(W.context_offsets(w0, 60 + seed))
    for s in range(S):
        sl = slice(int(w.cu_anchor[s]), int(w.cu_anchor[s + 1]))
        ends = w.anchors[sl].astype(np.int64) + (1 if inclusive else 0)
        L = lengths[s]
        for cs in range(0, L, w.chunk):
            cl = min(w.chunk, L - cs)
            got = OP.chunk_cost(ends, cs, cl, B, w.ctx_lo[sl])
            assert got == brute_mask_count(w, s, cs, cs + cl)
    # the items partition the masked pairs
    total = sum(brute_mask_count(w, s, 0, lengths[s]) for s in range(S))
    assert sum(it[-1] for it in OP.fwd_items(w)) == total * w.Hkv
    assert sum(it[-1] for it in OP.bwd_items(w)) == total * w.Hkv
