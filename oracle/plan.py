"""CPU reference for chunk costs and the LPT assignment.

Test infrastructure only (see the package docstring).

Cost model. The Split-KV abstract (arXiv:2611.05926) prices each context
key/value chunk by its realized attention cost, and the rit.work article on
Split-KV (paragraph on anchor sampling and load imbalance) says the planner
can compute every chunk's cost in advance because it sees all queries. The
realized masked work of chunk [cs, cs + cl) of a sample is the number of
(query, key) pairs of the mask that fall into it:

    cost = sum over anchors a_j > cs of  min(cl, a_j - cs) * B

(block j sees context keys [0, a_j), so it sees min(cl, a_j - cs) keys of
the chunk, for each of its B query rows). With the inclusive mask variant
(context [0, a_j]) the same formula runs on a_j + 1. With per-block context
offsets o_j (block j sees [o_j, a_j)) each block contributes the overlap of
its range with the chunk, max(0, min(cs + cl, a_j) - max(cs, o_j)) * B; with
every o_j = 0 that is the formula above.

Work items. The forward splits each chunk further by kv head g and by
"slab" sigma: ``bps = 128 // (B * group)`` consecutive draft blocks of one
sample, whose B*group*bps = 128 (query, head) rows share K/V. Item cost is
the formula above restricted to the slab's anchors (the formula is additive,
so a chunk's cost is the sum of its items). Item ids enumerate
(sample, chunk, slab, kv head) with the kv head fastest. The backward splits
each sample's keys into 128-key tiles; its items are (sample, tile, kv head)
with the same formula over all of the sample's anchors. Items of cost 0 are
dropped.

LPT (same passages): sort items by cost, most expensive first (ties: lower
item id first), and give each to the worker with the smallest load so far
(ties: lower worker id). The contiguous baseline gives worker w the items
[floor(w*n/m), floor((w+1)*n/m)) in id order.
"""
from __future__ import annotations

import heapq
import itertools
from typing import Dict, List, Sequence, Tuple

import numpy as np

TILE_ROWS = 128   # (query, head) rows per forward work item
KEY_TILE = 128    # keys per backward work item


def chunk_cost(anchors: Sequence[int], cs: int, cl: int, B: int,
               starts: Sequence[int] = None) -> int:
    """Realized masked pairs of key range [cs, cs+cl) for the given anchors
    (ends of the visible context). With ``starts`` (per-block context
    offsets) block j sees [starts[j], anchors[j]) instead of [0, anchors[j]),
    and contributes the overlap of that range with the chunk."""
    if starts is None:
        return int(sum(min(cl, int(a) - cs) * B for a in anchors if int(a) > cs))
    total = 0
    for a, o in zip(anchors, starts):
        total += max(0, min(cs + cl, int(a)) - max(cs, int(o))) * B
    return int(total)


def blocks_per_slab(w) -> int:
    group = w.Hq // w.Hkv
    if TILE_ROWS % (w.B * group) != 0:
        raise ValueError("B * (Hq/Hkv) must divide 128")
    return TILE_ROWS // (w.B * group)


def _sample_anchors(w, s: int) -> np.ndarray:
    """End of the visible context of each block of sample s: a_j, or a_j + 1
    when the context is inclusive ([0, a_j])."""
    anc = np.asarray(w.anchors[int(w.cu_anchor[s]):int(w.cu_anchor[s + 1])], np.int64)
    return anc + 1 if getattr(w, "mask_inclusive", False) else anc


def _sample_starts(w, s: int):
    """Start of the visible context of each block of sample s (None when the
    mask has no per-block context offsets)."""
    lo = getattr(w, "ctx_lo", None)
    if lo is None:
        return None
    return np.asarray(lo[int(w.cu_anchor[s]):int(w.cu_anchor[s + 1])], np.int64)


def fwd_items(w) -> List[Tuple[int, int, int, int, int, int]]:
    """(id, s, c, sigma, g, cost) for every forward item of positive cost."""
    bps = blocks_per_slab(w)
    out = []
    nid = 0
    for s in range(w.num_samples):
        L = int(w.cu_ctx[s + 1] - w.cu_ctx[s])
        anc = _sample_anchors(w, s)
        st = _sample_starts(w, s)
        nch = -(-L // w.chunk)
        nsl = -(-len(anc) // bps)
        for c in range(nch):
            cs = c * w.chunk
            cl = min(w.chunk, L - cs)
            for sg in range(nsl):
                cost = chunk_cost(anc[sg * bps:(sg + 1) * bps], cs, cl, w.B,
                                  None if st is None else st[sg * bps:(sg + 1) * bps])
                for g in range(w.Hkv):
                    if cost > 0:
                        out.append((nid, s, c, sg, g, cost))
                    nid += 1
    return out


def bwd_items(w) -> List[Tuple[int, int, int, int, int]]:
    """(id, s, key tile, g, cost) for every backward item of positive cost."""
    out = []
    nid = 0
    for s in range(w.num_samples):
        L = int(w.cu_ctx[s + 1] - w.cu_ctx[s])
        anc = _sample_anchors(w, s)
        st = _sample_starts(w, s)
        for kt in range(-(-L // KEY_TILE)):
            ks = kt * KEY_TILE
            cost = chunk_cost(anc, ks, min(KEY_TILE, L - ks), w.B, st)
            for g in range(w.Hkv):
                if cost > 0:
                    out.append((nid, s, kt, g, cost))
                nid += 1
    return out


def lpt(ids: Sequence[int], costs: Sequence[int], m: int):
    """Longest-processing-time-first assignment with fixed tie-breaks.

    Returns (worker_of[i], queues[w] as lists of positions i in input order,
    loads[w]). Queues are in assignment order (most expensive first).
    """
    n = len(ids)
    order = sorted(range(n), key=lambda i: (-int(costs[i]), int(ids[i])))
    heap = [(0, wk) for wk in range(m)]
    worker_of = [-1] * n
    queues: List[List[int]] = [[] for _ in range(m)]
    loads = [0] * m
    for i in order:
        load, wk = heapq.heappop(heap)
        worker_of[i] = wk
        queues[wk].append(i)
        loads[wk] = load + int(costs[i])
        heapq.heappush(heap, (loads[wk], wk))
    return worker_of, queues, loads


def lpt_linear(ids: Sequence[int], costs: Sequence[int], m: int):
    """Same rule as ``lpt`` with a linear argmin (independent cross-check)."""
    n = len(ids)
    order = sorted(range(n), key=lambda i: (-int(costs[i]), int(ids[i])))
    loads = [0] * m
    worker_of = [-1] * n
    for i in order:
        best = 0
        for wk in range(1, m):
            if loads[wk] < loads[best]:
                best = wk
        worker_of[i] = best
        loads[best] += int(costs[i])
    return worker_of, loads


def contiguous(costs_in_id_order: Sequence[int], m: int) -> List[int]:
    """Loads of the naive contiguous assignment (items in id order)."""
    n = len(costs_in_id_order)
    loads = []
    for wk in range(m):
        lo, hi = (wk * n) // m, ((wk + 1) * n) // m
        loads.append(int(sum(int(c) for c in costs_in_id_order[lo:hi])))
    return loads


def imbalance(loads: Sequence[int]) -> float:
    """max / mean - 1 over workers (0 for perfectly even loads)."""
    arr = np.asarray(loads, dtype=np.float64)
    mean = arr.mean()
    return float(arr.max() / mean - 1.0) if mean > 0 else 0.0


def optimal_makespan(costs: Sequence[int], m: int) -> int:
    """Exact minimum makespan by enumerating all m**n assignments."""
    c = np.asarray(costs, dtype=np.int64)
    n = len(c)
    if n == 0:
        return 0
    best = None
    for assign in itertools.product(range(m), repeat=n - 1):
        loads = np.zeros(m, np.int64)
        loads[0] = c[0]                     # symmetry: first item on worker 0
        np.add.at(loads, np.asarray(assign, dtype=np.int64), c[1:])
        mk = int(loads.max())
        if best is None or mk < best:
            best = mk
    return int(best)


def plan_summary(w, m: int) -> Dict[str, object]:
    """Costs, LPT and contiguous loads for the forward and backward items."""
    out = {}
    for kind, items in (("fwd", fwd_items(w)), ("bwd", bwd_items(w))):
        ids = [it[0] for it in items]
        costs = [it[-1] for it in items]
        worker_of, queues, loads = lpt(ids, costs, m)
        out[kind] = {
            "ids": ids, "costs": costs, "worker_of": worker_of, "queues": queues,
            "lpt_loads": loads, "contig_loads": contiguous(costs, m),
            "lpt_imbalance": imbalance(loads),
            "contig_imbalance": imbalance(contiguous(costs, m)),
        }
    return out
