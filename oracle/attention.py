"""Plain float64 masked cross-attention, forward and analytic backward.

Test infrastructure only (see the package docstring).

Definition (Split-KV paper, arXiv:2611.05926, abstract: draft queries attend
with a block-sparse mask to a longer context). For sample s, draft block j
with anchor a_j (sample-local), query head h and kv head g = h // (Hq/Hkv):

    keys_j   = [ Kc[cu_ctx[s] + k, g] for 0 <= k < a_j ] ++ [ Kd[j*B + t, g] for 0 <= t < B ]
    values_j = the same rows of Vc / Vd
    S        = scale * Q_rows . keys_j^T            (B x (a_j + B))
    LSE      = log sum_k exp(S)                      (natural log)
    P        = exp(S - LSE)
    O        = P . values_j

Backward of the loss sum(dO * O):

    dV_j = P^T dO          dP = dO . values_j^T        D = rowsum(dO * O)
    dS   = P * (dP - D)    dQ = scale * dS . keys_j    dK_j = scale * dS^T . Q_rows

dK_j / dV_j are scattered back onto the Kc/Vc and Kd/Vd rows they came from
and summed over the query heads of the kv group.

Mask variants (the pages say other diffusion drafters -- DFlash, Domino,
DSpark -- share this attention pattern, rit.work article, section "Когда метод
меняет инфраструктурный план"; their exact masks are not given, so two plain
variants are offered, selected by the workload's flags):

    inclusive       the context keys are 0 <= k <= a_j (a_j + 1 keys)
    causal block    query i of block j (row j*B + i) sees draft keys t <= i only
    context offsets block j's context starts at its own offset o_j:
                    o_j <= k < a_j (o_j <= k <= a_j when also inclusive)

Every input holds exactly the values the device sees (the compute-dtype
rounding happens before); slices are upcast to float64 before any
arithmetic, so float32 arrays of bf16-rounded values are accepted as well.
"""
from __future__ import annotations

from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np


def _logsumexp_rows(S: np.ndarray) -> np.ndarray:
    m = S.max(axis=1)
    return m + np.log(np.exp(S - m[:, None]).sum(axis=1))


def _blocks(w) -> Iterable[Tuple[int, int, int]]:
    """(global block j, sample s, anchor a_j) for every draft block."""
    for s in range(w.num_samples):
        for j in range(int(w.cu_anchor[s]), int(w.cu_anchor[s + 1])):
            yield j, s, int(w.anchors[j])


def _ctx_len(w, a: int) -> int:
    """End (exclusive) of the context keys the block with anchor a sees."""
    return a + 1 if getattr(w, "mask_inclusive", False) else a


def _ctx_range(w, j: int, a: int) -> Tuple[int, int]:
    """[lo, hi) of the sample-local context keys block j sees."""
    lo_arr = getattr(w, "ctx_lo", None)
    lo = 0 if lo_arr is None else int(lo_arr[j])
    hi = _ctx_len(w, a)
    return lo, max(lo, hi)


def _mask_draft(w, S: np.ndarray, n_ctx: int) -> np.ndarray:
    """Sets the scores of draft keys a causal block hides to -inf (in place).
    S is B x (n_ctx + B) with the draft keys last."""
    if getattr(w, "mask_causal_block", False):
        B = w.B
        hidden = np.triu(np.ones((B, B), bool), k=1)   # t > i
        S[:, n_ctx:][hidden] = -np.inf
    return S


def _head_sets(w, heads: Optional[Sequence[int]]):
    """Map kv head g -> list of query heads of that group to evaluate."""
    group = w.Hq // w.Hkv
    wanted = range(w.Hq) if heads is None else sorted(int(h) for h in heads)
    out = {}
    for h in wanted:
        out.setdefault(h // group, []).append(h)
    return out


def forward(w, Q, Kc, Vc, Kd, Vd, blocks=None, heads=None):
    """O [N_q, Hq, d] and LSE [Hq, N_q] (float64) by the plain definition.

    ``blocks`` / ``heads`` restrict the evaluation to a subset of draft blocks
    and query heads; rows outside it are left at 0 (O) and NaN (LSE).
    """
    B, scale = w.B, w.scale
    O = np.zeros(Q.shape, np.float64)
    LSE = np.full((w.Hq, Q.shape[0]), np.nan)
    sel = None if blocks is None else set(int(b) for b in blocks)
    hs = _head_sets(w, heads)
    for j, s, a in _blocks(w):
        if sel is not None and j not in sel:
            continue
        c0 = int(w.cu_ctx[s])
        lo, hi = _ctx_range(w, j, a)
        na = hi - lo
        rows = slice(j * B, (j + 1) * B)
        for g, hlist in hs.items():
            keys = np.concatenate([Kc[c0 + lo:c0 + hi, g], Kd[rows, g]], axis=0).astype(np.float64)
            vals = np.concatenate([Vc[c0 + lo:c0 + hi, g], Vd[rows, g]], axis=0).astype(np.float64)
            for h in hlist:
                S = _mask_draft(w, scale * (Q[rows, h].astype(np.float64) @ keys.T), na)
                lse = _logsumexp_rows(S)
                P = np.exp(S - lse[:, None])
                O[rows, h] = P @ vals
                LSE[h, rows] = lse
    return O, LSE


def backward(w, Q, Kc, Vc, Kd, Vd, dO, blocks=None, heads=None):
    """Gradients of sum(dO * O) w.r.t. Q, Kc, Vc, Kd, Vd (float64).

    Restricting ``blocks``/``heads`` gives the gradient of the loss restricted
    to those rows (equivalently: dO set to zero everywhere else).
    """
    B, scale = w.B, w.scale
    dQ = np.zeros(Q.shape, np.float64)
    dKc = np.zeros(Kc.shape, np.float64)
    dVc = np.zeros(Vc.shape, np.float64)
    dKd = np.zeros(Kd.shape, np.float64)
    dVd = np.zeros(Vd.shape, np.float64)
    sel = None if blocks is None else set(int(b) for b in blocks)
    hs = _head_sets(w, heads)
    for j, s, a in _blocks(w):
        if sel is not None and j not in sel:
            continue
        c0 = int(w.cu_ctx[s])
        lo, hi = _ctx_range(w, j, a)
        na = hi - lo
        rows = slice(j * B, (j + 1) * B)
        for g, hlist in hs.items():
            keys = np.concatenate([Kc[c0 + lo:c0 + hi, g], Kd[rows, g]], axis=0).astype(np.float64)
            vals = np.concatenate([Vc[c0 + lo:c0 + hi, g], Vd[rows, g]], axis=0).astype(np.float64)
            dK = np.zeros_like(keys)
            dV = np.zeros_like(vals)
            for h in hlist:
                q = Q[rows, h].astype(np.float64)
                do = dO[rows, h].astype(np.float64)
                S = _mask_draft(w, scale * (q @ keys.T), na)
                lse = _logsumexp_rows(S)
                P = np.exp(S - lse[:, None])
                O = P @ vals
                dV += P.T @ do
                dP = do @ vals.T
                D = (do * O).sum(axis=1)
                dS = P * (dP - D[:, None])
                dQ[rows, h] = scale * (dS @ keys)
                dK += scale * (dS.T @ q)
            dKc[c0 + lo:c0 + hi, g] += dK[:na]
            dVc[c0 + lo:c0 + hi, g] += dV[:na]
            dKd[rows, g] += dK[na:]
            dVd[rows, g] += dV[na:]
    return {"dQ": dQ, "dKc": dKc, "dVc": dVc, "dKd": dKd, "dVd": dVd}


def partial_forward(w, Q, Kc, Vc, Kd, Vd, lo: int, hi: int, draft: bool):
    """Attention of every row restricted to context keys [lo, hi) of its mask.

    Returns (lse [Hq, N_q], O [N_q, Hq, d]) where O is normalised over the
    subset; rows whose subset is empty get lse = -inf and O = 0. With
    ``draft`` the row's own B draft keys are the subset instead (lo/hi
    ignored). This is one "local part" of the split computation.
    """
    B, scale = w.B, w.scale
    group = w.Hq // w.Hkv
    nq = Q.shape[0]
    lse_out = np.full((w.Hq, nq), -np.inf)
    O_out = np.zeros(Q.shape, np.float64)
    for j, s, a in _blocks(w):
        c0 = int(w.cu_ctx[s])
        rows = slice(j * B, (j + 1) * B)
        for h in range(w.Hq):
            g = h // group
            if draft:
                keys, vals = Kd[rows, g], Vd[rows, g]
            else:
                r_lo, r_hi = _ctx_range(w, j, a)
                k0, k1 = max(lo, r_lo), min(hi, r_hi)
                if k1 <= k0:
                    continue
                keys, vals = Kc[c0 + k0:c0 + k1, g], Vc[c0 + k0:c0 + k1, g]
            keys = keys.astype(np.float64)
            S = scale * (Q[rows, h].astype(np.float64) @ keys.T)
            if draft:
                S = _mask_draft(w, S, 0)
            lse = _logsumexp_rows(S)
            lse_out[h, rows] = lse
            O_out[rows, h] = np.exp(S - lse[:, None]) @ vals.astype(np.float64)
    return lse_out, O_out


def merge(partials: List[Tuple[np.ndarray, np.ndarray]]):
    """Exact log-sum-exp merge of (lse, O) partials over disjoint key sets.

    LSE = log sum_c exp(lse_c);  O = sum_c exp(lse_c - LSE) * O_c.
    """
    lses = np.stack([p[0] for p in partials])            # [C, Hq, N_q]
    M = lses.max(axis=0)
    M_safe = np.where(np.isfinite(M), M, 0.0)
    wts = np.exp(lses - M_safe[None])                     # exp(-inf) = 0
    L = wts.sum(axis=0)
    LSE = M_safe + np.log(L)
    O = np.zeros_like(partials[0][1])
    for (lse_c, O_c), wc in zip(partials, wts):
        O += (wc / L).T[:, :, None] * O_c
    return O, LSE
