"""Plain float64 projections of the drafter layer around the attention.

Test infrastructure only (see the package docstring).

The Split-KV paper trains diffusion drafters whose draft blocks cross-attend
to the target model's context (arXiv:2611.05926, abstract; the rit.work
article, section "Когда метод меняет инфраструктурный план", names the
drafters that share the pattern). The pages give the attention, not the
layer's projections; the reading taken is the bias-free linear maps of an
attention layer with weights in a linear layer's [out, in] layout, the
context keys/values going through the same key/value weights as the draft
tokens:

    [Q | Kd | Vd] = Xd Wqkv^T        Wqkv = [Wq; Wk; Wv]   ((Hq + 2 Hkv) d rows)
    [Kc | Vc]     = Xc [Wk; Wv]^T
    Y             = O Wo^T

Backward of sum(dY * Y) and of the attention gradients (a linear map
X -> X W^T has input gradient dY W and weight gradient dY^T X):

    dO    = dY Wo                 dWo = dY^T O
    dXd   = dQ Wq + dKd Wk + dVd Wv
    dXc   = dKc Wk + dVc Wv
    dWq   = dQ^T Xd               dWk = dKd^T Xd + dKc^T Xc    dWv likewise

Heads are flattened: a [rows, heads, d] tensor is the [rows, heads * d]
matrix of its rows. Matrix products are numpy float64 matmuls.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

from . import attention


def _f64(x):
    return None if x is None else np.asarray(x, np.float64)


def split_weight(Wqkv, Hq: int, Hkv: int, d: int):
    """(Wq, Wk, Wv) row blocks of the stacked input weight."""
    W = _f64(Wqkv)
    qd, kd = Hq * d, Hkv * d
    assert W.shape[0] == qd + 2 * kd
    return W[:qd], W[qd:qd + kd], W[qd + kd:]


def in_forward(w, Xd, Xc, Wqkv) -> Dict[str, np.ndarray]:
    """Q, Kd, Vd [rows, heads, d] from Xd; Kc, Vc from Xc (if given)."""
    Wq, Wk, Wv = split_weight(Wqkv, w.Hq, w.Hkv, w.d)
    Xd = _f64(Xd)
    n = Xd.shape[0]
    out = {"Q": (Xd @ Wq.T).reshape(n, w.Hq, w.d),
           "Kd": (Xd @ Wk.T).reshape(n, w.Hkv, w.d),
           "Vd": (Xd @ Wv.T).reshape(n, w.Hkv, w.d)}
    if Xc is not None:
        Xc = _f64(Xc)
        t = Xc.shape[0]
        out["Kc"] = (Xc @ Wk.T).reshape(t, w.Hkv, w.d)
        out["Vc"] = (Xc @ Wv.T).reshape(t, w.Hkv, w.d)
    return out


def in_backward(w, Xd, Xc, Wqkv, dQ, dKd, dVd, dKc=None, dVc=None) -> Dict[str, np.ndarray]:
    """dXd, dXc (if Xc is given) and the stacked weight gradient dWqkv."""
    Wq, Wk, Wv = split_weight(Wqkv, w.Hq, w.Hkv, w.d)
    Xd = _f64(Xd)
    n = Xd.shape[0]
    dQ = _f64(dQ).reshape(n, -1)
    dKd = _f64(dKd).reshape(n, -1)
    dVd = _f64(dVd).reshape(n, -1)
    out = {"dXd": dQ @ Wq + dKd @ Wk + dVd @ Wv}
    dWq = dQ.T @ Xd
    dWk = dKd.T @ Xd
    dWv = dVd.T @ Xd
    if Xc is not None:
        Xc = _f64(Xc)
        t = Xc.shape[0]
        dKc = _f64(dKc).reshape(t, -1)
        dVc = _f64(dVc).reshape(t, -1)
        out["dXc"] = dKc @ Wk + dVc @ Wv
        dWk = dWk + dKc.T @ Xc
        dWv = dWv + dVc.T @ Xc
    out["dWqkv"] = np.concatenate([dWq, dWk, dWv], axis=0)
    return out


def out_forward(O, Wo) -> np.ndarray:
    """Y = O Wo^T with O flattened to [rows, heads * d]."""
    O = _f64(O)
    return O.reshape(O.shape[0], -1) @ _f64(Wo).T


def out_backward(O, Wo, dY) -> Dict[str, np.ndarray]:
    """dO (shaped like O) and dWo of the loss sum(dY * Y)."""
    O = _f64(O)
    n = O.shape[0]
    dY = _f64(dY)
    return {"dO": (dY @ _f64(Wo)).reshape(O.shape),
            "dWo": dY.T @ O.reshape(n, -1)}


def layer_forward(w, Xd, Xc, Wqkv, Wo) -> Dict[str, np.ndarray]:
    """The drafter layer: projections, exact masked cross-attention, output
    projection. Returns Y plus every intermediate."""
    p = in_forward(w, Xd, Xc, Wqkv)
    O, LSE = attention.forward(w, p["Q"], p["Kc"], p["Vc"], p["Kd"], p["Vd"])
    p.update({"O": O, "LSE": LSE, "Y": out_forward(O, Wo)})
    return p


def layer_backward(w, Xd, Xc, Wqkv, Wo, dY, fwd: Optional[Dict[str, np.ndarray]] = None,
                   attn_inputs: Optional[Dict[str, np.ndarray]] = None) -> Dict[str, np.ndarray]:
    """Gradients of sum(dY * Y) through the whole layer.

    ``attn_inputs`` optionally replaces the projected Q, Kc, Vc, Kd, Vd and O
    that the attention backward and the output projection's weight gradient
    read (a test passes the values a device computed, rounded as it stored
    them, so both sides differentiate at the same point)."""
    fwd = layer_forward(w, Xd, Xc, Wqkv, Wo) if fwd is None else fwd
    a = dict(fwd)
    if attn_inputs:
        a.update(attn_inputs)
    ob = out_backward(a["O"], Wo, dY)
    g = attention.backward(w, a["Q"], a["Kc"], a["Vc"], a["Kd"], a["Vd"], ob["dO"])
    ib = in_backward(w, Xd, Xc, Wqkv, g["dQ"], g["dKd"], g["dVd"], g["dKc"], g["dVc"])
    out = {"dO": ob["dO"], "dWo": ob["dWo"]}
    out.update(g)
    out.update(ib)
    return out
