"""GPU parity of the drafter layer's projections (splitkv_proj_*) against the
float64 oracle (oracle/projection.py), through the C ABI.

Tolerances. Activations and their gradients are stored in bf16: one rounding
of each output element (relative error at most 2^-9, about 1.1e-3 in
rel-L2 for a spread of values) on top of an fp32 accumulation of exact bf16
products, so rel-L2 <= 4e-3. Weight gradients are fp32 sums of up to N_q + T
exact products: rel-L2 <= 1e-4.
"""
import numpy as np
import pytest
import torch

import block_sparse_cross_gb300 as S
import oracle.projection as OP
import workloads as W
from gpu_case import Case, rel_l2

pytestmark = pytest.mark.gpu

BF16_REL = 4e-3
F32_REL = 1e-4


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda().to(torch.bfloat16)


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


class Layer:
    """One workload's problem (plan not needed for the projections) plus the
    layer's draws, on the device and, bf16-rounded, on the host."""

    def __init__(self, w, hidden=None, seed_offset=7):
        self.w = w
        self.H = W.default_hidden(w) if hidden is None else hidden
        t = W.layer_tensors(w, self.H, seed_offset)
        self.host = {k: W.round_to_bf16(v).astype(np.float64) for k, v in t.items()}
        self.dev = {k: _bf16(v) for k, v in t.items()}
        self.case = Case(w)
        self.kv = self.case.kv
        nq, T, w_ = w.n_q, w.total_ctx, w
        bf = dict(dtype=torch.bfloat16, device="cuda")
        self.Q = torch.full((nq, w_.Hq, w_.d), float("nan"), **bf)
        self.Kd = torch.full((nq, w_.Hkv, w_.d), float("nan"), **bf)
        self.Vd = torch.full((nq, w_.Hkv, w_.d), float("nan"), **bf)
        self.Kc = torch.full((T, w_.Hkv, w_.d), float("nan"), **bf)
        self.Vc = torch.full((T, w_.Hkv, w_.d), float("nan"), **bf)

    def in_forward(self, with_ctx=True):
        d = self.dev
        self.kv.proj_in_forward(self.H, d["Xd"], d["Xc"] if with_ctx else None, d["Wqkv"],
                                self.Q, self.Kc if with_ctx else None,
                                self.Vc if with_ctx else None, self.Kd, self.Vd)
        torch.cuda.synchronize()


def _check_status():
    st, s = S.splitkv_proj_status(clear=True)
    assert st == S.SPLITKV_OK and s == S.SPLITKV_OK, S.splitkv_status_string(s)


def _cases():
    return [
        pytest.param(W.config(0), None, id="cfg0-h128"),
        pytest.param(W.config(0), 320, id="cfg0-h320"),       # one full + one partial N tile
        pytest.param(W.custom(31, lengths=[3000, 1700], prompts=[500, 300], counts=[5, 2],
                              B=16, Hq=32, Hkv=8, d=128, chunk=1024), 192,
                     id="ragged-nq112-t4700-h192"),
        pytest.param(W.custom(32, lengths=[40000], prompts=[4000], counts=[6], B=8, Hq=8,
                              Hkv=2, d=64, chunk=1024), 256,
                     id="d64-t40000-h256"),                     # k-split weight gradients
    ]


@pytest.mark.parametrize("w,hidden", _cases())
def test_in_forward_matches_oracle(w, hidden):
    L = Layer(w, hidden)
    L.in_forward()
    _check_status()
    ref = OP.in_forward(w, L.host["Xd"], L.host["Xc"], L.host["Wqkv"])
    for k, t in (("Q", L.Q), ("Kd", L.Kd), ("Vd", L.Vd), ("Kc", L.Kc), ("Vc", L.Vc)):
        got = _np(t)
        assert np.isfinite(got).all(), k
        assert rel_l2(got, ref[k]) < BF16_REL, (k, rel_l2(got, ref[k]))


def test_in_forward_without_context_leaves_kc_vc_untouched():
    w = W.config(0)
    L = Layer(w)
    L.in_forward(with_ctx=False)
    _check_status()
    assert torch.isnan(L.Kc.float()).all() and torch.isnan(L.Vc.float()).all()
    ref = OP.in_forward(w, L.host["Xd"], None, L.host["Wqkv"])
    assert rel_l2(_np(L.Q), ref["Q"]) < BF16_REL


@pytest.mark.parametrize("w,hidden", _cases())
def test_in_backward_matches_oracle(w, hidden):
    L = Layer(w, hidden)
    rng = np.random.Generator(np.random.PCG64(77))
    nq, T = w.n_q, w.total_ctx
    g = {"dQ": (nq, w.Hq, w.d), "dKd": (nq, w.Hkv, w.d), "dVd": (nq, w.Hkv, w.d),
         "dKc": (T, w.Hkv, w.d), "dVc": (T, w.Hkv, w.d)}
    g32 = {k: W.round_to_bf16(rng.standard_normal(s, dtype=np.float32)) for k, s in g.items()}
    gd = {k: _bf16(v) for k, v in g32.items()}
    dXd = torch.empty(nq, L.H, dtype=torch.bfloat16, device="cuda")
    dXc = torch.empty(T, L.H, dtype=torch.bfloat16, device="cuda")
    dW = torch.full(((w.Hq + 2 * w.Hkv) * w.d, L.H), float("nan"), device="cuda")
    d = L.dev
    L.kv.proj_in_backward(L.H, d["Xd"], d["Xc"], d["Wqkv"], gd["dQ"], gd["dKc"], gd["dVc"],
                          gd["dKd"], gd["dVd"], dXd, dXc, dW)
    torch.cuda.synchronize()
    _check_status()
    ref = OP.in_backward(w, L.host["Xd"], L.host["Xc"], L.host["Wqkv"], g32["dQ"], g32["dKd"],
                         g32["dVd"], g32["dKc"], g32["dVc"])
    assert rel_l2(_np(dXd), ref["dXd"]) < BF16_REL
    assert rel_l2(_np(dXc), ref["dXc"]) < BF16_REL
    got = _np(dW)
    assert np.isfinite(got).all()
    qd, kd = w.Hq * w.d, w.Hkv * w.d
    for name, sl in (("dWq", slice(0, qd)), ("dWk", slice(qd, qd + kd)),
                     ("dWv", slice(qd + kd, qd + 2 * kd))):
        assert rel_l2(got[sl], ref["dWqkv"][sl]) < F32_REL, (name, rel_l2(got[sl], ref["dWqkv"][sl]))


@pytest.mark.parametrize("w,hidden", _cases()[:3])
def test_out_forward_backward_match_oracle(w, hidden):
    L = Layer(w, hidden)
    rng = np.random.Generator(np.random.PCG64(78))
    nq = w.n_q
    O32 = W.round_to_bf16(rng.standard_normal((nq, w.Hq, w.d), dtype=np.float32))
    O = _bf16(O32)
    Y = torch.empty(nq, L.H, dtype=torch.bfloat16, device="cuda")
    dO = torch.empty_like(O)
    dWo = torch.full((L.H, w.Hq * w.d), float("nan"), device="cuda")
    L.kv.proj_out_forward(L.H, O, L.dev["Wo"], Y)
    L.kv.proj_out_backward(L.H, O, L.dev["Wo"], L.dev["dY"], dO, dWo)
    torch.cuda.synchronize()
    _check_status()
    assert rel_l2(_np(Y), OP.out_forward(O32, L.host["Wo"])) < BF16_REL
    ref = OP.out_backward(O32, L.host["Wo"], L.host["dY"])
    assert rel_l2(_np(dO), ref["dO"]) < BF16_REL
    assert rel_l2(_np(dWo), ref["dWo"]) < F32_REL


@pytest.mark.parametrize("w,hidden", [
    pytest.param(W.config(0), None, id="cfg0"),
    pytest.param(W.custom(33, lengths=[5000, 2300], prompts=[1000, 200], counts=[4, 3],
                          B=16, Hq=32, Hkv=8, d=128, chunk=1024), 256, id="ragged-h256"),
])
def test_whole_layer_matches_oracle(w, hidden):
    """proj_in -> plan -> attention fwd -> proj_out, then the three backward
    passes, against the oracle differentiated at the device's own rounded
    intermediates (Q, K, V, O as the device stored them)."""
    L = Layer(w, hidden)
    L.in_forward()
    c = L.case
    nq = w.n_q
    O = torch.empty(nq, w.Hq, w.d, dtype=torch.bfloat16, device="cuda")
    LSE = torch.empty(w.Hq, nq, device="cuda")
    L.kv.plan()
    L.kv.forward(L.Q, L.Kc, L.Vc, L.Kd, L.Vd, O, LSE)
    Y = torch.empty(nq, L.H, dtype=torch.bfloat16, device="cuda")
    L.kv.proj_out_forward(L.H, O, L.dev["Wo"], Y)
    dO = torch.empty_like(O)
    dWo = torch.empty(L.H, w.Hq * w.d, device="cuda")
    L.kv.proj_out_backward(L.H, O, L.dev["Wo"], L.dev["dY"], dO, dWo)
    g = {k: torch.empty_like(v) for k, v in
         (("dQ", L.Q), ("dKc", L.Kc), ("dVc", L.Vc), ("dKd", L.Kd), ("dVd", L.Vd))}
    L.kv.backward(L.Q, L.Kc, L.Vc, L.Kd, L.Vd, O, LSE, dO, g["dQ"], g["dKc"], g["dVc"],
                  g["dKd"], g["dVd"])
    dXd = torch.empty(nq, L.H, dtype=torch.bfloat16, device="cuda")
    dXc = torch.empty(w.total_ctx, L.H, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty((w.Hq + 2 * w.Hkv) * w.d, L.H, device="cuda")
    d = L.dev
    L.kv.proj_in_backward(L.H, d["Xd"], d["Xc"], d["Wqkv"], g["dQ"], g["dKc"], g["dVc"],
                          g["dKd"], g["dVd"], dXd, dXc, dW)
    torch.cuda.synchronize()
    _check_status()
    assert L.kv.device_status() == S.SPLITKV_OK
    h = L.host
    at = {"Q": _np(L.Q), "Kc": _np(L.Kc), "Vc": _np(L.Vc), "Kd": _np(L.Kd), "Vd": _np(L.Vd),
          "O": _np(O)}
    fwd = OP.layer_forward(w, h["Xd"], h["Xc"], h["Wqkv"], h["Wo"])
    assert rel_l2(at["Q"], fwd["Q"]) < BF16_REL
    assert rel_l2(_np(Y), OP.out_forward(at["O"], h["Wo"])) < BF16_REL
    assert rel_l2(_np(Y), fwd["Y"]) < 1e-2
    ref = OP.layer_backward(w, h["Xd"], h["Xc"], h["Wqkv"], h["Wo"], h["dY"], fwd=fwd,
                            attn_inputs=at)
    for k, t in (("dXd", dXd), ("dXc", dXc), ("dWqkv", dW), ("dWo", dWo)):
        err = rel_l2(_np(t), ref[k])
        assert err < 1e-2, (k, err)


def test_no_draft_queries_and_no_context():
    """Problems without anchors (only the context projection and its
    gradients; dWq and dWo are zero) and calls without context hidden states."""
    w = W.custom(34, lengths=[2000], prompts=[100], counts=[0], B=16, Hq=32, Hkv=8, d=128,
                 chunk=1024)
    assert w.n_q == 0
    L = Layer(w, 192)
    d = L.dev
    L.kv.proj_in_forward(L.H, None, d["Xc"], d["Wqkv"], None, L.Kc, L.Vc, None, None)
    T = w.total_ctx
    rng = np.random.Generator(np.random.PCG64(79))
    g32 = {k: W.round_to_bf16(rng.standard_normal((T, w.Hkv, w.d), dtype=np.float32))
           for k in ("dKc", "dVc")}
    dXc = torch.empty(T, L.H, dtype=torch.bfloat16, device="cuda")
    dW = torch.full(((w.Hq + 2 * w.Hkv) * w.d, L.H), float("nan"), device="cuda")
    L.kv.proj_in_backward(L.H, None, d["Xc"], d["Wqkv"], None, _bf16(g32["dKc"]),
                          _bf16(g32["dVc"]), None, None, None, dXc, dW)
    dWo = torch.full((L.H, w.Hq * w.d), float("nan"), device="cuda")
    L.kv.proj_out_backward(L.H, None, d["Wo"], None, None, dWo)
    torch.cuda.synchronize()
    _check_status()
    h = L.host
    qd, kd = w.Hq * w.d, w.Hkv * w.d
    Wk, Wv = h["Wqkv"][qd:qd + kd], h["Wqkv"][qd + kd:]
    assert rel_l2(_np(L.Kc).reshape(T, -1), h["Xc"] @ Wk.T) < BF16_REL
    assert rel_l2(_np(L.Vc).reshape(T, -1), h["Xc"] @ Wv.T) < BF16_REL
    gk, gv = g32["dKc"].reshape(T, -1).astype(np.float64), g32["dVc"].reshape(T, -1).astype(np.float64)
    assert rel_l2(_np(dXc), gk @ Wk + gv @ Wv) < BF16_REL
    got = _np(dW)
    assert (got[:qd] == 0).all()
    assert rel_l2(got[qd:qd + kd], gk.T @ h["Xc"]) < F32_REL
    assert rel_l2(got[qd + kd:], gv.T @ h["Xc"]) < F32_REL
    assert (_np(dWo) == 0).all()
