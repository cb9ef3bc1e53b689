"""Pins for the float64 projection oracle, each independent of the oracle's code.

* brute force: explicit per-element sums, with the stacked weight's row
  blocks and the heads' column ranges indexed by hand
* a special case with a closed form: identity weights, so every projection
  is a slice of its input (pins the block boundaries of [Wq; Wk; Wv])
* central finite differences of the scalar losses the backward differentiates
* a library special case for the whole drafter layer: torch float64
  matmuls + scaled_dot_product_attention with an explicit mask, differentiated
  by autograd, against layer_forward / layer_backward
"""
import math

import numpy as np
import pytest
import torch

import oracle.projection as OP
import workloads as W


def tiny(seed=5, B=2, Hq=4, Hkv=2, d=3):
    return W.custom(seed, lengths=[11, 7], prompts=[2, 1], counts=[2, 2], B=B, Hq=Hq, Hkv=Hkv,
                    d=d, chunk=4)


def draws(w, hidden, seed=3):
    rng = np.random.Generator(np.random.PCG64(seed))
    nq, T = w.n_q, w.total_ctx
    rows = (w.Hq + 2 * w.Hkv) * w.d
    return {"Xd": rng.standard_normal((nq, hidden)), "Xc": rng.standard_normal((T, hidden)),
            "Wqkv": rng.standard_normal((rows, hidden)),
            "Wo": rng.standard_normal((hidden, w.Hq * w.d)),
            "dY": rng.standard_normal((nq, hidden))}


def test_in_forward_matches_explicit_sums():
    w = tiny()
    H = 5
    t = draws(w, H)
    out = OP.in_forward(w, t["Xd"], t["Xc"], t["Wqkv"])
    X, Xc, Wt = t["Xd"], t["Xc"], t["Wqkv"]
    qd, kd = w.Hq * w.d, w.Hkv * w.d
    for n in range(w.n_q):
        for h in range(w.Hq):
            for e in range(w.d):
                ref = sum(X[n, k] * Wt[h * w.d + e, k] for k in range(H))
                assert out["Q"][n, h, e] == pytest.approx(ref, abs=1e-12)
        for g in range(w.Hkv):
            for e in range(w.d):
                rk = sum(X[n, k] * Wt[qd + g * w.d + e, k] for k in range(H))
                rv = sum(X[n, k] * Wt[qd + kd + g * w.d + e, k] for k in range(H))
                assert out["Kd"][n, g, e] == pytest.approx(rk, abs=1e-12)
                assert out["Vd"][n, g, e] == pytest.approx(rv, abs=1e-12)
    for t_ in range(w.total_ctx):
        for g in range(w.Hkv):
            for e in range(w.d):
                rk = sum(Xc[t_, k] * Wt[qd + g * w.d + e, k] for k in range(H))
                rv = sum(Xc[t_, k] * Wt[qd + kd + g * w.d + e, k] for k in range(H))
                assert out["Kc"][t_, g, e] == pytest.approx(rk, abs=1e-12)
                assert out["Vc"][t_, g, e] == pytest.approx(rv, abs=1e-12)


def test_out_forward_matches_explicit_sums():
    w = tiny()
    H = 4
    t = draws(w, H)
    rng = np.random.Generator(np.random.PCG64(9))
    O = rng.standard_normal((w.n_q, w.Hq, w.d))
    Y = OP.out_forward(O, t["Wo"])
    for n in range(w.n_q):
        for o in range(H):
            ref = sum(O[n, h, e] * t["Wo"][o, h * w.d + e] for h in range(w.Hq) for e in range(w.d))
            assert Y[n, o] == pytest.approx(ref, abs=1e-12)


def test_identity_weight_slices_the_input():
    # hidden = (Hq + 2 Hkv) d and Wqkv = I: Q, K, V are consecutive column blocks
    w = tiny()
    qd, kd = w.Hq * w.d, w.Hkv * w.d
    H = qd + 2 * kd
    t = draws(w, H)
    out = OP.in_forward(w, t["Xd"], t["Xc"], np.eye(H))
    X, Xc = t["Xd"], t["Xc"]
    np.testing.assert_array_equal(out["Q"].reshape(w.n_q, -1), X[:, :qd])
    np.testing.assert_array_equal(out["Kd"].reshape(w.n_q, -1), X[:, qd:qd + kd])
    np.testing.assert_array_equal(out["Vd"].reshape(w.n_q, -1), X[:, qd + kd:])
    np.testing.assert_array_equal(out["Kc"].reshape(w.total_ctx, -1), Xc[:, qd:qd + kd])
    np.testing.assert_array_equal(out["Vc"].reshape(w.total_ctx, -1), Xc[:, qd + kd:])
    # and the weight gradient of sum(G * outputs) is G^T X, block by block
    rng = np.random.Generator(np.random.PCG64(4))
    g = {k: rng.standard_normal(v.shape) for k, v in out.items()}
    b = OP.in_backward(w, X, Xc, np.eye(H), g["Q"], g["Kd"], g["Vd"], g["Kc"], g["Vc"])
    Gd = np.concatenate([g["Q"].reshape(w.n_q, -1), g["Kd"].reshape(w.n_q, -1),
                         g["Vd"].reshape(w.n_q, -1)], axis=1)
    np.testing.assert_allclose(b["dXd"], Gd, atol=1e-13)
    np.testing.assert_allclose(b["dXc"][:, :qd], 0.0)


def _central(f, x, idx, h=1e-6):
    x0 = x[idx]
    x[idx] = x0 + h
    fp = f()
    x[idx] = x0 - h
    fm = f()
    x[idx] = x0
    return (fp - fm) / (2 * h)


def test_in_backward_matches_central_differences():
    w = tiny()
    H = 6
    t = draws(w, H)
    rng = np.random.Generator(np.random.PCG64(11))
    fwd = OP.in_forward(w, t["Xd"], t["Xc"], t["Wqkv"])
    G = {k: rng.standard_normal(v.shape) for k, v in fwd.items()}

    def loss():
        o = OP.in_forward(w, t["Xd"], t["Xc"], t["Wqkv"])
        return sum(float((G[k] * o[k]).sum()) for k in o)

    b = OP.in_backward(w, t["Xd"], t["Xc"], t["Wqkv"], G["Q"], G["Kd"], G["Vd"], G["Kc"], G["Vc"])
    for name, grad in (("Xd", "dXd"), ("Xc", "dXc"), ("Wqkv", "dWqkv")):
        x = t[name]
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in x.shape)
            fd = _central(loss, x, idx)
            assert b[grad][idx] == pytest.approx(fd, rel=1e-6, abs=1e-8), (name, idx)


def test_out_backward_matches_central_differences():
    w = tiny()
    H = 5
    t = draws(w, H)
    rng = np.random.Generator(np.random.PCG64(12))
    O = rng.standard_normal((w.n_q, w.Hq, w.d))

    def loss():
        return float((t["dY"] * OP.out_forward(O, t["Wo"])).sum())

    b = OP.out_backward(O, t["Wo"], t["dY"])
    for x, grad in ((O, "dO"), (t["Wo"], "dWo")):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in x.shape)
            assert b[grad][idx] == pytest.approx(_central(loss, x, idx), rel=1e-6, abs=1e-8)


def _torch_layer(w, t):
    """The drafter layer in torch float64 (matmuls + SDPA with an explicit
    mask over all keys), differentiated by autograd."""
    nq, T = w.n_q, w.total_ctx
    Hq, Hkv, d = w.Hq, w.Hkv, w.d
    group = Hq // Hkv
    mask = np.zeros((nq, T + nq), bool)
    block_sample = w.sample_of_block()
    for n in range(nq):
        j = n // w.B
        c0 = int(w.cu_ctx[block_sample[j]])
        mask[n, c0:c0 + int(w.anchors[j])] = True
        mask[n, T + j * w.B:T + (j + 1) * w.B] = True
    Xd = torch.tensor(t["Xd"], requires_grad=True)
    Xc = torch.tensor(t["Xc"], requires_grad=True)
    Wqkv = torch.tensor(t["Wqkv"], requires_grad=True)
    Wo = torch.tensor(t["Wo"], requires_grad=True)
    qd, kd = Hq * d, Hkv * d
    Wq, Wk, Wv = Wqkv[:qd], Wqkv[qd:qd + kd], Wqkv[qd + kd:]
    q = (Xd @ Wq.T).reshape(nq, Hq, d).permute(1, 0, 2)
    k = torch.cat([Xc @ Wk.T, Xd @ Wk.T], 0).reshape(T + nq, Hkv, d).permute(1, 0, 2)
    v = torch.cat([Xc @ Wv.T, Xd @ Wv.T], 0).reshape(T + nq, Hkv, d).permute(1, 0, 2)
    k = k.repeat_interleave(group, 0)
    v = v.repeat_interleave(group, 0)
    o = torch.nn.functional.scaled_dot_product_attention(
        q[None], k[None], v[None], attn_mask=torch.tensor(mask), scale=w.scale)[0]
    Y = o.permute(1, 0, 2).reshape(nq, qd) @ Wo.T
    (Y * torch.tensor(t["dY"])).sum().backward()
    return {"Y": Y.detach().numpy(), "dXd": Xd.grad.numpy(), "dXc": Xc.grad.numpy(),
            "dWqkv": Wqkv.grad.numpy(), "dWo": Wo.grad.numpy()}


@pytest.mark.parametrize("Hq,Hkv", [(2, 1), (4, 2)])
def test_layer_matches_torch_autograd(Hq, Hkv):
    w = tiny(Hq=Hq, Hkv=Hkv)
    t = draws(w, 7)
    ref = _torch_layer(w, t)
    fwd = OP.layer_forward(w, t["Xd"], t["Xc"], t["Wqkv"], t["Wo"])
    g = OP.layer_backward(w, t["Xd"], t["Xc"], t["Wqkv"], t["Wo"], t["dY"], fwd=fwd)
    np.testing.assert_allclose(fwd["Y"], ref["Y"], rtol=1e-11, atol=1e-11)
    for k in ("dXd", "dXc", "dWqkv", "dWo"):
        np.testing.assert_allclose(g[k], ref[k], rtol=1e-10, atol=1e-10, err_msg=k)


def test_layer_on_the_tiny_config_matches_torch_autograd():
    # the 64-query, 1024-key workload with its default width (Hq d = 128)
    w = W.config(0)
    t = {k: np.asarray(v, np.float64) for k, v in W.layer_tensors(w).items()}
    ref = _torch_layer(w, t)
    g = OP.layer_backward(w, t["Xd"], t["Xc"], t["Wqkv"], t["Wo"], t["dY"])
    for k in ("dXd", "dXc", "dWqkv", "dWo"):
        np.testing.assert_allclose(g[k], ref[k], rtol=1e-9, atol=1e-9, err_msg=k)


def test_without_context_hidden_states():
    w = tiny()
    t = draws(w, 4)
    out = OP.in_forward(w, t["Xd"], None, t["Wqkv"])
    assert set(out) == {"Q", "Kd", "Vd"}
    rng = np.random.Generator(np.random.PCG64(2))
    g = {k: rng.standard_normal(v.shape) for k, v in out.items()}
    b = OP.in_backward(w, t["Xd"], None, t["Wqkv"], g["Q"], g["Kd"], g["Vd"])
    assert "dXc" not in b and b["dWqkv"].shape == t["Wqkv"].shape


def test_layer_tensor_draws_are_seeded_and_scaled():
    w = W.config(1)
    a = W.layer_tensors(w, hidden=256, seed_offset=7)
    b = W.layer_tensors(w, hidden=256, seed_offset=7)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
    assert a["Xd"].shape == (w.n_q, 256) and a["Xc"].shape == (w.total_ctx, 256)
    assert a["Wqkv"].shape == ((w.Hq + 2 * w.Hkv) * w.d, 256)
    assert a["Wo"].shape == (256, w.Hq * w.d)
    # unit-variance projections: std(W) = 1/sqrt(fan-in)
    assert abs(float(a["Wqkv"].std()) * math.sqrt(256) - 1.0) < 0.02
    assert abs(float(a["Wo"].std()) * math.sqrt(w.Hq * w.d) - 1.0) < 0.02
