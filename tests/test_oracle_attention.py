"""Pins for the float64 attention oracle, each independent of the oracle's code.

* brute force: per-element explicit loops with a mask built from the set rule
* library special case: torch scaled_dot_product_attention (float64, CPU) with
  an explicit boolean mask over all keys, differentiated by autograd
* central finite differences of sum(dO * O)
* closed forms: constant values, a hand-derived row (tests/golden), B=1
  single-query textbook attention via scipy
* invariants: exactness of any KV split merged by log-sum-exp (the property
  the Split-KV pages claim), strict prefix mask, GQA head map
* the mask variants (inclusive context, causal draft block, per-block context
  offsets) through the same brute-force, SDPA, finite-difference and split
  pins, plus their boundary keys and the special cases that reduce to the
  plain mask (every offset 0) or to textbook attention over the draft keys
  alone (every offset at the end of the context)
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special as sps
import torch

import oracle.attention as OA
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f64(t):
    return {k: np.asarray(v, np.float64) for k, v in t.items()}


def tiny_workload(seed=7, B=2, Hq=4, Hkv=2, d=5):
    return W.custom(seed, lengths=[13, 9, 6], prompts=[3, 2, 0], counts=[3, 2, 0],
                    B=B, Hq=Hq, Hkv=Hkv, d=d, chunk=4)


def brute_force_forward(w, Q, Kc, Vc, Kd, Vd):
    """Explicit loops: every (row, key) pair checked against the set rule."""
    nq, Hq, d = Q.shape
    T = Kc.shape[0]
    group = Hq // w.Hkv
    O = np.zeros_like(Q)
    LSE = np.zeros((Hq, nq))
    block_sample = w.sample_of_block()
    for n in range(nq):
        j = n // w.B
        s = block_sample[j]
        a = int(w.anchors[j])
        o = 0 if w.ctx_lo is None else int(w.ctx_lo[j])
        c0, c1 = int(w.cu_ctx[s]), int(w.cu_ctx[s + 1])
        for h in range(Hq):
            g = h // group
            scores, vals = [], []
            for t in range(T):                       # every context row
                k = t - c0
                visible = (c0 <= t < c1 and (k <= a if w.mask_inclusive else k < a)
                           and k >= o)
                if visible:
                    scores.append(w.scale * sum(Q[n, h, x] * Kc[t, g, x] for x in range(d)))
                    vals.append(Vc[t, g])
            for t in range(nq):                      # every draft row
                if t // w.B == j and (not w.mask_causal_block or t % w.B <= n % w.B):
                    scores.append(w.scale * sum(Q[n, h, x] * Kd[t, g, x] for x in range(d)))
                    vals.append(Vd[t, g])
            mx = max(scores)
            e = [math.exp(sc - mx) for sc in scores]
            tot = sum(e)
            LSE[h, n] = mx + math.log(tot)
            for x in range(d):
                O[n, h, x] = sum(ei * v[x] for ei, v in zip(e, vals)) / tot
    return O, LSE


def sdpa_reference(w, t):
    """torch SDPA over all keys with an explicit boolean mask + autograd."""
    nq, Hq, d = t["Q"].shape
    T = t["Kc"].shape[0]
    group = Hq // w.Hkv
    mask = np.zeros((nq, T + nq), bool)
    block_sample = w.sample_of_block()
    for n in range(nq):
        j = n // w.B
        s = block_sample[j]
        c0 = int(w.cu_ctx[s])
        o = 0 if w.ctx_lo is None else int(w.ctx_lo[j])
        mask[n, c0 + o:c0 + int(w.anchors[j]) + (1 if w.mask_inclusive else 0)] = True
        for u in range(w.B):
            if not w.mask_causal_block or u <= n % w.B:
                mask[n, T + j * w.B + u] = True
    q = torch.tensor(t["Q"]).permute(1, 0, 2).requires_grad_(True)
    kc = torch.tensor(t["Kc"]).requires_grad_(True)
    vc = torch.tensor(t["Vc"]).requires_grad_(True)
    kd = torch.tensor(t["Kd"]).requires_grad_(True)
    vd = torch.tensor(t["Vd"]).requires_grad_(True)
    k = torch.cat([kc, kd], 0).permute(1, 0, 2).repeat_interleave(group, 0)
    v = torch.cat([vc, vd], 0).permute(1, 0, 2).repeat_interleave(group, 0)
    m = torch.tensor(mask)
    out = torch.nn.functional.scaled_dot_product_attention(
        q[None], k[None], v[None], attn_mask=m, scale=w.scale)[0]
    scores = (q @ k.transpose(1, 2)) * w.scale
    lse = torch.logsumexp(scores.masked_fill(~m, float("-inf")), dim=-1)
    dO = torch.tensor(t["dO"]).permute(1, 0, 2)
    (out * dO).sum().backward()
    return {
        "O": out.permute(1, 0, 2).detach().numpy(), "LSE": lse.detach().numpy(),
        "dQ": q.grad.permute(1, 0, 2).numpy(), "dKc": kc.grad.numpy(),
        "dVc": vc.grad.numpy(), "dKd": kd.grad.numpy(), "dVd": vd.grad.numpy(),
    }


def test_forward_matches_brute_force_loops():
    w = tiny_workload()
    t = _f64(W.tensors(w))
    O, LSE = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    Ob, LSEb = brute_force_forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-13)
    np.testing.assert_allclose(LSE, LSEb, rtol=0, atol=1e-13)


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (2, 1), (3, 3)])
def test_forward_backward_match_torch_sdpa(Hq, Hkv):
    w = tiny_workload(seed=11, Hq=Hq, Hkv=Hkv)
    t = _f64(W.tensors(w))
    ref = sdpa_reference(w, t)
    O, LSE = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    g = OA.backward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], t["dO"])
    np.testing.assert_allclose(O, ref["O"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, ref["LSE"], rtol=0, atol=1e-12)
    for k in ("dQ", "dKc", "dVc", "dKd", "dVd"):
        np.testing.assert_allclose(g[k], ref[k], rtol=0, atol=1e-12, err_msg=k)


def test_backward_matches_central_differences():
    w = W.custom(3, lengths=[96], prompts=[40], counts=[4], B=8, Hq=2, Hkv=1, d=16, chunk=32)
    t = _f64(W.tensors(w))
    g = OA.backward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], t["dO"])
    rng = np.random.default_rng(0)
    h = 1e-6

    def loss(tt):
        O, _ = OA.forward(w, tt["Q"], tt["Kc"], tt["Vc"], tt["Kd"], tt["Vd"])
        return float((O * tt["dO"]).sum())

    for name, gname in (("Q", "dQ"), ("Kc", "dKc"), ("Vc", "dVc"), ("Kd", "dKd"), ("Vd", "dVd")):
        arr = t[name]
        flat_idx = rng.choice(arr.size, size=12, replace=False)
        if name in ("Kc", "Vc"):  # include rows that some block sees
            flat_idx[:4] = np.arange(4) * w.d * w.Hkv
        for fi in flat_idx:
            idx = np.unravel_index(fi, arr.shape)
            tp = dict(t); tm = dict(t)
            tp[name] = arr.copy(); tp[name][idx] += h
            tm[name] = arr.copy(); tm[name][idx] -= h
            fd = (loss(tp) - loss(tm)) / (2 * h)
            an = g[gname][idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, idx, fd, an)


def test_constant_values_give_constant_output_and_zero_dq_dk():
    w = tiny_workload(seed=5)
    t = _f64(W.tensors(w))
    v = np.array([0.5, -1.25, 2.0, 3.0, -0.75])
    for name in ("Vc", "Vd"):
        t[name][:] = v
    O, _ = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    np.testing.assert_allclose(O, np.broadcast_to(v, O.shape), rtol=0, atol=1e-14)
    g = OA.backward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], t["dO"])
    for k in ("dQ", "dKc", "dKd"):
        assert np.abs(g[k]).max() <= 1e-13, k
    # all-ones values: O = sum of softmax weights = 1 for every row
    for name in ("Vc", "Vd"):
        t[name][:] = 1.0
    O, _ = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    np.testing.assert_allclose(O, 1.0, rtol=0, atol=1e-14)


def test_single_query_block_is_textbook_attention():
    w = W.custom(1, lengths=[40], prompts=[10], counts=[1], B=1, Hq=1, Hkv=1, d=8, chunk=16)
    t = _f64(W.tensors(w))
    a = int(w.anchors[0])
    keys = np.concatenate([t["Kc"][:a, 0], t["Kd"][:1, 0]])
    vals = np.concatenate([t["Vc"][:a, 0], t["Vd"][:1, 0]])
    s = keys @ t["Q"][0, 0] / math.sqrt(8)
    O, LSE = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    np.testing.assert_allclose(O[0, 0], sps.softmax(s) @ vals, rtol=0, atol=1e-13)
    assert abs(LSE[0, 0] - sps.logsumexp(s)) < 1e-13


def test_closed_form_golden():
    with open(os.path.join(GOLDEN, "closed_form_tiny.json")) as f:
        gold = json.load(f)
    w = W.Workload("golden", np.array([0, 3], np.int32), np.array([0, 1], np.int32),
                   np.array([2], np.int32), 1, 1, 1, 1, 2, 0)
    ln2, ln3 = math.log(2), math.log(3)
    t = {"Q": np.array([[[1.0]]]), "Kc": np.array([[[0.0]], [[ln2]], [[99.0]]]),
         "Vc": np.array([[[6.0]], [[12.0]], [[1000.0]]]), "Kd": np.array([[[ln3]]]),
         "Vd": np.array([[[-6.0]]]), "dO": np.array([[[1.0]]])}
    O, LSE = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    g = OA.backward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], t["dO"])
    ex = gold["expected"]
    assert abs(O[0, 0, 0] - ex["O"]) < 1e-14
    assert abs(LSE[0, 0] - math.log(6)) < 1e-14
    assert abs(g["dQ"][0, 0, 0] - (10 / 3 * ln2 - 4 * ln3)) < 1e-14
    np.testing.assert_allclose(g["dKc"][:, 0, 0], ex["dKc"], atol=1e-14)
    np.testing.assert_allclose(g["dKd"][:, 0, 0], ex["dKd"], atol=1e-14)
    np.testing.assert_allclose(g["dVc"][:, 0, 0], ex["dVc"], atol=1e-14)
    np.testing.assert_allclose(g["dVd"][:, 0, 0], ex["dVd"], atol=1e-14)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_any_kv_split_merges_to_unsplit_result(seed):
    """Exactness: local parts over disjoint key ranges + LSE merge == unsplit."""
    w = W.custom(100 + seed, lengths=[300, 170], prompts=[60, 20], counts=[5, 3],
                 B=4, Hq=4, Hkv=2, d=8, chunk=64)
    t = _f64(W.tensors(w))
    O, LSE = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, 300), size=6, replace=False))
    edges = [0, *cuts.tolist(), 300]
    parts = [OA.partial_forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], lo, hi, False)
             for lo, hi in zip(edges[:-1], edges[1:])]
    rng.shuffle(parts)                          # merge order must not matter
    parts.append(OA.partial_forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], 0, 0, True))
    Om, LSEm = OA.merge(parts)
    np.testing.assert_allclose(Om, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSEm, LSE, rtol=0, atol=1e-12)


def test_mask_is_strict_prefix_of_context():
    """Key a_j is invisible to block j, key a_j - 1 is visible."""
    w = W.custom(9, lengths=[50], prompts=[10], counts=[1], B=2, Hq=1, Hkv=1, d=4, chunk=16)
    t = _f64(W.tensors(w))
    a = int(w.anchors[0])
    base, _ = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    t2 = {k: v.copy() for k, v in t.items()}
    t2["Vc"][a] = 1e6                           # first invisible key
    o2, _ = OA.forward(w, t2["Q"], t2["Kc"], t2["Vc"], t2["Kd"], t2["Vd"])
    assert np.array_equal(base, o2)
    t3 = {k: v.copy() for k, v in t.items()}
    t3["Vc"][a - 1] = 1e6                       # last visible key
    o3, _ = OA.forward(w, t3["Q"], t3["Kc"], t3["Vc"], t3["Kd"], t3["Vd"])
    assert np.abs(o3 - base).max() > 1.0


def test_gqa_head_map():
    """Query head h reads kv head h // (Hq/Hkv)."""
    w = W.custom(4, lengths=[30], prompts=[5], counts=[2], B=2, Hq=4, Hkv=2, d=3, chunk=8)
    t = _f64(W.tensors(w))
    for name in ("Vc", "Vd"):
        t[name][:, 0] = 7.0
        t[name][:, 1] = -3.0
    O, _ = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    np.testing.assert_allclose(O[:, :2], 7.0, atol=1e-14)
    np.testing.assert_allclose(O[:, 2:], -3.0, atol=1e-14)


def test_subset_restriction_equals_masked_dO():
    w = tiny_workload(seed=21)
    t = _f64(W.tensors(w))
    heads, blocks = [1, 2], [0, 3]
    g_sub = OA.backward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], t["dO"],
                        blocks=blocks, heads=heads)
    dO = np.zeros_like(t["dO"])
    for j in blocks:
        for h in heads:
            dO[j * w.B:(j + 1) * w.B, h] = t["dO"][j * w.B:(j + 1) * w.B, h]
    g_full = OA.backward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], dO)
    for k in ("dKc", "dVc", "dKd", "dVd"):
        np.testing.assert_allclose(g_sub[k], g_full[k], atol=1e-13, err_msg=k)


MASKS = [(True, False), (False, True), (True, True)]


@pytest.mark.parametrize("inclusive,causal", MASKS)
def test_mask_variants_match_brute_force_loops(inclusive, causal):
    w = tiny_workload(seed=17).with_mask(inclusive, causal)
    t = _f64(W.tensors(w))
    O, LSE = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    Ob, LSEb = brute_force_forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-13)
    np.testing.assert_allclose(LSE, LSEb, rtol=0, atol=1e-13)


@pytest.mark.parametrize("inclusive,causal", MASKS)
def test_mask_variants_match_torch_sdpa(inclusive, causal):
    w = tiny_workload(seed=23, B=3).with_mask(inclusive, causal)
    t = _f64(W.tensors(w))
    ref = sdpa_reference(w, t)
    O, LSE = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    g = OA.backward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], t["dO"])
    np.testing.assert_allclose(O, ref["O"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, ref["LSE"], rtol=0, atol=1e-12)
    for k in ("dQ", "dKc", "dVc", "dKd", "dVd"):
        np.testing.assert_allclose(g[k], ref[k], rtol=0, atol=1e-12, err_msg=k)


def test_mask_variants_backward_matches_central_differences():
    w = W.custom(31, lengths=[80], prompts=[30], counts=[3], B=4, Hq=2, Hkv=1, d=8,
                 chunk=32).with_mask(True, True)
    t = _f64(W.tensors(w))
    g = OA.backward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], t["dO"])
    rng = np.random.default_rng(3)
    h = 1e-6

    def loss(tt):
        O, _ = OA.forward(w, tt["Q"], tt["Kc"], tt["Vc"], tt["Kd"], tt["Vd"])
        return float((O * tt["dO"]).sum())

    for name, gname in (("Q", "dQ"), ("Kc", "dKc"), ("Vc", "dVc"), ("Kd", "dKd"), ("Vd", "dVd")):
        arr = t[name]
        flat_idx = rng.choice(arr.size, size=10, replace=False)
        if name in ("Kc", "Vc"):  # the anchor rows themselves (visible only when inclusive)
            flat_idx[:3] = [int(a) * w.d * w.Hkv for a in w.anchors]
        for fi in flat_idx:
            idx = np.unravel_index(fi, arr.shape)
            tp = dict(t); tm = dict(t)
            tp[name] = arr.copy(); tp[name][idx] += h
            tm[name] = arr.copy(); tm[name][idx] -= h
            fd = (loss(tp) - loss(tm)) / (2 * h)
            assert abs(fd - g[gname][idx]) <= 1e-6 * max(1.0, abs(g[gname][idx])), (name, idx)


@pytest.mark.parametrize("inclusive,causal", MASKS)
def test_mask_variants_any_kv_split_merges_to_unsplit_result(inclusive, causal):
    w = W.custom(140, lengths=[300, 170], prompts=[60, 20], counts=[5, 3], B=4, Hq=4, Hkv=2,
                 d=8, chunk=64).with_mask(inclusive, causal)
    t = _f64(W.tensors(w))
    O, LSE = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    edges = [0, 37, 64, 128, 200, 300]
    parts = [OA.partial_forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], lo, hi, False)
             for lo, hi in zip(edges[:-1], edges[1:])]
    parts.append(OA.partial_forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], 0, 0, True))
    Om, LSEm = OA.merge(parts)
    np.testing.assert_allclose(Om, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSEm, LSE, rtol=0, atol=1e-12)


def test_inclusive_mask_sees_the_anchor_key_and_no_further():
    w = W.custom(9, lengths=[50], prompts=[10], counts=[1], B=2, Hq=1, Hkv=1, d=4,
                 chunk=16).with_mask(True, False)
    t = _f64(W.tensors(w))
    a = int(w.anchors[0])
    base, _ = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    t2 = {k: v.copy() for k, v in t.items()}
    t2["Vc"][a + 1] = 1e6                       # first invisible key
    o2, _ = OA.forward(w, t2["Q"], t2["Kc"], t2["Vc"], t2["Kd"], t2["Vd"])
    assert np.array_equal(base, o2)
    t3 = {k: v.copy() for k, v in t.items()}
    t3["Vc"][a] = 1e6                           # the anchor key is now visible
    o3, _ = OA.forward(w, t3["Q"], t3["Kc"], t3["Vc"], t3["Kd"], t3["Vd"])
    assert np.abs(o3 - base).max() > 1.0


def test_causal_block_first_query_sees_one_draft_key():
    """Query 0 of a causal block sees draft key 0 only; the last query sees all B."""
    w = W.custom(12, lengths=[40], prompts=[8], counts=[1], B=4, Hq=1, Hkv=1, d=4,
                 chunk=16).with_mask(False, True)
    t = _f64(W.tensors(w))
    base, _ = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    t2 = {k: v.copy() for k, v in t.items()}
    t2["Vd"][1:4] = 1e6                         # draft keys 1..3
    o2, _ = OA.forward(w, t2["Q"], t2["Kc"], t2["Vc"], t2["Kd"], t2["Vd"])
    assert np.array_equal(base[0], o2[0])       # query 0: unchanged
    assert np.abs(o2[3] - base[3]).max() > 1.0  # query 3 sees them


# ---- per-block context offsets ---------------------------------------------
OFFSET_MASKS = [(False, False), (True, False), (False, True), (True, True)]


def offset_workload(seed, inclusive=False, causal=False, B=2, Hq=4, Hkv=2, d=5):
    w = tiny_workload(seed=seed, B=B, Hq=Hq, Hkv=Hkv, d=d).with_mask(inclusive, causal)
    return w.with_ctx_offsets(W.context_offsets(w, seed + 1000))


@pytest.mark.parametrize("inclusive,causal", OFFSET_MASKS)
def test_context_offsets_match_brute_force_loops(inclusive, causal):
    w = offset_workload(41, inclusive, causal)
    assert (w.ctx_lo > 0).any()
    t = _f64(W.tensors(w))
    O, LSE = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    Ob, LSEb = brute_force_forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-13)
    np.testing.assert_allclose(LSE, LSEb, rtol=0, atol=1e-13)


@pytest.mark.parametrize("inclusive,causal", OFFSET_MASKS)
def test_context_offsets_match_torch_sdpa(inclusive, causal):
    w = offset_workload(43, inclusive, causal, B=3)
    t = _f64(W.tensors(w))
    ref = sdpa_reference(w, t)
    O, LSE = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    g = OA.backward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], t["dO"])
    np.testing.assert_allclose(O, ref["O"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, ref["LSE"], rtol=0, atol=1e-12)
    for k in ("dQ", "dKc", "dVc", "dKd", "dVd"):
        np.testing.assert_allclose(g[k], ref[k], rtol=0, atol=1e-12, err_msg=k)


def test_context_offsets_backward_matches_central_differences():
    w0 = W.custom(47, lengths=[80], prompts=[30], counts=[3], B=4, Hq=2, Hkv=1, d=8, chunk=32)
    lo = np.array([int(a) // 3 for a in w0.anchors], np.int32)
    w = w0.with_ctx_offsets(lo)
    t = _f64(W.tensors(w))
    g = OA.backward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], t["dO"])
    rng = np.random.default_rng(5)
    h = 1e-6

    def loss(tt):
        O, _ = OA.forward(w, tt["Q"], tt["Kc"], tt["Vc"], tt["Kd"], tt["Vd"])
        return float((O * tt["dO"]).sum())

    for name, gname in (("Q", "dQ"), ("Kc", "dKc"), ("Vc", "dVc"), ("Kd", "dKd"), ("Vd", "dVd")):
        arr = t[name]
        flat_idx = rng.choice(arr.size, size=10, replace=False)
        if name in ("Kc", "Vc"):  # the offset rows (first visible) and the ones just before
            flat_idx[:3] = [int(o) * w.d * w.Hkv for o in lo]
            flat_idx[3:6] = [max(int(o) - 1, 0) * w.d * w.Hkv for o in lo]
        for fi in flat_idx:
            idx = np.unravel_index(fi, arr.shape)
            tp = dict(t); tm = dict(t)
            tp[name] = arr.copy(); tp[name][idx] += h
            tm[name] = arr.copy(); tm[name][idx] -= h
            fd = (loss(tp) - loss(tm)) / (2 * h)
            assert abs(fd - g[gname][idx]) <= 1e-6 * max(1.0, abs(g[gname][idx])), (name, idx)


@pytest.mark.parametrize("inclusive,causal", OFFSET_MASKS)
def test_context_offsets_any_kv_split_merges_to_unsplit_result(inclusive, causal):
    w0 = W.custom(150, lengths=[300, 170], prompts=[60, 20], counts=[5, 3], B=4, Hq=4, Hkv=2,
                  d=8, chunk=64).with_mask(inclusive, causal)
    w = w0.with_ctx_offsets(W.context_offsets(w0, 151))
    t = _f64(W.tensors(w))
    O, LSE = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    edges = [0, 37, 64, 128, 200, 300]
    parts = [OA.partial_forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], lo, hi, False)
             for lo, hi in zip(edges[:-1], edges[1:])]
    parts.append(OA.partial_forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], 0, 0, True))
    Om, LSEm = OA.merge(parts)
    np.testing.assert_allclose(Om, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSEm, LSE, rtol=0, atol=1e-12)


def test_context_offset_key_is_the_first_visible_one():
    w0 = W.custom(9, lengths=[50], prompts=[10], counts=[1], B=2, Hq=1, Hkv=1, d=4, chunk=16)
    o = int(w0.anchors[0]) // 2
    w = w0.with_ctx_offsets(np.array([o], np.int32))
    t = _f64(W.tensors(w))
    base, _ = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    t2 = {k: v.copy() for k, v in t.items()}
    t2["Vc"][o - 1] = 1e6                       # last key before the offset: invisible
    o2, _ = OA.forward(w, t2["Q"], t2["Kc"], t2["Vc"], t2["Kd"], t2["Vd"])
    assert np.array_equal(base, o2)
    t3 = {k: v.copy() for k, v in t.items()}
    t3["Vc"][o] = 1e6                           # the offset key itself: visible
    o3, _ = OA.forward(w, t3["Q"], t3["Kc"], t3["Vc"], t3["Kd"], t3["Vd"])
    assert np.abs(o3 - base).max() > 1.0


def test_zero_offsets_reduce_to_the_plain_mask():
    w = tiny_workload(seed=53)
    wz = w.with_ctx_offsets(np.zeros_like(w.anchors))
    t = _f64(W.tensors(w))
    a = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    b = OA.forward(wz, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_offset_at_the_context_end_leaves_textbook_attention_over_the_draft_keys():
    w0 = W.custom(57, lengths=[60], prompts=[10], counts=[2], B=4, Hq=2, Hkv=1, d=6, chunk=16)
    w = w0.with_ctx_offsets(w0.anchors.copy())   # o_j = a_j: no context key at all
    t = _f64(W.tensors(w))
    O, LSE = OA.forward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"])
    for j in range(2):
        rows = slice(4 * j, 4 * j + 4)
        for h in range(2):
            s = t["Q"][rows, h] @ t["Kd"][rows, 0].T * w.scale
            np.testing.assert_allclose(O[rows, h], sps.softmax(s, axis=1) @ t["Vd"][rows, 0],
                                       rtol=0, atol=1e-13)
            np.testing.assert_allclose(LSE[h, rows], sps.logsumexp(s, axis=1), rtol=0, atol=1e-13)
    g = OA.backward(w, t["Q"], t["Kc"], t["Vc"], t["Kd"], t["Vd"], t["dO"])
    assert np.abs(g["dKc"]).max() == 0.0 and np.abs(g["dVc"]).max() == 0.0
