"""The seeded input generators: determinism and structural constraints."""
import numpy as np
import pytest

import workloads as W


@pytest.mark.parametrize("idx,sweep", [(0, 0), (1, 0), (2, 0), (3, 0), (4, 0), (4, 4)])
def test_config_constraints(idx, sweep):
    w = W.config(idx, sweep)
    again = W.config(idx, sweep)
    assert np.array_equal(w.anchors, again.anchors)
    assert np.array_equal(w.cu_ctx, again.cu_ctx)
    lens = np.diff(w.cu_ctx)
    counts = np.diff(w.cu_anchor)
    for s in range(w.num_samples):
        a = w.anchors[w.cu_anchor[s]:w.cu_anchor[s + 1]]
        assert np.all(np.diff(a) > 0), "anchors strictly increasing"
        assert a.min() >= 0 and a.max() <= lens[s] - w.B
    if idx in (0, 1, 2, 4):
        L = int(lens[0])
        prompt = {0: 512, 1: 4096, 2: 8192}.get(idx, L // 8)
        assert w.anchors.min() >= prompt
    if idx == 3:
        assert w.num_samples == 8 and counts.sum() == 256 and counts.min() >= 1
        assert np.all(lens % 128 == 0) and lens.min() >= 2048 and lens.max() <= 65536
    assert w.n_q == w.B * counts.sum()


def test_tensor_draws_deterministic_and_independent():
    w = W.config(0)
    a = W.tensors(w)
    b = W.tensors(w)
    for k in a:
        assert np.array_equal(a[k], b[k])
    assert a["Q"].shape == (w.n_q, w.Hq, w.d)
    assert a["Kc"].shape == (w.total_ctx, w.Hkv, w.d)
    assert not np.array_equal(a["Q"][:1], a["dO"][:1])


def test_round_to_bf16_ties_to_even():
    # 1 + 2^-8 is halfway between bf16 neighbours 1 and 1 + 2^-7 -> even (1.0)
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 0.0], np.float32)
    y = W.round_to_bf16(x)
    assert y[0] == 1.0
    assert y[1] == np.float32(1.0 + 2 * 2.0 ** -7)
    assert y[2] == -2.5 and y[3] == 0.0
