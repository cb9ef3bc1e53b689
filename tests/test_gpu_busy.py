"""Measured per-CTA busy stamps of the persistent attention kernels
(splitkv_busy_read), against the plan they ran."""
import numpy as np
import pytest

import block_sparse_cross_gb300 as S
import workloads as W
from gpu_case import Case

pytestmark = pytest.mark.gpu

KERNELS = (S.SPLITKV_K_FWD_ATTN, S.SPLITKV_K_BWD_DQ, S.SPLITKV_K_BWD_DKDV)


@pytest.mark.parametrize("cfg,dtype", [(0, "fp32"), (0, "bf16"), (1, "bf16")])
def test_busy_stamps_cover_every_worker(cfg, dtype):
    c = Case(W.config(cfg), dtype=dtype).plan().forward().backward()
    assert c.status() == 0
    st = c.kv.stats()
    spans = {}
    for kid in KERNELS:
        ns = c.kv.busy_ns(kid).astype(np.int64)
        assert ns.shape == (st.workers, 2)
        busy = ns[:, 1] - ns[:, 0]
        assert (busy > 0).all(), kid          # every CTA stamped its start and its end
        assert busy.max() < 10_000_000_000, kid  # < 10 s: stamps of this launch
        spans[kid] = (ns[:, 0].min(), ns[:, 1].max())
    # the launches ran in stream order: forward, then dQ, then dK/dV
    assert spans[KERNELS[0]][1] <= spans[KERNELS[1]][0]
    assert spans[KERNELS[1]][1] <= spans[KERNELS[2]][0]


def test_busy_read_rejects_small_buffers():
    c = Case(W.config(0), dtype="bf16").plan().forward()
    ns = np.zeros(2, np.uint64)
    st, w = S.splitkv_busy_read(c.kv.prob, c.kv.plan_ws, S.SPLITKV_K_FWD_ATTN, ns)
    assert st == S.SPLITKV_EINVAL and w == c.kv.stats().workers
