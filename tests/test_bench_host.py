"""Host-side logic of bench.py (no GPU): the gate that reports a kernel's DRAM
traffic only for the source and workload it was captured on, and the
algorithmic byte and pair counts the roofline figures divide by."""
import math
import os
import re

import numpy as np
import pytest

import bench
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _profile_fields(kernel):
    text = open(os.path.join(ROOT, "profiles", f"{kernel}_ncu.md")).read()
    sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text).group(1)
    work = re.search(r"traffic_workload:\s*(\S+)", text).group(1)
    nbytes = float(re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text).group(1))
    return sha, work, nbytes


def test_traffic_is_reported_only_for_its_source_and_workload():
    sha, work, nbytes = _profile_fields("bwd_dkdv")
    assert nbytes > 0
    assert bench.profile_traffic("bwd_dkdv", sha, work) == nbytes
    other = ("0" if sha[0] != "0" else "1") + sha[1:]
    assert bench.profile_traffic("bwd_dkdv", other, work) is None
    assert bench.profile_traffic("bwd_dkdv", sha, work + "_other") is None
    assert bench.profile_traffic("no_such_kernel", sha, work) is None


def test_kernel_source_sha_is_stable_and_hex():
    a, b = bench.kernel_source_sha(), bench.kernel_source_sha()
    assert a == b and re.fullmatch(r"[0-9a-f]{64}", a)


@pytest.mark.parametrize("spec", [
    ([300, 1000, 129], [0, 100, 10], [3, 9, 2], 16, 8, 2, 128, 256),
    ([1500], [200], [33], 1, 4, 1, 64, 384),
])
def test_row_kernel_bytes_count_every_partial_row_once(spec):
    L, P, A, B, Hq, Hkv, d, chunk = spec
    w = W.custom(11, L, P, A, B=B, Hq=Hq, Hkv=Hkv, d=d, chunk=chunk)
    # count the chunk partial rows block by block, chunk by chunk
    part_rows = 0
    for j in range(w.total_anchors):
        a = int(w.anchors[j])
        for c in range(0, a, chunk):  # chunks that hold at least one key below a_j
            part_rows += B * Hq
    assert part_rows == sum(math.ceil(int(a) / chunk) for a in w.anchors) * B * Hq
    rows = w.n_q * Hq
    rb = bench.row_kernel_bytes(w)
    merge = (part_rows * (d + 1) * 4            # partial O and lse, fp32
             + rows * (2 * d + 2 * d + 4)        # Q read, O written (bf16), LSE written
             + w.total_anchors * Hkv * 2 * B * d * 2)  # the block's draft keys and values
    reduce = part_rows * d * 4 + rows * (4 * d + 2 * d)  # partials, draft term; dQ written
    assert rb == {"merge": merge, "dq_reduce": reduce}


def test_context_pairs_plus_draft_pairs_are_the_masked_pairs():
    w = W.config(1)
    draft = w.total_anchors * w.B * w.B  # every query sees its block's B draft keys
    assert bench.context_pairs(w) + draft == w.masked_pairs()
    # useful FLOP of the step: 14 d per masked pair and head
    assert w.useful_flop(14) == w.Hq * w.d * 14 * w.masked_pairs()
    assert w.useful_flop(12) * 14 == w.useful_flop(14) * 12


def test_sample_flop_of_all_blocks_is_the_step():
    w = W.config(1)
    assert bench.sample_flop(w, np.arange(w.total_anchors)) == w.useful_flop(14)
