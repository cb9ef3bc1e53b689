"""Seeded synthetic workloads for anchor-masked block-sparse cross-attention.

This module only draws random inputs: sample lengths, prompt lengths, anchor
positions and the N(0,1) tensors Q, Kc, Vc, Kd, Vd, dO. It holds none of the
attention arithmetic, so both the float64 oracle (``oracle/``) and the CUDA
path (``block_sparse_cross_gb300``) can consume the same draws without sharing
any code of the method.

Shapes follow the drafter-training workload that the Split-KV paper
(arXiv:2611.05926, abstract) describes: a short set of draft queries, built
by anchor sampling, attends with a block-sparse mask to a much longer context.
The pages give no sizes; the five configurations below are the workload set
this library is measured on.

Conventions (all arrays are numpy):
  cu_ctx    int32 [S+1]   offsets of each sample's context rows in Kc/Vc
  cu_anchor int32 [S+1]   offsets of each sample's anchors in ``anchors``
  anchors   int32 [NA]    sample-local anchor positions, sorted ascending
  Q, dO     [N_q, Hq, d]  N_q = B * NA; block j owns rows [j*B, (j+1)*B)
  Kc, Vc    [T, Hkv, d]   T = cu_ctx[S]
  Kd, Vd    [N_q, Hkv, d] keys/values of the draft tokens themselves
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

SEED_BASE = 20261100


@dataclasses.dataclass(frozen=True)
class Workload:
    """One seeded draw of the problem metadata plus its shape parameters."""

    name: str
    cu_ctx: np.ndarray
    cu_anchor: np.ndarray
    anchors: np.ndarray
    B: int
    Hq: int
    Hkv: int
    d: int
    chunk: int
    seed: int
    # mask variants (the default is the strict prefix [0, a_j) plus all B
    # draft keys): inclusive context [0, a_j]; draft keys causal within the
    # block (query i of a block sees draft keys t <= i)
    mask_inclusive: bool = False
    mask_causal_block: bool = False
    # per-block context offsets: block j sees context keys from ctx_lo[j] on
    # (sample-local, 0 <= ctx_lo[j] <= the end of its visible context);
    # None = every block's context starts at key 0
    ctx_lo: Optional[np.ndarray] = None

    @property
    def num_samples(self) -> int:
        return int(self.cu_ctx.shape[0] - 1)

    @property
    def total_ctx(self) -> int:
        return int(self.cu_ctx[-1])

    @property
    def total_anchors(self) -> int:
        return int(self.cu_anchor[-1])

    @property
    def n_q(self) -> int:
        return self.B * self.total_anchors

    @property
    def max_ctx(self) -> int:
        lens = np.diff(self.cu_ctx)
        return int(lens.max()) if lens.size else 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def sample_of_block(self) -> np.ndarray:
        """Sample index of every draft block (global block order)."""
        return np.repeat(np.arange(self.num_samples), np.diff(self.cu_anchor))

    def with_mask(self, inclusive: bool = False, causal_block: bool = False) -> "Workload":
        """The same draw with another mask variant."""
        tag = ("_incl" if inclusive else "") + ("_causal" if causal_block else "")
        return dataclasses.replace(self, name=self.name + tag, mask_inclusive=inclusive,
                                   mask_causal_block=causal_block)

    def with_ctx_offsets(self, ctx_lo: np.ndarray, tag: str = "_off") -> "Workload":
        """The same draw with per-block context offsets ``ctx_lo``."""
        lo = np.asarray(ctx_lo, np.int32)
        if lo.shape != self.anchors.shape:
            raise ValueError("one offset per draft block")
        return dataclasses.replace(self, name=self.name + tag, ctx_lo=lo)

    def context_ends(self) -> np.ndarray:
        """End (exclusive) of every block's visible context: a_j, or a_j + 1
        when inclusive."""
        return self.anchors.astype(np.int64) + (1 if self.mask_inclusive else 0)

    def context_starts(self) -> np.ndarray:
        """Start of every block's visible context (0 without offsets)."""
        if self.ctx_lo is None:
            return np.zeros(self.anchors.shape, np.int64)
        return self.ctx_lo.astype(np.int64)

    def masked_pairs(self) -> int:
        """(query, key) pairs per query head: sum over blocks of B*(a_j + B)
        (B*(a_j + 1) context pairs when inclusive, B*(a_j - o_j) with context
        offsets, B*(B+1)/2 draft pairs when causal within the block)."""
        ctx = np.maximum(self.context_ends() - self.context_starts(), 0)
        draft = self.B * (self.B + 1) // 2 if self.mask_causal_block else self.B * self.B
        return int((self.B * ctx + draft).sum())

    def useful_flop(self, per_pair_per_dim: int = 14) -> int:
        """Useful FLOP of fwd+bwd: Hq * d * c * pairs (c=14: 4 fwd + 10 bwd)."""
        return int(self.Hq * self.d * per_pair_per_dim * self.masked_pairs())


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _uniform_anchors(rng, lo: int, hi: int, count: int) -> np.ndarray:
    """``count`` distinct integers from [lo, hi], sorted."""
    if hi - lo + 1 < count:
        raise ValueError("anchor range smaller than anchor count")
    a = rng.choice(np.arange(lo, hi + 1, dtype=np.int64), size=count, replace=False)
    return np.sort(a).astype(np.int32)


def single_sample(name: str, seed: int, L: int, prompt: int, A: int, B: int,
                  Hq: int, Hkv: int, d: int, chunk: int) -> Workload:
    """One sample; ``A`` anchors drawn without replacement from [prompt, L-B]."""
    rng = _rng(seed)
    anchors = _uniform_anchors(rng, prompt, L - B, A)
    return Workload(name, np.array([0, L], np.int32), np.array([0, A], np.int32),
                    anchors, B, Hq, Hkv, d, chunk, seed)


def _largest_remainder(total: int, weights: np.ndarray, lo: np.ndarray,
                       hi: np.ndarray) -> np.ndarray:
    """Apportion ``total`` integers proportionally to ``weights``.

    Largest-remainder (Hamilton) apportionment, then each share is clamped to
    [lo, hi] and the surplus or deficit is moved one unit at a time between
    the samples with the largest/smallest remainders that still have room.
    """
    w = weights.astype(np.float64)
    quota = total * w / w.sum()
    share = np.floor(quota).astype(np.int64)
    rem = quota - share
    order = np.lexsort((np.arange(len(w)), -rem))  # largest remainder first
    for i in order[: total - int(share.sum())]:
        share[i] += 1
    share = np.clip(share, lo, hi)
    diff = total - int(share.sum())
    while diff != 0:
        if diff > 0:
            cand = [i for i in order if share[i] < hi[i]]
            share[cand[0]] += 1
            diff -= 1
        else:
            cand = [i for i in order[::-1] if share[i] > lo[i]]
            share[cand[0]] -= 1
            diff += 1
    return share


def packed_varlen(name: str, seed: int, S: int = 8, median: int = 16384,
                  sigma: float = 1.0, lmin: int = 2048, lmax: int = 65536,
                  total_anchors: int = 256, B: int = 16, Hq: int = 32,
                  Hkv: int = 8, d: int = 128, chunk: int = 1024) -> Workload:
    """Packed batch of ``S`` samples with Beta(3,1)-skewed anchors.

    Lengths: lognormal around ``median`` (sigma on ln L), rounded to the
    nearest multiple of 128, clamped to [lmin, lmax]. Prompt fraction f_s is
    uniform on [0.1, 0.7], P_s = round(f_s * L_s). The anchor budget is split
    in proportion to response length (L_s - P_s) by largest remainder with
    1 <= A_s <= L_s - B - P_s + 1. Positions a = P + floor(u * (L - B - P + 1))
    with u ~ Beta(3, 1) (density rising toward the response end); duplicates
    are redrawn, then sorted.
    """
    rng = _rng(seed)
    raw = np.exp(rng.normal(math.log(median), sigma, size=S))
    L = np.clip(np.round(raw / 128.0).astype(np.int64) * 128, lmin, lmax)
    f = rng.uniform(0.1, 0.7, size=S)
    P = np.round(f * L).astype(np.int64)
    room = L - B - P + 1
    A = _largest_remainder(total_anchors, (L - P), np.ones(S, np.int64), room)
    anchors = []
    for s in range(S):
        chosen: set = set()
        span = int(room[s])
        while len(chosen) < A[s]:
            need = int(A[s]) - len(chosen)
            u = rng.beta(3.0, 1.0, size=need)
            for x in (P[s] + np.floor(u * span).astype(np.int64)):
                x = int(min(x, P[s] + span - 1))
                if x not in chosen and len(chosen) < A[s]:
                    chosen.add(x)
        anchors.append(np.sort(np.fromiter(chosen, np.int64)))
    cu_ctx = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    cu_anchor = np.concatenate([[0], np.cumsum(A)]).astype(np.int32)
    return Workload(name, cu_ctx, cu_anchor, np.concatenate(anchors).astype(np.int32),
                    B, Hq, Hkv, d, chunk, seed)


SWEEP_L = (16384, 32768, 65536, 131072, 262144)


def config(idx: int, sweep: int = 0) -> Workload:
    """The five measured workloads, by index.

    0: tiny, L=1024, prompt 512, A=8, B=8, Hq=2/Hkv=1, d=64, chunk 256
    1: L=16384, prompt 4096, A=64, B=16, Hq=32/Hkv=8, d=128, chunk 1024
    2: L=65536, prompt 8192, A=256, B=16, Hq=32/Hkv=8, d=128, chunk 2048
    3: packed varlen, 8 samples, 256 anchors total, chunk 1024
    4: fixed query budget sweep, L in SWEEP_L[sweep], prompt L/8, A=512, chunk 2048
    """
    seed = SEED_BASE + 10 * idx + sweep
    if idx == 0:
        return single_sample("cfg0", seed, 1024, 512, 8, 8, 2, 1, 64, 256)
    if idx == 1:
        return single_sample("cfg1", seed, 16384, 4096, 64, 16, 32, 8, 128, 1024)
    if idx == 2:
        return single_sample("cfg2", seed, 65536, 8192, 256, 16, 32, 8, 128, 2048)
    if idx == 3:
        return packed_varlen("cfg3", seed)
    if idx == 4:
        L = SWEEP_L[sweep]
        return single_sample(f"cfg4_L{L}", seed, L, L // 8, 512, 16, 32, 8, 128, 2048)
    raise ValueError(f"unknown config {idx}")


def custom(seed: int, lengths: Sequence[int], prompts: Sequence[int],
           counts: Sequence[int], B: int, Hq: int, Hkv: int, d: int,
           chunk: int, name: str = "custom") -> Workload:
    """Arbitrary small workloads for fuzzing: uniform anchors per sample."""
    rng = _rng(seed)
    anchors: List[np.ndarray] = []
    for L, P, A in zip(lengths, prompts, counts):
        if A == 0:
            anchors.append(np.zeros(0, np.int32))
        else:
            anchors.append(_uniform_anchors(rng, P, L - B, A))
    cu_ctx = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    cu_anchor = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    flat = np.concatenate(anchors).astype(np.int32) if anchors else np.zeros(0, np.int32)
    return Workload(name, cu_ctx, cu_anchor, flat, B, Hq, Hkv, d, chunk, seed)


def tensors(w: Workload, seed_offset: int = 1, dtype=np.float32,
            with_grad: bool = True) -> dict:
    """N(0,1) draws for Q, Kc, Vc, Kd, Vd (and dO), in that order.

    Drawn in float32 from their own PCG64 stream (seed + ``seed_offset``
    * 1_000_003) so that metadata and tensors are independent streams. The
    caller rounds them to the compute dtype; the oracle then upcasts the
    rounded values to float64 so both sides see identical inputs.
    """
    rng = _rng(w.seed + seed_offset * 1_000_003)
    nq, T = w.n_q, w.total_ctx
    out = {
        "Q": rng.standard_normal((nq, w.Hq, w.d), dtype=dtype),
        "Kc": rng.standard_normal((T, w.Hkv, w.d), dtype=dtype),
        "Vc": rng.standard_normal((T, w.Hkv, w.d), dtype=dtype),
        "Kd": rng.standard_normal((nq, w.Hkv, w.d), dtype=dtype),
        "Vd": rng.standard_normal((nq, w.Hkv, w.d), dtype=dtype),
    }
    if with_grad:
        out["dO"] = rng.standard_normal((nq, w.Hq, w.d), dtype=dtype)
    return out


def default_hidden(w: Workload) -> int:
    """Model width of the drafter layer around the attention: Hq * d (the
    pages give none; this is the usual width of an attention layer whose
    heads tile the model dimension, e.g. 32 x 128 = 4096)."""
    return w.Hq * w.d


def layer_tensors(w: Workload, hidden: Optional[int] = None, seed_offset: int = 7,
                  dtype=np.float32) -> dict:
    """Inputs of the drafter layer's projections, from their own PCG64 stream.

    Xd [N_q, hidden] and Xc [T, hidden] (hidden states of the draft tokens and
    of the context) and dY [N_q, hidden] (upstream gradient of the layer
    output) are N(0,1); the stacked input weight Wqkv [(Hq + 2 Hkv) d, hidden]
    is N(0, 1/hidden) and the output weight Wo [hidden, Hq d] N(0, 1/(Hq d)),
    so that the projected Q, K, V and the output have unit variance like the
    attention's own N(0,1) draws.
    """
    H = default_hidden(w) if hidden is None else int(hidden)
    rng = _rng(w.seed + seed_offset * 1_000_003)
    nq, T = w.n_q, w.total_ctx
    rows = (w.Hq + 2 * w.Hkv) * w.d
    return {
        "Xd": rng.standard_normal((nq, H), dtype=dtype),
        "Xc": rng.standard_normal((T, H), dtype=dtype),
        "Wqkv": (rng.standard_normal((rows, H), dtype=dtype) / np.float32(math.sqrt(H))),
        "Wo": (rng.standard_normal((H, w.Hq * w.d), dtype=dtype) /
               np.float32(math.sqrt(w.Hq * w.d))),
        "dY": rng.standard_normal((nq, H), dtype=dtype),
    }


def context_offsets(w: Workload, seed: int, window: Optional[int] = None) -> np.ndarray:
    """Seeded per-block context offsets for the context-offset mask variant.

    With ``window`` each block keeps the last ``window`` keys of its visible
    context (o_j = max(0, end_j - window)); otherwise o_j is uniform on
    [0, end_j] (the empty context end_j included), end_j = a_j (+1 when
    inclusive)."""
    ends = w.anchors.astype(np.int64) + (1 if w.mask_inclusive else 0)
    if window is not None:
        return np.maximum(ends - int(window), 0).astype(np.int32)
    rng = _rng(seed)
    return np.floor(rng.random(ends.shape) * (ends + 1)).astype(np.int32)


def subset(w: Workload, n_heads: int, n_anchors: int, seed: int) -> tuple:
    """Seeded subset (query heads, global block indices) for spot checks."""
    rng = _rng(seed)
    heads = np.sort(rng.choice(w.Hq, size=min(n_heads, w.Hq), replace=False))
    blocks = np.sort(rng.choice(w.total_anchors, size=min(n_anchors, w.total_anchors),
                                replace=False))
    return heads.astype(np.int64), blocks.astype(np.int64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even).

    Returns float32 arrays holding exactly representable bf16 values, the same
    values ``torch.Tensor.to(torch.bfloat16)`` produces for finite inputs.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    # finite inputs: bits + 0x8000 stays below 2**32, so uint32 arithmetic is exact
    out = (bits >> np.uint32(16)) & np.uint32(1)
    out += np.uint32(0x7FFF)
    out += bits
    out &= np.uint32(0xFFFF0000)
    return out.view(np.float32).reshape(x.shape)
