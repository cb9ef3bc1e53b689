"""Test helper: one problem on the GPU driven through the C ABI, and the
matching float64 oracle inputs (the same dt-rounded values).

Every output and both workspaces are carved from buffers that start filled
with 0xFF bytes (NaN in fp32 and bf16) and run GUARD_BYTES past the end of
the tensor. Outputs are re-poisoned before every call that writes them and
the workspaces before every call that uses them, so a row a kernel never
writes, or a workspace slot read before it is written, shows up as NaN; the
guard bytes past each buffer must still hold 0xFF after every call, so a
write past the end of any output or workspace fails the test.
"""
import numpy as np
import torch

import block_sparse_cross_gb300 as S
import workloads as W

TOL = {  # rel-L2 / max-abs bounds for bf16 inputs with fp32 accumulation
    "O_rel": 5e-3, "O_abs": 2e-2, "LSE_abs": 1e-3, "grad_rel": 1e-2,
}
GUARD_BYTES = 4096
POISON = 0xFF


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a))


def mask_flags(w):
    """Problem flags of the workload's mask variant."""
    return ((S.SPLITKV_FLAG_MASK_INCLUSIVE if w.mask_inclusive else 0) |
            (S.SPLITKV_FLAG_MASK_CAUSAL_BLOCK if w.mask_causal_block else 0))


def assert_no_debug_violations(kv):
    """Under the index-checking debug build (SPLITKV_DEBUG=1), no kernel that
    read this plan found an index out of range; a no-op in the release build."""
    assert S.DEBUG_BUILD == bool(S.splitkv_build_flags() & S.SPLITKV_BUILD_DEBUG)
    if S.DEBUG_BUILD:
        st = kv.stats()
        assert st.debug_violations == 0, (st.debug_violations, st.debug_site, st.debug_index)


class Guarded:
    """A device tensor at the start of a poisoned buffer with a guard tail."""

    def __init__(self, shape, dtype, device="cuda"):
        itemsize = torch.empty(0, dtype=dtype).element_size()
        self.nbytes = int(np.prod(shape)) * itemsize
        self.buf = torch.full((self.nbytes + GUARD_BYTES,), POISON, dtype=torch.uint8,
                              device=device)
        self.t = self.buf[:self.nbytes].view(dtype).view(*shape) if self.nbytes else \
            torch.empty(shape, dtype=dtype, device=device)

    def poison(self):
        self.buf[:self.nbytes].fill_(POISON)

    def guard_ok(self) -> bool:
        return bool((self.buf[self.nbytes:] == POISON).all().item())


class Case:
    def __init__(self, w, dtype="bf16", flags=0, num_workers=0, seed_offset=1):
        self.w = w
        flags |= mask_flags(w)
        t = W.tensors(w, seed_offset)
        self.dtype = dtype
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        # oracle view: exactly the values the device holds
        self.host = {k: (W.round_to_bf16(v) if dtype == "bf16" else v) for k, v in t.items()}
        self.dev = {k: torch.from_numpy(v).cuda().to(tdt).contiguous() for k, v in t.items()}
        self.cu_ctx = torch.from_numpy(w.cu_ctx.astype(np.int32)).cuda()
        self.cu_anchor = torch.from_numpy(w.cu_anchor.astype(np.int32)).cuda()
        self.anchors = torch.from_numpy(w.anchors.astype(np.int32)).cuda()
        self.ctx_lo = (None if w.ctx_lo is None
                       else torch.from_numpy(w.ctx_lo.astype(np.int32)).cuda())
        self.kv = S.SplitKV(self.cu_ctx, self.cu_anchor, self.anchors, w.total_ctx,
                            w.total_anchors, w.max_ctx, w.B, w.Hq, w.Hkv, w.d, w.chunk, w.scale,
                            S.SPLITKV_BF16 if dtype == "bf16" else S.SPLITKV_FP32,
                            num_workers=num_workers, flags=flags, ctx_lo=self.ctx_lo)
        # both workspaces replaced by poisoned, guarded buffers of the same size
        self.g_plan = Guarded((self.kv.plan_bytes,), torch.uint8)
        self.g_work = Guarded((self.kv.work_bytes,), torch.uint8)
        self.kv.plan_ws = self.g_plan.t
        self.kv.work = self.g_work.t
        nq = w.n_q
        self.g_out = {"O": Guarded((nq, w.Hq, w.d), tdt),
                      "LSE": Guarded((w.Hq, nq), torch.float32)}
        self.g_grads = {"dQ": Guarded(self.dev["Q"].shape, tdt),
                        "dKc": Guarded(self.dev["Kc"].shape, tdt),
                        "dVc": Guarded(self.dev["Vc"].shape, tdt),
                        "dKd": Guarded(self.dev["Kd"].shape, tdt),
                        "dVd": Guarded(self.dev["Vd"].shape, tdt)}
        self.O = self.g_out["O"].t
        self.LSE = self.g_out["LSE"].t
        self.grads = {k: g.t for k, g in self.g_grads.items()}
        self.written = set()  # outputs some call has written since their poisoning

    def guarded(self):
        return [self.g_plan, self.g_work, *self.g_out.values(), *self.g_grads.values()]

    def plan(self):
        self.g_plan.poison()
        self.kv.plan()
        return self

    def forward(self):
        d = self.dev
        self.g_work.poison()
        for g in self.g_out.values():
            g.poison()
        self.written |= set(self.g_out)
        self.kv.forward(d["Q"], d["Kc"], d["Vc"], d["Kd"], d["Vd"], self.O, self.LSE)
        return self

    def backward(self, dO=None):
        d = self.dev
        g = self.grads
        self.g_work.poison()
        for x in self.g_grads.values():
            x.poison()
        self.written |= set(self.g_grads)
        self.kv.backward(d["Q"], d["Kc"], d["Vc"], d["Kd"], d["Vd"], self.O, self.LSE,
                         d["dO"] if dO is None else dO, g["dQ"], g["dKc"], g["dVc"], g["dKd"],
                         g["dVd"])
        return self

    def status(self):
        return self.kv.device_status()

    def check_guards(self):
        torch.cuda.synchronize()
        names = ["plan_ws", "work", *self.g_out, *self.g_grads]
        bad = [n for n, g in zip(names, self.guarded()) if not g.guard_ok()]
        assert not bad, f"guard bytes overwritten past: {bad}"

    def numpy(self, finite=True):
        """Outputs as float numpy arrays; checks the guards and (by default)
        that every element of every output a call has written is finite (no
        poison NaN left)."""
        self.check_guards()
        assert_no_debug_violations(self.kv)
        out = {"O": self.O.float().cpu().numpy(), "LSE": self.LSE.cpu().numpy()}
        for k, v in self.grads.items():
            out[k] = v.float().cpu().numpy()
        if finite:
            bad = [k for k, v in out.items() if k in self.written and not np.isfinite(v).all()]
            assert not bad, f"unwritten (NaN) or non-finite elements in {bad}"
        return out
