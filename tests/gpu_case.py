"""Test helper: one problem on the GPU driven through the C ABI, and the
matching float64 oracle inputs (the same dt-rounded values)."""
import numpy as np
import torch

import block_sparse_cross_gb300 as S
import workloads as W

TOL = {  # rel-L2 / max-abs bounds for bf16 inputs with fp32 accumulation
    "O_rel": 5e-3, "O_abs": 2e-2, "LSE_abs": 1e-3, "grad_rel": 1e-2,
}


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a))


def mask_flags(w):
    """Problem flags of the workload's mask variant."""
    return ((S.SPLITKV_FLAG_MASK_INCLUSIVE if w.mask_inclusive else 0) |
            (S.SPLITKV_FLAG_MASK_CAUSAL_BLOCK if w.mask_causal_block else 0))


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
        self.kv = S.SplitKV(self.cu_ctx, self.cu_anchor, self.anchors, w.total_ctx,
                            w.total_anchors, w.max_ctx, w.B, w.Hq, w.Hkv, w.d, w.chunk, w.scale,
                            S.SPLITKV_BF16 if dtype == "bf16" else S.SPLITKV_FP32,
                            num_workers=num_workers, flags=flags)
        nq = w.n_q
        self.O = torch.zeros(nq, w.Hq, w.d, dtype=tdt, device="cuda")
        self.LSE = torch.zeros(w.Hq, nq, dtype=torch.float32, device="cuda")
        self.grads = {
            "dQ": torch.zeros_like(self.dev["Q"]), "dKc": torch.zeros_like(self.dev["Kc"]),
            "dVc": torch.zeros_like(self.dev["Vc"]), "dKd": torch.zeros_like(self.dev["Kd"]),
            "dVd": torch.zeros_like(self.dev["Vd"]),
        }

    def plan(self):
        self.kv.plan()
        return self

    def forward(self):
        d = self.dev
        self.kv.forward(d["Q"], d["Kc"], d["Vc"], d["Kd"], d["Vd"], self.O, self.LSE)
        return self

    def backward(self, dO=None):
        d = self.dev
        g = self.grads
        self.kv.backward(d["Q"], d["Kc"], d["Vc"], d["Kd"], d["Vd"], self.O, self.LSE,
                         d["dO"] if dO is None else dO, g["dQ"], g["dKc"], g["dVc"], g["dKd"],
                         g["dVd"])
        return self

    def status(self):
        return self.kv.device_status()

    def numpy(self):
        torch.cuda.synchronize()
        out = {"O": self.O.float().cpu().numpy(), "LSE": self.LSE.cpu().numpy()}
        for k, v in self.grads.items():
            out[k] = v.float().cpu().numpy()
        return out
