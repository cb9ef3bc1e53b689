#!/usr/bin/env python
"""Throughput of the split-KV hot path on GB300: one step = plan + forward +
backward of anchor-masked block-sparse cross-attention over one batch.

Metric: useful (masked) fwd+bwd TFLOP/s, FLOP = Hq * d * 14 * sum_j B*(a_j+B)
(4 forward + 10 backward per (query, key) pair per head and dim, the draft
self-block included), also as % of the dense bf16 tensor peak, plus the
planned LPT imbalance against naive contiguous assignment.

Default workload: the largest single-GPU configuration, config 4 at
L = 262144 (one sample, prompt 32768, 512 anchors x B = 16 = 8192 draft
queries, Hq 32 / Hkv 8, d 128, chunk 2048, bf16, seeded N(0,1) inputs,
68.7 useful TFLOP per step). K + V are 1 GiB > L2, so every step streams them
from HBM. The same line carries a record per configuration (configs 1, 2,
the three config-3 draws and every config-4 length): useful TFLOP/s and %
of the burst bf16 peak, per-kernel times and TFLOP/s, HBM GB/s of the merge
and dQ-reduce kernels, skip rate, and LPT against contiguous imbalance,
planned and measured.

N > 1 GPUs (torchrun): every rank runs its own independent batch (weak
scaling, no data-path collective); gloo is used only for the barrier and the
max-over-ranks timing reduction.

--impl reference times the float64 CPU oracle (oracle/) on the host cores,
each step a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "useful masked cross-attn fwd+bwd TFLOP/s, % of bf16 TC peak; LPT imbalance"
UNIT = "TFLOP/s"
FALLBACK_PEAK = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
# algorithmic FLOP per (context pair, head, dim) of each attention kernel
KERNEL_FLOP_PER_PAIR_DIM = {"fwd_attention": 4, "bwd_dq": 6, "bwd_dkdv": 8}


def workload_desc(w) -> str:
    lens = np.diff(w.cu_ctx)
    return (f"{w.name}: {w.num_samples} sample(s), L={'/'.join(map(str, lens[:8]))}, "
            f"{w.total_anchors} anchors x B={w.B} = {w.n_q} queries, Hq={w.Hq}/Hkv={w.Hkv}, "
            f"d={w.d}, chunk={w.chunk}")


def context_pairs(w) -> int:
    return int((w.B * w.anchors.astype(np.int64)).sum())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except Exception:
        return FALLBACK_PEAK, "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class Dist:
    def __init__(self):
        self.rank, self.world, self.local = dist_env()
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def aggregate(d: "Dist", flop_step: float, steps: int, ms_local: float):
    """Whole-job throughput of a weak-scaling run: every rank times its own
    `steps` steps (ms_local per step); the job's step time is the slowest
    rank's, and the value is the FLOP all ranks did over that time.
    Returns (TFLOP/s, ms per step)."""
    ms = d.max(ms_local)
    return d.sum(flop_step) * steps / (ms * steps * 1e-3) / 1e12, ms


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", self.gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(nm)
        if not sm:
            return None
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


def profile_traffic(kernel: str, source_sha: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source and on this workload (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_ncu.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_w = re.search(r"traffic_workload:\s*(\S+)", text)
    if not m_sha or not m_b or not m_w or m_sha.group(1) != source_sha or m_w.group(1) != workload:
        return None
    return float(m_b.group(1))


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for f in ("attn_tc.cu", "tc_common.cuh", "common.cuh", "layout.h"):
        with open(os.path.join(ROOT, "block_sparse_cross_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(w, host, blocks):
    """(seconds, O, LSE, dQ) of the oracle's fwd+bwd restricted to `blocks`."""
    import oracle.attention as OA
    t0 = time.perf_counter()
    O, LSE = OA.forward(w, host["Q"], host["Kc"], host["Vc"], host["Kd"], host["Vd"],
                        blocks=blocks)
    g = OA.backward(w, host["Q"], host["Kc"], host["Vc"], host["Kd"], host["Vd"], host["dO"],
                    blocks=blocks)
    return time.perf_counter() - t0, O, LSE, g["dQ"]


def oracle_sample_seconds(w, host, blocks):
    return oracle_sample(w, host, blocks)[0]


def oracle_errors(w, blocks, ref, outs):
    """Errors of the GPU outputs against the oracle on the sampled blocks' rows
    (O, LSE and dQ rows are exact per row; dK/dV sum over all blocks)."""
    _, O, LSE, dQ = ref
    rows = np.concatenate([np.arange(int(j) * w.B, (int(j) + 1) * w.B) for j in blocks])

    def rel(a, b):
        den = np.linalg.norm(b)
        return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a))
    Og = outs["O"].float().cpu().numpy()[rows].astype(np.float64)
    Lg = outs["LSE"].cpu().numpy()[:, rows].astype(np.float64)
    dQg = outs["dQ"].float().cpu().numpy()[rows].astype(np.float64)
    return {"rows": int(rows.size), "heads": int(w.Hq),
            "O_rel_l2": rel(Og, O[rows]), "O_max_abs": float(np.abs(Og - O[rows]).max()),
            "LSE_max_abs": float(np.abs(Lg - LSE[:, rows]).max()),
            "dQ_rel_l2": rel(dQg, dQ[rows])}


def sample_flop(w, blocks) -> int:
    a = w.anchors[np.asarray(blocks, np.int64)].astype(np.int64)
    return int(w.Hq * w.d * 14 * (w.B * (a + w.B)).sum())


def oracle_threads() -> int:
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(v, "").isdigit():
            return int(os.environ[v])
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def calibrate_blocks(w, host, target_s: float, rng_seed: int):
    """Seeded block sample whose oracle fwd+bwd takes about target_s."""
    rng = np.random.default_rng(rng_seed)
    order = rng.permutation(w.total_anchors)
    cum = np.cumsum([sample_flop(w, [b]) for b in order])
    n = 1
    ref = oracle_sample(w, host, order[:n])
    for _ in range(4):
        t = ref[0]
        if 0.6 * target_s <= t <= 1.5 * target_s or (t < target_s and n == w.total_anchors):
            break
        rate = cum[n - 1] / max(t, 1e-6)            # oracle FLOP/s on this sample
        n = int(np.clip(np.searchsorted(cum, rate * target_s, side="right"), 1, w.total_anchors))
        ref = oracle_sample(w, host, order[:n])
    calibrate_blocks.last = ref
    return np.sort(order[:n]), ref[0]


def host_inputs(w, seed_offset=1):
    t = W.tensors(w, seed_offset)
    return {k: W.round_to_bf16(v) for k, v in t.items()}


def run_reference(args, d: Dist):
    if d.rank != 0:
        return 0
    w = W.config(args.config, args.sweep)
    host = host_inputs(w)
    budget = max(20.0, min(150.0, args.reference_budget_s))
    per_step = budget / max(1, args.steps + args.warmup)
    blocks, _ = calibrate_blocks(w, host, per_step, w.seed + 99)
    for _ in range(args.warmup):
        oracle_sample_seconds(w, host, blocks)
    times = [oracle_sample_seconds(w, host, blocks) for _ in range(args.steps)]
    flop = sample_flop(w, blocks)
    v = flop / statistics.mean(times) / 1e12
    cores = oracle_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(w), "sample": f"{len(blocks)} of {w.total_anchors} draft blocks, all {w.Hq} heads, fwd+bwd"},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{len(blocks)} seeded draft blocks x {w.Hq} heads of {w.name}, float64 numpy fwd+bwd"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_ours(args, d: Dist):
    import torch
    import block_sparse_cross_gb300 as S

    torch.cuda.set_device(d.local)
    dev = torch.device("cuda", d.local)
    w = W.config(args.config, args.sweep)
    t32 = W.tensors(w, seed_offset=1 + d.rank)  # independent batch per rank
    names_in = ("Q", "Kc", "Vc", "Kd", "Vd", "dO")
    pinned = {k: torch.from_numpy(t32[k]).to(torch.bfloat16).pin_memory() for k in names_in}
    del t32
    gpu = {k: v.to(dev) for k, v in pinned.items()}
    meta_host = [torch.from_numpy(a.astype(np.int32)).pin_memory()
                 for a in (w.cu_ctx, w.cu_anchor, w.anchors)]
    meta = [m.to(dev) for m in meta_host]
    flags = S.SPLITKV_FLAG_CONTIGUOUS if args.contiguous else 0
    kv = S.SplitKV(*meta, w.total_ctx, w.total_anchors, w.max_ctx, w.B, w.Hq, w.Hkv, w.d,
                   w.chunk, w.scale, flags=flags)
    outs = {"O": torch.empty_like(gpu["Q"]), "LSE": torch.empty(w.Hq, w.n_q, device=dev),
            "dQ": torch.empty_like(gpu["Q"]), "dKc": torch.empty_like(gpu["Kc"]),
            "dVc": torch.empty_like(gpu["Vc"]), "dKd": torch.empty_like(gpu["Kd"]),
            "dVd": torch.empty_like(gpu["Vd"])}
    out_host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}

    def step():
        kv.plan()
        kv.forward(gpu["Q"], gpu["Kc"], gpu["Vc"], gpu["Kd"], gpu["Vd"], outs["O"], outs["LSE"])
        kv.backward(gpu["Q"], gpu["Kc"], gpu["Vc"], gpu["Kd"], gpu["Vd"], outs["O"], outs["LSE"],
                    gpu["dO"], outs["dQ"], outs["dKc"], outs["dVc"], outs["dKd"], outs["dVd"])

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if kv.device_status() != S.SPLITKV_OK:
        raise RuntimeError("device status " + S.splitkv_status_string(kv.device_status()))
    st = kv.stats()

    # ---- device-timed region (inputs resident) ----
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(d.local)
    sampler = ClockSampler(gpu_id)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    S.splitkv_profile_enable(True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    S.splitkv_profile_enable(False)
    clocks = sampler.stop()
    d.barrier()
    ms_local = e0.elapsed_time(e1) / args.steps
    flop_step = w.useful_flop(14)
    value, ms = aggregate(d, flop_step, args.steps, ms_local)
    pst, ktimes = S.splitkv_profile_read()
    busy = busy_imbalance(kv, S)
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAK["bf16_tflops"]))
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAK["bf16_tflops_sustained"]))

    # ---- per-kernel roofline from the live CUDA-event brackets ----
    cp = context_pairs(w)
    row_bytes = row_kernel_bytes(w)
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAK["hbm_gbs"]))
    kernels = {}
    for name, (launches, tot) in ktimes.items():
        if launches == 0:
            continue
        # the planner and the draft-block prologue are several launches per
        # call: their figure per step is the one to compare
        per_launch = tot / launches
        entry = {"launches": launches, "ms_total": tot, "ms_per_launch": per_launch,
                 "ms_per_step": tot / args.steps}
        if name in KERNEL_FLOP_PER_PAIR_DIM:
            f = KERNEL_FLOP_PER_PAIR_DIM[name] * w.d * w.Hq * cp
            entry["tflops"] = f / (per_launch * 1e-3) / 1e12
        if name in row_bytes:
            entry["hbm_gbs"] = row_bytes[name] / (per_launch * 1e-3) / 1e9
            entry["hbm_frac"] = entry["hbm_gbs"] / hbm_peak
            entry["bytes"] = row_bytes[name]
        kernels[name] = entry
    attn = {k: v for k, v in kernels.items() if k in KERNEL_FLOP_PER_PAIR_DIM}
    dom = max(attn, key=lambda k: attn[k]["ms_total"])
    sha = kernel_source_sha()
    traffic = profile_traffic(dom, sha, w.name)
    roofline = {"kernel": dom, "bound": "tensor", "achieved": attn[dom]["tflops"], "peak": peak,
                "unit": "TFLOP/s", "frac": attn[dom]["tflops"] / peak, "traffic": traffic,
                "peak_source": f"bf16_tflops (burst) of {peak_src}",
                "frac_of_sustained": attn[dom]["tflops"] / peak_sus,
                "flop_per_launch": KERNEL_FLOP_PER_PAIR_DIM[dom] * w.d * w.Hq * cp}
    launches_total = sum(v["launches"] for v in kernels.values())
    fwd_ms = sum(kernels.get(k, {}).get("ms_total", 0.0) for k in ("fwd_attention", "merge")) / args.steps
    bwd_ms = sum(kernels.get(k, {}).get("ms_total", 0.0)
                 for k in ("bwd_draft", "bwd_dq", "bwd_dkdv", "dq_reduce", "zero_uncovered")) / args.steps
    plan_ms = kernels.get("plan", {}).get("ms_total", 0.0) / args.steps

    # ---- end to end through the public API with host buffers ----
    # Every step copies its inputs from pinned host memory and its outputs
    # back. Pipelined (the `e2e` key): two device buffer sets; step i's inputs
    # are copied on an H2D stream while step i-1 computes, and its outputs on
    # a D2H stream while step i+1 computes, each copy ordered against the
    # compute that last used its buffer set by CUDA events. Serial
    # (`e2e_serial`): copy in, compute, copy out on one stream.
    e2e = e2e_serial = None
    if not args.no_e2e:
        h2d = sum(v.numel() * v.element_size() for v in pinned.values()) + \
            sum(m.numel() * m.element_size() for m in meta_host)
        d2h = sum(v.numel() * v.element_size() for v in outs.values())
        # each buffer set has its own metadata copy and its own problem handle
        # (plan and work workspaces), so a copy never writes what a running
        # step reads
        meta2 = [torch.empty_like(m) for m in meta]
        kv2 = S.SplitKV(*meta2, w.total_ctx, w.total_anchors, w.max_ctx, w.B, w.Hq, w.Hkv, w.d,
                        w.chunk, w.scale, flags=flags)
        sets = [(gpu, outs, meta, kv),
                ({k: torch.empty_like(v) for k, v in gpu.items()},
                 {k: torch.empty_like(v) for k, v in outs.items()}, meta2, kv2)]

        def step_on(g, o, kvb):
            kvb.plan()
            kvb.forward(g["Q"], g["Kc"], g["Vc"], g["Kd"], g["Vd"], o["O"], o["LSE"])
            kvb.backward(g["Q"], g["Kc"], g["Vc"], g["Kd"], g["Vd"], o["O"], o["LSE"],
                         g["dO"], o["dQ"], o["dKc"], o["dVc"], o["dKd"], o["dVd"])

        def copy_in(g, m):
            for k in names_in:
                g[k].copy_(pinned[k], non_blocking=True)
            for dm, mh in zip(m, meta_host):
                dm.copy_(mh, non_blocking=True)

        def copy_out(o):
            for k in o:
                out_host[k].copy_(o[k], non_blocking=True)

        def run_pipelined(steps):
            comp = torch.cuda.current_stream()
            s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
            done = [None, None]    # compute that last read / wrote set b
            copied = [None, None]  # D2H that last read set b's outputs
            for i in range(steps):
                b = i % 2
                g, o, m, kvb = sets[b]
                with torch.cuda.stream(s_in):
                    if done[b] is not None:
                        s_in.wait_event(done[b])
                    copy_in(g, m)
                    ready = torch.cuda.Event()
                    ready.record(s_in)
                comp.wait_event(ready)
                if copied[b] is not None:
                    comp.wait_event(copied[b])
                step_on(g, o, kvb)
                done[b] = torch.cuda.Event()
                done[b].record(comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done[b])
                    copy_out(o)
                    copied[b] = torch.cuda.Event()
                    copied[b].record(s_out)
            torch.cuda.synchronize()

        def run_serial(steps):
            for _ in range(steps):
                copy_in(gpu, meta)
                step_on(gpu, outs, kv)
                copy_out(outs)
            torch.cuda.synchronize()

        res = {}
        for name, fn in (("pipelined", run_pipelined), ("serial", run_serial)):
            fn(2)  # warm-up (streams, events)
            d.barrier()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn(args.steps)
            t = d.max(time.perf_counter() - t0)
            res[name] = {"value": d.sum(flop_step) * args.steps / t / 1e12, "unit": UNIT,
                         "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                         "ms_per_step": 1e3 * t / args.steps}
        e2e = dict(res["pipelined"], overlap="two device buffer sets; step i's kernels overlap "
                   "the H2D copy of step i+1 and the D2H copy of step i-1 (own streams)")
        e2e_serial = res["serial"]
        for kvb in (kv, kv2):
            if kvb.device_status() != S.SPLITKV_OK:
                raise RuntimeError("device status " + S.splitkv_status_string(kvb.device_status()))
        del sets, kv2, meta2

    # ---- CPU oracle baseline (rank 0, N = 1), and the errors of the GPU
    # outputs against it on the same sampled rows ----
    cpu = None
    errors = None
    if d.rank == 0 and d.world == 1 and not args.no_cpu_baseline:
        host = {k: v.float().numpy() for k, v in pinned.items()}
        blocks, _ = calibrate_blocks(w, host, args.cpu_target_s, w.seed + 99)
        ref = oracle_sample(w, host, blocks)
        t = ref[0]
        cpu = {"value": sample_flop(w, blocks) / t / 1e12, "unit": UNIT,
               "cores": oracle_threads(), "kind": "oracle",
               "sample": f"{len(blocks)} seeded draft blocks x {w.Hq} heads of {w.name} "
                         f"({t:.1f} s), float64 numpy fwd+bwd"}
        errors = oracle_errors(w, blocks, ref, outs)

    kv_mib = int(2 * w.total_ctx * w.Hkv * w.d * 2 / 2**20)
    per_config = None
    if d.rank == 0 and d.world == 1 and not args.no_configs:
        del kv, gpu, outs
        torch.cuda.empty_cache()
        per_config = {}
        for cfg, sweep in CONFIG_RECORDS:
            wc = w if (cfg, sweep) == (args.config, args.sweep) else W.config(cfg, sweep)
            key = f"{wc.name}_draw{sweep}" if cfg == 3 else wc.name
            per_config[key] = measure_config(wc, dev, S, torch, args.config_steps, peak)
            torch.cuda.empty_cache()

    if d.rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": d.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": workload_desc(w), "global_batch": d.world * w.n_q,
                       "seq_len": int(w.max_ctx), "parallelism": f"replicas x{d.world}",
                       "l2": f"inputs larger than L2 (K+V {kv_mib} MiB per step)",
                       "step": "plan + forward + backward"},
            "pct_of_peak": 100.0 * value / d.world / peak,
            "strict": {"value": value * 12.0 / 14.0, "unit": UNIT,
                       "pct_of_peak": 100.0 * value * 12.0 / 14.0 / d.world / peak,
                       "note": "the same step counted as 4 d forward + 8 d backward FLOP per "
                               "masked pair and head (the headline counts 4 d + 10 d)"},
            "fwd_bwd": {"ms": ms - plan_ms,
                        "tflops": flop_step / ((ms - plan_ms) * 1e-3) / 1e12,
                        "pct_of_peak": 100.0 * flop_step / ((ms - plan_ms) * 1e-3) / 1e12 / peak,
                        "note": "the step without the plan (timed on its own: one plan serves "
                                "every layer that shares the mask)"},
            "peak": {"bf16_tflops": peak, "source": f"bf16_tflops (burst) of {peak_src}",
                     "pct_of_sustained": 100.0 * value / d.world / peak_sus},
            "plan": "contiguous" if args.contiguous else "lpt",
            "lpt_imbalance": {"fwd": st.fwd_lpt_imbalance, "bwd": st.bwd_lpt_imbalance},
            "busy_imbalance": busy,
            "contiguous_imbalance": {"fwd": st.fwd_contig_imbalance, "bwd": st.bwd_contig_imbalance},
            "skip_rate": 1.0 - st.fwd_tiles / max(1, st.dense_tiles),
            "phase_ms": {"plan": plan_ms, "fwd": fwd_ms, "bwd": bwd_ms},
            "phase_tflops": {"fwd": w.useful_flop(4) / (fwd_ms * 1e-3) / 1e12 if fwd_ms else None,
                             "bwd": w.useful_flop(10) / (bwd_ms * 1e-3) / 1e12 if bwd_ms else None},
            "kernels": kernels,
            "roofline": roofline,
            "gpu_launches": launches_total,
            "clocks": clocks,
            "e2e": e2e,
            "e2e_serial": e2e_serial,
            "cpu_baseline": cpu,
            "oracle_errors": errors,
            "per_config": per_config,
        }
        print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Per-configuration records (in the bench line)
# ---------------------------------------------------------------------------
CONFIG_RECORDS = [(1, 0), (2, 0), (3, 0), (3, 1), (3, 2), (4, 0), (4, 1), (4, 2), (4, 3), (4, 4)]


def row_kernel_bytes(w) -> dict:
    """Algorithmic HBM bytes of one merge and one dQ-reduce launch.

    A (query, head) row of draft block j has nact_j = ceil(a_j / C) chunk
    partials. The merge reads each partial row once ((d + 1) fp32: O and
    lse), the row's Q (bf16) and, once per (block, kv head), the block's B
    draft keys and values, and writes O (bf16) and LSE (fp32). The dQ reduce
    reads each partial dQ row (d fp32) and the row's draft term (d fp32) and
    writes dQ (bf16)."""
    nact = -(-w.anchors.astype(np.int64) // w.chunk)
    part_rows = int(nact.sum()) * w.B * w.Hq
    rows = w.n_q * w.Hq
    merge = (part_rows * (4 * w.d + 4) + rows * (2 * w.d + 2 * w.d + 4) +
             w.total_anchors * w.Hkv * 2 * w.B * w.d * 2)
    reduce = part_rows * 4 * w.d + rows * (4 * w.d + 2 * w.d)
    return {"merge": merge, "dq_reduce": reduce}


def measure_config(w, dev, S, torch, steps, peak):
    """One configuration: plan + forward + backward steps with the LPT plan
    and with the contiguous plan, CUDA events around `steps` steps (3 untimed
    first), the library's per-launch event brackets for the kernel split,
    and the per-CTA busy stamps of the last launch of each attention kernel."""
    cp = context_pairs(w)
    rb = row_kernel_bytes(w)
    hbm_peak = float(load_peaks()[0].get("hbm_gbs", FALLBACK_PEAK["hbm_gbs"]))
    rec = {"workload": workload_desc(w), "useful_tflop_per_step": w.useful_flop(14) / 1e12,
           "steps": steps}
    for mode, flags in (("lpt", 0), ("contiguous", S.SPLITKV_FLAG_CONTIGUOUS)):
        kv, keep, fwd, bwd = _setup(w, dev, flags, S, torch)

        def step():
            kv.plan()
            fwd()
            bwd()
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        S.splitkv_profile_enable(True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            step()
        b.record()
        torch.cuda.synchronize()
        S.splitkv_profile_enable(False)
        if kv.device_status() != S.SPLITKV_OK:
            raise RuntimeError(f"{w.name} {mode}: " +
                               S.splitkv_status_string(kv.device_status()))
        ms = a.elapsed_time(b) / steps
        _, kt = S.splitkv_profile_read()
        st = kv.stats()
        busy = {k: v["imbalance"] for k, v in busy_imbalance(kv, S).items()}
        tf = w.useful_flop(14) / (ms * 1e-3) / 1e12
        # fwd + bwd alone: the plan depends on the metadata only and one plan
        # serves every layer that shares the mask, so it is timed on its own
        plan_ms = kt["plan"][1] / steps if kt["plan"][0] else 0.0
        tf_fb = w.useful_flop(14) / ((ms - plan_ms) * 1e-3) / 1e12
        r = {"ms_per_step": ms, "tflops": tf, "pct_of_peak": 100.0 * tf / peak,
             "tflops_strict": w.useful_flop(12) / (ms * 1e-3) / 1e12,
             "plan_ms": plan_ms, "fwd_bwd_ms": ms - plan_ms, "fwd_bwd_tflops": tf_fb,
             "fwd_bwd_pct_of_peak": 100.0 * tf_fb / peak, "busy_imbalance": busy}
        if mode == "lpt":
            kern = {}
            for name, (launches, tot) in kt.items():
                if launches == 0:
                    continue
                e = {"ms_per_step": tot / steps}
                if name in KERNEL_FLOP_PER_PAIR_DIM:
                    f = KERNEL_FLOP_PER_PAIR_DIM[name] * w.d * w.Hq * cp
                    e["tflops"] = f / (tot / steps * 1e-3) / 1e12
                    e["frac_of_peak"] = e["tflops"] / peak
                if name in rb:
                    e["hbm_gbs"] = rb[name] / (tot / steps * 1e-3) / 1e9
                    e["hbm_frac"] = e["hbm_gbs"] / hbm_peak
                    e["bytes"] = rb[name]
                kern[name] = e
            r["kernels"] = kern
            r["skip_rate"] = 1.0 - st.fwd_tiles / max(1, st.dense_tiles)
            r["planned_imbalance"] = {
                "lpt": {"fwd": st.fwd_lpt_imbalance, "bwd": st.bwd_lpt_imbalance},
                "contiguous": {"fwd": st.fwd_contig_imbalance, "bwd": st.bwd_contig_imbalance}}
        rec[mode] = r
        del kv, keep
        torch.cuda.empty_cache()
    rec["speedup_lpt_over_contiguous"] = rec["contiguous"]["ms_per_step"] / rec["lpt"]["ms_per_step"]
    return rec


# ---------------------------------------------------------------------------
# Studies (one JSON line per workload)
# ---------------------------------------------------------------------------
def _setup(w, dev, flags, S, torch):
    t32 = W.tensors(w, seed_offset=1)
    gpu = {k: torch.from_numpy(t32[k]).to(torch.bfloat16).to(dev)
           for k in ("Q", "Kc", "Vc", "Kd", "Vd", "dO")}
    del t32
    meta = [torch.from_numpy(a.astype(np.int32)).to(dev) for a in (w.cu_ctx, w.cu_anchor, w.anchors)]
    kv = S.SplitKV(*meta, w.total_ctx, w.total_anchors, w.max_ctx, w.B, w.Hq, w.Hkv, w.d,
                   w.chunk, w.scale, flags=flags)
    outs = {"O": torch.empty_like(gpu["Q"]), "LSE": torch.empty(w.Hq, w.n_q, device=dev),
            "dQ": torch.empty_like(gpu["Q"]), "dKc": torch.empty_like(gpu["Kc"]),
            "dVc": torch.empty_like(gpu["Vc"]), "dKd": torch.empty_like(gpu["Kd"]),
            "dVd": torch.empty_like(gpu["Vd"])}

    def fwd():
        kv.forward(gpu["Q"], gpu["Kc"], gpu["Vc"], gpu["Kd"], gpu["Vd"], outs["O"], outs["LSE"])

    def bwd():
        kv.backward(gpu["Q"], gpu["Kc"], gpu["Vc"], gpu["Kd"], gpu["Vd"], outs["O"], outs["LSE"],
                    gpu["dO"], outs["dQ"], outs["dKc"], outs["dVc"], outs["dKd"], outs["dVd"])
    return kv, (gpu, outs, meta), fwd, bwd


def _event_ms(fn, n, torch):
    """Mean device time of fn over n calls (3 untimed calls first)."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(n):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def run_study(args, d):
    """balance: the single-GPU analogue of the pages' balancing speedup — step
    time (plan + fwd + bwd) with the LPT plan against the contiguous plan.
    planner: planning time against the item count, next to the forward time."""
    import torch
    import block_sparse_cross_gb300 as S
    if d.rank != 0:
        return 0
    torch.cuda.set_device(d.local)
    dev = torch.device("cuda", d.local)
    n = max(3, min(args.steps, 10))
    if args.study == "balance":
        cases = [(3, 0), (3, 1), (3, 2)] + [(4, k) for k in range(5)]
    else:
        cases = [(1, 0), (2, 0), (3, 0)] + [(4, k) for k in range(5)]
    for cfg, sweep in cases:
        w = W.config(cfg, sweep)
        line = {"study": args.study, "workload": workload_desc(w), "steps": n}
        if args.study == "balance":
            for mode, flags in (("lpt", 0), ("contiguous", S.SPLITKV_FLAG_CONTIGUOUS)):
                kv, keep, fwd, bwd = _setup(w, dev, flags, S, torch)

                def step():
                    kv.plan()
                    fwd()
                    bwd()
                ms = _event_ms(step, n, torch)
                if kv.device_status() != S.SPLITKV_OK:
                    raise RuntimeError(S.splitkv_status_string(kv.device_status()))
                st = kv.stats()
                line[mode] = {
                    "ms_per_step": ms,
                    "tflops": w.useful_flop(14) / (ms * 1e-3) / 1e12,
                    "planned_imbalance": {
                        "fwd": st.fwd_contig_imbalance if flags else st.fwd_lpt_imbalance,
                        "bwd": st.bwd_contig_imbalance if flags else st.bwd_lpt_imbalance},
                    "busy_imbalance": {k: v["imbalance"] for k, v in busy_imbalance(kv, S).items()},
                }
                del kv, keep
                torch.cuda.empty_cache()
            line["speedup_lpt_over_contiguous"] = line["contiguous"]["ms_per_step"] / line["lpt"]["ms_per_step"]
        else:
            kv, keep, fwd, bwd = _setup(w, dev, 0, S, torch)
            plan_ms = _event_ms(kv.plan, n, torch)
            fwd_ms = _event_ms(fwd, n, torch)
            st = kv.stats()
            line.update({"fwd_items": st.fwd_items, "bwd_items": st.bwd_items,
                         "workers": st.workers, "plan_ms": plan_ms, "fwd_ms": fwd_ms,
                         "plan_over_fwd": plan_ms / fwd_ms})
            del kv, keep
            torch.cuda.empty_cache()
        print(json.dumps(line), flush=True)
    return 0


def proj_flop(w, H):
    """FLOP of the drafter layer's projections (2 per multiply-add)."""
    nq, T = w.n_q, w.total_ctx
    qd, kd = w.Hq * w.d, w.Hkv * w.d
    in_fwd = 2 * nq * H * (qd + 2 * kd) + 2 * T * H * 2 * kd
    out_fwd = 2 * nq * H * qd
    return {"in_fwd": in_fwd, "in_bwd": 2 * in_fwd, "out_fwd": out_fwd, "out_bwd": 2 * out_fwd}


def run_projection_study(args, d):
    """The drafter layer's projections (splitkv_proj_*) at configs 1 and 2
    with hidden = Hq d: each call's device time and TFLOP/s against the
    measured burst bf16 peak, the same products through torch.matmul
    (cuBLAS) for context, and the whole layer step (projections + plan +
    attention forward and backward)."""
    import torch
    import block_sparse_cross_gb300 as S
    if d.rank != 0:
        return 0
    torch.cuda.set_device(d.local)
    dev = torch.device("cuda", d.local)
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAK["bf16_tflops"]))
    n = max(3, min(args.steps, 20))
    for cfg in [int(c) for c in args.proj_configs.split(",")]:
        w = W.config(cfg)
        H = W.default_hidden(w)
        kv, keep, fwd, bwd = _setup(w, dev, 0, S, torch)
        t = W.layer_tensors(w, H)
        x = {k: torch.from_numpy(v).to(dev).to(torch.bfloat16) for k, v in t.items()}
        del t
        nq, T = w.n_q, w.total_ctx
        qd, kd = w.Hq * w.d, w.Hkv * w.d
        bf = dict(dtype=torch.bfloat16, device=dev)
        gpu, outs, _ = keep
        a = {k: gpu[k] for k in ("Q", "Kc", "Vc", "Kd", "Vd")}
        O, LSE = outs["O"], outs["LSE"]
        Y = torch.empty(nq, H, **bf)
        dO = torch.empty(nq, w.Hq, w.d, **bf)
        g = {k: torch.empty_like(v) for k, v in a.items()}
        dXd = torch.empty(nq, H, **bf)
        dXc = torch.empty(T, H, **bf)
        dW = torch.empty(qd + 2 * kd, H, device=dev)
        dWo = torch.empty(H, qd, device=dev)
        calls = {
            "in_fwd": lambda: kv.proj_in_forward(H, x["Xd"], x["Xc"], x["Wqkv"], a["Q"], a["Kc"],
                                                 a["Vc"], a["Kd"], a["Vd"]),
            "out_fwd": lambda: kv.proj_out_forward(H, O, x["Wo"], Y),
            "out_bwd": lambda: kv.proj_out_backward(H, O, x["Wo"], x["dY"], dO, dWo),
            "in_bwd": lambda: kv.proj_in_backward(H, x["Xd"], x["Xc"], x["Wqkv"], g["Q"], g["Kc"],
                                                  g["Vc"], g["Kd"], g["Vd"], dXd, dXc, dW),
        }
        fl = proj_flop(w, H)
        line = {"study": "projection", "workload": workload_desc(w), "hidden": H, "steps": n,
                "peak": peak, "peak_source": f"bf16_tflops (burst) of {src}",
                "l2": "context hidden states and their gradient are larger than L2; "
                      "the draft-side operands stay L2-resident between calls"}
        for name, fn in calls.items():
            S.splitkv_profile_enable(True)
            ms = _event_ms(fn, n, torch)
            S.splitkv_profile_enable(False)
            _, kt = S.splitkv_profile_read()
            tf = fl[name] / (ms * 1e-3) / 1e12
            line[name] = {"ms": ms, "tflops": tf, "frac": tf / peak,
                          "launches_per_call": kt["projection"][0] / (n + 3)}
        st, ds = S.splitkv_proj_status(clear=True)
        if st != S.SPLITKV_OK or ds != S.SPLITKV_OK:
            raise RuntimeError("projection status " + S.splitkv_status_string(ds))
        # the same products through torch.matmul (cuBLAS), operands pre-packed
        Wkv = x["Wqkv"][qd:]
        gq = torch.randn(nq, qd + 2 * kd, **bf)
        gc = torch.randn(T, 2 * kd, **bf)
        Of = O.reshape(nq, qd)
        cub = {
            "in_fwd": lambda: (x["Xd"] @ x["Wqkv"].t(), x["Xc"] @ Wkv.t()),
            "out_fwd": lambda: Of @ x["Wo"].t(),
            "out_bwd": lambda: (x["dY"] @ x["Wo"], x["dY"].t() @ Of),
            "in_bwd": lambda: (gq @ x["Wqkv"], gc @ Wkv, gq.t() @ x["Xd"], gc.t() @ x["Xc"]),
        }
        line["cublas"] = {}
        for name, fn in cub.items():
            ms = _event_ms(fn, n, torch)
            line["cublas"][name] = {"ms": ms, "tflops": fl[name] / (ms * 1e-3) / 1e12}
        del gq, gc

        def layer():
            calls["in_fwd"]()
            kv.plan()
            kv.forward(a["Q"], a["Kc"], a["Vc"], a["Kd"], a["Vd"], O, LSE)
            calls["out_fwd"]()
            calls["out_bwd"]()
            kv.backward(a["Q"], a["Kc"], a["Vc"], a["Kd"], a["Vd"], O, LSE, dO, g["Q"], g["Kc"],
                        g["Vc"], g["Kd"], g["Vd"])
            calls["in_bwd"]()
        ms = _event_ms(layer, n, torch)
        if kv.device_status() != S.SPLITKV_OK:
            raise RuntimeError(S.splitkv_status_string(kv.device_status()))
        attn = w.useful_flop(14)
        proj = sum(fl.values())
        line["layer"] = {"ms": ms, "useful_tflop": (attn + proj) / 1e12,
                         "attention_tflop": attn / 1e12, "projection_tflop": proj / 1e12,
                         "tflops": (attn + proj) / (ms * 1e-3) / 1e12}
        print(json.dumps(line), flush=True)
        del kv, keep, gpu, outs, x, a, g
        torch.cuda.empty_cache()
    return 0


def _oracle_line(w, host, blocks, seconds, full: bool) -> dict:
    f_sample = sample_flop(w, blocks)
    f_total = w.useful_flop(14)
    return {"workload": workload_desc(w), "threads": oracle_threads(),
            "blocks": f"{len(blocks)} of {w.total_anchors}", "seconds": seconds,
            "tflops": f_sample / seconds / 1e12,
            "full_seconds": seconds if full else seconds * f_total / f_sample,
            "full": "measured" if full else "linear extrapolation by masked-pair count"}


def run_oracle_study(args, d):
    """The float64 oracle timed on this machine's host cores (a reported
    baseline only): the whole problem for configs 0, 1 and 3 (each under ten
    minutes on 16 cores), a seeded block sample with a labelled linear
    extrapolation by masked-pair count for configs 2 and 4 (L = 16k and
    256k), and single-thread times for configs 0 and 1 (a child process with
    one BLAS thread)."""
    if d.rank != 0:
        return 0
    if args.study == "oracle-1t":  # the child: one case, BLAS limited to one thread
        w = W.config(args.config)
        host = host_inputs(w)
        if args.config == 0:
            blocks = np.arange(w.total_anchors)
            t = oracle_sample_seconds(w, host, blocks)
        else:
            blocks, t = calibrate_blocks(w, host, 8.0, w.seed + 99)
        print(json.dumps(_oracle_line(w, host, blocks, t, args.config == 0)), flush=True)
        return 0
    cases = [(0, 0, True), (1, 0, True), (2, 0, False), (3, 0, True), (4, 0, False), (4, 4, False)]
    for cfg, sweep, full in cases:
        w = W.config(cfg, sweep)
        host = host_inputs(w)
        if full:
            blocks = np.arange(w.total_anchors)
            oracle_sample_seconds(w, host, blocks[:1])  # warm
            t = oracle_sample_seconds(w, host, blocks)
        else:
            blocks, t = calibrate_blocks(w, host, 8.0, w.seed + 99)
        line = {"study": "oracle"}
        line.update(_oracle_line(w, host, blocks, t, full))
        if cfg <= 1:
            env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1",
                       MKL_NUM_THREADS="1")
            r = subprocess.run([sys.executable, os.path.abspath(__file__), "--study", "oracle-1t",
                                "--config", str(cfg)], env=env, capture_output=True, text=True,
                               timeout=600)
            if r.returncode == 0 and r.stdout.strip():
                one = json.loads(r.stdout.strip().splitlines()[-1])
                line["single_thread"] = {k: one[k] for k in ("threads", "blocks", "seconds",
                                                             "tflops", "full_seconds", "full")}
        print(json.dumps(line), flush=True)
    return 0


def busy_imbalance(kv, S):
    """Measured load balance of the latest launch of each persistent attention
    kernel: per-CTA busy time (end - start %globaltimer) max / mean - 1."""
    out = {}
    for name, kid in (("fwd_attention", S.SPLITKV_K_FWD_ATTN), ("bwd_dq", S.SPLITKV_K_BWD_DQ),
                      ("bwd_dkdv", S.SPLITKV_K_BWD_DKDV)):
        ns = kv.busy_ns(kid).astype(np.int64)
        b = (ns[:, 1] - ns[:, 0]).astype(np.float64)
        out[name] = {"imbalance": float(b.max() / b.mean() - 1.0), "busy_max_ms": float(b.max() * 1e-6),
                     "busy_mean_ms": float(b.mean() * 1e-6),
                     "span_ms": float((ns[:, 1].max() - ns[:, 0].min()) * 1e-6)}
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--sweep", type=int, default=4)
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration records")
    ap.add_argument("--config-steps", type=int, default=10,
                    help="timed steps of each per-configuration record")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-target-s", type=float, default=15.0)
    ap.add_argument("--reference-budget-s", type=float, default=120.0)
    ap.add_argument("--contiguous", action="store_true",
                    help="contiguous item assignment instead of LPT")
    ap.add_argument("--study", choices=("balance", "planner", "projection", "oracle", "oracle-1t"),
                    help="balance: step time with LPT vs contiguous plans (configs 3, 4); "
                         "planner: plan time vs item count next to the forward (configs 1-4); "
                         "projection: the drafter layer's projection GEMMs and the whole "
                         "layer step (configs 1, 2); oracle: the float64 oracle on the host "
                         "cores, whole problems and extrapolated samples, one thread and all")
    ap.add_argument("--proj-configs", default="1,2",
                    help="configs of --study projection (comma-separated)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    d = Dist()
    try:
        if args.study == "projection":
            rc = run_projection_study(args, d)
        elif args.study in ("oracle", "oracle-1t"):
            rc = run_oracle_study(args, d)
        elif args.study:
            rc = run_study(args, d)
        else:
            rc = run_reference(args, d) if args.impl == "reference" else run_ours(args, d)
    finally:
        d.close()
    return rc


if __name__ == "__main__":
    sys.exit(main())
