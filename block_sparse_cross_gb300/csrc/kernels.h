// Host-side launchers of every kernel (defined in the .cu files).
#pragma once
#include <cuda_runtime.h>

#include "layout.h"

namespace skv {

// plan.cu
cudaError_t launch_plan(const ProbDev& P, const PlanPtrs& pp, const PlanCaps& caps,
                        cudaStream_t st);

// attn_simt.cu — CUDA-core attention (fp32 problems, or SPLITKV_FLAG_CUDA_CORE)
cudaError_t launch_fwd_simt(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                            const void* Q, const void* Kc, const void* Vc, cudaStream_t st);
cudaError_t launch_bwd_dq_simt(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                               const void* Q, const void* Kc, const void* Vc, const void* dO,
                               const float* LSE, cudaStream_t st);
cudaError_t launch_bwd_dkdv_simt(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                                 const void* Q, const void* Kc, const void* Vc, const void* dO,
                                 const float* LSE, void* dKc, void* dVc, cudaStream_t st);

// attn_tc.cu — tcgen05 / TMEM / TMA attention (bf16)
cudaError_t launch_fwd_tc(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                          const void* Q, const void* Kc, const void* Vc, cudaStream_t st);
cudaError_t launch_bwd_dq_tc(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                             const void* Q, const void* Kc, const void* Vc, const void* dO,
                             const float* LSE, cudaStream_t st);
// dQ != nullptr: the kernel also reduces the dQ partials into dQ (bf16) and
// zeroes the dK/dV rows of key tiles no block sees
cudaError_t launch_bwd_dkdv_tc(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                               const void* Q, const void* Kc, const void* Vc, const void* dO,
                               const float* LSE, void* dKc, void* dVc, void* dQ,
                               cudaStream_t st);

// rows.cu — HBM-bound row kernels
cudaError_t launch_merge(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                         const void* Q, const void* Kd, const void* Vd, void* O, float* LSE,
                         cudaStream_t st);
cudaError_t launch_bwd_draft(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                             const void* Q, const void* Kd, const void* Vd, const void* O,
                             const float* LSE, const void* dO, void* dKd, void* dVd,
                             int64_t nsl_cap, cudaStream_t st);
// draft.cu — the draft-block products of the merge and of the backward
// prologue as mma.sync tiles (bf16, B in {8, 16, 32}, 16 <= B * group <= 128);
// launch_merge / launch_bwd_draft use them when draft_mma_supported(P).
bool draft_mma_supported(const ProbDev& P);
cudaError_t launch_merge_draft(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                               const void* Q, const void* Kd, const void* Vd, void* O, float* LSE,
                               cudaStream_t st);
cudaError_t launch_bwd_draft_mma(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                                 const void* Q, const void* Kd, const void* Vd, const void* O,
                                 const float* LSE, const void* dO, void* dKd, void* dVd,
                                 cudaStream_t st);
// Kernel launches launch_bwd_draft makes for this problem.
int bwd_draft_launches(const ProbDev& P, int64_t nsl_cap);
// nsl_cap: the host bound on slabs (the grid covers every slab and kv head)
cudaError_t launch_dq_reduce(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk, void* dQ,
                             int64_t nsl_cap, cudaStream_t st);
// ncb_cap: the host bound on backward candidates (sample, key tile)
cudaError_t launch_zero_uncovered(const ProbDev& P, const PlanPtrs& pp, int64_t ncb_cap,
                                  void* dKc, void* dVc, cudaStream_t st);

// proj.cu — grouped tcgen05 GEMM of the drafter layer's projections.
constexpr int kProjMaxParts = 3, kProjMaxSegs = 3, kProjMaxDst = 3;

// Columns [col0, col0 + ncols) of a product go to ptr[row * ld + (c - col0)].
struct ProjDst {
  void* ptr;
  int col0, ncols;
  int64_t ld;
};

// A row-major [rows][cols] bf16 tensor read by one segment.
struct ProjOperand {
  const void* ptr;
  int64_t rows, cols;
};

// One product C[M, N] = sum over segments s of A_s B_s (host description).
//   K-major A: a[s] is [M rows][K cols]; MN-major A: [K rows][M cols];
//   likewise B with N. The part's first row of C is row a_off of A's M
//   extent and its first column is b_off of B's N extent; segment s covers
//   K coordinates [k0_a[s], k0_a[s] + klen[s]) of a[s] and [k0_b[s], ...) of
//   b[s]. A segment whose K range ends inside its tensor must have
//   klen % 64 == 0 (the last k block is padded with the tensor's zero fill).
//   ksplit > 1 splits K into that many slices added with fp32 atomics
//   (out_f32 only; the output must be zeroed first).
struct ProjSpec {
  int64_t M, N;
  int a_mn, b_mn;
  int64_t a_off, b_off;
  int nseg;
  ProjOperand a[kProjMaxSegs], b[kProjMaxSegs];
  int64_t k0_a[kProjMaxSegs], k0_b[kProjMaxSegs], klen[kProjMaxSegs];
  int ksplit, out_f32, ndst;
  ProjDst dst[kProjMaxDst];
};

// Device form of a part (built by launch_proj).
struct ProjSeg {
  int kb0, a_k, b_k;
};
struct ProjPart {
  int M, N, mt, nt, a_mn, b_mn, a_off, b_off, nseg, nkb, ksplit, kb_per_split, unit0, out_f32,
      ndst;
  ProjSeg seg[kProjMaxSegs];
  ProjDst dst[kProjMaxDst];
};
struct ProjGroup {
  int nparts, units;
  ProjPart part[kProjMaxParts];
};

cudaError_t launch_proj(const ProjSpec* parts, int nparts, cudaStream_t st);

// selftest.cu — a wait that nothing satisfies; *status = what the kernel
// reported (SPLITKV_ETIMEOUT when the bounded wait gave up). Synchronises st.
cudaError_t run_wait_probe(int* status, cudaStream_t st);
// Reads (and optionally clears) the projections' device status word.
cudaError_t proj_status(int* status, bool clear);

}  // namespace skv
