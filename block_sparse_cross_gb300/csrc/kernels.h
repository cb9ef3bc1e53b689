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
cudaError_t launch_bwd_dkdv_tc(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                               const void* Q, const void* Kc, const void* Vc, const void* dO,
                               const float* LSE, void* dKc, void* dVc, cudaStream_t st);

// rows.cu — HBM-bound row kernels
cudaError_t launch_merge(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                         const void* Q, const void* Kd, const void* Vd, void* O, float* LSE,
                         cudaStream_t st);
cudaError_t launch_bwd_draft(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                             const void* Q, const void* Kd, const void* Vd, const void* O,
                             const float* LSE, const void* dO, void* dKd, void* dVd,
                             int64_t nsl_cap, cudaStream_t st);
cudaError_t launch_dq_reduce(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk, void* dQ,
                             cudaStream_t st);
cudaError_t launch_zero_uncovered(const ProbDev& P, const PlanPtrs& pp, void* dKc, void* dVc,
                                  cudaStream_t st);

}  // namespace skv
