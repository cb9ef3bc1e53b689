// Small device helpers shared by the kernels.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "layout.h"

namespace skv {

__device__ __forceinline__ void latch(PlanHeader* h, int code) {
  atomicCAS(&h->status, 0, code);
}

// Index checks of the debug build (compiled with -DSKV_DEBUG=1): a failed
// check counts itself in the plan header, keeps the first failure's site and
// index there, and the caller skips the access. In the release build a check
// is the constant true: its condition is not even evaluated.
enum DebugSite : int {
  kDbgFwdSlot = 1,       // forward partial slot written (tensor-core or CUDA-core kernel)
  kDbgDqSlot = 2,        // dQ partial slot written
  kDbgKvRow = 3,         // dK/dV context row written
  kDbgQueue = 4,         // a CTA's queue range [q0, q1) within the plan's items
  kDbgMergeSlot = 5,     // partial slots a merge row reads
  kDbgReduceSlot = 6,    // partial slots a dQ-reduce row reads
  kDbgQueryRow = 7,      // O / LSE / dQ query row written
  kDbgPlanScatter = 8,   // a planner scatter position (sorted order, LPT pick, queue entry)
  kDbgDraftRow = 9,      // draft key/value gradient row written
  kDbgZeroRow = 10,      // context row zeroed
};
#ifdef SKV_DEBUG
static __device__ __noinline__ bool skv_dbg_fail(const PlanHeader* h, int site, int64_t idx) {
  PlanHeader* w = const_cast<PlanHeader*>(h);
  atomicAdd((unsigned long long*)&w->dbg_count, 1ull);
  const unsigned long long code =
      ((unsigned long long)site << 48) | ((unsigned long long)idx & 0xffffffffffffull);
  atomicCAS((unsigned long long*)&w->dbg_first, 0ull, code);
  return false;
}
#define SKV_OK(cond, h, site, idx) ((cond) || ::skv::skv_dbg_fail((h), (site), (int64_t)(idx)))
#else
#define SKV_OK(cond, h, site, idx) true
#endif

// The end of worker w's queue range [qoff[w], qoff[w + 1]): the range is
// made empty when the debug build finds it outside the plan's n entries.
__device__ __forceinline__ int queue_end(const int32_t* qoff, int w, int64_t n,
                                         const PlanHeader* h) {
  const int q0 = qoff[w], q1 = qoff[w + 1];
  return SKV_OK(q0 >= 0 && q0 <= q1 && q1 <= n, h, kDbgQueue, w) ? q1 : q0;
}

__device__ __forceinline__ int read_status(const PlanHeader* h) {
  return *(volatile const int32_t*)&h->status;
}

// True when the plan is valid and was built for this problem; otherwise
// latches SPLITKV_EPLAN (mismatch) and the caller skips its work.
__device__ __forceinline__ bool plan_ok(const ProbDev& P, const PlanHeader* H) {
  if (read_status(H) != 0) return false;
  if (H->problem_hash != P.hash || H->magic != kPlanMagic) {
    if (threadIdx.x == 0) latch(const_cast<PlanHeader*>(H), SPLITKV_EPLAN);
    return false;
  }
  return true;
}

// CTA-uniform version of plan_ok (one thread reads, all agree).
__device__ __forceinline__ bool plan_ok_cta(const ProbDev& P, const PlanHeader* H) {
  __shared__ int ok_flag;
  if (threadIdx.x == 0) ok_flag = plan_ok(P, H) ? 1 : 0;
  __syncthreads();
  return ok_flag != 0;
}

// Start (which = 0) or end (1) stamp of this worker's CTA in the plan's busy
// table; slot 0 = forward, 1 = dQ, 2 = dK/dV attention launch.
__device__ __forceinline__ void stamp_busy(const ProbDev& P, const PlanPtrs& pp, int slot,
                                           int which) {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  pp.busy_ns[((size_t)slot * P.workers + blockIdx.x) * 2 + which] = t;
}

// Last index s in [0, n) with off[s] <= x (off non-decreasing, off[0] <= x).
__device__ __forceinline__ int seg_of(const int32_t* off, int n, int64_t x) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if ((int64_t)off[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

template <typename T> __device__ __forceinline__ float ld_f(const T* p);
template <> __device__ __forceinline__ float ld_f<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ void st_f(T* p, float v);
template <> __device__ __forceinline__ void st_f<float>(float* p, float v) { *p = v; }
template <> __device__ __forceinline__ void st_f<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

// Block-wide exclusive scan (blockDim.x a multiple of 32, <= 1024).
// `ws` is 32 shared slots. Returns the exclusive prefix; *total = block sum.
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* ws, T* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[wid] = x;
  __syncthreads();
  if (wid == 0) {
    T w = lane < nw ? ws[lane] : T(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    ws[lane] = w;
  }
  __syncthreads();
  T pre = (wid > 0 ? ws[wid - 1] : T(0)) + x - v;
  *total = ws[nw - 1];
  __syncthreads();
  return pre;
}

// Sample / slab / row geometry of a forward item's 128 rows.
// Row r of an item = (draft block b of the slab, query qi in the block,
// head-in-group hg) with r = (b * B + qi) * group + hg.
struct RowInfo {
  int n;        // global query index, or -1 if the row is padding
  int h;        // query head
  int anchor;   // end of the row's visible context (0 for padding rows)
  int lo;       // start of the row's visible context (0 for padding rows)
};

__device__ __forceinline__ RowInfo row_info(const ProbDev& P, int first_block, int nblk, int g,
                                            int r) {
  RowInfo ri;
  const int per_blk = P.B * P.group;
  const int b = r / per_blk;
  if (b >= nblk) {
    ri.n = -1; ri.h = 0; ri.anchor = 0; ri.lo = 0;
    return ri;
  }
  const int qi = (r / P.group) % P.B;
  const int hg = r % P.group;
  ri.n = (first_block + b) * P.B + qi;
  ri.h = g * P.group + hg;
  ri.anchor = P.anchors[first_block + b];
  ri.lo = P.ctx_lo[first_block + b];
  return ri;
}

}  // namespace skv
