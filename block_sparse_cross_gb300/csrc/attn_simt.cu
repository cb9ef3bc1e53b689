// CUDA-core (FMA) attention kernels of the split: the product path for fp32
// problems (exact fp32 products; the tf32 tensor path would round inputs to
// 10 mantissa bits) and, behind SPLITKV_FLAG_CUDA_CORE, an independent GPU
// implementation the tensor-core kernels are cross-checked against.
//
// They consume the same plan and produce the same partials as the tcgen05
// kernels:
//   forward  item (sample s, chunk c, slab, kv head g): for its 128 rows, the
//            softmax over the chunk's visible keys -> (lse_c, O_c normalised)
//   dQ       same items: dQ_c = sum over the chunk's keys of dS * k (unscaled)
//   dK/dV    item (sample, 128-key tile, kv head): the tile's keys accumulate
//            dV += P^T dO and dK += dS^T Q over every slab that sees them.
// This is the local part / normalisation reconciliation split of the rit.work
// article on Split-KV (section "Split-KV двигает запросы, а не ключи и
// значения"), applied to KV chunks on one GPU.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace skv {

namespace {

constexpr int kSimtKeys = 32;  // keys staged per step

template <typename T, int D>
__global__ void __launch_bounds__(128) fwd_simt_kernel(ProbDev P, PlanPtrs pp, WorkPtrs wk,
                                                       const T* __restrict__ Q,
                                                       const T* __restrict__ Kc,
                                                       const T* __restrict__ Vc) {
  extern __shared__ float sm[];
  float* qT = sm;                      // [D][128]
  float* ks = qT + D * kRows;          // [32][D]
  float* vs = ks + kSimtKeys * D;      // [32][D]
  if (!plan_ok_cta(P, pp.hdr)) return;
  if (threadIdx.x == 0) stamp_busy(P, pp, 0, 0);
  const int w = blockIdx.x;
  const int r = threadIdx.x;
  const int q0 = pp.f_qoff[w];
  const int q1 = queue_end(pp.f_qoff, w, (int64_t)pp.hdr->n_fwd_items * P.Hkv, pp.hdr);
  for (int qi = q0; qi < q1; ++qi) {
    const QEntry e = pp.f_queue[qi];
    const int first = pp.sl_first[e.slab], nblk = pp.sl_nblk[e.slab];
    const RowInfo ri = row_info(P, first, nblk, e.g, r);
    const int c0 = P.cu_ctx[e.s];
    const int L = P.cu_ctx[e.s + 1] - c0;
    const int amax = P.anchors[first + nblk - 1];
    const int cs = e.c * P.chunk;
    const int ke = min(min(cs + P.chunk, L), amax);
    __syncthreads();
    {
      const T* qp = Q + ((size_t)(ri.n < 0 ? 0 : ri.n) * P.Hq + ri.h) * D;
#pragma unroll 8
      for (int x = 0; x < D; ++x) qT[x * kRows + r] = ri.n >= 0 ? ld_f(qp + x) * P.scale : 0.f;
    }
    float m = -INFINITY, l = 0.f;
    float acc[D];
#pragma unroll
    for (int x = 0; x < D; ++x) acc[x] = 0.f;
    for (int kb = cs; kb < ke; kb += kSimtKeys) {
      __syncthreads();
      for (int idx = r; idx < kSimtKeys * D; idx += kRows) {
        const int t = idx / D, x = idx % D, key = kb + t;
        float kv = 0.f, vv = 0.f;
        if (key < ke) {
          const size_t off = ((size_t)(c0 + key) * P.Hkv + e.g) * D + x;
          kv = ld_f(Kc + off);
          vv = ld_f(Vc + off);
        }
        ks[t * D + x] = kv;
        vs[t * D + x] = vv;
      }
      __syncthreads();
      const int nt = min(kSimtKeys, min(ke, ri.anchor) - kb);
      for (int t = max(0, ri.lo - kb); t < nt; ++t) {  // keys [lo, end) of the row
        float sdot = 0.f;
#pragma unroll
        for (int x = 0; x < D; ++x) sdot = fmaf(qT[x * kRows + r], ks[t * D + x], sdot);
        if (sdot > m) {
          const float f = expf(m - sdot);
          l = l * f + 1.f;
#pragma unroll
          for (int x = 0; x < D; ++x) acc[x] = fmaf(acc[x], f, vs[t * D + x]);
          m = sdot;
        } else {
          const float p = expf(sdot - m);
          l += p;
#pragma unroll
          for (int x = 0; x < D; ++x) acc[x] = fmaf(p, vs[t * D + x], acc[x]);
        }
      }
    }
    const size_t slot = (size_t)(pp.sl_slot[e.slab] + e.c) * P.Hkv + e.g;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    if (SKV_OK(slot < (size_t)pp.hdr->n_slot_base * P.Hkv, pp.hdr, kDbgFwdSlot, slot)) {
#pragma unroll
      for (int x = 0; x < D; x += 4)
        *(float4*)(wk.part_o + part_off(slot, r, x, D)) =
            make_float4(acc[x] * inv, acc[x + 1] * inv, acc[x + 2] * inv, acc[x + 3] * inv);
      wk.part_lse[slot * kRows + r] = l > 0.f ? m + logf(l) : -INFINITY;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) stamp_busy(P, pp, 0, 1);
}

template <typename T, int D>
__global__ void __launch_bounds__(128) bwd_dq_simt_kernel(ProbDev P, PlanPtrs pp, WorkPtrs wk,
                                                          const T* __restrict__ Q,
                                                          const T* __restrict__ Kc,
                                                          const T* __restrict__ Vc,
                                                          const T* __restrict__ dO,
                                                          const float* __restrict__ LSE) {
  extern __shared__ float sm[];
  float* qT = sm;                      // [D][128]
  float* doT = qT + D * kRows;         // [D][128]
  float* ks = doT + D * kRows;         // [32][D]
  float* vs = ks + kSimtKeys * D;      // [32][D]
  if (!plan_ok_cta(P, pp.hdr)) return;
  if (threadIdx.x == 0) stamp_busy(P, pp, 1, 0);
  const int w = blockIdx.x;
  const int r = threadIdx.x;
  const int q0 = pp.f_qoff[w];
  const int q1 = queue_end(pp.f_qoff, w, (int64_t)pp.hdr->n_fwd_items * P.Hkv, pp.hdr);
  for (int qi = q0; qi < q1; ++qi) {
    const QEntry e = pp.f_queue[qi];
    const int first = pp.sl_first[e.slab], nblk = pp.sl_nblk[e.slab];
    const RowInfo ri = row_info(P, first, nblk, e.g, r);
    const int c0 = P.cu_ctx[e.s];
    const int L = P.cu_ctx[e.s + 1] - c0;
    const int amax = P.anchors[first + nblk - 1];
    const int cs = e.c * P.chunk;
    const int ke = min(min(cs + P.chunk, L), amax);
    float lse = 0.f, Dr = 0.f;
    __syncthreads();
    {
      const size_t ro = ((size_t)(ri.n < 0 ? 0 : ri.n) * P.Hq + ri.h) * D;
#pragma unroll 8
      for (int x = 0; x < D; ++x) {
        qT[x * kRows + r] = ri.n >= 0 ? ld_f(Q + ro + x) * P.scale : 0.f;
        doT[x * kRows + r] = ri.n >= 0 ? ld_f(dO + ro + x) : 0.f;
      }
      if (ri.n >= 0) {
        lse = LSE[(size_t)ri.h * P.NQ + ri.n];
        Dr = wk.dvec[(size_t)ri.h * P.NQ + ri.n];
      }
    }
    float acc[D];
#pragma unroll
    for (int x = 0; x < D; ++x) acc[x] = 0.f;
    for (int kb = cs; kb < ke; kb += kSimtKeys) {
      __syncthreads();
      for (int idx = r; idx < kSimtKeys * D; idx += kRows) {
        const int t = idx / D, x = idx % D, key = kb + t;
        float kv = 0.f, vv = 0.f;
        if (key < ke) {
          const size_t off = ((size_t)(c0 + key) * P.Hkv + e.g) * D + x;
          kv = ld_f(Kc + off);
          vv = ld_f(Vc + off);
        }
        ks[t * D + x] = kv;
        vs[t * D + x] = vv;
      }
      __syncthreads();
      const int nt = min(kSimtKeys, min(ke, ri.anchor) - kb);
      for (int t = max(0, ri.lo - kb); t < nt; ++t) {  // keys [lo, end) of the row
        float sdot = 0.f, dp = 0.f;
#pragma unroll
        for (int x = 0; x < D; ++x) {
          sdot = fmaf(qT[x * kRows + r], ks[t * D + x], sdot);
          dp = fmaf(doT[x * kRows + r], vs[t * D + x], dp);
        }
        const float p = expf(sdot - lse);
        const float ds = p * (dp - Dr);
#pragma unroll
        for (int x = 0; x < D; ++x) acc[x] = fmaf(ds, ks[t * D + x], acc[x]);
      }
    }
    const size_t slot = (size_t)(pp.sl_slot[e.slab] + e.c) * P.Hkv + e.g;
    if (SKV_OK(slot < (size_t)pp.hdr->n_slot_base * P.Hkv, pp.hdr, kDbgDqSlot, slot)) {
#pragma unroll
      for (int x = 0; x < D; x += 4)
        *(float4*)(wk.part_o + part_off(slot, r, x, D)) =
            make_float4(acc[x], acc[x + 1], acc[x + 2], acc[x + 3]);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) stamp_busy(P, pp, 1, 1);
}

constexpr int kRowBatch = 32;

// 256 threads: key kl = tid / 2 of the tile, half = tid % 2 owns dims
// [half*D/2, (half+1)*D/2). Dot products combine the halves with a shuffle.
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_dkdv_simt_kernel(ProbDev P, PlanPtrs pp, WorkPtrs wk,
                                                            const T* __restrict__ Q,
                                                            const T* __restrict__ Kc,
                                                            const T* __restrict__ Vc,
                                                            const T* __restrict__ dO,
                                                            const float* __restrict__ LSE,
                                                            T* __restrict__ dKc,
                                                            T* __restrict__ dVc) {
  constexpr int HD = D / 2;
  constexpr int RS = 2 * (HD + 1);     // row stride of the staged rows (padded halves)
  extern __shared__ float sm[];
  float* kv_k = sm;                    // [HD][128][2]
  float* kv_v = kv_k + D * kRows;      // [HD][128][2]
  float* qs = kv_v + D * kRows;        // [kRowBatch][RS]
  float* dos = qs + kRowBatch * RS;    // [kRowBatch][RS]
  float* lse_s = dos + kRowBatch * RS; // [kRowBatch]
  float* d_s = lse_s + kRowBatch;      // [kRowBatch]
  int* anc_s = (int*)(d_s + kRowBatch);// [kRowBatch]
  int* lo_s = anc_s + kRowBatch;       // [kRowBatch]
  if (!plan_ok_cta(P, pp.hdr)) return;
  if (threadIdx.x == 0) stamp_busy(P, pp, 2, 0);
  const int w = blockIdx.x;
  const int tid = threadIdx.x;
  const int kl = tid >> 1, half = tid & 1;
  const int q0 = pp.b_qoff[w];
  const int q1 = queue_end(pp.b_qoff, w, (int64_t)pp.hdr->n_bwd_items * P.Hkv, pp.hdr);
  for (int qi = q0; qi < q1; ++qi) {
    const QEntry e = pp.b_queue[qi];
    const int s = e.s, g = e.g;
    const int c0 = P.cu_ctx[s];
    const int L = P.cu_ctx[s + 1] - c0;
    const int ks0 = e.c * kKeyTile;
    const int key = ks0 + kl;
    __syncthreads();
    for (int idx = tid; idx < kRows * D; idx += blockDim.x) {
      const int t = idx / D, x = idx % D;
      float kv = 0.f, vv = 0.f;
      if (ks0 + t < L) {
        const size_t off = ((size_t)(c0 + ks0 + t) * P.Hkv + g) * D + x;
        kv = ld_f(Kc + off);
        vv = ld_f(Vc + off);
      }
      const int hx = x / HD, xl = x % HD;
      kv_k[(xl * kRows + t) * 2 + hx] = kv;
      kv_v[(xl * kRows + t) * 2 + hx] = vv;
    }
    float dk[HD], dv[HD];
#pragma unroll
    for (int x = 0; x < HD; ++x) dk[x] = dv[x] = 0.f;
    // active slabs of the sample: those whose last anchor exceeds ks0
    const int sl0 = pp.s_slab_off[s], sl1 = pp.s_slab_off[s + 1];
    int lo = sl0, hi = sl1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (P.anchors[pp.sl_first[mid] + pp.sl_nblk[mid] - 1] > ks0) hi = mid; else lo = mid + 1;
    }
    for (int sg = lo; sg < sl1; ++sg) {
      const int first = pp.sl_first[sg], nblk = pp.sl_nblk[sg];
      for (int rb = 0; rb < kRows; rb += kRowBatch) {
        __syncthreads();
        for (int idx = tid; idx < kRowBatch * D; idx += blockDim.x) {
          const int rr = idx / D, x = idx % D;
          const RowInfo ri = row_info(P, first, nblk, g, rb + rr);
          float qv = 0.f, dv_ = 0.f;
          if (ri.n >= 0) {
            const size_t ro = ((size_t)ri.n * P.Hq + ri.h) * D + x;
            qv = ld_f(Q + ro);
            dv_ = ld_f(dO + ro);
          }
          const int o = rr * RS + (x / HD) * (HD + 1) + (x % HD);
          qs[o] = qv;
          dos[o] = dv_;
          if (x == 0) {
            lse_s[rr] = ri.n >= 0 ? LSE[(size_t)ri.h * P.NQ + ri.n] : 0.f;
            d_s[rr] = ri.n >= 0 ? wk.dvec[(size_t)ri.h * P.NQ + ri.n] : 0.f;
            anc_s[rr] = ri.anchor;
            lo_s[rr] = ri.lo;
          }
        }
        __syncthreads();
        for (int rr = 0; rr < kRowBatch; ++rr) {
          const float* qrow = qs + rr * RS + half * (HD + 1);
          const float* drow = dos + rr * RS + half * (HD + 1);
          float ps = 0.f, pd = 0.f;
#pragma unroll
          for (int x = 0; x < HD; ++x) {
            ps = fmaf(qrow[x], kv_k[(x * kRows + kl) * 2 + half], ps);
            pd = fmaf(drow[x], kv_v[(x * kRows + kl) * 2 + half], pd);
          }
          ps += __shfl_xor_sync(0xffffffffu, ps, 1);
          pd += __shfl_xor_sync(0xffffffffu, pd, 1);
          const float p =
              (key < anc_s[rr] && key >= lo_s[rr]) ? expf(ps * P.scale - lse_s[rr]) : 0.f;
          const float ds = p * (pd - d_s[rr]);
#pragma unroll
          for (int x = 0; x < HD; ++x) {
            dv[x] = fmaf(p, drow[x], dv[x]);
            dk[x] = fmaf(ds, qrow[x], dk[x]);
          }
        }
      }
    }
    if (key < L && SKV_OK((int64_t)c0 + key < P.T && g >= 0 && g < P.Hkv, pp.hdr, kDbgKvRow,
                          (int64_t)c0 + key)) {
      const size_t off = ((size_t)(c0 + key) * P.Hkv + g) * D + half * HD;
#pragma unroll
      for (int x = 0; x < HD; ++x) {
        st_f(dKc + off + x, dk[x] * P.scale);
        st_f(dVc + off + x, dv[x]);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) stamp_busy(P, pp, 2, 1);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_fwd_simt(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                            const void* Q, const void* Kc, const void* Vc, cudaStream_t st) {
  auto go = [&](auto tag, auto dtag) -> cudaError_t {
    using T = decltype(tag);
    constexpr int D = decltype(dtag)::value;
    auto k = fwd_simt_kernel<T, D>;
    const size_t smem = sizeof(float) * (D * kRows + 2 * kSimtKeys * D);
    cudaError_t err = set_smem(k, smem);
    if (err != cudaSuccess) return err;
    k<<<P.workers, kRows, smem, st>>>(P, pp, wk, (const T*)Q, (const T*)Kc, (const T*)Vc);
    return cudaGetLastError();
  };
  using D64 = std::integral_constant<int, 64>;
  using D128 = std::integral_constant<int, 128>;
  if (P.dtype == SPLITKV_FP32) return P.d == 64 ? go(float(), D64()) : go(float(), D128());
  return P.d == 64 ? go(__nv_bfloat16(), D64()) : go(__nv_bfloat16(), D128());
}

cudaError_t launch_bwd_dq_simt(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                               const void* Q, const void* Kc, const void* Vc, const void* dO,
                               const float* LSE, cudaStream_t st) {
  auto go = [&](auto tag, auto dtag) -> cudaError_t {
    using T = decltype(tag);
    constexpr int D = decltype(dtag)::value;
    auto k = bwd_dq_simt_kernel<T, D>;
    const size_t smem = sizeof(float) * (2 * D * kRows + 2 * kSimtKeys * D);
    cudaError_t err = set_smem(k, smem);
    if (err != cudaSuccess) return err;
    k<<<P.workers, kRows, smem, st>>>(P, pp, wk, (const T*)Q, (const T*)Kc, (const T*)Vc,
                                      (const T*)dO, LSE);
    return cudaGetLastError();
  };
  using D64 = std::integral_constant<int, 64>;
  using D128 = std::integral_constant<int, 128>;
  if (P.dtype == SPLITKV_FP32) return P.d == 64 ? go(float(), D64()) : go(float(), D128());
  return P.d == 64 ? go(__nv_bfloat16(), D64()) : go(__nv_bfloat16(), D128());
}

cudaError_t launch_bwd_dkdv_simt(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                                 const void* Q, const void* Kc, const void* Vc, const void* dO,
                                 const float* LSE, void* dKc, void* dVc, cudaStream_t st) {
  auto go = [&](auto tag, auto dtag) -> cudaError_t {
    using T = decltype(tag);
    constexpr int D = decltype(dtag)::value;
    constexpr int HD = D / 2;
    auto k = bwd_dkdv_simt_kernel<T, D>;
    const size_t smem =
        sizeof(float) * (2 * D * kRows + 2 * kRowBatch * 2 * (HD + 1) + 4 * kRowBatch);
    cudaError_t err = set_smem(k, smem);
    if (err != cudaSuccess) return err;
    k<<<P.workers, 256, smem, st>>>(P, pp, wk, (const T*)Q, (const T*)Kc, (const T*)Vc,
                                    (const T*)dO, LSE, (T*)dKc, (T*)dVc);
    return cudaGetLastError();
  };
  using D64 = std::integral_constant<int, 64>;
  using D128 = std::integral_constant<int, 128>;
  if (P.dtype == SPLITKV_FP32) return P.d == 64 ? go(float(), D64()) : go(float(), D128());
  return P.d == 64 ? go(__nv_bfloat16(), D64()) : go(__nv_bfloat16(), D128());
}

}  // namespace skv
