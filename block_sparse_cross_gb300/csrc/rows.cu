// Row kernels of the split (HBM-bound, CUDA cores):
//
//  merge        per (query, head): the draft-block partial over the block's
//               own B draft keys, then the exact log-sum-exp merge of every
//               chunk partial of the row in ascending chunk order, then the
//               draft partial — the "reconcile the normalisation" step of the
//               rit.work article on Split-KV (section "Split-KV двигает
//               запросы, а не ключи и значения"); exact, so the result equals
//               the single-device attention.
//  bwd_prep     per (query, head): D = rowsum(dO * O), the softmax weights
//               P and gradients dS of the row's B draft keys and the draft
//               term of dQ (fp32, unscaled).
//  bwd_draft_kv per (draft block, kv head): dKd, dVd of the B x B draft
//               self-block, summed over the block's rows and the group's
//               heads in fixed order.
//  dq_reduce    per (query, head): dQ = scale * (sum over chunk partials in
//               ascending chunk order + draft term); the query gradients are
//               what moves between shards in the article's description.
//  zero         context rows that no draft block sees get dK = dV = 0.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace skv {

namespace {

struct RowGeom {
  int slab;     // global slab index
  int r;        // row inside the slab's 128-row item
  int anchor;
  int c_lo;     // chunks whose keys the row sees: [c_lo, nact), empty when its
  int nact;     // visible context [lo, anchor) is (nact = ceil(anchor / C))
};

__device__ __forceinline__ RowGeom row_geom(const ProbDev& P, const PlanPtrs& pp, int n, int h) {
  RowGeom G;
  const int j = n / P.B, qi = n % P.B;
  const int s = seg_of(P.cu_anchor, P.S, j);
  const int lj = j - P.cu_anchor[s];
  G.slab = pp.s_slab_off[s] + lj / P.bps;
  const int b = lj % P.bps;
  G.r = (b * P.B + qi) * P.group + (h % P.group);
  G.anchor = P.anchors[j];
  G.nact = (G.anchor + P.chunk - 1) / P.chunk;
  const int lo = P.ctx_lo[j];
  G.c_lo = lo >= G.anchor ? G.nact : lo / P.chunk;
  return G;
}

template <typename T, int EPL>
__device__ __forceinline__ void ld_vec(const T* p, float* v) {
#pragma unroll
  for (int i = 0; i < EPL; ++i) v[i] = ld_f(p + i);
}
template <typename T, int EPL>
__device__ __forceinline__ void st_vec(T* p, const float* v) {
#pragma unroll
  for (int i = 0; i < EPL; ++i) st_f(p + i, v[i]);
}

// Eight consecutive outputs in one store (16 bytes of bf16, or 2 x 16 bytes
// of fp32); p aligned accordingly.
__device__ __forceinline__ void st8(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 u;
  __nv_bfloat162 t;
  t = __floats2bfloat162_rn(v[0], v[1]); u.x = *(uint32_t*)&t;
  t = __floats2bfloat162_rn(v[2], v[3]); u.y = *(uint32_t*)&t;
  t = __floats2bfloat162_rn(v[4], v[5]); u.z = *(uint32_t*)&t;
  t = __floats2bfloat162_rn(v[6], v[7]); u.w = *(uint32_t*)&t;
  *(uint4*)p = u;
}
__device__ __forceinline__ void st8(float* p, const float (&v)[8]) {
  *(float4*)p = make_float4(v[0], v[1], v[2], v[3]);
  *(float4*)(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Reduce-scatter of 16 per-lane partial sums over the warp: afterwards lanes
// 2k and 2k+1 both hold the warp total of value k (k = (lane >> 1) & 15).
// Each halving step sends the half this lane gives up to its partner and
// adds the half it keeps: 8 + 4 + 2 + 1 + 1 = 16 shuffles, against 5 per
// value for a full all-reduce of each.
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int lane) {
  float w[8];
  {
    const bool b = (lane >> 4) & 1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float keep = b ? v[i + 8] : v[i], send = b ? v[i] : v[i + 8];
      w[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
  }
  {
    const bool b = (lane >> 3) & 1;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float keep = b ? w[i + 4] : w[i], send = b ? w[i] : w[i + 4];
      w[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
  }
  {
    const bool b = (lane >> 2) & 1;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float keep = b ? w[i + 2] : w[i], send = b ? w[i] : w[i + 2];
      w[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
  }
  float x;
  {
    const bool b = (lane >> 1) & 1;
    const float keep = b ? w[1] : w[0], send = b ? w[0] : w[1];
    x = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  return x + __shfl_xor_sync(0xffffffffu, x, 1);
}

constexpr int kDraftBM = 32, kDraftRM = 64;

// EPL consecutive floats of shared memory (16- or 8-byte aligned) in one load.
template <int EPL>
__device__ __forceinline__ void lds_vec(const float* p, float (&v)[EPL]) {
  if constexpr (EPL == 4) {
    const float4 t = *(const float4*)p;
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else {
    static_assert(EPL == 2, "head dim 64 or 128");
    const float2 t = *(const float2*)p;
    v[0] = t.x; v[1] = t.y;
  }
}

// Merge of one (query n, head h) row by one warp; lane owns dims
// [lane*EPL, lane*EPL + EPL). kd_row / vd_row(t, v) fetch this lane's dims of
// draft key / value t of the row's block (from global memory or shared).
template <typename T, int D, typename KF, typename VF>
__device__ __forceinline__ void merge_row(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                                          const T* __restrict__ Q, T* __restrict__ O,
                                          float* __restrict__ LSE, int n, int h, int lane,
                                          KF kd_row, VF vd_row) {
  constexpr int EPL = D / 32;
  const int g = h / P.group;
  const RowGeom G = row_geom(P, pp, n, h);
  const int x0 = lane * EPL;
  const bool causal = (P.flags & SPLITKV_FLAG_MASK_CAUSAL_BLOCK) != 0;
  // draft partial over the block's draft keys the row sees: all B
  // (bidirectional within the block), or t <= n % B for a causal block
  float q[EPL], od[EPL];
  ld_vec<T, EPL>(Q + ((size_t)n * P.Hq + h) * D + x0, q);
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    q[i] *= P.scale;
    od[i] = 0.f;
  }
  // Sixteen draft keys per pass: each lane pair ends with one key's score
  // (reduce-scatter), the pass's maximum and sum combine over the 16 pairs,
  // and each key's weight is broadcast from its pair to accumulate o_d.
  float md = -INFINITY, ld = 0.f;
  constexpr int KT = 16;
  const int kl = (lane >> 1) & 15;  // the key this lane's pair holds
  for (int t0 = 0; t0 < P.B; t0 += KT) {
    float sc[KT];
    {
      float kv[KT][EPL];
#pragma unroll
      for (int u = 0; u < KT; ++u) kd_row(min(t0 + u, P.B - 1), kv[u]);
#pragma unroll
      for (int u = 0; u < KT; ++u) {
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) part = fmaf(q[i], kv[u][i], part);
        sc[u] = part;
      }
    }
    // draft key t is visible to query i = n % B of its block (all t, or t <= i
    // for a causal block)
    const bool valid = t0 + kl < P.B && (!causal || t0 + kl <= n % P.B);
    const float s_all = reduce_scatter16(sc, lane);  // every lane takes part in the shuffles
    const float s_mine = valid ? s_all : -INFINITY;
    float mg = s_mine;
#pragma unroll
    for (int o = 2; o < 32; o <<= 1) mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, o));
    const float m_new = fmaxf(md, mg);
    const float f = (md == -INFINITY) ? 0.f : expf(md - m_new);
    const float pm = valid ? expf(s_mine - m_new) : 0.f;
    float lg = pm;
#pragma unroll
    for (int o = 2; o < 32; o <<= 1) lg += __shfl_xor_sync(0xffffffffu, lg, o);
    ld = ld * f + lg;
#pragma unroll
    for (int i = 0; i < EPL; ++i) od[i] *= f;
    // keys past B repeat the last key's values with weight 0
    float vv[KT][EPL];
#pragma unroll
    for (int u = 0; u < KT; ++u) vd_row(min(t0 + u, P.B - 1), vv[u]);
#pragma unroll
    for (int u = 0; u < KT; ++u) {
      const float pu = __shfl_sync(0xffffffffu, pm, 2 * u);
#pragma unroll
      for (int i = 0; i < EPL; ++i) od[i] = fmaf(pu, vv[u][i], od[i]);
    }
    md = m_new;
  }
  const float lse_d = md + logf(ld);
  // One pass over the chunk partials in ascending chunk order, then the
  // draft partial: a running maximum Mr and normaliser Sr, the weighted sum
  // rescaled when the maximum grows. Lane c of each group of 32 chunks holds
  // chunk c's lse; the group's lse values and its first eight partial rows
  // are loaded together, eight rows in flight per step.
  // the row reads partial slots slot0 + c, c in [c_lo, nhi), of its slab
  const bool slab_ok =
      SKV_OK(G.slab >= 0 && G.slab < pp.hdr->n_slabs, pp.hdr, kDbgMergeSlot, G.slab);
  const size_t slot0 = slab_ok ? (size_t)pp.sl_slot[G.slab] : 0;
  const int nhi = slab_ok && SKV_OK(slot0 + (size_t)G.nact <= (size_t)pp.hdr->n_slot_base, pp.hdr,
                                    kDbgMergeSlot, slot0 + G.nact)
                      ? G.nact
                      : G.c_lo;
  const float* plse = wk.part_lse + (slot0 * P.Hkv + g) * kRows + G.r;  // chunk c at c * Hkv * 128
  const size_t cstride = (size_t)P.Hkv * kRows;
  const float* pbase = wk.part_o + part_off(slot0 * P.Hkv + g, G.r, x0, D);
  const size_t ostride = cstride * D;  // between chunks of the row
  constexpr int U = 8;
  auto load_rows = [&](int cb, int c0, int nc, float (&v)[U][EPL]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = min(c0 + u, nc - 1);  // clamped rows get weight 0
      const float* po = pbase + (size_t)(cb + c) * ostride;
      if constexpr (EPL == 4) {  // 16-byte aligned: row * D * 4 and lane * 16 bytes
        const float4 t = *(const float4*)po;
        v[u][0] = t.x; v[u][1] = t.y; v[u][2] = t.z; v[u][3] = t.w;
      } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i) v[u][i] = po[i];
      }
    }
  };
  float acc[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
  float Mr = -INFINITY, Sr = 0.f;
  for (int cb = G.c_lo; cb < nhi; cb += 32) {
    const int nc = min(32, nhi - cb);
    const float lc = lane < nc ? plse[(cb + lane) * cstride] : -INFINITY;
    float v[U][EPL];
    load_rows(cb, 0, nc, v);
    const float Mn = fmaxf(Mr, warp_max(lc));
    const float f = Mr == -INFINITY ? 0.f : expf(Mr - Mn);
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] *= f;
    const float e = lc == -INFINITY ? 0.f : expf(lc - Mn);  // this lane's chunk weight
    Sr = Sr * f + warp_sum(e);
    Mr = Mn;
    for (int c0 = 0; c0 < nc; c0 += U) {
      if (c0 > 0) load_rows(cb, c0, nc, v);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float wgt = __shfl_sync(0xffffffffu, e, min(c0 + u, 31));
        if (c0 + u < nc) {
#pragma unroll
          for (int i = 0; i < EPL; ++i) acc[i] = fmaf(wgt, v[u][i], acc[i]);
        }
      }
    }
  }
  {  // the draft partial (its lse is finite: every row sees a draft key)
    const float Mn = fmaxf(Mr, lse_d);
    const float f = Mr == -INFINITY ? 0.f : expf(Mr - Mn);
    const float ed = expf(lse_d - Mn);
    Sr = Sr * f + ed;
    Mr = Mn;
    const float wd = ed / ld;
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] = fmaf(wd, od[i], acc[i] * f);
  }
  const float invS = 1.f / Sr;
#pragma unroll
  for (int i = 0; i < EPL; ++i) acc[i] *= invS;
  const float M = Mr, Ls = Sr;
  st_vec<T, EPL>(O + ((size_t)n * P.Hq + h) * D + x0, acc);
  if (lane == 0) LSE[(size_t)h * P.NQ + n] = M + logf(Ls);
}

// One warp per (query n, head h), draft keys and values read from global
// memory (any B).
template <typename T, int D>
__global__ void __launch_bounds__(256) merge_kernel(ProbDev P, PlanPtrs pp, WorkPtrs wk,
                                                    const T* __restrict__ Q,
                                                    const T* __restrict__ Kd,
                                                    const T* __restrict__ Vd,
                                                    T* __restrict__ O, float* __restrict__ LSE) {
  constexpr int EPL = D / 32;
  if (read_status(pp.hdr) != 0) return;
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wid >= P.NQ * P.Hq) return;
  const int n = (int)(wid / P.Hq), h = (int)(wid % P.Hq);
  const size_t kv0 = ((size_t)(n / P.B) * P.B * P.Hkv + h / P.group) * D + lane * EPL;
  const size_t kvs = (size_t)P.Hkv * D;  // between draft rows
  merge_row<T, D>(P, pp, wk, Q, O, LSE, n, h, lane,
                  [&](int t, float (&v)[EPL]) { ld_vec<T, EPL>(Kd + kv0 + t * kvs, v); },
                  [&](int t, float (&v)[EPL]) { ld_vec<T, EPL>(Vd + kv0 + t * kvs, v); });
}

// One CTA per (draft block j, kv head g) for B <= kDraftBM: the block's draft
// keys and values are staged in shared memory once, and the eight warps
// merge the block's B * group rows in turn.
template <typename T, int D>
__global__ void __launch_bounds__(256) merge_block_kernel(ProbDev P, PlanPtrs pp, WorkPtrs wk,
                                                          const T* __restrict__ Q,
                                                          const T* __restrict__ Kd,
                                                          const T* __restrict__ Vd,
                                                          T* __restrict__ O,
                                                          float* __restrict__ LSE) {
  constexpr int EPL = D / 32;
  extern __shared__ float sm[];
  float* kd_s = sm;                   // [B][D]
  float* vd_s = kd_s + kDraftBM * D;  // [B][D]
  if (read_status(pp.hdr) != 0) return;
  const int B = P.B, Gs = P.group, R = B * Gs;
  const int j = blockIdx.x, g = blockIdx.y;
  if (!SKV_OK(j < P.NA && g < P.Hkv, pp.hdr, kDbgDraftRow, j)) return;  // CTA-uniform
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < B * D; i += blockDim.x) {
    const size_t o = ((size_t)(j * B + i / D) * P.Hkv + g) * D + i % D;
    kd_s[i] = ld_f(Kd + o);
    vd_s[i] = ld_f(Vd + o);
  }
  __syncthreads();
  const int x0 = lane * EPL;
  for (int r = warp; r < R; r += 8)
    merge_row<T, D>(P, pp, wk, Q, O, LSE, j * B + r / Gs, g * Gs + r % Gs, lane,
                    [&](int t, float (&v)[EPL]) { lds_vec<EPL>(kd_s + t * D + x0, v); },
                    [&](int t, float (&v)[EPL]) { lds_vec<EPL>(vd_s + t * D + x0, v); });
}

// Backward prologue, one warp per (query n, head h):
//   D = rowsum(dO * O); for each of the block's B draft keys t the row sees
//   (all B, or t <= n % B for a causal block):
//   P_t = exp(scale q.kd_t - LSE), dS_t = P_t (dO.vd_t - D); the draft term
//   of dQ = sum_t dS_t kd_t (fp32, unscaled). P_t and dS_t are kept for the
//   draft key/value gradients.
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(ProbDev P, PlanPtrs pp, WorkPtrs wk,
                                                       const T* __restrict__ Q,
                                                       const T* __restrict__ Kd,
                                                       const T* __restrict__ Vd,
                                                       const T* __restrict__ O,
                                                       const float* __restrict__ LSE,
                                                       const T* __restrict__ dO) {
  constexpr int EPL = D / 32;
  if (read_status(pp.hdr) != 0) return;
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wid >= P.NQ * P.Hq) return;
  const int n = (int)(wid / P.Hq), h = (int)(wid % P.Hq);
  const int g = h / P.group;
  const int j = n / P.B;
  const int x0 = lane * EPL;
  const size_t row = ((size_t)n * P.Hq + h) * D + x0;
  const bool causal = (P.flags & SPLITKV_FLAG_MASK_CAUSAL_BLOCK) != 0;
  float q[EPL], dov[EPL], tmp[EPL];
  ld_vec<T, EPL>(Q + row, q);
  ld_vec<T, EPL>(dO + row, dov);
  ld_vec<T, EPL>(O + row, tmp);
  float dd = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) dd = fmaf(dov[i], tmp[i], dd);
  const float Dr = warp_sum(dd);
  const float lse = LSE[(size_t)h * P.NQ + n];
  if (lane == 0) wk.dvec[(size_t)h * P.NQ + n] = Dr;
  float* prow = wk.draft_p + ((size_t)n * P.Hq + h) * P.B;
  float* srow = wk.draft_ds + ((size_t)n * P.Hq + h) * P.B;
  float acc[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
  // Sixteen draft keys per pass: the scores and dP values are reduce-scattered
  // so that lane pair k holds key t0 + k; it computes P and dS, and dS is
  // broadcast back for the draft term of dQ.
  constexpr int KT = 16;
  const int kl = (lane >> 1) & 15;
  for (int t0 = 0; t0 < P.B; t0 += KT) {
    float kd[KT][EPL], sp[KT], dp[KT];
#pragma unroll
    for (int u = 0; u < KT; ++u) {
      const int t = min(t0 + u, P.B - 1);
      const size_t kro = ((size_t)(j * P.B + t) * P.Hkv + g) * D + x0;
      float vd[EPL];
      ld_vec<T, EPL>(Kd + kro, kd[u]);
      ld_vec<T, EPL>(Vd + kro, vd);
      sp[u] = 0.f;
      dp[u] = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        sp[u] = fmaf(q[i], kd[u][i], sp[u]);
        dp[u] = fmaf(dov[i], vd[i], dp[u]);
      }
    }
    const float s_mine = reduce_scatter16(sp, lane);
    const float dp_mine = reduce_scatter16(dp, lane);
    const int t_mine = t0 + kl;
    const bool valid = t_mine < P.B && (!causal || t_mine <= n % P.B);
    const float pt = valid ? expf(s_mine * P.scale - lse) : 0.f;
    const float ds = pt * (dp_mine - Dr);
    if (t_mine < P.B && (lane & 1) == 0) {  // 0 for keys a causal block hides
      prow[t_mine] = pt;
      srow[t_mine] = ds;
    }
#pragma unroll
    for (int u = 0; u < KT; ++u) {  // dS of keys past B is 0
      const float du = __shfl_sync(0xffffffffu, ds, 2 * u);
#pragma unroll
      for (int i = 0; i < EPL; ++i) acc[i] = fmaf(du, kd[u][i], acc[i]);
    }
  }
  float* dqd = wk.dq_draft + row;
#pragma unroll
  for (int i = 0; i < EPL; ++i) dqd[i] = acc[i];
}

// Draft key/value gradients, one CTA per (draft block j, kv head g), one
// thread per head dim x: dVd[t] = sum_r P_t(r) dO_r, dKd[t] = scale *
// sum_r dS_t(r) q_r over the block's B * group rows r in fixed order.
template <typename T, int D>
__global__ void __launch_bounds__(D) bwd_draft_kv_kernel(ProbDev P, PlanPtrs pp, WorkPtrs wk,
                                                         const T* __restrict__ Q,
                                                         const T* __restrict__ dO,
                                                         T* __restrict__ dKd,
                                                         T* __restrict__ dVd) {
  constexpr int TC = 16;  // draft keys per pass
  extern __shared__ float sm[];
  const int B = P.B, R = B * P.group;
  float* ps = sm;            // [R][B]
  float* dss = ps + R * B;   // [R][B]
  const int j = blockIdx.x, g = blockIdx.y;
  if (!SKV_OK(j < P.NA && g < P.Hkv, pp.hdr, kDbgDraftRow, j)) return;  // CTA-uniform
  const int x = threadIdx.x;
  if (read_status(pp.hdr) != 0) return;  // every thread reads the same word
  for (int idx = x; idx < R * B; idx += blockDim.x) {
    const int r = idx / B, t = idx % B;
    const int n = j * B + r / P.group, h = g * P.group + r % P.group;
    const size_t o = ((size_t)n * P.Hq + h) * B + t;
    ps[idx] = wk.draft_p[o];
    dss[idx] = wk.draft_ds[o];
  }
  __syncthreads();
  for (int t0 = 0; t0 < B; t0 += TC) {
    float av[TC], ak[TC];
#pragma unroll
    for (int k = 0; k < TC; ++k) av[k] = ak[k] = 0.f;
    for (int r = 0; r < R; ++r) {
      const int n = j * B + r / P.group, h = g * P.group + r % P.group;
      const size_t o = ((size_t)n * P.Hq + h) * D + x;
      const float dov = ld_f(dO + o), qv = ld_f(Q + o);
#pragma unroll
      for (int k = 0; k < TC; ++k) {
        if (t0 + k < B) {
          av[k] = fmaf(ps[r * B + t0 + k], dov, av[k]);
          ak[k] = fmaf(dss[r * B + t0 + k], qv, ak[k]);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < TC; ++k) {
      if (t0 + k < B) {
        const size_t o = ((size_t)(j * B + t0 + k) * P.Hkv + g) * D + x;
        st_f(dVd + o, av[k]);
        st_f(dKd + o, ak[k] * P.scale);
      }
    }
  }
}

// The whole backward of one draft block's B x B self-attention block for one
// kv head, in one CTA (blocks with B <= 32 and B * group <= 64 rows): the
// block's draft keys and values are staged once in shared memory; warp w
// takes rows w, w + 8, ...: D = rowsum(dO * O), the B scores and dP values
// (reduce-scattered over the lanes), P = exp(scale q.kd_t - LSE) (0 for keys
// a causal block hides), dS = P (dP - D), and the row's draft term of dQ =
// sum_t dS_t kd_t (fp32, unscaled); then one thread per (head dim, key
// group) sums dVd[t] = sum_r P_t(r) dO_r and dKd[t] = scale * sum_r dS_t(r)
// q_r over the rows in fixed order.
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_draft_block_kernel(ProbDev P, PlanPtrs pp, WorkPtrs wk,
                                                              const T* __restrict__ Q,
                                                              const T* __restrict__ Kd,
                                                              const T* __restrict__ Vd,
                                                              const T* __restrict__ O,
                                                              const float* __restrict__ LSE,
                                                              const T* __restrict__ dO,
                                                              T* __restrict__ dKd,
                                                              T* __restrict__ dVd) {
  constexpr int EPL = D / 32;
  extern __shared__ float sm[];
  float* kd_s = sm;                      // [B][D]
  float* vd_s = kd_s + kDraftBM * D;     // [B][D]
  float* ps = vd_s + kDraftBM * D;       // [R][kDraftBM]  P
  float* dss = ps + kDraftRM * kDraftBM; // [R][kDraftBM]  dS
  if (read_status(pp.hdr) != 0) return;
  const int B = P.B, G = P.group, R = B * G;
  const int j = blockIdx.x, g = blockIdx.y;
  if (!SKV_OK(j < P.NA && g < P.Hkv, pp.hdr, kDbgDraftRow, j)) return;  // CTA-uniform
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool causal = (P.flags & SPLITKV_FLAG_MASK_CAUSAL_BLOCK) != 0;
  for (int i = threadIdx.x; i < B * D; i += blockDim.x) {
    const size_t o = ((size_t)(j * B + i / D) * P.Hkv + g) * D + i % D;
    kd_s[i] = ld_f(Kd + o);
    vd_s[i] = ld_f(Vd + o);
  }
  __syncthreads();
  const int x0 = lane * EPL;
  const int kl = (lane >> 1) & 15;  // the key this lane's pair holds after a reduce-scatter
  // rows are prefetched one step ahead: their loads overlap the previous row
  auto row_of = [&](int rr) {
    return ((size_t)(j * B + rr / G) * P.Hq + g * G + rr % G) * D + x0;
  };
  auto lse_of = [&](int rr) { return LSE[(size_t)(g * G + rr % G) * P.NQ + j * B + rr / G]; };
  float qn[EPL], don[EPL], onx[EPL], lsen = 0.f;
  if (warp < R) {
    ld_vec<T, EPL>(Q + row_of(warp), qn);
    ld_vec<T, EPL>(dO + row_of(warp), don);
    ld_vec<T, EPL>(O + row_of(warp), onx);
    lsen = lse_of(warp);
  }
  for (int r = warp; r < R; r += 8) {
    const int n = j * B + r / G, h = g * G + r % G;
    const size_t row = ((size_t)n * P.Hq + h) * D + x0;
    float q[EPL], dov[EPL], ov[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      q[i] = qn[i];
      dov[i] = don[i];
      ov[i] = onx[i];
    }
    const float lse = lsen;
    if (r + 8 < R) {
      ld_vec<T, EPL>(Q + row_of(r + 8), qn);
      ld_vec<T, EPL>(dO + row_of(r + 8), don);
      ld_vec<T, EPL>(O + row_of(r + 8), onx);
      lsen = lse_of(r + 8);
    }
    float dd = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) dd = fmaf(dov[i], ov[i], dd);
    const float Dr = warp_sum(dd);
    if (lane == 0) wk.dvec[(size_t)h * P.NQ + n] = Dr;
    float acc[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
    for (int t0 = 0; t0 < B; t0 += 16) {
      float sp[16], dp[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int t = min(t0 + u, B - 1);
        float kr[EPL], vr[EPL];
        lds_vec<EPL>(kd_s + t * D + x0, kr);
        lds_vec<EPL>(vd_s + t * D + x0, vr);
        sp[u] = 0.f;
        dp[u] = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          sp[u] = fmaf(q[i], kr[i], sp[u]);
          dp[u] = fmaf(dov[i], vr[i], dp[u]);
        }
      }
      const float s_mine = reduce_scatter16(sp, lane);
      const float dp_mine = reduce_scatter16(dp, lane);
      const int t_mine = t0 + kl;
      const bool valid = t_mine < B && (!causal || t_mine <= n % B);
      const float pt = valid ? expf(s_mine * P.scale - lse) : 0.f;
      const float ds = pt * (dp_mine - Dr);
      if (t_mine < B && (lane & 1) == 0) {  // 0 for keys a causal block hides
        ps[r * kDraftBM + t_mine] = pt;
        dss[r * kDraftBM + t_mine] = ds;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {  // dS of keys past B is 0
        const float du = __shfl_sync(0xffffffffu, ds, 2 * u);
        float kr[EPL];
        lds_vec<EPL>(kd_s + min(t0 + u, B - 1) * D + x0, kr);
#pragma unroll
        for (int i = 0; i < EPL; ++i) acc[i] = fmaf(du, kr[i], acc[i]);
      }
    }
    float* dqd = wk.dq_draft + row;
#pragma unroll
    for (int i = 0; i < EPL; ++i) dqd[i] = acc[i];
  }
  __syncthreads();
  // dVd and dKd: thread (x, key group); groups of 16 keys at a time
  constexpr int KG = 256 / D;  // key groups (2 at d = 128, 4 at d = 64)
  const int x = threadIdx.x % D, kg = threadIdx.x / D;
  for (int t0 = kg * 16; t0 < B; t0 += KG * 16) {
    float av[16], ak[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) av[k] = ak[k] = 0.f;
#pragma unroll 4
    for (int r = 0; r < R; ++r) {
      const int n = j * B + r / G, h = g * G + r % G;
      const size_t o = ((size_t)n * P.Hq + h) * D + x;
      const float dv = ld_f(dO + o), qv = ld_f(Q + o);
      const float* pr = ps + r * kDraftBM + t0;
      const float* sr = dss + r * kDraftBM + t0;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        if (t0 + k < B) {
          av[k] = fmaf(pr[k], dv, av[k]);
          ak[k] = fmaf(sr[k], qv, ak[k]);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      if (t0 + k < B) {
        const size_t o = ((size_t)(j * B + t0 + k) * P.Hkv + g) * D + x;
        st_f(dVd + o, av[k]);
        st_f(dKd + o, ak[k] * P.scale);
      }
    }
  }
}

// Row table of every (slab, kv head) for the dK/dV kernel, which streams it
// with the slab's Q / dO tiles: -LSE*log2(e) (-inf on padding rows, so their
// P is 0 without masking), D, and the row's anchor.
__global__ void __launch_bounds__(128) slab_rowinfo_kernel(ProbDev P, PlanPtrs pp, WorkPtrs wk,
                                                           const float* __restrict__ LSE) {
  const int sg = blockIdx.x, g = blockIdx.y, r = threadIdx.x;
  if (sg == 0 && g == 0 && r == 0) *wk.red_next = 0;  // the dK/dV kernel's task counter
  if (sg >= pp.hdr->n_slabs || read_status(pp.hdr) != 0) return;
  const RowInfo ri = row_info(P, pp.sl_first[sg], pp.sl_nblk[sg], g, r);
  float* rec = wk.rowinfo + ((size_t)sg * P.Hkv + g) * kRowInfoFloats;
  if (ri.n >= 0) {
    rec[r] = -LSE[(size_t)ri.h * P.NQ + ri.n] * 1.4426950408889634f;
    rec[kRows + r] = wk.dvec[(size_t)ri.h * P.NQ + ri.n];
  } else {
    rec[r] = -INFINITY;
    rec[kRows + r] = 0.f;
  }
  ((int*)rec)[2 * kRows + r] = ri.anchor;
  ((int*)rec)[3 * kRows + r] = ri.lo;
}

// dQ = scale * (sum of the row's chunk partials in ascending chunk order +
// its draft term), one CTA per (slab, kv head, half of the slab's 128-row
// tile): four threads per row (thread t: row 64 z + t % 64, 8-dim groups
// t / 64 + 4i), so that a warp reads 32 consecutive rows of one group, 1 KB
// contiguous, from each partial slot.
template <typename T, int D>
__global__ void __launch_bounds__(256) dq_reduce_kernel(ProbDev P, PlanPtrs pp, WorkPtrs wk,
                                                        T* __restrict__ dQ) {
  constexpr int kGroups = D / 32;
  if (read_status(pp.hdr) != 0) return;
  const int sg = blockIdx.x, g = blockIdx.y;
  if (sg >= pp.hdr->n_slabs) return;
  const int r = 64 * blockIdx.z + threadIdx.x % 64, q = threadIdx.x / 64;
  const RowInfo ri = row_info(P, pp.sl_first[sg], pp.sl_nblk[sg], g, r);
  if (ri.n < 0) return;  // padding row of the slab's tile
  const int na = (ri.anchor + P.chunk - 1) / P.chunk;
  const int c_lo = ri.lo >= ri.anchor ? na : ri.lo / P.chunk;
  const size_t slot0 = (size_t)pp.sl_slot[sg];
  // the row reads partial slots slot0 + c, c in [c_lo, nact), of its slab
  const int nact = SKV_OK(slot0 + (size_t)na <= (size_t)pp.hdr->n_slot_base, pp.hdr, kDbgReduceSlot,
                          slot0 + na)
                       ? na
                       : c_lo;
  const float* prow = wk.part_o + part_off(slot0 * P.Hkv + g, r, 8 * q, D);
  const size_t ostride = (size_t)P.Hkv * kRows * D;  // between chunks of the row
  float acc[kGroups][8];
#pragma unroll
  for (int i = 0; i < kGroups; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
#pragma unroll 2
  for (int c = c_lo; c < nact; ++c) {
    const float* pc = prow + (size_t)c * ostride;
#pragma unroll
    for (int i = 0; i < kGroups; ++i) {
      const float4 a = *(const float4*)(pc + (size_t)(4 * i) * kRows * 8);
      const float4 b = *(const float4*)(pc + (size_t)(4 * i) * kRows * 8 + 4);
      acc[i][0] += a.x; acc[i][1] += a.y; acc[i][2] += a.z; acc[i][3] += a.w;
      acc[i][4] += b.x; acc[i][5] += b.y; acc[i][6] += b.z; acc[i][7] += b.w;
    }
  }
  if (!SKV_OK(ri.n < P.NQ && ri.h >= 0 && ri.h < P.Hq, pp.hdr, kDbgQueryRow, ri.n)) return;
  const size_t row = ((size_t)ri.n * P.Hq + ri.h) * D + 8 * q;
#pragma unroll
  for (int i = 0; i < kGroups; ++i) {
    const float* dd = wk.dq_draft + row + 32 * i;
    const float4 a = *(const float4*)dd, b = *(const float4*)(dd + 4);
    float v[8] = {(acc[i][0] + a.x) * P.scale, (acc[i][1] + a.y) * P.scale,
                  (acc[i][2] + a.z) * P.scale, (acc[i][3] + a.w) * P.scale,
                  (acc[i][4] + b.x) * P.scale, (acc[i][5] + b.y) * P.scale,
                  (acc[i][6] + b.z) * P.scale, (acc[i][7] + b.w) * P.scale};
    st8(dQ + row + 32 * i, v);
  }
}

// Key tiles that no block sees (backward candidates of cost 0: past a
// sample's last visible key, every tile of a sample without anchors, and
// with per-block context offsets any tile outside every block's range) are
// in no backward item; their key/value gradients are zero. A CTA takes eight
// candidates at a time (one cost read per warp) and zeroes each tile of cost
// 0 among them with all its threads, in 16-byte stores.
template <typename T>
__global__ void __launch_bounds__(256) zero_uncovered_kernel(ProbDev P, PlanPtrs pp,
                                                             T* __restrict__ dKc,
                                                             T* __restrict__ dVc) {
  __shared__ int unseen[8];
  if (read_status(pp.hdr) != 0) return;
  const int ncand = pp.hdr->n_bwd_cand;
  const int warp = threadIdx.x >> 5;
  const size_t row16 = (size_t)P.Hkv * P.d * sizeof(T) / 16;  // d in {64, 128}: whole 16 B units
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int base = blockIdx.x * 8; base < ncand; base += gridDim.x * 8) {
    if ((threadIdx.x & 31) == 0) {
      const int cand = base + warp;
      unseen[warp] = cand < ncand && pp.b_cost[cand] == 0;
    }
    __syncthreads();
    for (int w = 0; w < 8; ++w) {
      if (!unseen[w]) continue;  // CTA-uniform
      const int cand = base + w;
      const int s = seg_of(pp.s_bcand_off, P.S, cand);
      const int kt = cand - pp.s_bcand_off[s];
      const int c0 = P.cu_ctx[s], L = P.cu_ctx[s + 1] - c0;
      const int k0 = kt * kKeyTile, k1 = min(L, k0 + kKeyTile);
      if (!SKV_OK(k0 >= 0 && (int64_t)c0 + k1 <= P.T, pp.hdr, kDbgZeroRow, (int64_t)c0 + k1))
        continue;  // CTA-uniform
      const size_t lo = (size_t)(c0 + k0) * row16, hi = (size_t)(c0 + k1) * row16;
      for (size_t i = lo + threadIdx.x; i < hi; i += blockDim.x) {
        ((uint4*)dKc)[i] = z;
        ((uint4*)dVc)[i] = z;
      }
    }
    __syncthreads();  // the flags are rewritten by the next group
  }
}

template <typename F>
cudaError_t dispatch(const ProbDev& P, F&& f) {
  using D64 = std::integral_constant<int, 64>;
  using D128 = std::integral_constant<int, 128>;
  if (P.dtype == SPLITKV_FP32) return P.d == 64 ? f(float(), D64()) : f(float(), D128());
  return P.d == 64 ? f(__nv_bfloat16(), D64()) : f(__nv_bfloat16(), D128());
}

}  // namespace

cudaError_t launch_merge(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                         const void* Q, const void* Kd, const void* Vd, void* O, float* LSE,
                         cudaStream_t st) {
  return dispatch(P, [&](auto tag, auto dtag) -> cudaError_t {
    using T = decltype(tag);
    constexpr int D = decltype(dtag)::value;
    const int64_t warps = P.NQ * P.Hq;
    if (warps == 0) return cudaSuccess;
    if (draft_mma_supported(P)) return launch_merge_draft(P, pp, wk, Q, Kd, Vd, O, LSE, st);
    if (P.B <= kDraftBM) {
      const size_t smem = sizeof(float) * 2 * kDraftBM * D;
      merge_block_kernel<T, D><<<dim3((unsigned)P.NA, (unsigned)P.Hkv), 256, smem, st>>>(
          P, pp, wk, (const T*)Q, (const T*)Kd, (const T*)Vd, (T*)O, LSE);
    } else {
      merge_kernel<T, D><<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(
          P, pp, wk, (const T*)Q, (const T*)Kd, (const T*)Vd, (T*)O, LSE);
    }
    return cudaGetLastError();
  });
}

int bwd_draft_launches(const ProbDev& P, int64_t nsl_cap) {
  if (P.NQ * P.Hq == 0) return 0;
  const bool fused = draft_mma_supported(P) || (P.B <= kDraftBM && P.B * P.group <= kDraftRM);
  return (fused ? 1 : 2) + (nsl_cap > 0 ? 1 : 0);
}

cudaError_t launch_bwd_draft(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                             const void* Q, const void* Kd, const void* Vd, const void* O,
                             const float* LSE, const void* dO, void* dKd, void* dVd,
                             int64_t nsl_cap, cudaStream_t st) {
  return dispatch(P, [&](auto tag, auto dtag) -> cudaError_t {
    using T = decltype(tag);
    constexpr int D = decltype(dtag)::value;
    const int64_t warps = P.NQ * P.Hq;
    if (warps == 0) return cudaSuccess;
    cudaError_t err;
    dim3 grid((unsigned)P.NA, (unsigned)P.Hkv);
    if (draft_mma_supported(P)) {
      err = launch_bwd_draft_mma(P, pp, wk, Q, Kd, Vd, O, LSE, dO, dKd, dVd, st);
      if (err != cudaSuccess) return err;
    } else if (P.B <= kDraftBM && P.B * P.group <= kDraftRM) {
      // one CTA per (draft block, kv head) does the whole draft-block backward
      const size_t smem = sizeof(float) * (2 * kDraftBM * D + 2 * kDraftRM * kDraftBM);
      auto k = bwd_draft_block_kernel<T, D>;
      err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
      k<<<grid, 256, smem, st>>>(P, pp, wk, (const T*)Q, (const T*)Kd, (const T*)Vd, (const T*)O,
                                 LSE, (const T*)dO, (T*)dKd, (T*)dVd);
    } else {  // larger blocks: one warp per row, then one CTA per (block, kv head)
      bwd_prep_kernel<T, D><<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(
          P, pp, wk, (const T*)Q, (const T*)Kd, (const T*)Vd, (const T*)O, LSE, (const T*)dO);
      err = cudaGetLastError();
      if (err != cudaSuccess) return err;
      const size_t smem = sizeof(float) * 2 * (size_t)P.B * P.group * P.B;
      auto k = bwd_draft_kv_kernel<T, D>;
      err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
      k<<<grid, D, smem, st>>>(P, pp, wk, (const T*)Q, (const T*)dO, (T*)dKd, (T*)dVd);
    }
    err = cudaGetLastError();
    if (err != cudaSuccess || nsl_cap == 0) return err;
    slab_rowinfo_kernel<<<dim3((unsigned)nsl_cap, (unsigned)P.Hkv), kRows, 0, st>>>(P, pp, wk, LSE);
    return cudaGetLastError();
  });
}

cudaError_t launch_dq_reduce(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk, void* dQ,
                             int64_t nsl_cap, cudaStream_t st) {
  return dispatch(P, [&](auto tag, auto dtag) -> cudaError_t {
    using T = decltype(tag);
    constexpr int D = decltype(dtag)::value;
    if (P.NQ * P.Hq == 0 || nsl_cap == 0) return cudaSuccess;
    dq_reduce_kernel<T, D><<<dim3((unsigned)nsl_cap, (unsigned)P.Hkv, 2), 256, 0, st>>>(
        P, pp, wk, (T*)dQ);
    return cudaGetLastError();
  });
}

cudaError_t launch_zero_uncovered(const ProbDev& P, const PlanPtrs& pp, int64_t ncb_cap,
                                  void* dKc, void* dVc, cudaStream_t st) {
  if (P.T == 0 || ncb_cap == 0) return cudaSuccess;
  const int64_t g8 = (ncb_cap + 7) / 8;  // 8 warps per CTA, one candidate per warp at a time
  const unsigned grid = (unsigned)(g8 < 1024 ? g8 : 1024);
  if (P.dtype == SPLITKV_FP32)
    zero_uncovered_kernel<float><<<grid, 256, 0, st>>>(P, pp, (float*)dKc, (float*)dVc);
  else
    zero_uncovered_kernel<__nv_bfloat16>
        <<<grid, 256, 0, st>>>(P, pp, (__nv_bfloat16*)dKc, (__nv_bfloat16*)dVc);
  return cudaGetLastError();
}

}  // namespace skv
