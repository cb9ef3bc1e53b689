// Draft-block work of the row kernels on the tensor cores (bf16 problems).
//
// Every draft block j attends to the B keys of its own draft tokens besides
// its visible context (bidirectional within the block, or causal with
// SPLITKV_FLAG_MASK_CAUSAL_BLOCK). Per (draft block, kv head) that is a set
// of small dense products over the block's R = B * group (query, head) rows:
//
//   forward   S = Q Kd^T [R x B], P = exp(S - m), O_d = P Vd [R x D]
//   backward  S, dP = dO Vd^T, P = exp(S - LSE), dS = P (dP - D),
//             dQ_d = dS Kd [R x D], dVd = P^T dO, dKd = scale dS^T Q [B x D]
//
// The row kernels used to form these products one row at a time with warp
// shuffles; here one CTA stages the block's rows in shared memory and runs
// them as mma.sync m16n8k16 tiles (bf16 operands, fp32 accumulation), so
// the rows are no longer walked one dependent global-memory round trip at a
// time. Warp w owns rows [16w, 16w + 16) of the block (m16 tile).
//
//  merge_draft_kernel   the draft partial, then the exact log-sum-exp merge
//                       with the row's chunk partials in ascending chunk
//                       order ("reconcile the normalisation", rit.work
//                       article on Split-KV, section "Split-KV двигает
//                       запросы, а не ключи и значения"), O and LSE.
//  bwd_draft_mma_kernel D = rowsum(dO * O), the draft self-block backward
//                       (draft term of dQ, dKd, dVd summed over the block's
//                       rows and the group's heads).
//
// Row r of a CTA is (query j*B + r / group, head g*group + r % group), the
// order of the forward items' rows, so a CTA's rows are consecutive rows of
// its slab's partial tiles.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace skv {

namespace {

constexpr float kLog2eD = 1.4426950408889634f;
constexpr float kLn2D = 0.6931471805599453f;

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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

// Eight consecutive floats (32-byte aligned) in one 256-bit load.
__device__ __forceinline__ void ld_global_v8(const float* p, float (&v)[8]) {
  asm volatile("ld.global.nc.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
                 "=f"(v[6]), "=f"(v[7])
               : "l"(p));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t lds32(const __nv_bfloat16* p) {
  return *(const uint32_t*)p;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Four 8x8 bf16 matrices, transposed: thread i gives the address of row i % 8
// of matrix i / 8 (16 contiguous bytes); r[m] = {M_m[2t][g], M_m[2t+1][g]}
// with g = lane / 4, t = lane % 4 — the mma operand pairs of a matrix stored
// with the K dimension along its rows.
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const __nv_bfloat16* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}

// Shared-memory strides (bf16 elements) of one (block, kv head) CTA. Rows
// are padded by 8 elements (16 bytes) so that the eight rows of every 8x8
// fragment load fall into distinct banks.
template <int D>
struct DraftGeom {
  int B, B16, R;
  int ld_row;  // D + 8: [row or key][D] tiles
  int ld_key;  // B16 + 8: [row][key] tiles (P, dS)
  __device__ __forceinline__ DraftGeom(int B_, int R_)
      : B(B_), B16(B_ <= 16 ? 16 : 32), R(R_), ld_row(D + 8), ld_key((B_ <= 16 ? 16 : 32) + 8) {}
};

// Stages rows [R][D] of a [N][H][D] bf16 tensor: row r = (n0 + r / G, h0 + r % G).
template <int D>
__device__ __forceinline__ void stage_rows(__nv_bfloat16* dst, int ld, const __nv_bfloat16* src,
                                           int n0, int h0, int G, int H, int R) {
  constexpr int V = D / 8;  // uint4 per row
  for (int i = threadIdx.x; i < R * V; i += blockDim.x) {
    const int r = i / V, c = i % V;
    const uint4 v = *(const uint4*)(src + ((size_t)(n0 + r / G) * H + h0 + r % G) * D + 8 * c);
    *(uint4*)(dst + r * ld + 8 * c) = v;
  }
}

// Stages the block's draft keys (or values) [B16][D], rows past B zero.
template <int D>
__device__ __forceinline__ void stage_keys(__nv_bfloat16* dst, int ld, const __nv_bfloat16* src,
                                           int t0, int g, int Hkv, int B, int B16) {
  constexpr int V = D / 8;
  for (int i = threadIdx.x; i < B16 * V; i += blockDim.x) {
    const int t = i / V, c = i % V;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (t < B) v = *(const uint4*)(src + ((size_t)(t0 + t) * Hkv + g) * D + 8 * c);
    *(uint4*)(dst + t * ld + 8 * c) = v;
  }
}

__device__ __forceinline__ float dot8_bf16(const uint4& a, const uint4& b) {
  const uint32_t x[4] = {a.x, a.y, a.z, a.w}, y[4] = {b.x, b.y, b.z, b.w};
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 u = __bfloat1622float2(*(const __nv_bfloat162*)&x[k]);
    const float2 v = __bfloat1622float2(*(const __nv_bfloat162*)&y[k]);
    s = fmaf(u.x, v.x, fmaf(u.y, v.y, s));
  }
  return s;
}

// S[16 x B16] of warp tile w: A = rows [16w, 16w + 16) of `rows` ([R][D]),
// B = keys ([B16][D], K contiguous: the "col" operand read directly).
template <int D, int NT>
__device__ __forceinline__ void tile_scores(float (&s)[NT][4], const __nv_bfloat16* rows,
                                            const __nv_bfloat16* keys, int ld, int w, int lane) {
  const int gr = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int i = 0; i < 4; ++i) s[n][i] = 0.f;
  const __nv_bfloat16* a_lo = rows + (16 * w + gr) * ld + 2 * tq;
  const __nv_bfloat16* a_hi = a_lo + 8 * ld;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    uint32_t a[4];
    a[0] = lds32(a_lo + 16 * kk);
    a[1] = lds32(a_hi + 16 * kk);
    a[2] = lds32(a_lo + 16 * kk + 8);
    a[3] = lds32(a_hi + 16 * kk + 8);
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const __nv_bfloat16* bp = keys + (8 * n + gr) * ld + 16 * kk + 2 * tq;
      mma16816(s[n], a, lds32(bp), lds32(bp + 8));
    }
  }
}

// acc[16 x D] += A[16 x 16*KS] * Bm[16*KS x D]: A given as fragments (one per
// 16-deep k step), Bm row-major in shared memory ([k][D], K along rows).
template <int D, int KS>
__device__ __forceinline__ void tile_times_rows(float (&acc)[D / 8][4], const uint32_t (&a)[KS][4],
                                                const __nv_bfloat16* Bm, int ld, int lane) {
  const int m = lane >> 3, r = lane & 7;
#pragma unroll
  for (int kk = 0; kk < KS; ++kk)
#pragma unroll
    for (int n = 0; n < D / 8; n += 2) {
      uint32_t b[4];
      ldsm_x4_t(b, Bm + (16 * kk + (m & 1) * 8 + r) * ld + 8 * (n + (m >> 1)));
      mma16816(acc[n], a[kk], b[0], b[1]);
      mma16816(acc[n + 1], a[kk], b[2], b[3]);
    }
}

// ===========================================================================
// Forward: draft partial + merge, one CTA per (draft block, kv head)
// ===========================================================================
// Phase 1 (tensor cores, warp tile = 16 rows): the draft partial of every
// row, normalised (O_d / l_d), into shared memory with its lse (log2 units).
// Phase 2 (one warp per row, lanes over the head dim, the whole row's
// partial data in flight while the previous row is combined): the exact
// log-sum-exp merge, starting from the draft partial, chunks ascending.
template <int D, int NT>
__global__ void __launch_bounds__(512, 2) merge_draft_kernel(ProbDev P, PlanPtrs pp, WorkPtrs wk,
                                                          const __nv_bfloat16* __restrict__ Q,
                                                          const __nv_bfloat16* __restrict__ Kd,
                                                          const __nv_bfloat16* __restrict__ Vd,
                                                          __nv_bfloat16* __restrict__ O,
                                                          float* __restrict__ LSE) {
  constexpr int kGroups = D / 32;  // 8-dim groups per thread in phase 2 (4 threads per row)
  extern __shared__ __align__(16) uint8_t smem_raw[];
  if (read_status(pp.hdr) != 0) return;
  const int G = P.group, R = P.B * G;
  const DraftGeom<D> geo(P.B, R);
  // [Qs | Ks] then Vs; Od (the draft partials, fp32) reuses the Qs / Ks bytes
  // once the scores are formed
  const size_t od_bytes = sizeof(float) * (size_t)R * D;
  const size_t qk_bytes = sizeof(__nv_bfloat16) * (size_t)(R + geo.B16) * geo.ld_row;
  const size_t v_off = od_bytes > qk_bytes ? od_bytes : qk_bytes;
  __nv_bfloat16* Qs = (__nv_bfloat16*)smem_raw;                  // [R][D + 8]
  __nv_bfloat16* Ks = Qs + R * geo.ld_row;                        // [B16][D + 8]
  __nv_bfloat16* Vs = (__nv_bfloat16*)(smem_raw + v_off);         // [B16][D + 8]
  float* Od = (float*)smem_raw;                                    // [R][D]
  float* lsed = (float*)(smem_raw + v_off + sizeof(__nv_bfloat16) * geo.B16 * geo.ld_row);  // [R]
  const int j = blockIdx.x, g = blockIdx.y;
  if (!SKV_OK(j < P.NA && g < P.Hkv, pp.hdr, kDbgDraftRow, j)) return;  // CTA-uniform
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, tq = lane & 3;
  stage_rows<D>(Qs, geo.ld_row, Q, j * P.B, g * G, G, P.Hq, R);
  stage_keys<D>(Ks, geo.ld_row, Kd, j * P.B, g, P.Hkv, P.B, geo.B16);
  stage_keys<D>(Vs, geo.ld_row, Vd, j * P.B, g, P.Hkv, P.B, geo.B16);
  __syncthreads();

  // ---- phase 1: draft partial of rows 16w .. 16w + 15 ----
  // P V_d is formed in two halves of the head dim (fewer live registers); the
  // normalised result goes to Od, which aliases the staged tiles, so each
  // half is written only after every warp has read them.
  const bool causal = (P.flags & SPLITKV_FLAG_MASK_CAUSAL_BLOCK) != 0;
  const int w = warp;  // warps 0 .. R/16 - 1 take one 16-row tile each
  const bool tile_warp = w < R / 16;
  const int r_lo = 16 * w + gr, r_hi = r_lo + 8;
  uint32_t a[NT / 2][4];  // P as the A operand, 16 draft keys per k step
  float il_lo = 0.f, il_hi = 0.f;
  if (tile_warp) {
    float sc[NT][4];
    tile_scores<D, NT>(sc, Qs, Ks, geo.ld_row, w, lane);
    const int qi_lo = r_lo / G, qi_hi = r_hi / G;
    float m_lo = -INFINITY, m_hi = -INFINITY;
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = 8 * n + 2 * tq + (i & 1);
        const bool vis = t < P.B && (!causal || t <= (i < 2 ? qi_lo : qi_hi));
        sc[n][i] = vis ? sc[n][i] * P.scale_log2 : -INFINITY;
        if (i < 2) m_lo = fmaxf(m_lo, sc[n][i]); else m_hi = fmaxf(m_hi, sc[n][i]);
      }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      m_lo = fmaxf(m_lo, __shfl_xor_sync(0xffffffffu, m_lo, o));
      m_hi = fmaxf(m_hi, __shfl_xor_sync(0xffffffffu, m_hi, o));
    }
    float l_lo = 0.f, l_hi = 0.f;
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sc[n][i] = exp2f(sc[n][i] - (i < 2 ? m_lo : m_hi));  // 0 on hidden keys
        if (i < 2) l_lo += sc[n][i]; else l_hi += sc[n][i];
      }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      l_lo += __shfl_xor_sync(0xffffffffu, l_lo, o);
      l_hi += __shfl_xor_sync(0xffffffffu, l_hi, o);
    }
    il_lo = 1.f / l_lo;
    il_hi = 1.f / l_hi;
    if (tq == 0) {
      lsed[r_lo] = m_lo + log2f(l_lo);
      lsed[r_hi] = m_hi + log2f(l_hi);
    }
#pragma unroll
    for (int kk = 0; kk < NT / 2; ++kk) {
      a[kk][0] = pack2(sc[2 * kk][0], sc[2 * kk][1]);
      a[kk][1] = pack2(sc[2 * kk][2], sc[2 * kk][3]);
      a[kk][2] = pack2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      a[kk][3] = pack2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
    }
  }
  __syncthreads();  // every warp has its scores: Od may overwrite Qs / Ks
  if (tile_warp) {
    constexpr int H = D / 2;
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
      float acc[H / 8][4];
#pragma unroll
      for (int n = 0; n < H / 8; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[n][i] = 0.f;
      tile_times_rows<H, NT / 2>(acc, a, Vs + hh * H, geo.ld_row, lane);
#pragma unroll
      for (int n = 0; n < H / 8; ++n) {  // Od is [D/8][R][8], like a partial slot
        const int k = hh * (H / 8) + n;
        *(float2*)(Od + (k * R + r_lo) * 8 + 2 * tq) =
            make_float2(acc[n][0] * il_lo, acc[n][1] * il_lo);
        *(float2*)(Od + (k * R + r_hi) * 8 + 2 * tq) =
            make_float2(acc[n][2] * il_hi, acc[n][3] * il_hi);
      }
    }
  }
  __syncthreads();

  // ---- phase 2: merge, four threads per row (thread t: row t % R, 8-dim
  // groups t / R + 4i), so that a warp reads 32 consecutive rows of a group,
  // 1 KB contiguous, per load ----
  const int s = seg_of(P.cu_anchor, P.S, j);
  const int lj = j - P.cu_anchor[s];
  const int slab = pp.s_slab_off[s] + lj / P.bps;
  const int rbase = (lj % P.bps) * R;
  // the block sees chunks [c_lo, nact) (none when its context [lo, end) is empty)
  const int na = (P.anchors[j] + P.chunk - 1) / P.chunk;
  const int c_lo = P.ctx_lo[j] >= P.anchors[j] ? na : P.ctx_lo[j] / P.chunk;
  const bool slab_ok = SKV_OK(slab >= 0 && slab < pp.hdr->n_slabs, pp.hdr, kDbgMergeSlot, slab);
  const size_t slot0 = slab_ok ? (size_t)pp.sl_slot[slab] : 0;
  // the block's rows read partial slots slot0 + c, c in [c_lo, nact)
  const int nact = slab_ok && SKV_OK(slot0 + (size_t)na <= (size_t)pp.hdr->n_slot_base, pp.hdr,
                                     kDbgMergeSlot, slot0 + na)
                       ? na
                       : c_lo;
  const size_t cstride = (size_t)P.Hkv * kRows;  // between chunks of a row
  const size_t ostride = cstride * D;
  const int r = threadIdx.x % R, q = threadIdx.x / R;
  const float* plse = wk.part_lse + (slot0 * P.Hkv + g) * kRows + rbase + r;
  const float* prow = wk.part_o + part_off(slot0 * P.Hkv + g, rbase + r, 8 * q, D);
  // pass A: the row's largest lse (log2 units), the draft partial's included
  const float ld = lsed[r];
  float M = ld;
#pragma unroll 4
  for (int c = c_lo; c < nact; ++c) M = fmaxf(M, plse[(size_t)c * cstride] * kLog2eD);
  // pass B: O = (2^(ld - M) O_d + sum_c 2^(lse_c - M) O_c) / T, chunks ascending
  float acc[kGroups][8];
  float T = exp2f(ld - M);
#pragma unroll
  for (int i = 0; i < kGroups; ++i) {
    const float* od = Od + ((q + 4 * i) * R + r) * 8;
    const float4 a = *(const float4*)od, b = *(const float4*)(od + 4);
    acc[i][0] = a.x * T; acc[i][1] = a.y * T; acc[i][2] = a.z * T; acc[i][3] = a.w * T;
    acc[i][4] = b.x * T; acc[i][5] = b.y * T; acc[i][6] = b.z * T; acc[i][7] = b.w * T;
  }
#pragma unroll 2
  for (int c = c_lo; c < nact; ++c) {
    const float w = exp2f(plse[(size_t)c * cstride] * kLog2eD - M);
    T += w;
    const float* pc = prow + (size_t)c * ostride;
#pragma unroll
    for (int i = 0; i < kGroups; ++i) {
      float v[8];
      ld_global_v8(pc + (size_t)(4 * i) * kRows * 8, v);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(w, v[e], acc[i][e]);
    }
  }
  const float inv = 1.f / T;
  const int n = j * P.B + r / G, h = g * G + r % G;
  __nv_bfloat16* o = O + ((size_t)n * P.Hq + h) * D + 8 * q;
#pragma unroll
  for (int i = 0; i < kGroups; ++i) {
    uint4 pk;
    pk.x = pack2(acc[i][0] * inv, acc[i][1] * inv);
    pk.y = pack2(acc[i][2] * inv, acc[i][3] * inv);
    pk.z = pack2(acc[i][4] * inv, acc[i][5] * inv);
    pk.w = pack2(acc[i][6] * inv, acc[i][7] * inv);
    *(uint4*)(o + 32 * i) = pk;
  }
  if (q == 0) LSE[(size_t)h * P.NQ + n] = (M + log2f(T)) * kLn2D;
}

// ===========================================================================
// Backward prologue: D and the draft self-block backward
// ===========================================================================
template <int D, int NT>
__global__ void __launch_bounds__(256) bwd_draft_mma_kernel(
    ProbDev P, PlanPtrs pp, WorkPtrs wk, const __nv_bfloat16* __restrict__ Q,
    const __nv_bfloat16* __restrict__ Kd, const __nv_bfloat16* __restrict__ Vd,
    const __nv_bfloat16* __restrict__ O, const float* __restrict__ LSE,
    const __nv_bfloat16* __restrict__ dO, __nv_bfloat16* __restrict__ dKd,
    __nv_bfloat16* __restrict__ dVd) {
  constexpr int V = D / 8;  // uint4 per row
  extern __shared__ __align__(16) uint8_t smem_raw[];
  if (read_status(pp.hdr) != 0) return;
  const int G = P.group, R = P.B * G;
  const DraftGeom<D> geo(P.B, R);
  __nv_bfloat16* Qs = (__nv_bfloat16*)smem_raw;        // [R][D + 8]
  __nv_bfloat16* dOs = Qs + R * geo.ld_row;             // [R][D + 8]
  __nv_bfloat16* Ks = dOs + R * geo.ld_row;             // [B16][D + 8]
  __nv_bfloat16* Vs = Ks + geo.B16 * geo.ld_row;        // [B16][D + 8]
  __nv_bfloat16* Ps = Vs + geo.B16 * geo.ld_row;        // [R][B16 + 8]  P
  __nv_bfloat16* dSs = Ps + R * geo.ld_key;             // [R][B16 + 8]  dS
  float* Dr = (float*)(dSs + R * geo.ld_key);           // [R]
  const int j = blockIdx.x, g = blockIdx.y;
  if (!SKV_OK(j < P.NA && g < P.Hkv, pp.hdr, kDbgDraftRow, j)) return;  // CTA-uniform
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, tq = lane & 3;
  const int nw = blockDim.x >> 5;
  stage_rows<D>(Qs, geo.ld_row, Q, j * P.B, g * G, G, P.Hq, R);
  stage_keys<D>(Ks, geo.ld_row, Kd, j * P.B, g, P.Hkv, P.B, geo.B16);
  stage_keys<D>(Vs, geo.ld_row, Vd, j * P.B, g, P.Hkv, P.B, geo.B16);
  // dO staged together with D_r = rowsum(dO * O): the V consecutive threads
  // of a row (lanes of one warp: blockDim and V divide each other) sum their
  // 8-element products by shuffles
  for (int base = 0; base < R * V; base += blockDim.x) {  // uniform trip count: every
    const int i = base + threadIdx.x;                     // lane reaches the shuffles
    const int r = i / V, c = i % V;
    float part = 0.f;
    if (i < R * V) {
      const size_t off = ((size_t)(j * P.B + r / G) * P.Hq + g * G + r % G) * D + 8 * c;
      const uint4 d = *(const uint4*)(dO + off);
      const uint4 o = *(const uint4*)(O + off);
      *(uint4*)(dOs + r * geo.ld_row + 8 * c) = d;
      part = dot8_bf16(d, o);
    }
#pragma unroll
    for (int k = V / 2; k > 0; k >>= 1) part += __shfl_xor_sync(0xffffffffu, part, k);
    if (i < R * V && c == 0) {
      Dr[r] = part;
      wk.dvec[(size_t)(g * G + r % G) * P.NQ + j * P.B + r / G] = part;
    }
  }
  __syncthreads();

  // ---- per warp tile (rows 16w .. 16w + 15): P, dS, draft term of dQ ----
  const bool causal = (P.flags & SPLITKV_FLAG_MASK_CAUSAL_BLOCK) != 0;
  for (int w = warp; w < R / 16; w += nw) {
    float s[NT][4], dp[NT][4];
    tile_scores<D, NT>(s, Qs, Ks, geo.ld_row, w, lane);
    tile_scores<D, NT>(dp, dOs, Vs, geo.ld_row, w, lane);
    const int r_lo = 16 * w + gr, r_hi = r_lo + 8;
    const int qi_lo = r_lo / G, qi_hi = r_hi / G;
    const int n_lo = j * P.B + qi_lo, n_hi = j * P.B + qi_hi;
    const int h_lo = g * G + r_lo % G, h_hi = g * G + r_hi % G;
    const float nl_lo = -LSE[(size_t)h_lo * P.NQ + n_lo] * kLog2eD;
    const float nl_hi = -LSE[(size_t)h_hi * P.NQ + n_hi] * kLog2eD;
    const float D_lo = Dr[r_lo], D_hi = Dr[r_hi];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = 8 * n + 2 * tq + (i & 1);
        const bool hi = i >= 2;
        const bool vis = t < P.B && (!causal || t <= (hi ? qi_hi : qi_lo));
        const float p = vis ? exp2f(fmaf(s[n][i], P.scale_log2, hi ? nl_hi : nl_lo)) : 0.f;
        s[n][i] = p;
        dp[n][i] = p * (dp[n][i] - (hi ? D_hi : D_lo));  // dS
      }
      *(uint32_t*)(Ps + r_lo * geo.ld_key + 8 * n + 2 * tq) = pack2(s[n][0], s[n][1]);
      *(uint32_t*)(Ps + r_hi * geo.ld_key + 8 * n + 2 * tq) = pack2(s[n][2], s[n][3]);
      *(uint32_t*)(dSs + r_lo * geo.ld_key + 8 * n + 2 * tq) = pack2(dp[n][0], dp[n][1]);
      *(uint32_t*)(dSs + r_hi * geo.ld_key + 8 * n + 2 * tq) = pack2(dp[n][2], dp[n][3]);
    }
    // draft term of dQ = dS Kd (fp32, unscaled)
    uint32_t a[NT / 2][4];
#pragma unroll
    for (int kk = 0; kk < NT / 2; ++kk) {
      a[kk][0] = pack2(dp[2 * kk][0], dp[2 * kk][1]);
      a[kk][1] = pack2(dp[2 * kk][2], dp[2 * kk][3]);
      a[kk][2] = pack2(dp[2 * kk + 1][0], dp[2 * kk + 1][1]);
      a[kk][3] = pack2(dp[2 * kk + 1][2], dp[2 * kk + 1][3]);
    }
    float acc[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[n][i] = 0.f;
    tile_times_rows<D, NT / 2>(acc, a, Ks, geo.ld_row, lane);
    float* q_lo = wk.dq_draft + ((size_t)n_lo * P.Hq + h_lo) * D + 2 * tq;
    float* q_hi = wk.dq_draft + ((size_t)n_hi * P.Hq + h_hi) * D + 2 * tq;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      *(float2*)(q_lo + 8 * n) = make_float2(acc[n][0], acc[n][1]);
      *(float2*)(q_hi + 8 * n) = make_float2(acc[n][2], acc[n][3]);
    }
  }
  __syncthreads();

  // ---- dVd = P^T dO, dKd = scale dS^T Q: [B16 x D], K = R rows ----
  // unit u = (which, 16-key tile mt, pair of 8-column tiles); the A operand
  // P^T / dS^T comes from the [row][key] tiles by transposed fragment loads
  const int m8 = lane >> 3, r8 = lane & 7;
  const int mtiles = geo.B16 / 16;
  const int per = mtiles * (D / 16);
  for (int u = warp; u < 2 * per; u += nw) {
    const int which = u / per, rest = u % per;
    const int mt = rest / (D / 16), nt = 2 * (rest % (D / 16));
    const __nv_bfloat16* A = which == 0 ? Ps : dSs;    // [row][key]
    const __nv_bfloat16* Bm = which == 0 ? dOs : Qs;   // [row][d]
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    for (int kk = 0; kk < R / 16; ++kk) {
      uint32_t a[4], b[4];
      // a0: keys 0-7 x rows 0-7, a1: keys 8-15 x rows 0-7, a2: keys 0-7 x rows
      // 8-15, a3: keys 8-15 x rows 8-15 (of this 16 x 16 step)
      ldsm_x4_t(a, A + (16 * kk + (m8 >> 1) * 8 + r8) * geo.ld_key + 16 * mt + (m8 & 1) * 8);
      ldsm_x4_t(b, Bm + (16 * kk + (m8 & 1) * 8 + r8) * geo.ld_row + 8 * (nt + (m8 >> 1)));
      mma16816(c0, a, b[0], b[1]);
      mma16816(c1, a, b[2], b[3]);
    }
    const float f = which == 0 ? 1.f : P.scale;
    __nv_bfloat16* dst = which == 0 ? dVd : dKd;
    const int t_lo = 16 * mt + gr, t_hi = t_lo + 8;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float* c = q == 0 ? c0 : c1;
      const int col = 8 * (nt + q) + 2 * tq;
      if (t_lo < P.B)
        *(uint32_t*)(dst + ((size_t)(j * P.B + t_lo) * P.Hkv + g) * D + col) =
            pack2(c[0] * f, c[1] * f);
      if (t_hi < P.B)
        *(uint32_t*)(dst + ((size_t)(j * P.B + t_hi) * P.Hkv + g) * D + col) =
            pack2(c[2] * f, c[3] * f);
    }
  }
}

template <int D>
size_t merge_smem(int B, int R) {
  const int B16 = B <= 16 ? 16 : 32;
  const size_t qk = sizeof(__nv_bfloat16) * (size_t)(R + B16) * (D + 8);
  const size_t od = sizeof(float) * (size_t)R * D;
  return (qk > od ? qk : od) + sizeof(__nv_bfloat16) * (size_t)B16 * (D + 8) + sizeof(float) * R;
}

template <int D>
size_t bwd_smem(int B, int R) {
  const int B16 = B <= 16 ? 16 : 32;
  return sizeof(__nv_bfloat16) * ((size_t)(2 * R + 2 * B16) * (D + 8) + (size_t)2 * R * (B16 + 8)) +
         sizeof(float) * R;
}

template <typename F>
cudaError_t dispatch_mma(const ProbDev& P, F&& f) {
  using D64 = std::integral_constant<int, 64>;
  using D128 = std::integral_constant<int, 128>;
  using N2 = std::integral_constant<int, 2>;
  using N4 = std::integral_constant<int, 4>;
  const bool wide = P.B > 16;
  if (P.d == 64) return wide ? f(D64(), N4()) : f(D64(), N2());
  return wide ? f(D128(), N4()) : f(D128(), N2());
}

}  // namespace

// bf16 problems on the tensor-core path (SPLITKV_FLAG_CUDA_CORE keeps the
// fp32 CUDA-core row kernels, an independent check of these).
bool draft_mma_supported(const ProbDev& P) {
  const int R = P.B * P.group;
  return P.dtype == SPLITKV_BF16 && !(P.flags & SPLITKV_FLAG_CUDA_CORE) &&
         (P.B == 8 || P.B == 16 || P.B == 32) && R >= 16 &&
         R % 16 == 0 && R <= kRows && (P.d == 64 || P.d == 128);
}

cudaError_t launch_merge_draft(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                               const void* Q, const void* Kd, const void* Vd, void* O, float* LSE,
                               cudaStream_t st) {
  return dispatch_mma(P, [&](auto dtag, auto ntag) -> cudaError_t {
    constexpr int D = decltype(dtag)::value;
    constexpr int NT = decltype(ntag)::value;
    const int R = P.B * P.group;
    const size_t smem = merge_smem<D>(P.B, R);
    auto k = merge_draft_kernel<D, NT>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<dim3((unsigned)P.NA, (unsigned)P.Hkv), 4 * R, smem, st>>>(
        P, pp, wk, (const __nv_bfloat16*)Q, (const __nv_bfloat16*)Kd, (const __nv_bfloat16*)Vd,
        (__nv_bfloat16*)O, LSE);
    return cudaGetLastError();
  });
}

cudaError_t launch_bwd_draft_mma(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                                 const void* Q, const void* Kd, const void* Vd, const void* O,
                                 const float* LSE, const void* dO, void* dKd, void* dVd,
                                 cudaStream_t st) {
  return dispatch_mma(P, [&](auto dtag, auto ntag) -> cudaError_t {
    constexpr int D = decltype(dtag)::value;
    constexpr int NT = decltype(ntag)::value;
    const int R = P.B * P.group;
    const size_t smem = bwd_smem<D>(P.B, R);
    auto k = bwd_draft_mma_kernel<D, NT>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // eight warps whatever R: shared memory holds four CTAs per SM, so the
    // extra warps double the loads in flight during staging (the kernel is
    // latency-bound: 4 warps per CTA left 16 warps per SM, 24 % occupancy)
    const int threads = 256;
    k<<<dim3((unsigned)P.NA, (unsigned)P.Hkv), threads, smem, st>>>(
        P, pp, wk, (const __nv_bfloat16*)Q, (const __nv_bfloat16*)Kd, (const __nv_bfloat16*)Vd,
        (const __nv_bfloat16*)O, LSE, (const __nv_bfloat16*)dO, (__nv_bfloat16*)dKd,
        (__nv_bfloat16*)dVd);
    return cudaGetLastError();
  });
}

}  // namespace skv
