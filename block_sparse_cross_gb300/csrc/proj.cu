// Tensor-core GEMMs of the drafter layer's projections around the attention
// (tcgen05 / TMEM / TMA, bf16 inputs, fp32 accumulation).
//
// One persistent kernel computes a group of up to three products ("parts")
//     C_p[M_p, N_p] = sum over segments s of A_ps * B_ps      (along K)
// tiled 128 x 256 with 64-deep k blocks. Each operand is K-major (rows = M or
// N, K contiguous: X and the weights of a forward projection) or MN-major
// (rows = K: a weight read along its output dimension, or the activations
// and gradients of a weight-gradient product); the choice is per part. The
// epilogue writes the columns of C to up to three destination tensors, so
// one launch over the stacked weight [Wq; Wk; Wv] lands Q, Kd and Vd directly
// in the attention's [rows, heads, d] layouts, and the backward sums
// dQ Wq + dKd Wk + dVd Wv (three segments) in one accumulator.
//
// Work units are (part, k slice, output tile); parts are ordered by unit
// length (longest first) and CTA c takes units c, c + grid, ... A part whose
// K is much longer than the others' (the context rows of dWk, dWv) is split
// into k slices whose fp32 results are added with vector atomics into a
// zeroed output; every other output is written once.
//
// Every CTA loads its own A and B tiles into its own shared memory, from
// the tensors its own call was given.
//
// Warp roles (256 threads, one CTA per SM): warp 0 loads A and B tiles with
// TMA into a 4-stage ring, warp 1 issues the MMAs (one elected lane) into one
// of two 256-column TMEM accumulators, warp 2 owns the TMEM allocation, warps
// 4..7 are the epilogue (warp w reads TMEM lane quadrant w % 4, one output row
// per thread) and overlap the next unit's main loop. Every wait is bounded;
// on a timeout the CTA drains its copies and MMAs, frees TMEM and latches
// SPLITKV_ETIMEOUT in a device status word (splitkv_proj_status).
#include <cudaTypedefs.h>
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace skv {

namespace {

using namespace tc;

constexpr int kGM = 128, kGN = 256, kGK = 64;  // output tile, k block
constexpr int kGStages = 4;
constexpr int kGThreads = 256;
constexpr int kGEpiWarp0 = 4;
constexpr uint32_t kGA = kGM * kGK * 2;  // 16 KB: A tile of one stage
constexpr uint32_t kGB = kGN * kGK * 2;  // 32 KB: B tile of one stage
constexpr uint32_t kGStage = kGA + kGB;
constexpr uint32_t kGChunk = 64 * kGK * 2;  // 8 KB: [64 k rows][64 columns] of an MN-major tile
constexpr uint32_t kGBars = kGStages * kGStage;
constexpr uint32_t kGSmem = kGBars + 256 + 1024;  // + barriers, alignment slack
constexpr uint64_t kGDrainNs = 100000000ull;

__device__ int g_proj_status;  // first device error of any projection launch

struct GemmMaps {
  CUtensorMap a[kProjMaxParts][kProjMaxSegs];
  CUtensorMap b[kProjMaxParts][kProjMaxSegs];
};

struct GUnit {
  int p, m0, n0, kb_lo, kb_hi;
};

// Unit u of a group: part p, k slice s, output tile (mt, nt), n fastest so
// that CTAs running side by side share the A rows.
__device__ __forceinline__ GUnit decode_unit(const ProjGroup& G, int u) {
  int p = 0;
  while (p + 1 < G.nparts && u >= G.part[p + 1].unit0) ++p;
  const ProjPart& P = G.part[p];
  int r = u - P.unit0;
  const int per_slice = P.mt * P.nt;
  const int s = r / per_slice;
  r -= s * per_slice;
  const int mt = r / P.nt;
  GUnit U;
  U.p = p;
  U.m0 = mt * kGM;
  U.n0 = (r - mt * P.nt) * kGN;
  U.kb_lo = s * P.kb_per_split;
  U.kb_hi = min(P.nkb, U.kb_lo + P.kb_per_split);
  return U;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ bool gwait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool mine = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, mine);
}

__global__ void __launch_bounds__(kGThreads, 1)
    proj_gemm_kernel(const __grid_constant__ GemmMaps maps, const ProjGroup G) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + kGBars);
  uint64_t* full = bars;                    // [stages] TMA -> MMA
  uint64_t* empty = full + kGStages;        // [stages] MMA -> TMA
  uint64_t* acc_full = empty + kGStages;    // [2] MMA -> epilogue
  uint64_t* acc_empty = acc_full + 2;       // [2] epilogue (4 warps) -> MMA
  uint64_t* mma_drain = acc_empty + 2;
  uint32_t* tmem_slot = (uint32_t*)(mma_drain + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGStages; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(acc_full + i, 1);
      mbar_init(acc_empty + i, 4);
    }
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer (whole warp waits, one lane issues) ----------------
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < G.units && ok; u += gridDim.x) {
      const GUnit U = decode_unit(G, u);
      const ProjPart& P = G.part[U.p];
      int sg = 0;
      for (int kb = U.kb_lo; kb < U.kb_hi; ++kb, ++it) {
        while (sg + 1 < P.nseg && kb >= P.seg[sg + 1].kb0) ++sg;
        const ProjSeg& S = P.seg[sg];
        const int k = (kb - S.kb0) * kGK;
        const uint32_t st = it % kGStages, ph = it / kGStages;
        if (ph > 0 && !(ok = gwait(empty + st, (ph - 1) & 1, abort_flag))) break;
        uint8_t* sa = smem + st * kGStage;
        uint8_t* sb = sa + kGA;
        if (elect_one()) {
          mbar_expect_tx(full + st, kGStage);
          const CUtensorMap* ma = &maps.a[U.p][sg];
          const CUtensorMap* mb = &maps.b[U.p][sg];
          if (P.a_mn) {
            for (int i = 0; i < kGM / 64; ++i)
              tma_load_2d(sa + i * kGChunk, ma, full + st, P.a_off + U.m0 + 64 * i, S.a_k + k);
          } else {
            tma_load_2d(sa, ma, full + st, S.a_k + k, P.a_off + U.m0);
          }
          if (P.b_mn) {
            for (int i = 0; i < kGN / 64; ++i)
              tma_load_2d(sb + i * kGChunk, mb, full + st, P.b_off + U.n0 + 64 * i, S.b_k + k);
          } else {
            tma_load_2d(sb, mb, full + st, S.b_k + k, P.b_off + U.n0);
          }
        }
        __syncwarp();
      }
    }
    if (!ok) {  // let every copy in flight land before the CTA exits
      for (uint32_t j = it > (uint32_t)kGStages ? it - kGStages : 0; j < it; ++j)
        mbar_wait_drain(full + j % kGStages, (j / kGStages) & 1, kGDrainNs);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    uint32_t it = 0, nu = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < G.units && ok; u += gridDim.x, ++nu) {
      const GUnit U = decode_unit(G, u);
      const ProjPart& P = G.part[U.p];
      const uint32_t ab = nu & 1, au = nu >> 1;
      if (au > 0 && !(ok = gwait(acc_empty + ab, (au - 1) & 1, abort_flag))) break;
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(kGM, kGN, P.a_mn != 0, P.b_mn != 0);
      const uint32_t d_tmem = tmem + ab * kGN;
      for (int kb = U.kb_lo; kb < U.kb_hi; ++kb, ++it) {
        const uint32_t st = it % kGStages, ph = it / kGStages;
        if (!(ok = gwait(full + st, ph & 1, abort_flag))) break;
        tc_fence_after();
        if (elect_one()) {
          const uint32_t sa = smem_u32(smem + st * kGStage), sb = sa + kGA;
          // MN-major: 8 KB per 64 columns (LBO), 1 KB per 8 k rows (SBO),
          // 2 KB per 16-row k step; K-major: 1 KB per 8 rows, 32 B per k step.
          const uint64_t ad = P.a_mn ? sdesc_sw128(sa, kGChunk, 1024u) : desc_kmajor0(sa);
          const uint64_t bd = P.b_mn ? sdesc_sw128(sb, kGChunk, 1024u) : desc_kmajor0(sb);
#pragma unroll
          for (int kk = 0; kk < kGK / 16; ++kk) {
            const uint32_t ao = P.a_mn ? (uint32_t)kk * 2048u : (uint32_t)kk * 32u;
            const uint32_t bo = P.b_mn ? (uint32_t)kk * 2048u : (uint32_t)kk * 32u;
            mma_ss(d_tmem, ad + (ao >> 4), bd + (bo >> 4), idesc,
                   (kb > U.kb_lo || kk > 0) ? 1u : 0u);
          }
          mma_commit(empty + st);  // frees the stage once these MMAs have read it
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) mma_commit(acc_full + ab);
      __syncwarp();
    }
    if (elect_one()) mma_commit(mma_drain);  // every MMA of this CTA is done
    __syncwarp();
    mbar_wait_drain(mma_drain, 0, kGDrainNs);
  } else if (warp >= kGEpiWarp0) {
    // ---------------- epilogue: one output row per thread ----------------
    const int q = warp & 3;
    uint32_t nu = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < G.units && ok; u += gridDim.x, ++nu) {
      const GUnit U = decode_unit(G, u);
      const ProjPart& P = G.part[U.p];
      const uint32_t ab = nu & 1, au = nu >> 1;
      if (!(ok = gwait(acc_full + ab, au & 1, abort_flag))) break;
      tc_fence_after();
      const int row = U.m0 + q * 32 + lane;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + ab * kGN;
      for (int c = 0; c < kGN / 32; ++c) {
        const int col = U.n0 + c * 32;
        if (col >= P.N) break;  // warp-uniform
        uint32_t r[32];
        tmem_ld32(taddr + c * 32, r);
        tmem_ld_wait(r);
        if (row >= P.M) continue;
        int di = 0;
        while (di + 1 < P.ndst && col >= P.dst[di + 1].col0) ++di;
        const ProjDst& D = P.dst[di];
        const size_t off = (size_t)row * D.ld + (col - D.col0);
        if (!P.out_f32) {
          uint4* dst = (uint4*)((__nv_bfloat16*)D.ptr + off);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(r[8 * j + 0]), __uint_as_float(r[8 * j + 1]));
            v.y = pack_bf16(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3]));
            v.z = pack_bf16(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5]));
            v.w = pack_bf16(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7]));
            dst[j] = v;
          }
        } else if (P.ksplit == 1) {
          float* dst = (float*)D.ptr + off;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            st_global_v8(dst + 8 * j, __uint_as_float(r[8 * j]), __uint_as_float(r[8 * j + 1]),
                         __uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3]),
                         __uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5]),
                         __uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7]));
        } else {
          float4* dst = (float4*)((float*)D.ptr + off);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            atomicAdd(dst + j, make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                           __uint_as_float(r[4 * j + 2]),
                                           __uint_as_float(r[4 * j + 3])));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + ab);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0 && *abort_flag) atomicCAS(&g_proj_status, 0, (int)SPLITKV_ETIMEOUT);
}

// ---- host -------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

// 2-D bf16 map over a row-major [rows][cols] tensor with a {64, box_rows} box.
cudaError_t map_2d(CUtensorMap* m, const void* base, int64_t cols, int64_t rows,
                   uint32_t box_rows) {
  auto fn = encode_tiled();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

cudaError_t launch_proj(const ProjSpec* parts, int nparts, cudaStream_t st) {
  if (nparts < 1 || nparts > kProjMaxParts) return cudaErrorInvalidValue;
  // longest units first (ties: caller's order), so the short ones fill the tail
  int order[kProjMaxParts];
  int64_t len[kProjMaxParts];
  for (int i = 0; i < nparts; ++i) {
    const ProjSpec& s = parts[i];
    int64_t nkb = 0;
    for (int j = 0; j < s.nseg; ++j) nkb += (s.klen[j] + kGK - 1) / kGK;
    const int ks = s.ksplit < 1 ? 1 : s.ksplit;
    len[i] = (nkb + ks - 1) / ks;
    order[i] = i;
  }
  for (int i = 1; i < nparts; ++i)
    for (int j = i; j > 0 && len[order[j]] > len[order[j - 1]]; --j) {
      const int t = order[j];
      order[j] = order[j - 1];
      order[j - 1] = t;
    }
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  GemmMaps maps;
  memset(&maps, 0, sizeof(maps));
  ProjGroup G;
  memset(&G, 0, sizeof(G));
  int64_t units = 0;
  for (int oi = 0; oi < nparts; ++oi) {
    const ProjSpec& s = parts[order[oi]];
    ProjPart& P = G.part[oi];
    if (s.nseg < 1 || s.nseg > kProjMaxSegs || s.ndst < 1 || s.ndst > kProjMaxDst ||
        s.M < 1 || s.N < 1)
      return cudaErrorInvalidValue;
    P.M = (int)s.M;
    P.N = (int)s.N;
    P.mt = (int)((s.M + kGM - 1) / kGM);
    P.nt = (int)((s.N + kGN - 1) / kGN);
    P.a_mn = s.a_mn;
    P.b_mn = s.b_mn;
    P.a_off = (int)s.a_off;
    P.b_off = (int)s.b_off;
    P.nseg = s.nseg;
    int kb = 0;
    for (int j = 0; j < s.nseg; ++j) {
      P.seg[j].kb0 = kb;
      P.seg[j].a_k = (int)s.k0_a[j];
      P.seg[j].b_k = (int)s.k0_b[j];
      kb += (int)((s.klen[j] + kGK - 1) / kGK);
      // K-major: [rows][K] with a {64 k, 128 | 256 rows} box; MN-major:
      // [K rows][cols] with {64 columns, 64 k rows} boxes.
      cudaError_t e = map_2d(&maps.a[oi][j], s.a[j].ptr, s.a[j].cols, s.a[j].rows,
                             s.a_mn ? 64u : (uint32_t)kGM);
      if (e != cudaSuccess) return e;
      e = map_2d(&maps.b[oi][j], s.b[j].ptr, s.b[j].cols, s.b[j].rows,
                 s.b_mn ? 64u : (uint32_t)kGN);
      if (e != cudaSuccess) return e;
    }
    P.nkb = kb;
    const int ks = s.ksplit < 1 ? 1 : s.ksplit;
    P.kb_per_split = (kb + ks - 1) / ks;
    P.ksplit = (kb + P.kb_per_split - 1) / P.kb_per_split;
    P.out_f32 = s.out_f32;
    P.ndst = s.ndst;
    for (int j = 0; j < s.ndst; ++j) P.dst[j] = s.dst[j];
    P.unit0 = (int)units;
    units += (int64_t)P.mt * P.nt * P.ksplit;
  }
  G.nparts = nparts;
  if (units == 0) return cudaSuccess;
  if (units >= (1LL << 31)) return cudaErrorInvalidValue;
  G.units = (int)units;
  const int grid = (int)std::min<int64_t>(units, sms);
  cudaError_t e = cudaFuncSetAttribute(proj_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kGSmem);
  if (e != cudaSuccess) return e;
  proj_gemm_kernel<<<grid, kGThreads, kGSmem, st>>>(maps, G);
  return cudaGetLastError();
}

cudaError_t proj_status(int* status, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(status, g_proj_status, sizeof(int));
  if (e == cudaSuccess && clear) {
    const int z = 0;
    e = cudaMemcpyToSymbol(g_proj_status, &z, sizeof(int));
  }
  return e;
}

}  // namespace skv
