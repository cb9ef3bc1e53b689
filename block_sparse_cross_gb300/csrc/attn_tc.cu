// Tensor-core (tcgen05 / TMEM / TMA) attention kernels of the split, bf16
// inputs, fp32 accumulation. Same items and partial layout as the CUDA-core
// kernels (attn_simt.cu):
//
//  fwd    item (sample, chunk, slab, kv head) = 128 (query, head) rows x the
//         chunk's visible keys. Per 128-key tile: S = Q K^T (SS MMA into
//         TMEM), online softmax in registers, P (bf16) written back over S,
//         O += P V (TS MMA, A from TMEM). Emits the chunk partial
//         (lse_c, O_c / l_c) of every row: the local part of attention that
//         the rit.work article on Split-KV (section "Split-KV двигает
//         запросы, а не ключи и значения") assigns to each KV shard.
//  dq     same items: S = Q K^T, dP = dO V^T, dS = P (dP - D) with
//         P = exp(S*scale - LSE), dQ_c += dS K (TS MMA). Emits the fp32 dQ
//         partial of the chunk (the query gradient that moves).
//  dkdv   item (sample, 128-key tile, kv head): the tile stays put (local
//         K/V gradients) while every slab of rows that sees it streams by:
//         S^T = K Q^T, dP^T = V dO^T, dV += P^T dO, dK += dS^T Q.
//
// Warp roles (320 threads): warp 0 issues TMA, warp 1 allocates TMEM and
// issues every MMA (the warp runs the control loop, one elected lane issues),
// warps 2..9 do the softmax and the epilogue: warp w owns TMEM lane quadrant
// w % 4 (one row (fwd/dq) or one key (dkdv) per thread) and one half of the
// 128 columns. All waits are bounded (tc_common.cuh); on a
// timeout the CTA winds down, drains its copies and MMAs, frees TMEM and
// latches SPLITKV_ETIMEOUT.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace skv {

namespace {

using namespace tc;

constexpr int kNS = 2;               // pipeline stages
// Warps 0 (TMA), 1 (MMA), 2..9 (softmax) in every kernel; the forward and
// dQ kernels add warp 10 (a second MMA issuer), warps 11..14 (epilogue, one
// per TMEM lane quadrant) and warp 15 (V loads).
constexpr int kThreads = 512;    // forward and dQ
constexpr int kVWarp = 15;
// dK / dV: warps 2..17 are the softmax (four per TMEM lane quadrant, one
// 32-row quarter of the slab each; on config 4 at L = 262144 this ran 2 %
// faster than two half-row warps per quadrant), warp 18 loads dO, warp 19
// sums the dQ kernel's chunk partials into dQ while the tensor pipe works
// (the reduction reads HBM, the rest of the kernel hardly does). Twenty
// warps put five on each SM sub-partition, which leaves 96 registers a
// thread; a 21st warp would cut that to 80.
constexpr int kKvSoftmaxWarps = 16;
constexpr int kKvDoWarp = 2 + kKvSoftmaxWarps;
constexpr int kKvRedWarp = kKvDoWarp + 1;
constexpr int kThreadsKv = 32 * (kKvRedWarp + 1);
// the reduction streams [128 rows][8] fp32 pieces (4 KB, one dims group of a
// partial tile, contiguous) through a ring of shared-memory stages
constexpr int kRedStages = 6;
constexpr uint32_t kRedPieceBytes = kRows * 8u * 4u;
// Stages read before they are refilled together, and the pause between polls
// of a stage not yet filled. On one box, at config 4 L = 262144, polling
// without a pause and refilling every stage at once ran the kernel 1.7 %
// slower than these values (the warp's issue slots are the softmax warps').
constexpr int kRedRefill = 3;
constexpr uint32_t kRedSleepNs = 200;
constexpr int kEpiWarp0 = 11;
constexpr int kSoftmaxWarps = 8;  // two per TMEM lane quadrant, one column half each
constexpr uint32_t kSubBytes = 16384; // one [128 rows][64 bf16] swizzled sub-tile
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kDrainNs = 100000000ull;

using FwdItem = FwdRec;

// The planner's decoded record of queue position p (read-only here). The
// loads are volatile asm so that they stay where they are written: every
// role issues the next item's record load when the current item starts and
// uses it one item later, off the item boundary's critical path.
__device__ __forceinline__ FwdRec ld_rec(const FwdRec* p) {
  FwdRec R;
  asm volatile("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(R.n0), "=r"(R.g), "=r"(R.row0), "=r"(R.cs)
               : "l"(p));
  asm volatile("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4 + 16];"
               : "=r"(R.ntiles), "=r"(R.first), "=r"(R.nblk), "=r"(R.slot)
               : "l"(p));
  return R;
}
__device__ __forceinline__ int ld_int_early(const int* p) {
  int v;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_float_early(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// Row r of an item (as row_info), with the anchor load issued now.
__device__ __forceinline__ RowInfo row_info_early(const ProbDev& P, const FwdRec& I, int r) {
  RowInfo ri;
  const int per_blk = P.B * P.group;
  const int b = r / per_blk;
  if (b >= I.nblk) {
    ri.n = -1; ri.h = 0; ri.anchor = 0; ri.lo = 0;
    return ri;
  }
  ri.n = (I.first + b) * P.B + (r / P.group) % P.B;
  ri.h = I.g * P.group + r % P.group;
  ri.anchor = ld_int_early(P.anchors + I.first + b);
  ri.lo = ld_int_early(P.ctx_lo + I.first + b);
  return ri;
}

// TMEM column of the packed bf16 A operand (P, dS, P^T, dS^T) for k step kk
// of a 128-key tile: each softmax column half h writes its 64 keys as 32
// packed columns at 64h, inside its own half of the fp32 tile it read, so
// the two halves never write where the other still reads.
__device__ __forceinline__ uint32_t a_col(int kk) { return (uint32_t)(kk * 8 + (kk >= 4 ? 32 : 0)); }
// The same for the dK/dV kernel's P^T and dS^T: softmax quarter q (rows
// 32q .. 32q + 31 of the slab) writes its 32 rows as 16 packed columns at the
// start of its own 32 fp32 columns.
__device__ __forceinline__ uint32_t kv_acol(int kk) { return (uint32_t)(32 * (kk >> 1) + 8 * (kk & 1)); }

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool mine = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, mine);
}

// The first 1024-byte boundary at or after p, a pointer into the dynamic
// shared array. It is reached by pointer arithmetic on p so that the compiler
// still knows the result points to shared memory: an integer round trip
// would turn every access through it into a generic load or store.
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

// ===========================================================================
// Forward
// ===========================================================================
// Two 128-column S buffers and two O accumulators fill the 512 TMEM columns
// at d = 128. Each softmax warp owns one 64-key half of every tile and keeps
// its own running maximum, row sum and O accumulator (O_h += P_h V_h, the
// keys of half h), so the two halves never meet during an item; the
// epilogue combines (m_0, l_0, O_0) and (m_1, l_1, O_1) once per item. The K
// stage, S buffer and V stage of tile t all have index t % 2.
constexpr int kFwdNK = 2, kFwdNV = 2;

template <int D>
struct FwdLayout {
  static constexpr int kSub = D / 64;
  static constexpr uint32_t tile = kSub * kSubBytes;  // one 128 x D bf16 tile
  static constexpr uint32_t q = 0;  // two Q tiles: item i uses i % 2
  static constexpr uint32_t k0 = 2 * tile;
  static constexpr uint32_t v0 = k0 + kFwdNK * tile;
  static constexpr uint32_t lm = v0 + kFwdNV * tile;  // [4][128] floats: l_0, l_1, m_0, m_1
  static constexpr uint32_t bars = lm + 2048;
  static constexpr uint32_t total = bars + 512 + 1024;  // + alignment slack
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, ProbDev P, PlanPtrs pp, WorkPtrs wk) {
  using Lay = FwdLayout<D>;
  constexpr int kSub = Lay::kSub;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = (uint64_t*)(smem + Lay::bars);
  // Tile t (counted over the CTA's items) uses index b = t % 2. S of tile t
  // is issued once both PV halves of tile t-2 are done (sfree); PV half h of
  // tile t once that half's P is written (p_ready[b][h]). The K stage is
  // free when S is done (s_full), the V stage when PV is done (sfree). Item
  // i's Q is in buffer i % 2, so the next item's Q lands while this item's
  // last tiles run.
  static_assert(kFwdNK == 2 && kFwdNV == 2, "ring sizes tied to the S buffers");
  uint64_t* q_full = bars + 0;          // [2]
  uint64_t* q_empty = bars + 2;         // [2] the item's last S is done
  uint64_t* k_full = bars + 4;          // [2]
  uint64_t* v_full = k_full + 2;        // [2]
  uint64_t* s_full = v_full + 2;        // [2] S of tile t is in buffer t % 2
  uint64_t* p_ready = s_full + 2;       // [2][2] P of half h written over its S half
  uint64_t* sfree = p_ready + 4;        // [2] both PV halves of tile t are done
  uint64_t* o_free = sfree + 2;         // the epilogue has read O_0, O_1 and the row sums
  uint64_t* lm_ready = o_free + 1;      // the softmax has written the item's (m, l)
  uint64_t* mma_drain = lm_ready + 1;   // [2] one per issuing warp
  uint64_t* stg_free = mma_drain + 2;   // [2] the epilogue is done with Q buffer b as staging
  uint32_t* tmem_slot = (uint32_t*)(bars + 32);
  volatile int* abort_flag = (volatile int*)(bars + 33);

  if (!plan_ok_cta(P, pp.hdr)) return;
  if (threadIdx.x == 0) stamp_busy(P, pp, 0, 0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(q_full + b, 1);
      mbar_init(q_empty + b, 1);
      mbar_init(k_full + b, 1);
      mbar_init(v_full + b, 1);
      mbar_init(s_full + b, 1);
      mbar_init(p_ready + 2 * b, kSoftmaxWarps / 2);
      mbar_init(p_ready + 2 * b + 1, kSoftmaxWarps / 2);
      mbar_init(sfree + b, 1);
    }
    mbar_init(o_free, 4);
    mbar_init(stg_free, 4);
    mbar_init(stg_free + 1, 4);
    mbar_init(lm_ready, kSoftmaxWarps);
    mbar_init(mma_drain, 1);
    mbar_init(mma_drain + 1, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 256;  // two S buffers, then O_0 and O_1 (D columns each)
  float* lm = (float*)(smem + Lay::lm);
  const int q0 = pp.f_qoff[blockIdx.x];
  const int q1 = queue_end(pp.f_qoff, blockIdx.x, (int64_t)pp.hdr->n_fwd_items * P.Hkv, pp.hdr);

  if (warp == 0) {
    // ---------------- TMA producer: Q and K (V comes from warp 15) ----------------
    {  // the whole warp runs the loop and waits; one elected lane issues the copies
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      uint32_t nq = 0, nk = 0;
      bool ok = true;
      FwdItem In = q0 < q1 ? ld_rec(pp.f_rec + q0) : FwdItem{};
      for (int qi = q0; qi < q1 && ok; ++qi) {
        const FwdItem I = In;
        if (qi + 1 < q1) In = ld_rec(pp.f_rec + qi + 1);  // lands during this item
        const uint32_t qb = nq & 1;
        // buffer qb is free once the last S of item nq - 2 is done
        if (nq >= 2 && !(ok = warp_wait(q_empty + qb, ((nq >> 1) - 1) & 1, abort_flag))) break;
        // ... and once the epilogue of that item has used it as staging
        if (nq >= 2 && !(ok = warp_wait(stg_free + qb, ((nq >> 1) - 1) & 1, abort_flag))) break;
        if (elect_one()) {
          mbar_expect_tx(q_full + qb, Lay::tile);
          for (int i = 0; i < kSub; ++i)
            tma_load_3d(smem + Lay::q + qb * Lay::tile + i * kSubBytes, &tmQ, q_full + qb, 64 * i,
                        I.g * P.group, I.n0);
        }
        __syncwarp();
        ++nq;
        for (int t = 0; t < I.ntiles; ++t) {
          const uint32_t s = nk % kFwdNK, u = nk / kFwdNK;
          // stage s is free once S of tile nk - 2 is done
          if (u > 0 && !(ok = warp_wait(s_full + s, (u - 1) & 1, abort_flag))) break;
          uint8_t* kb = smem + Lay::k0 + s * Lay::tile;
          if (elect_one()) {
            mbar_expect_tx(k_full + s, Lay::tile);
            for (int i = 0; i < kSub; ++i)
              tma_load_3d(kb + i * kSubBytes, &tmK, k_full + s, 64 * i, I.g, I.row0 + t * kKeyTile);
          }
          __syncwarp();
          ++nk;
        }
      }
      if (!ok) {  // let every copy in flight land before the CTA exits
        for (uint32_t j = nq > 2u ? nq - 2 : 0; j < nq; ++j)
          mbar_wait_drain(q_full + (j & 1), (j >> 1) & 1, kDrainNs);
        for (uint32_t j = nk > (uint32_t)kFwdNK ? nk - kFwdNK : 0; j < nk; ++j)
          mbar_wait_drain(k_full + j % kFwdNK, (j / kFwdNK) & 1, kDrainNs);
      }
    }
  } else if (warp == kVWarp) {
    // ---------------- V producer: its own warp, so that it runs in parallel
    // with the Q/K producer instead of taking turns with it ----------------
    {  // the whole warp runs the loop and waits; one elected lane issues the copies
      tma_prefetch_desc(&tmV);
      uint32_t nv = 0;
      bool ok = true;
      FwdItem In = q0 < q1 ? ld_rec(pp.f_rec + q0) : FwdItem{};
      for (int qi = q0; qi < q1 && ok; ++qi) {
        const FwdItem I = In;
        if (qi + 1 < q1) In = ld_rec(pp.f_rec + qi + 1);  // lands during this item
        for (int t = 0; t < I.ntiles; ++t) {
          const uint32_t s = nv % kFwdNV, u = nv / kFwdNV;
          // stage s is free once both PV halves of tile nv - 2 are done
          if (u > 0 && !(ok = warp_wait(sfree + s, (u - 1) & 1, abort_flag))) break;
          uint8_t* vb = smem + Lay::v0 + s * Lay::tile;
          if (elect_one()) {
            mbar_expect_tx(v_full + s, Lay::tile);
            for (int i = 0; i < kSub; ++i)
              tma_load_3d(vb + i * kSubBytes, &tmV, v_full + s, 64 * i, I.g, I.row0 + t * kKeyTile);
          }
          __syncwarp();
          ++nv;
        }
      }
      if (!ok) {
        for (uint32_t j = nv > (uint32_t)kFwdNV ? nv - kFwdNV : 0; j < nv; ++j)
          mbar_wait_drain(v_full + j % kFwdNV, (j / kFwdNV) & 1, kDrainNs);
      }
    }
  } else if (warp == 1) {
    // ---------------- S issuer: the whole warp, one elected lane issues ----------------
    // A commit holds its thread until the MMAs it tracks are nearly done, so
    // S and PV are issued by two warps: while one waits on its commit the
    // other keeps the tensor pipe fed.
    constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
    uint32_t ns = 0, nit = 0;
    bool ok = true;
    FwdItem In = q0 < q1 ? ld_rec(pp.f_rec + q0) : FwdItem{};
    for (int qi = q0; qi < q1 && ok; ++qi, ++nit) {
      const FwdItem I = In;
      if (qi + 1 < q1) In = ld_rec(pp.f_rec + qi + 1);  // lands during this item
      const uint32_t qb = nit & 1;
      if (!(ok = warp_wait(q_full + qb, (nit >> 1) & 1, abort_flag))) break;
      const uint64_t qd0 = desc_kmajor0(smem_u32(smem + Lay::q + qb * Lay::tile));
      for (int t = 0; t < I.ntiles; ++t, ++ns) {
        const uint32_t b = ns & 1;
        if (!(ok = warp_wait(k_full + b, (ns >> 1) & 1, abort_flag))) break;
        if (ns >= 2 && !(ok = warp_wait(sfree + b, ((ns >> 1) - 1) & 1, abort_flag))) break;
        tc_fence_after();
        const uint64_t kd0 = desc_kmajor0(smem_u32(smem + Lay::k0 + b * Lay::tile));
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tS + b * 128, qd0 + (kmajor_off(kk) >> 4), kd0 + (kmajor_off(kk) >> 4), kIdS,
                   kk > 0 ? 1u : 0u);
          mma_commit(s_full + b);  // also frees K stage b
          if (t == I.ntiles - 1) mma_commit(q_empty + qb);
        }
        __syncwarp();
      }
    }
    if (elect_one()) mma_commit(mma_drain);
    __syncwarp();
    mbar_wait_drain(mma_drain, 0, kDrainNs);
  } else if (warp == kSoftmaxWarps + 2) {
    // ---------------- PV issuer: O_h += P_h V_h, half by half ----------------
    constexpr uint32_t kIdPV = idesc_bf16(128, D, false, true);
    uint32_t np = 0, nit = 0;
    bool ok = true;
    FwdItem In = q0 < q1 ? ld_rec(pp.f_rec + q0) : FwdItem{};
    for (int qi = q0; qi < q1 && ok; ++qi, ++nit) {
      const FwdItem I = In;
      if (qi + 1 < q1) In = ld_rec(pp.f_rec + qi + 1);  // lands during this item
      for (int t = 0; t < I.ntiles && ok; ++t, ++np) {
        const uint32_t b = np & 1;
        if (!(ok = warp_wait(v_full + b, (np >> 1) & 1, abort_flag))) break;
        if (t == 0 && nit > 0 && !(ok = warp_wait(o_free, (nit - 1) & 1, abort_flag))) break;
        const uint64_t vd0 = desc_mnmajor0(smem_u32(smem + Lay::v0 + b * Lay::tile));
        const uint32_t ta = tS + b * 128;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!(ok = warp_wait(p_ready + 2 * b + h, (np >> 1) & 1, abort_flag))) break;
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
              mma_ts(tO + h * D, ta + a_col(kk), vd0 + (mnmajor_off(kk) >> 4), kIdPV,
                     (t == 0 && kk == 4 * h) ? 0u : 1u);
            if (h == 1) mma_commit(sfree + b);  // both halves; also frees V stage b
          }
          __syncwarp();
        }
      }
    }
    if (elect_one()) mma_commit(mma_drain + 1);
    __syncwarp();
    mbar_wait_drain(mma_drain + 1, 0, kDrainNs);
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ---------------- epilogue (warps 11..14): one lane quadrant each ----------------
    // Waits for the item's last PV and its (m, l) per half and combines the
    // halves (O = sum_h 2^(m_h - m) O_h / l, l = sum_h 2^(m_h - m) l_h). The
    // accumulators are read out of TMEM before anything is written to global
    // memory, and released at once (the next item's first PV overwrites them
    // and waits for that): columns [0, D/2) go to a staging row in the item's
    // Q buffer (free: the item's S are all done, and the next Q load into it
    // waits for stg_free), columns [D/2, D) stay in registers. Then the chunk
    // partial (O / l, lse) is written out. The softmax warps never wait for it.
    constexpr int DH = D / 2;   // staged columns per row
    constexpr int NC = DH / 4;  // 16-byte chunks per staged row (swizzled by row)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    uint32_t ns = 0, nit = 0;
    bool ok = true;
    FwdItem In = q0 < q1 ? ld_rec(pp.f_rec + q0) : FwdItem{};
    for (int qi = q0; qi < q1 && ok; ++qi, ++nit) {
      const FwdItem I = In;
      if (qi + 1 < q1) In = ld_rec(pp.f_rec + qi + 1);  // lands during this item
      ns += I.ntiles;
      const uint32_t pt = ns - 1;  // the item's last tile
      if (!(ok = warp_wait(lm_ready, nit & 1, abort_flag))) break;
      if (!(ok = warp_wait(sfree + (pt & 1), (pt >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      const float m0 = lm[256 + r], m1 = lm[384 + r];  // log2 units
      const float m = fmaxf(m0, m1);
      const float w0 = m0 == -INFINITY ? 0.f : ex2(m0 - m);
      const float w1 = m1 == -INFINITY ? 0.f : ex2(m1 - m);
      const float lt = lm[r] * w0 + lm[128 + r] * w1;
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float f0 = w0 * inv, f1 = w1 * inv;
      const bool sok = SKV_OK(I.slot >= 0 && (int64_t)I.slot < (int64_t)pp.hdr->n_slot_base * P.Hkv,
                              pp.hdr, kDbgFwdSlot, I.slot);
      const uint32_t qb = nit & 1;
      float* stg = (float*)(smem + Lay::q + qb * Lay::tile) + r * DH;
      auto chunk = [&](int ch) { return 4 * (ch ^ (r & (NC - 1))); };
#pragma unroll 1
      for (int c = 0; c < DH; c += 16) {
        uint32_t a[16], b[16];
        tmem_ld16(tO + lane_base + c, a);
        tmem_ld16(tO + D + lane_base + c, b);
        tmem_ld_wait16(a);
        tmem_ld_wait16(b);
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          float4 v;
          v.x = fmaf(__uint_as_float(a[j]), f0, __uint_as_float(b[j]) * f1);
          v.y = fmaf(__uint_as_float(a[j + 1]), f0, __uint_as_float(b[j + 1]) * f1);
          v.z = fmaf(__uint_as_float(a[j + 2]), f0, __uint_as_float(b[j + 2]) * f1);
          v.w = fmaf(__uint_as_float(a[j + 3]), f0, __uint_as_float(b[j + 3]) * f1);
          *(float4*)(stg + chunk((c + j) / 4)) = v;
        }
      }
      float oh[DH];
#pragma unroll
      for (int c = 0; c < DH; c += 16) {
        uint32_t a[16], b[16];
        tmem_ld16(tO + lane_base + DH + c, a);
        tmem_ld16(tO + D + lane_base + DH + c, b);
        tmem_ld_wait16(a);
        tmem_ld_wait16(b);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          oh[c + j] = fmaf(__uint_as_float(a[j]), f0, __uint_as_float(b[j]) * f1);
      }
      tc_fence_before();  // O and the row statistics are in registers and staging
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
      if (sok) {
#pragma unroll
        for (int i = 0; i < DH; i += 8)
          st_global_v8(wk.part_o + part_off(I.slot, r, DH + i, D), oh[i], oh[i + 1], oh[i + 2],
                       oh[i + 3], oh[i + 4], oh[i + 5], oh[i + 6], oh[i + 7]);
#pragma unroll
        for (int i = 0; i < DH; i += 8) {
          const float4 x = *(const float4*)(stg + chunk(i / 4));
          const float4 y = *(const float4*)(stg + chunk(i / 4 + 1));
          st_global_v8(wk.part_o + part_off(I.slot, r, i, D), x.x, x.y, x.z, x.w, y.x, y.y, y.z,
                       y.w);
        }
        wk.part_lse[(size_t)I.slot * kRows + r] = lt > 0.f ? (m + log2f(lt)) * kLn2 : -INFINITY;
      }
      fence_proxy_async_shared();  // the staging reads come before the next TMA load here
      __syncwarp();
      if (lane == 0) mbar_arrive(stg_free + qb);
    }
  } else {
    // ---------------- softmax (warps 2..9) ----------------
    // Warp w owns TMEM lane quadrant w % 4 (rows r) and key half hf of every
    // tile, with its own running maximum m_run (log2 units), row sum l and
    // accumulator O_hf; lazy rescale keeps exponents <= 2^8.
    const int wq = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const float sl2 = P.scale_log2;
    const uint32_t tOh = tO + hf * D + lane_base;
    uint32_t ns = 0;
    bool ok = true;
    // The next item's record is loaded when an item starts and the row's
    // anchor once its first tile is done, so neither load is waited for at
    // the item boundary.
    FwdItem In{};
    RowInfo rin{};
    if (q0 < q1) {
      In = ld_rec(pp.f_rec + q0);
      rin = row_info_early(P, In, r);
    }
    for (int qi = q0, nit = 0; qi < q1 && ok; ++qi, ++nit) {
      const FwdItem I = In;
      const RowInfo ri = rin;
      bool row_next = qi + 1 >= q1;  // the next item's row is loaded (or not needed)
      if (!row_next) In = ld_rec(pp.f_rec + qi + 1);
      float m_run = -INFINITY, l = 0.f;
      for (int t = 0; t < I.ntiles; ++t, ++ns) {
        const uint32_t sb = ns & 1;
        if (!(ok = warp_wait(s_full + sb, (ns >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        // the row sees keys [llo, lim) of this half (padding rows, beyond the
        // slab's blocks, compute on whatever Q rows the tile box holds; their
        // partials are never read)
        const int kt0 = I.cs + t * kKeyTile;
        const int lim = (ri.n < 0 ? kKeyTile : min(max(ri.anchor - kt0, 0), kKeyTile)) - 64 * hf;
        const int llo = (ri.n < 0 ? 0 : min(max(ri.lo - kt0, 0), kKeyTile)) - 64 * hf;
        const uint32_t sa = tS + lane_base + sb * 128 + 64 * hf;
        uint32_t x[64];  // raw scores of this half row (masked entries -> -inf)
        tmem_ld_row<64>(sa, x);
        if (!__all_sync(0xffffffffu, lim >= 64 && llo <= 0)) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i >= lim || i < llo) x[i] = __float_as_uint(-INFINITY);
        }
        // row max of this half: eight chains of three-input maxima
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = __uint_as_float(x[k]);
#pragma unroll
        for (int i = 8; i < 56; i += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mx[k] = max3f(mx[k], __uint_as_float(x[i + k]), __uint_as_float(x[i + 8 + k]));
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], __uint_as_float(x[56 + k]));
        const float mt =
            fmaxf(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], max3f(mx[5], mx[6], mx[7]))) * sl2;
        const float m_new = fmaxf(m_run, mt);
        float fac = 1.f;
        bool resc = false;
        if (t == 0) {
          m_run = m_new;
        } else if (m_new > m_run + 8.f) {  // lazy rescale: keep exponents <= 2^8
          fac = ex2(m_run - m_new);
          resc = true;
          m_run = m_new;
        }
        const float nmu = (m_run == -INFINITY) ? 0.f : -m_run;
        // P = 2^(x * scale*log2(e) - m) two columns per packed instruction
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nmux2 = f2_pack(nmu, nmu);
        uint64_t lsum[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) lsum[k] = 0ull;  // (+0.f, +0.f)
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float y0, y1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1])), sl2x2,
                           nmux2),
                    y0, y1);
          const float p0 = ex2(y0), p1 = ex2(y1);
          lsum[i & 3] = f2_add(lsum[i & 3], f2_pack(p0, p1));
          pk[i] = pack_bf16(p0, p1);
        }
        float ls;
        {
          const uint64_t a = f2_add(f2_add(lsum[0], lsum[1]), f2_add(lsum[2], lsum[3]));
          float a0, a1;
          f2_unpack(a, a0, a1);
          ls = a0 + a1;
        }
        l = (t == 0) ? ls : l * fac + ls;
        tmem_st32(tS + lane_base + sb * 128 + 64 * hf, pk);  // packed P of this half: a_col()
        tmem_st_wait();
        // O_hf holds the PVs of tiles before t only once the PV of tile t-1
        // is done; wait for it only when O_hf must be rescaled (rare).
        if (t > 0 && __any_sync(0xffffffffu, resc)) {
          const uint32_t pt = ns - 1;
          if (!(ok = warp_wait(sfree + (pt & 1), (pt >> 1) & 1, abort_flag))) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 64; ++c) {
            uint32_t v[64];
            tmem_ld_row<64>(tOh + 64 * c, v);
#pragma unroll
            for (int i = 0; i < 64; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * fac);
            tmem_st64(tOh + 64 * c, v);
            tmem_st_wait();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_ready + 2 * sb + hf);
        if (!row_next) {
          rin = row_info_early(P, In, r);
          row_next = true;
        }
      }
      if (!ok) break;
      // hand (m, l) of this half to the epilogue once it has read the previous item's
      if (nit > 0 && !(ok = warp_wait(o_free, (nit - 1) & 1, abort_flag))) break;
      lm[hf * 128 + r] = l;
      lm[256 + hf * 128 + r] = m_run;
      __syncwarp();
      if (lane == 0) mbar_arrive(lm_ready);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0) {
    if (*abort_flag) latch(pp.hdr, SPLITKV_ETIMEOUT);
    stamp_busy(P, pp, 0, 1);
  }
}

// ===========================================================================
// dQ (same items as the forward)
// ===========================================================================
// Q and dO are constant over an item, so they are copied once per item from
// their shared-memory tiles into TMEM and S = Q K^T, dP = dO V^T run as TS
// MMAs: only K and V are read from shared memory (16 KB per k step instead
// of 32 KB), which is what bounds these 128x128 products. TMEM: two
// 128-column regions, tile t using region t % 2 for S, then dP (written over
// S once the softmax has loaded it), then dS (bf16, over dP); the dQ
// accumulator (D columns); Q and dO (D / 2 packed columns each).
// K is read by S (early) and by dQ (late) of its tile, V only by dP: a ring
// of three K tiles and a ring of two V tiles, each released after its last
// reader.
constexpr int kDqNK = 3, kDqNV = 2;

template <int D>
struct DqLayout {
  static constexpr int kSub = D / 64;
  static constexpr uint32_t tile = kSub * kSubBytes;
  static constexpr uint32_t q = 0;
  static constexpr uint32_t dO = tile;
  static constexpr uint32_t k0 = 2 * tile;
  static constexpr uint32_t v0 = k0 + kDqNK * tile;
  static constexpr uint32_t bars = v0 + kDqNV * tile;
  static constexpr uint32_t total = bars + 512 + 1024;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                     const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     ProbDev P, PlanPtrs pp, WorkPtrs wk, const float* __restrict__ LSE) {
  using Lay = DqLayout<D>;
  constexpr int kSub = Lay::kSub;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = (uint64_t*)(smem + Lay::bars);
  uint64_t* q_full = bars + 0;          // Q, dO of the item in shared memory
  uint64_t* q_empty = bars + 1;         // ... copied to TMEM (the copies are done)
  uint64_t* k_full = bars + 2;          // [kDqNK]
  uint64_t* k_empty = k_full + kDqNK;
  // V is read only by dP: V stage and dp_full of tile t are both t % 2, so
  // dP's commit frees the V stage.
  static_assert(kDqNV == 2, "V ring size tied to dp_full");
  uint64_t* v_full = k_empty + kDqNK;   // [kDqNV]
  uint64_t* s_full = v_full + kDqNV;    // S of tile t is in its region
  uint64_t* s_read = s_full + 1;        // softmax has loaded S: dP may overwrite it
  uint64_t* dp_full = s_read + 1;       // [2] dP of tile t (by tile parity)
  uint64_t* p_ready = dp_full + 2;      // [2] softmax wrote dS (bf16) over dP of tile t
  uint64_t* rfree = p_ready + 2;        // [2] the dQ MMA of tile t has read dS: region free
  uint64_t* qt_empty = rfree + 2;       // the item's S and dP MMAs are done with Q, dO in TMEM
  uint64_t* dq_done = qt_empty + 1;
  uint64_t* dq_free = dq_done + 1;
  uint64_t* mma_drain = dq_free + 1;    // [2] one per issuing warp
  uint32_t* tmem_slot = (uint32_t*)(bars + 32);
  volatile int* abort_flag = (volatile int*)(bars + 33);

  if (!plan_ok_cta(P, pp.hdr)) return;
  if (threadIdx.x == 0) stamp_busy(P, pp, 1, 0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kDqNK; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
    }
    for (int s = 0; s < kDqNV; ++s) mbar_init(v_full + s, 1);
    mbar_init(s_full, 1);
    mbar_init(s_read, kSoftmaxWarps);
    for (int b = 0; b < 2; ++b) {
      mbar_init(dp_full + b, 1);
      mbar_init(p_ready + b, kSoftmaxWarps);
      mbar_init(rfree + b, 1);
    }
    mbar_init(qt_empty, 1);
    mbar_init(dq_done, 1);
    mbar_init(dq_free, 4);
    mbar_init(mma_drain, 1);
    mbar_init(mma_drain + 1, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // regions: tmem + 128 * (t % 2)
  const uint32_t tdQ = tmem + 256;           // D columns
  const uint32_t tQ = tdQ + D;               // D / 2 columns: Q, bf16 pairs
  const uint32_t tdO = tQ + D / 2;           // D / 2 columns: dO
  const int q0 = pp.f_qoff[blockIdx.x];
  const int q1 = queue_end(pp.f_qoff, blockIdx.x, (int64_t)pp.hdr->n_fwd_items * P.Hkv, pp.hdr);

  if (warp == 0) {
    // ---------------- TMA producer: Q, dO and K (V comes from warp 15) ----------------
    {  // the whole warp runs the loop and waits; one elected lane issues the copies
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmdO);
      tma_prefetch_desc(&tmK);
      uint32_t nq = 0, nk = 0;
      bool ok = true;
      FwdItem In = q0 < q1 ? ld_rec(pp.f_rec + q0) : FwdItem{};
      for (int qi = q0; qi < q1 && ok; ++qi) {
        const FwdItem I = In;
        if (qi + 1 < q1) In = ld_rec(pp.f_rec + qi + 1);  // lands during this item
        if (nq > 0 && !(ok = warp_wait(q_empty, (nq - 1) & 1, abort_flag))) break;
        if (elect_one()) {
          mbar_expect_tx(q_full, 2 * Lay::tile);
          for (int i = 0; i < kSub; ++i) {
            tma_load_3d(smem + Lay::q + i * kSubBytes, &tmQ, q_full, 64 * i, I.g * P.group, I.n0);
            tma_load_3d(smem + Lay::dO + i * kSubBytes, &tmdO, q_full, 64 * i, I.g * P.group, I.n0);
          }
        }
        __syncwarp();
        ++nq;
        for (int t = 0; t < I.ntiles; ++t) {
          const uint32_t s = nk % kDqNK, u = nk / kDqNK;
          if (u > 0 && !(ok = warp_wait(k_empty + s, (u - 1) & 1, abort_flag))) break;
          uint8_t* kb = smem + Lay::k0 + s * Lay::tile;
          if (elect_one()) {
            mbar_expect_tx(k_full + s, Lay::tile);
            for (int i = 0; i < kSub; ++i)
              tma_load_3d(kb + i * kSubBytes, &tmK, k_full + s, 64 * i, I.g, I.row0 + t * kKeyTile);
          }
          __syncwarp();
          ++nk;
        }
      }
      if (!ok) {
        if (nq > 0) mbar_wait_drain(q_full, (nq - 1) & 1, kDrainNs);
        for (uint32_t j = nk > (uint32_t)kDqNK ? nk - kDqNK : 0; j < nk; ++j)
          mbar_wait_drain(k_full + j % kDqNK, (j / kDqNK) & 1, kDrainNs);
      }
    }
  } else if (warp == kVWarp) {
    // ---------------- V producer (its own warp) ----------------
    {  // the whole warp runs the loop and waits; one elected lane issues the copies
      tma_prefetch_desc(&tmV);
      uint32_t nv = 0;
      bool ok = true;
      FwdItem In = q0 < q1 ? ld_rec(pp.f_rec + q0) : FwdItem{};
      for (int qi = q0; qi < q1 && ok; ++qi) {
        const FwdItem I = In;
        if (qi + 1 < q1) In = ld_rec(pp.f_rec + qi + 1);  // lands during this item
        for (int t = 0; t < I.ntiles; ++t) {
          const uint32_t s = nv % kDqNV, u = nv / kDqNV;
          if (u > 0 && !(ok = warp_wait(dp_full + s, (u - 1) & 1, abort_flag))) break;
          uint8_t* vb = smem + Lay::v0 + s * Lay::tile;
          if (elect_one()) {
            mbar_expect_tx(v_full + s, Lay::tile);
            for (int i = 0; i < kSub; ++i)
              tma_load_3d(vb + i * kSubBytes, &tmV, v_full + s, 64 * i, I.g, I.row0 + t * kKeyTile);
          }
          __syncwarp();
          ++nv;
        }
      }
      if (!ok) {
        for (uint32_t j = nv > (uint32_t)kDqNV ? nv - kDqNV : 0; j < nv; ++j)
          mbar_wait_drain(v_full + j % kDqNV, (j / kDqNV) & 1, kDrainNs);
      }
    }
  } else if (warp == 1) {
    // ---------------- S and dP issuer (whole warp, one elected lane) ----------------
    // S of tile t lands on the region the dQ MMA of tile t-2 read (rfree);
    // dP of tile t lands on S once the softmax has loaded it (s_read).
    constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
    const uint64_t qsd0 = desc_kmajor0(smem_u32(smem + Lay::q));
    const uint64_t dosd0 = desc_kmajor0(smem_u32(smem + Lay::dO));
    uint32_t gt = 0, nit = 0;  // gt: tiles issued (K and V ring index)
    bool ok = true;
    FwdItem In = q0 < q1 ? ld_rec(pp.f_rec + q0) : FwdItem{};
    for (int qi = q0; qi < q1 && ok; ++qi, ++nit) {
      const FwdItem I = In;
      if (qi + 1 < q1) In = ld_rec(pp.f_rec + qi + 1);  // lands during this item
      // Q and dO of the item into TMEM: asynchronous shared-memory -> TMEM
      // copies, one per 16-element k step, once the previous item's S and dP
      // are done with the columns; the item's first S follows them in issue
      // order, which orders it after the copies.
      if (!(ok = warp_wait(q_full, nit & 1, abort_flag))) break;
      if (nit > 0 && !(ok = warp_wait(qt_empty, (nit - 1) & 1, abort_flag))) break;
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          tmem_cp_128x256b(tQ + kk * 8, qsd0 + (kmajor_off(kk) >> 4));
          tmem_cp_128x256b(tdO + kk * 8, dosd0 + (kmajor_off(kk) >> 4));
        }
        mma_commit(q_empty);  // the shared-memory tiles may take the next item
      }
      __syncwarp();
      for (int t = 0; t < I.ntiles; ++t, ++gt) {
        const uint32_t ks = gt % kDqNK, vs = gt % kDqNV, b = gt & 1;
        const uint32_t tR = tmem + 128 * b;
        if (!(ok = warp_wait(k_full + ks, (gt / kDqNK) & 1, abort_flag))) break;
        if (gt >= 2 && !(ok = warp_wait(rfree + b, ((gt >> 1) - 1) & 1, abort_flag))) break;
        tc_fence_after();
        const uint64_t kd0 = desc_kmajor0(smem_u32(smem + Lay::k0 + ks * Lay::tile));
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ts(tR, tQ + kk * 8, kd0 + (kmajor_off(kk) >> 4), kIdS, kk > 0 ? 1u : 0u);
          mma_commit(s_full);
        }
        __syncwarp();
        if (!(ok = warp_wait(v_full + vs, (gt / kDqNV) & 1, abort_flag))) break;
        if (!(ok = warp_wait(s_read, gt & 1, abort_flag))) break;
        tc_fence_after();
        const uint64_t vd0 = desc_kmajor0(smem_u32(smem + Lay::v0 + vs * Lay::tile));
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ts(tR, tdO + kk * 8, vd0 + (kmajor_off(kk) >> 4), kIdS, kk > 0 ? 1u : 0u);
          mma_commit(dp_full + (gt & 1));  // also frees V stage vs == gt % 2
          if (t == I.ntiles - 1) mma_commit(qt_empty);  // Q and dO in TMEM are free
        }
        __syncwarp();
      }
    }
    if (elect_one()) mma_commit(mma_drain);
    __syncwarp();
    mbar_wait_drain(mma_drain, 0, kDrainNs);
  } else if (warp == kSoftmaxWarps + 2) {
    // ---------------- dQ issuer ----------------
    constexpr uint32_t kIdQ = idesc_bf16(128, D, false, true);
    uint32_t gt = 0, nit = 0;
    bool ok = true;
    FwdItem In = q0 < q1 ? ld_rec(pp.f_rec + q0) : FwdItem{};
    for (int qi = q0; qi < q1 && ok; ++qi, ++nit) {
      const FwdItem I = In;
      if (qi + 1 < q1) In = ld_rec(pp.f_rec + qi + 1);  // lands during this item
      for (int t = 0; t < I.ntiles; ++t, ++gt) {
        const uint32_t b = gt & 1;
        if (!(ok = warp_wait(p_ready + b, (gt >> 1) & 1, abort_flag))) break;
        if (t == 0 && nit > 0 && !(ok = warp_wait(dq_free, (nit - 1) & 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t ks = gt % kDqNK;
        const uint64_t kd0 = desc_mnmajor0(smem_u32(smem + Lay::k0 + ks * Lay::tile));
        const uint32_t tR = tmem + 128 * b;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kKeyTile / 16; ++kk)
            mma_ts(tdQ, tR + a_col(kk), kd0 + (mnmajor_off(kk) >> 4), kIdQ,
                   (t == 0 && kk == 0) ? 0u : 1u);
          mma_commit(rfree + b);
          mma_commit(k_empty + ks);
          if (t == I.ntiles - 1) mma_commit(dq_done);
        }
        __syncwarp();
      }
    }
    if (elect_one()) mma_commit(mma_drain + 1);
    __syncwarp();
    mbar_wait_drain(mma_drain + 1, 0, kDrainNs);
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ---------------- epilogue (warps 11..14): one lane quadrant each ----------------
    // Writes each item's dQ partial once its last dQ MMA is done, releasing
    // the accumulator right after loading it.
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    bool ok = true;
    auto write_dq = [&](const FwdItem& I, uint32_t it) -> bool {
      if (!warp_wait(dq_done, it & 1, abort_flag)) return false;
      tc_fence_after();
      const bool sok = SKV_OK(I.slot >= 0 && (int64_t)I.slot < (int64_t)pp.hdr->n_slot_base * P.Hkv,
                              pp.hdr, kDbgDqSlot, I.slot);
#pragma unroll 1
      for (int h = 0; h < D / 64; ++h) {  // 64 columns at a time (register budget)
        uint32_t v[64];
        tmem_ld_row<64>(tdQ + lane_base + 64 * h, v);
        if (h == D / 64 - 1) {  // dQ is in registers: the next item may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dq_free);
        }
#pragma unroll
        for (int i = 0; i < 64; i += 8)
          if (sok)
            st_global_v8(wk.part_o + part_off(I.slot, r, 64 * h + i, D), __uint_as_float(v[i]),
                       __uint_as_float(v[i + 1]),
                       __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]),
                       __uint_as_float(v[i + 4]), __uint_as_float(v[i + 5]),
                       __uint_as_float(v[i + 6]), __uint_as_float(v[i + 7]));
      }
      return true;
    };
    uint32_t nit = 0;
    FwdItem In = q0 < q1 ? ld_rec(pp.f_rec + q0) : FwdItem{};
    for (int qi = q0; qi < q1 && ok; ++qi, ++nit) {
      const FwdItem I = In;
      if (qi + 1 < q1) In = ld_rec(pp.f_rec + qi + 1);  // lands during this item
      ok = write_dq(I, nit);
    }
  } else {
    // softmax (warps 2..9): lane quadrant warp % 4, column half hf
    const int wq = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const float sl2 = P.scale_log2;
    uint32_t gt = 0, nit = 0;
    bool ok = true;
    // The next item's record, row and row statistics are loaded after this
    // item's last tile (two dependent loads: the decoded record, then the
    // row's anchor, LSE and D; keeping them across the tiles would cost the
    // registers this role does not have).
    FwdItem In{};
    RowInfo rin{};
    float nl2n = -INFINITY, Drn = 0.f;
    auto load_next = [&](int qn) {
      In = ld_rec(pp.f_rec + qn);
      rin = row_info_early(P, In, r);
      // padding rows: -inf exponent offset makes their P exactly 0
      nl2n = -INFINITY;
      Drn = 0.f;
      if (rin.n >= 0) {
        nl2n = -ld_float_early(LSE + (size_t)rin.h * P.NQ + rin.n) * kLog2e;
        Drn = ld_float_early(wk.dvec + (size_t)rin.h * P.NQ + rin.n);
      }
    };
    if (q0 < q1) load_next(q0);
    for (int qi = q0; qi < q1 && ok; ++qi, ++nit) {
      const FwdItem I = In;
      const RowInfo ri = rin;
      const float nl2 = nl2n, Dr = Drn;
      for (int t = 0; t < I.ntiles; ++t, ++gt) {
        if (!(ok = warp_wait(s_full, gt & 1, abort_flag))) break;
        tc_fence_after();
        const int kt0 = I.cs + t * kKeyTile;
        const int lim = (ri.n < 0 ? kKeyTile : min(max(ri.anchor - kt0, 0), kKeyTile)) - 64 * hf;
        const int llo = (ri.n < 0 ? 0 : min(max(ri.lo - kt0, 0), kKeyTile)) - 64 * hf;
        // S, then dP, then dS of this tile: region gt % 2, this half's columns
        const uint32_t sa = tmem + 128 * (gt & 1) + lane_base + 64 * hf;
        const uint32_t pa = sa;
        // phase 1 (while dP of this tile and dQ of the previous one run):
        // P = exp(S * scale - LSE) on the row's visible keys, kept as bf16
        uint32_t pk[32];
        {
          uint32_t sv[64];
          tmem_ld_row<64>(sa, sv);
          tc_fence_before();  // S is in registers: dP may overwrite it
          __syncwarp();
          if (lane == 0) mbar_arrive(s_read);
          if (__all_sync(0xffffffffu, lim >= 64 && llo <= 0)) {
            const uint64_t sl2x2 = f2_pack(sl2, sl2), nl2x2 = f2_pack(nl2, nl2);
#pragma unroll
            for (int i = 0; i < 64; i += 2) {
              float y0, y1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), sl2x2,
                               nl2x2),
                        y0, y1);
              pk[i / 2] = pack_bf16(ex2(y0), ex2(y1));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 64; i += 2) {
              const float p0 =
                  (i < lim && i >= llo) ? ex2(fmaf(__uint_as_float(sv[i]), sl2, nl2)) : 0.f;
              const float p1 = (i + 1 < lim && i + 1 >= llo)
                                   ? ex2(fmaf(__uint_as_float(sv[i + 1]), sl2, nl2))
                                   : 0.f;
              pk[i / 2] = pack_bf16(p0, p1);
            }
          }
        }
        // phase 2: dS = P * (dP - D), written over this half's dP columns
        if (!(ok = warp_wait(dp_full + (gt & 1), (gt >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        {
          const uint64_t dr2 = f2_pack(Dr, Dr);
#pragma unroll
          for (int c = 0; c < 2; ++c) {  // 32 columns at a time (register budget)
            uint32_t dv[32];
            tmem_ld_row<32>(pa + 32 * c, dv);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const uint32_t pp2 = pk[16 * c + i / 2];
              const uint64_t d2 =
                  f2_mul(f2_pack(__uint_as_float(pp2 << 16), __uint_as_float(pp2 & 0xffff0000u)),
                         f2_sub(f2_pack(__uint_as_float(dv[i]), __uint_as_float(dv[i + 1])), dr2));
              float d0, d1;
              f2_unpack(d2, d0, d1);
              pk[16 * c + i / 2] = pack_bf16(d0, d1);
            }
          }
        }
        tmem_st32(pa, pk);  // packed dS of this half: columns a_col() of the dP region
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_ready + (gt & 1));
      }
      if (!ok) break;
      if (qi + 1 < q1) load_next(qi + 1);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0) {
    if (*abort_flag) latch(pp.hdr, SPLITKV_ETIMEOUT);
    stamp_busy(P, pp, 1, 1);
  }
}

// ===========================================================================
// dK / dV (backward items: one 128-key tile, all slabs that see it)
// ===========================================================================
template <int D>
struct KvLayout {
  static constexpr int kSub = D / 64;
  static constexpr uint32_t k = 0;
  static constexpr uint32_t v = kSub * kSubBytes;
  static constexpr uint32_t stage0 = 2 * kSub * kSubBytes;
  static constexpr uint32_t info_off = 2 * kSub * kSubBytes;       // inside a stage
  static constexpr uint32_t stage_bytes = 2 * kSub * kSubBytes + 2048;  // Q, dO, row table
  static constexpr uint32_t bars = stage0 + kNS * stage_bytes;
  static constexpr uint32_t red = bars + 512;  // the dQ reduction's ring, then its draft rows
  static constexpr uint32_t total = red + (kRedStages + 1) * kRedPieceBytes + 1024;
};
static_assert(KvLayout<128>::total <= 232448, "dK/dV shared memory above the per-CTA limit");

using KvItem = BwdRec;

__device__ __forceinline__ BwdRec ld_brec(const BwdRec* p) {
  BwdRec R;
  asm volatile("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(R.s), "=r"(R.g), "=r"(R.c0), "=r"(R.L)
               : "l"(p));
  asm volatile("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4 + 16];"
               : "=r"(R.ks0), "=r"(R.sl_lo), "=r"(R.sl_hi), "=r"(R.pad)
               : "l"(p));
  return R;
}

// Waits like warp_wait; with kRedSleepNs > 0 the warp pauses between polls,
// leaving its issue slots to the softmax warps of its SM sub-partition.
__device__ __forceinline__ bool red_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  bool mine;
  if (kRedSleepNs == 0) {
    mine = mbar_wait(bar, parity, abort);
  } else {
    mine = mbar_try_wait(bar, parity);
    const uint64_t t0 = mine ? 0 : globaltimer();
    for (uint32_t it = 1; !mine; ++it) {
      __nanosleep(kRedSleepNs);
      if ((mine = mbar_try_wait(bar, parity))) break;
      if ((it & 15) == 0) {
        if (*abort) break;
        if (globaltimer() - t0 > kWaitTimeoutNs) {
          *abort = 1;
          break;
        }
      }
    }
  }
  return __all_sync(0xffffffffu, mine);
}

// dQ = scale * (the row's chunk partials summed in ascending chunk order +
// its draft term), run by the reduction warp of the dK/dV kernel. Tasks are
// (slab, kv head) pairs, taken from a counter in the work workspace so that
// the CTAs finish their shares together. For each 8-dim group of the slab's
// 128 x d partial tiles, the chunks that any of its rows reads are copied one
// 4 KB piece at a time into a ring of kRedStages shared-memory stages (with
// an evict-first L2 policy: each partial is read once); lane l sums rows
// l + 32 i over the chunks of each row's own range only and writes the
// group's 8 dims of each row, whose draft term was copied into shared memory
// while the chunks streamed. The warp alone reads the ring, so stages are
// refilled as soon as the warp has read kRedRefill of them (one proxy fence
// orders those reads before the copies), and the copies run in ring order
// across tasks. The sums run in the same order as the standalone dq_reduce
// kernel, so the result is the same bit for bit.
template <int D>
__device__ __forceinline__ void kv_dq_reduce(const ProbDev& P, const PlanPtrs& pp,
                                             const WorkPtrs& wk, __nv_bfloat16* __restrict__ dQ,
                                             float* ring, uint64_t* full, volatile int* abort_flag,
                                             int lane) {
  constexpr int kPieces = D / 8;
  constexpr uint32_t kPieceFloats = kRedPieceBytes / 4;
  const int ntask = pp.hdr->n_slabs * P.Hkv;
  const size_t cstride = (size_t)P.Hkv * kRows * D;  // floats between chunk tiles
  const uint64_t policy = l2_evict_first_policy();
  float* dbuf = ring + kRedStages * kPieceFloats;  // [128 rows][8] draft term of one piece
  uint32_t cs = 0, cpar = 0;  // ring stage of the next copy to read, and its phase parity
  uint32_t is = 0;            // ring stage of the next copy to issue
  int pend = 0;               // stages read since the last proxy fence
  bool ok = true;
  int t = __shfl_sync(0xffffffffu, lane == 0 ? atomicAdd(wk.red_next, 1) : 0, 0);
  while (t < ntask && ok) {
    // the next task is claimed now; the answer is needed only at the end
    const int tn = lane == 0 ? atomicAdd(wk.red_next, 1) : 0;
    const int sg = t / P.Hkv, g = t - sg * P.Hkv;
    const int first = pp.sl_first[sg], nblk = pp.sl_nblk[sg];
    const size_t slot0 = (size_t)pp.sl_slot[sg];
    // chunk range [clo, cend) and output row of rows lane + 32 i
    int clo[4], cend[4], qrow[4];
    int cmin = 0x7fffffff, cmax = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const RowInfo ri = row_info(P, first, nblk, g, lane + 32 * i);
      clo[i] = cend[i] = 0;
      qrow[i] = -1;
      if (ri.n >= 0) {
        const int na = (ri.anchor + P.chunk - 1) / P.chunk;
        clo[i] = ri.lo >= ri.anchor ? na : ri.lo / P.chunk;
        cend[i] = SKV_OK(slot0 + (size_t)na <= (size_t)pp.hdr->n_slot_base, pp.hdr,
                         kDbgReduceSlot, slot0 + na)
                      ? na
                      : clo[i];
        if (cend[i] > clo[i]) {
          cmin = min(cmin, clo[i]);
          cmax = max(cmax, cend[i]);
        }
        if (SKV_OK(ri.n < P.NQ && ri.h >= 0 && ri.h < P.Hq, pp.hdr, kDbgQueryRow, ri.n))
          qrow[i] = ri.n * P.Hq + ri.h;
      }
    }
    cmin = (int)__reduce_min_sync(0xffffffffu, (uint32_t)cmin);
    cmax = (int)__reduce_max_sync(0xffffffffu, (uint32_t)cmax);
    const int nch = cmax > cmin ? cmax - cmin : 0;
    if (nch == 0) cmin = 0;       // no row reads a partial: only the draft term
    const int K = kPieces * nch;  // copies of this task: dims group-major, then chunk
    // the next copy to issue: dims group ip of chunk cmin + ic, into stage is
    const float* tile0 = wk.part_o + part_off((slot0 + cmin) * P.Hkv + g, 0, 0, D);
    int ip = 0, ic = 0, issued = 0;
    auto issue = [&]() {
      if (elect_one()) {
        mbar_expect_tx(full + is, kRedPieceBytes);
        bulk_load_hint(ring + is * kPieceFloats, tile0 + (size_t)ic * cstride + ip * kPieceFloats,
                       kRedPieceBytes, full + is, policy);
      }
      __syncwarp();
      ++issued;
      if (++is == (uint32_t)kRedStages) is = 0;
      if (++ic == nch) {
        ic = 0;
        ++ip;
      }
    };
    if (K > 0 && pend > 0) {  // stages read by the previous task are refilled now
      fence_proxy_async_shared();
      __syncwarp();
      pend = 0;
    }
    for (int k = 0; k < K && k < kRedStages; ++k) issue();
    int k = 0;  // copies read
    for (int p = 0; p < kPieces && ok; ++p) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (qrow[i] < 0) continue;
        const float* src = wk.dq_draft + (size_t)qrow[i] * D + 8 * p;
        cp_async16(dbuf + (lane + 32 * i) * 8, src);
        cp_async16(dbuf + (lane + 32 * i) * 8 + 4, src + 4);
      }
      float acc[4][8];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
      for (int c = cmin; c < cmin + nch; ++c) {
        if (!(ok = red_wait(full + cs, cpar, abort_flag))) break;
        const float* sp = ring + cs * kPieceFloats;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (c >= clo[i] && c < cend[i]) {
            const int r = lane + 32 * i;
            const float4 a = *(const float4*)(sp + r * 8);
            const float4 b = *(const float4*)(sp + r * 8 + 4);
            float* o = acc[i];
            o[0] += a.x; o[1] += a.y; o[2] += a.z; o[3] += a.w;
            o[4] += b.x; o[5] += b.y; o[6] += b.z; o[7] += b.w;
          }
        }
        ++k;
        if (++pend >= kRedRefill && issued < K) {  // refill the stages just read
          fence_proxy_async_shared();
          __syncwarp();
          for (; pend > 0 && issued < K; --pend) issue();
          pend = 0;
        }
        if (++cs == (uint32_t)kRedStages) {
          cs = 0;
          cpar ^= 1u;
        }
      }
      cp_async_wait_all();
      if (!ok) break;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (qrow[i] < 0) continue;
        const size_t row = (size_t)qrow[i] * D + 8 * p;
        const float4 a = *(const float4*)(dbuf + (lane + 32 * i) * 8);
        const float4 b = *(const float4*)(dbuf + (lane + 32 * i) * 8 + 4);
        uint4 w;
        w.x = pack_bf16((acc[i][0] + a.x) * P.scale, (acc[i][1] + a.y) * P.scale);
        w.y = pack_bf16((acc[i][2] + a.z) * P.scale, (acc[i][3] + a.w) * P.scale);
        w.z = pack_bf16((acc[i][4] + b.x) * P.scale, (acc[i][5] + b.y) * P.scale);
        w.w = pack_bf16((acc[i][6] + b.z) * P.scale, (acc[i][7] + b.w) * P.scale);
        *(uint4*)(dQ + row) = w;
      }
    }
    if (!ok) {
      // copies issued and not read land before the CTA exits: the one the
      // warp gave up on (stage cs) and those after it in ring order
      uint32_t st = cs, par = cpar;
      for (int i = k; i < issued; ++i) {
        mbar_wait_drain(full + st, par, kDrainNs);
        if (++st == (uint32_t)kRedStages) {
          st = 0;
          par ^= 1u;
        }
      }
    }
    t = __shfl_sync(0xffffffffu, tn, 0);
  }
}

// Key tiles that no block sees (backward candidates of cost 0) are in no
// backward item; their dK and dV rows are zero. Run by the reduction warp of
// the dK/dV kernel after its dQ tasks: candidate c on CTA c mod the grid,
// 16-byte stores.
template <int D>
__device__ __forceinline__ void kv_zero_unseen(const ProbDev& P, const PlanPtrs& pp,
                                               __nv_bfloat16* __restrict__ dKc,
                                               __nv_bfloat16* __restrict__ dVc, int lane) {
  const int ncand = pp.hdr->n_bwd_cand;
  const size_t row16 = (size_t)P.Hkv * D * 2 / 16;  // 16-byte units of a key row
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int cand = blockIdx.x; cand < ncand; cand += gridDim.x) {
    if (pp.b_cost[cand] != 0) continue;  // warp-uniform
    const int s = seg_of(pp.s_bcand_off, P.S, cand);
    const int kt = cand - pp.s_bcand_off[s];
    const int c0 = P.cu_ctx[s], L = P.cu_ctx[s + 1] - c0;
    const int k0 = kt * kKeyTile, k1 = min(L, k0 + kKeyTile);
    if (!SKV_OK(k0 >= 0 && (int64_t)c0 + k1 <= P.T, pp.hdr, kDbgZeroRow, (int64_t)c0 + k1))
      continue;
    const size_t lo = (size_t)(c0 + k0) * row16, hi = (size_t)(c0 + k1) * row16;
    for (size_t i = lo + lane; i < hi; i += 32) {
      ((uint4*)dKc)[i] = z;
      ((uint4*)dVc)[i] = z;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreadsKv, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                       const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       ProbDev P, PlanPtrs pp, WorkPtrs wk, const float* __restrict__ LSE,
                       __nv_bfloat16* __restrict__ dKc, __nv_bfloat16* __restrict__ dVc,
                       __nv_bfloat16* __restrict__ dQ) {
  using Lay = KvLayout<D>;
  constexpr int kSub = Lay::kSub;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = (uint64_t*)(smem + Lay::bars);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 1;
  uint64_t* st_full = bars + 2;        // [kNS]
  uint64_t* st_empty = st_full + kNS;  // [kNS]
  uint64_t* s_full = st_empty + kNS;   // S^T of a slab is in TMEM
  uint64_t* dp_full = s_full + 1;      // dP^T of a slab is in TMEM
  uint64_t* p_ready = dp_full + 1;     // softmax wrote P^T (bf16) over S^T
  uint64_t* ds_ready = p_ready + 1;    // softmax wrote dS^T (bf16) over dP^T
  uint64_t* acc_done = ds_ready + 1;
  uint64_t* acc_free = acc_done + 1;
  uint64_t* mma_drain = acc_free + 1;
  uint64_t* red_full = bars + 16;   // [kRedStages] a partial piece is in its stage
  static_assert(16 + kRedStages <= 32, "reduction barriers below the TMEM slot");
  uint32_t* tmem_slot = (uint32_t*)(bars + 32);
  volatile int* abort_flag = (volatile int*)(bars + 33);

  if (!plan_ok_cta(P, pp.hdr)) return;
  if (threadIdx.x == 0) stamp_busy(P, pp, 2, 0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    // st_full takes one arrival from each of the two producer warps
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int s = 0; s < kNS; ++s) {
      mbar_init(st_full + s, 2);
      mbar_init(st_empty + s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_ready, kKvSoftmaxWarps);
    mbar_init(ds_ready, kKvSoftmaxWarps);
    mbar_init(acc_done, 1);
    mbar_init(acc_free, kKvSoftmaxWarps);
    mbar_init(mma_drain, 1);
    for (int s = 0; s < kRedStages; ++s) mbar_init(red_full + s, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;
  const int q0 = pp.b_qoff[blockIdx.x];
  const int q1 = queue_end(pp.b_qoff, blockIdx.x, (int64_t)pp.hdr->n_bwd_items * P.Hkv, pp.hdr);

  if (warp == kKvRedWarp) {
    // ---------------- dQ reduction and the zero rows (independent of the
    // items) ----------------
    if (dQ != nullptr) {
      kv_dq_reduce<D>(P, pp, wk, dQ, (float*)(smem + Lay::red), red_full, abort_flag, lane);
      kv_zero_unseen<D>(P, pp, dKc, dVc, lane);
    }
  } else if (warp == 0) {
    // ---------------- producer: K/V per item, then Q and the slab's row table
    // (one bulk copy of the precomputed record) per slab; dO comes from
    // warp 10 ----------------
    {  // the whole warp runs the loop and waits; one elected lane issues the copies
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmdO);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint32_t nkv = 0, nst = 0;
      bool ok = true;
      KvItem In = q0 < q1 ? ld_brec(pp.b_rec + q0) : KvItem{};
      for (int qi = q0; qi < q1 && ok; ++qi) {
        const KvItem I = In;
        if (qi + 1 < q1) In = ld_brec(pp.b_rec + qi + 1);  // lands during this item
        if (nkv > 0 && !(ok = warp_wait(kv_empty, (nkv - 1) & 1, abort_flag))) break;
        if (elect_one()) {
          mbar_expect_tx(kv_full, 2 * kSub * kSubBytes);
          for (int i = 0; i < kSub; ++i) {
            tma_load_3d(smem + Lay::k + i * kSubBytes, &tmK, kv_full, 64 * i, I.g, I.c0 + I.ks0);
            tma_load_3d(smem + Lay::v + i * kSubBytes, &tmV, kv_full, 64 * i, I.g, I.c0 + I.ks0);
          }
        }
        __syncwarp();
        ++nkv;
        for (int sg = I.sl_lo; sg < I.sl_hi; ++sg) {
          const uint32_t s = nst % kNS, u = nst / kNS;
          if (u > 0 && !(ok = warp_wait(st_empty + s, (u - 1) & 1, abort_flag))) break;
          uint8_t* sb = smem + Lay::stage0 + s * Lay::stage_bytes;
          const int n0 = pp.sl_first[sg] * P.B;
          if (elect_one()) {
            mbar_expect_tx(st_full + s, kSub * kSubBytes + kRowInfoFloats * 4);
            for (int i = 0; i < kSub; ++i)
              tma_load_3d(sb + i * kSubBytes, &tmQ, st_full + s, 64 * i, I.g * P.group, n0);
            bulk_load(sb + Lay::info_off, wk.rowinfo + ((size_t)sg * P.Hkv + I.g) * kRowInfoFloats,
                      kRowInfoFloats * 4, st_full + s);
          }
          __syncwarp();
          ++nst;
        }
      }
      if (!ok) {
        if (nkv > 0) mbar_wait_drain(kv_full, (nkv - 1) & 1, kDrainNs);
        for (uint32_t j = nst > (uint32_t)kNS ? nst - kNS : 0; j < nst; ++j)
          mbar_wait_drain(st_full + j % kNS, (j / kNS) & 1, kDrainNs);
      }
    }
  } else if (warp == kKvDoWarp) {
    // ---------------- dO producer: its own warp, so that it runs in parallel
    // with the Q producer instead of taking turns with it ----------------
    {  // the whole warp runs the loop and waits; one elected lane issues the copies
      tma_prefetch_desc(&tmdO);
      uint32_t nst = 0;
      bool ok = true;
      KvItem In = q0 < q1 ? ld_brec(pp.b_rec + q0) : KvItem{};
      for (int qi = q0; qi < q1 && ok; ++qi) {
        const KvItem I = In;
        if (qi + 1 < q1) In = ld_brec(pp.b_rec + qi + 1);  // lands during this item
        for (int sg = I.sl_lo; sg < I.sl_hi; ++sg) {
          const uint32_t s = nst % kNS, u = nst / kNS;
          if (u > 0 && !(ok = warp_wait(st_empty + s, (u - 1) & 1, abort_flag))) break;
          uint8_t* sb = smem + Lay::stage0 + s * Lay::stage_bytes;
          const int n0 = pp.sl_first[sg] * P.B;
          if (elect_one()) {
            mbar_expect_tx(st_full + s, kSub * kSubBytes);
            for (int i = 0; i < kSub; ++i)
              tma_load_3d(sb + (kSub + i) * kSubBytes, &tmdO, st_full + s, 64 * i, I.g * P.group, n0);
          }
          __syncwarp();
          ++nst;
        }
      }
      if (!ok) {
        for (uint32_t j = nst > (uint32_t)kNS ? nst - kNS : 0; j < nst; ++j)
          mbar_wait_drain(st_full + j % kNS, (j / kNS) & 1, kDrainNs);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (whole warp, one elected lane) ----------------
    // Per slab: S^T, dP^T, [P^T ready] dV, S^T of the next slab, [dS^T ready]
    // dK — the next S^T is queued before dK so the tensor pipe has work
    // while the softmax warps turn dP^T into dS^T. TMEM reuse is safe
    // because tcgen05 MMAs of one thread execute in issue order. Every
    // 128x128 product here reads both operands from shared memory, whose
    // bandwidth the MMAs of one slab already fill, so a single in-order
    // issuer loses nothing to a second one.
    constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
    constexpr uint32_t kIdKV = idesc_bf16(128, D, false, true);
    const uint64_t kd0 = desc_kmajor0(smem_u32(smem + Lay::k));
    const uint64_t vd0 = desc_kmajor0(smem_u32(smem + Lay::v));
    auto issue_s = [&](uint32_t stage) {
      const uint64_t qd0 = desc_kmajor0(smem_u32(smem + Lay::stage0 + stage * Lay::stage_bytes));
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tS, kd0 + (kmajor_off(kk) >> 4), qd0 + (kmajor_off(kk) >> 4), kIdS,
                 kk > 0 ? 1u : 0u);
        mma_commit(s_full);
      }
      __syncwarp();
    };
    uint32_t nst = 0, nit = 0;
    bool ok = true;
    KvItem In = q0 < q1 ? ld_brec(pp.b_rec + q0) : KvItem{};
    for (int qi = q0; qi < q1 && ok; ++qi, ++nit) {
      const KvItem I = In;
      if (qi + 1 < q1) In = ld_brec(pp.b_rec + qi + 1);  // lands during this item
      if (!(ok = warp_wait(kv_full, nit & 1, abort_flag))) break;
      if (!(ok = warp_wait(st_full + nst % kNS, (nst / kNS) & 1, abort_flag))) break;
      tc_fence_after();
      issue_s(nst % kNS);
      for (int sg = I.sl_lo; sg < I.sl_hi; ++sg, ++nst) {
        const uint32_t s = nst % kNS;
        const uint32_t q_addr = smem_u32(smem + Lay::stage0 + s * Lay::stage_bytes);
        const uint32_t do_addr = q_addr + kSub * kSubBytes;
        const bool first = (sg == I.sl_lo), last = (sg == I.sl_hi - 1);
        const uint64_t dod0 = desc_kmajor0(do_addr);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tP, vd0 + (kmajor_off(kk) >> 4), dod0 + (kmajor_off(kk) >> 4), kIdS,
                   kk > 0 ? 1u : 0u);
          mma_commit(dp_full);
          if (last) mma_commit(kv_empty);  // K and V are not read after this
        }
        __syncwarp();
        if (!(ok = warp_wait(p_ready, nst & 1, abort_flag))) break;
        if (first && nit > 0 && !(ok = warp_wait(acc_free, (nit - 1) & 1, abort_flag))) break;
        tc_fence_after();
        const uint64_t dom0 = desc_mnmajor0(do_addr);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kRows / 16; ++kk)
            mma_ts(tdV, tS + kv_acol(kk), dom0 + (mnmajor_off(kk) >> 4), kIdKV,
                   (first && kk == 0) ? 0u : 1u);
        }
        __syncwarp();
        if (!last) {
          const uint32_t s2 = (nst + 1) % kNS;
          if (!(ok = warp_wait(st_full + s2, ((nst + 1) / kNS) & 1, abort_flag))) break;
          tc_fence_after();
          issue_s(s2);
        }
        if (!(ok = warp_wait(ds_ready, nst & 1, abort_flag))) break;
        tc_fence_after();
        const uint64_t qm0 = desc_mnmajor0(q_addr);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kRows / 16; ++kk)
            mma_ts(tdK, tP + kv_acol(kk), qm0 + (mnmajor_off(kk) >> 4), kIdKV,
                   (first && kk == 0) ? 0u : 1u);
          mma_commit(st_empty + s);
          if (last) mma_commit(acc_done);
        }
        __syncwarp();
      }
    }
    if (elect_one()) mma_commit(mma_drain);
    __syncwarp();
    mbar_wait_drain(mma_drain, 0, kDrainNs);
  } else {
    // softmax + epilogue (warps 2..17): key lane quadrant warp % 4, row
    // quarter qr (32 rows of the slab; a quarter of dK and dV's columns in
    // the epilogue)
    constexpr int OQ = D / 4;
    const int wq = warp & 3;
    const int qr = (warp - 2) >> 2;
    const int r = wq * 32 + lane;  // key of the tile owned by this thread
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const float sl2 = P.scale_log2;
    // with per-block context offsets every element is checked against its
    // row's [lo, end); otherwise a key below the slab's first anchor is seen
    // by every row
    const bool offsets = (P.flags & SPLITKV_FLAG_MASK_CONTEXT_OFFSET) != 0;
    uint32_t nst = 0, nit = 0;
    bool ok = true;
    KvItem In = q0 < q1 ? ld_brec(pp.b_rec + q0) : KvItem{};
    for (int qi = q0; qi < q1 && ok; ++qi, ++nit) {
      const KvItem I = In;
      if (qi + 1 < q1) In = ld_brec(pp.b_rec + qi + 1);  // lands during this item
      const int key = I.ks0 + r;
      for (int sg = I.sl_lo; sg < I.sl_hi; ++sg, ++nst) {
        const uint32_t s = nst % kNS;
        // row table of the stage: acquire it through the stage barrier
        // (already complete; it cannot advance before this slab's dS^T is
        // consumed), then wait for S^T.
        if (!(ok = warp_wait(st_full + s, (nst / kNS) & 1, abort_flag))) break;
        if (!(ok = warp_wait(s_full, nst & 1, abort_flag))) break;
        tc_fence_after();
        const uint8_t* sb = smem + Lay::stage0 + s * Lay::stage_bytes;
        const float* nl2 = (const float*)(sb + Lay::info_off) + 32 * qr;  // -LSE*log2(e)
        const float* dvv = nl2 + kRows;
        const int* anc = (const int*)(dvv + kRows);   // end of each row's visible context
        const int* alo = anc + kRows;                 // start of each row's visible context
        const int* anc0 = anc - 32 * qr;  // the slab's first row: its smallest anchor
        // phase 1: P^T = exp(S^T * scale - LSE) on visible (key, row) pairs.
        // Rows are ordered by block and anchors rise with the block, so a key
        // below the slab's first anchor is seen by every row (padding rows give
        // 0 through their -inf): no per-element mask on such warps.
        uint32_t pk[16];
        {
          uint32_t sv[32];
          tmem_ld_row<32>(tS + lane_base + 32 * qr, sv);
          if (!offsets && __all_sync(0xffffffffu, key < anc0[0])) {
            const uint64_t sl2x2 = f2_pack(sl2, sl2);
            const uint64_t* nl2x2 = (const uint64_t*)nl2;  // (row c, row c + 1) pairs
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              float y0, y1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2,
                               nl2x2[c / 2]),
                        y0, y1);
              pk[c / 2] = pack_bf16(ex2(y0), ex2(y1));
            }
          } else {
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const float p0 = (key < anc[c] && key >= alo[c])
                                   ? ex2(fmaf(__uint_as_float(sv[c]), sl2, nl2[c]))
                                   : 0.f;
              const float p1 = (key < anc[c + 1] && key >= alo[c + 1])
                                   ? ex2(fmaf(__uint_as_float(sv[c + 1]), sl2, nl2[c + 1]))
                                   : 0.f;
              pk[c / 2] = pack_bf16(p0, p1);
            }
          }
        }
        tmem_st16(tS + lane_base + 32 * qr, pk);  // packed P^T of this quarter: kv_acol()
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_ready);
        // phase 2: dS^T = P^T * (dP^T - D)
        if (!(ok = warp_wait(dp_full, nst & 1, abort_flag))) break;
        tc_fence_after();
        {
          uint32_t dv[32];
          tmem_ld_row<32>(tP + lane_base + 32 * qr, dv);
          const uint64_t* dvv2 = (const uint64_t*)dvv;  // (row c, row c + 1) pairs
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const uint32_t pp2 = pk[c / 2];
            const uint64_t d2 =
                f2_mul(f2_pack(__uint_as_float(pp2 << 16), __uint_as_float(pp2 & 0xffff0000u)),
                       f2_sub(f2_pack(__uint_as_float(dv[c]), __uint_as_float(dv[c + 1])), dvv2[c / 2]));
            float d0, d1;
            f2_unpack(d2, d0, d1);
            pk[c / 2] = pack_bf16(d0, d1);
          }
        }
        tmem_st16(tP + lane_base + 32 * qr, pk);  // packed dS^T of this quarter
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ds_ready);
      }
      if (!ok) break;
      if (!(ok = warp_wait(acc_done, nit & 1, abort_flag))) break;
      tc_fence_after();
      const bool valid =
          key < I.L && SKV_OK((int64_t)I.c0 + key < P.T && I.g >= 0 && I.g < P.Hkv, pp.hdr,
                              kDbgKvRow, (int64_t)I.c0 + key);
      const size_t off = ((size_t)(I.c0 + key) * P.Hkv + I.g) * D + OQ * qr;
      for (int which = 0; which < 2; ++which) {  // dV, then dK (scaled)
        uint32_t a[OQ];
        tmem_ld_row<OQ>((which == 0 ? tdV : tdK) + lane_base + OQ * qr, a);
        if (which == 1) {  // both accumulators read: the next item may overwrite them
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_free);
        }
        const float f = which == 0 ? 1.f : P.scale;
        __nv_bfloat16* dst = (which == 0 ? dVc : dKc) + off;
        if (valid) {
#pragma unroll
          for (int i = 0; i < OQ; i += 8) {
            uint4 pv;
            pv.x = pack_bf16(__uint_as_float(a[i]) * f, __uint_as_float(a[i + 1]) * f);
            pv.y = pack_bf16(__uint_as_float(a[i + 2]) * f, __uint_as_float(a[i + 3]) * f);
            pv.z = pack_bf16(__uint_as_float(a[i + 4]) * f, __uint_as_float(a[i + 5]) * f);
            pv.w = pack_bf16(__uint_as_float(a[i + 6]) * f, __uint_as_float(a[i + 7]) * f);
            *(uint4*)(dst + i) = pv;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0) {
    if (*abort_flag) latch(pp.hdr, SPLITKV_ETIMEOUT);
    stamp_busy(P, pp, 2, 1);
  }
}

// ===========================================================================
// Host side: tensor maps and launches
// ===========================================================================
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 3-D bf16 map over [n2][n1][n0] (n0 contiguous) with a {64, b1, b2} box.
cudaError_t make_map(CUtensorMap* m, const void* base, uint64_t n0, uint64_t n1, uint64_t n2,
                     uint32_t b1, uint32_t b2) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {n0, n1, n2};
  const cuuint64_t strides[2] = {n0 * 2, n0 * n1 * 2};
  const cuuint32_t box[3] = {64, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

struct Maps {
  CUtensorMap q, dO, k, v;
};

cudaError_t make_maps(const ProbDev& P, const void* Q, const void* dO, const void* Kc,
                      const void* Vc, Maps* m) {
  const uint32_t rows_q = (uint32_t)(P.bps * P.B);
  cudaError_t e = make_map(&m->q, Q, P.d, P.Hq, P.NQ, P.group, rows_q);
  if (e == cudaSuccess && dO) e = make_map(&m->dO, dO, P.d, P.Hq, P.NQ, P.group, rows_q);
  if (e == cudaSuccess) e = make_map(&m->k, Kc, P.d, P.Hkv, P.T, 1, kKeyTile);
  if (e == cudaSuccess) e = make_map(&m->v, Vc, P.d, P.Hkv, P.T, 1, kKeyTile);
  return e;
}

template <typename K>
cudaError_t prep(K kernel, size_t smem) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

}  // namespace

cudaError_t launch_fwd_tc(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                          const void* Q, const void* Kc, const void* Vc, cudaStream_t st) {
  if (P.T == 0) return cudaErrorInvalidValue;
  Maps m;
  cudaError_t e = make_maps(P, Q, nullptr, Kc, Vc, &m);
  if (e != cudaSuccess) return e;
  if (P.d == 128) {
    auto k = fwd_tc_kernel<128>;
    if ((e = prep(k, FwdLayout<128>::total)) != cudaSuccess) return e;
    k<<<P.workers, kThreads, FwdLayout<128>::total, st>>>(m.q, m.k, m.v, P, pp, wk);
  } else {
    auto k = fwd_tc_kernel<64>;
    if ((e = prep(k, FwdLayout<64>::total)) != cudaSuccess) return e;
    k<<<P.workers, kThreads, FwdLayout<64>::total, st>>>(m.q, m.k, m.v, P, pp, wk);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq_tc(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                             const void* Q, const void* Kc, const void* Vc, const void* dO,
                             const float* LSE, cudaStream_t st) {
  if (P.T == 0) return cudaErrorInvalidValue;
  Maps m;
  cudaError_t e = make_maps(P, Q, dO, Kc, Vc, &m);
  if (e != cudaSuccess) return e;
  if (P.d == 128) {
    auto k = bwd_dq_tc_kernel<128>;
    if ((e = prep(k, DqLayout<128>::total)) != cudaSuccess) return e;
    k<<<P.workers, kThreads, DqLayout<128>::total, st>>>(m.q, m.dO, m.k, m.v, P, pp, wk, LSE);
  } else {
    auto k = bwd_dq_tc_kernel<64>;
    if ((e = prep(k, DqLayout<64>::total)) != cudaSuccess) return e;
    k<<<P.workers, kThreads, DqLayout<64>::total, st>>>(m.q, m.dO, m.k, m.v, P, pp, wk, LSE);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv_tc(const ProbDev& P, const PlanPtrs& pp, const WorkPtrs& wk,
                               const void* Q, const void* Kc, const void* Vc, const void* dO,
                               const float* LSE, void* dKc, void* dVc, void* dQ,
                               cudaStream_t st) {
  Maps m;
  cudaError_t e = make_maps(P, Q, dO, Kc, Vc, &m);
  if (e != cudaSuccess) return e;
  if (P.d == 128) {
    auto k = bwd_dkdv_tc_kernel<128>;
    if ((e = prep(k, KvLayout<128>::total)) != cudaSuccess) return e;
    k<<<P.workers, kThreadsKv, KvLayout<128>::total, st>>>(m.q, m.dO, m.k, m.v, P, pp, wk, LSE,
                                                          (__nv_bfloat16*)dKc, (__nv_bfloat16*)dVc,
                                                          (__nv_bfloat16*)dQ);
  } else {
    auto k = bwd_dkdv_tc_kernel<64>;
    if ((e = prep(k, KvLayout<64>::total)) != cudaSuccess) return e;
    k<<<P.workers, kThreadsKv, KvLayout<64>::total, st>>>(m.q, m.dO, m.k, m.v, P, pp, wk, LSE,
                                                         (__nv_bfloat16*)dKc, (__nv_bfloat16*)dVc,
                                                         (__nv_bfloat16*)dQ);
  }
  return cudaGetLastError();
}

}  // namespace skv
