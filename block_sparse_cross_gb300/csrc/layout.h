// Workspace layouts shared by the host API and the kernels.
//
// Plan workspace: a header (status word, counts) followed by the per-sample,
// per-slab, per-item and per-worker arrays the planner fills. Every offset is
// a pure function of host-known scalars, so the host can rebuild the typed
// pointers on every call without reading the device.
//
// Work workspace: fp32 partials of the split computation.
#pragma once
#include <stddef.h>
#include <stdint.h>

#include "../../include/splitkv.h"

namespace skv {

constexpr int kRows = 128;      // (query, head) rows per work item / MMA tile
constexpr int kKeyTile = 128;   // keys per tile; backward items own one tile
constexpr int kMaxGroupsPerLane = 8;   // LPT kernel: groups <= 32 * 8
constexpr int kMaxWorkers = 4096;
constexpr int32_t kPlanMagic = 0x53504b56;  // "SPKV"

struct PlanHeader {
  int32_t magic;
  int32_t status;          // latched device status (first error wins)
  int32_t workers;         // m persistent CTAs
  int32_t groups;          // m / Hkv
  int32_t n_slabs;
  int32_t n_fwd_cand;      // (sample, chunk, slab) candidates
  int32_t n_fwd_items;     // ... of positive cost
  int32_t n_slot_base;     // sum over slabs of active chunks (slots / Hkv)
  int32_t n_bwd_cand;      // (sample, key tile) candidates
  int32_t n_bwd_items;
  int32_t flags;
  int32_t pad0;
  int64_t fwd_total_cost;  // per kv head
  int64_t bwd_total_cost;
  int64_t fwd_tiles;       // per kv head
  int64_t dense_tiles;     // per kv head
  uint64_t problem_hash;
  // index checks of the debug build (SKV_DEBUG): failed checks since the
  // plan, and the first one as (site << 48) | (index & (2^48 - 1)); zero in
  // the release build
  int64_t dbg_count;
  int64_t dbg_first;
  int64_t pad1[5];
};
static_assert(sizeof(PlanHeader) % 16 == 0, "header alignment");

// A queue entry: one item for one worker.
//   forward : {sample, chunk, global slab index, kv head}
//   backward: {sample, key tile, unused, kv head}
struct __align__(16) QEntry {
  int32_t s, c, slab, g;
};

// A forward / dQ queue entry decoded once by the planner, so that a kernel
// role reads an item with one 32-byte load instead of chasing the slab and
// anchor tables at every item boundary.
//   n0      first query row of the slab      g      kv head
//   row0    first context row of the chunk   cs     chunk start (sample-local)
//   ntiles  128-key tiles below the slab's last visible key
//   first   first draft block of the slab    nblk   blocks in the slab
//   slot    partial slot of (slab, chunk, kv head)
struct __align__(16) FwdRec {
  int32_t n0, g, row0, cs, ntiles, first, nblk, slot;
};

// A dK/dV queue entry decoded once by the planner:
//   s, g     sample, kv head          c0, L   first context row, length of s
//   ks0      the key tile's first key (sample-local)
//   sl_lo    first slab whose last visible key lies beyond ks0
//   sl_hi    end of the sample's slabs
struct __align__(16) BwdRec {
  int32_t s, g, c0, L, ks0, sl_lo, sl_hi, pad;
};

struct PlanCaps {
  int64_t S, NA, NSL, NCF, NCB, M, Hkv;
};

struct PlanPtrs {
  PlanHeader* hdr;
  // per sample [S+1]
  int32_t* s_nch;
  int32_t* s_nsl;
  int32_t* s_nkt;
  int32_t* s_cand_off;
  int32_t* s_slab_off;
  int32_t* s_bcand_off;
  // per slab [NSL+1]
  int32_t* sl_sample;
  int32_t* sl_first;       // first global draft block
  int32_t* sl_nblk;
  int32_t* sl_nact;        // active chunks: ceil(max anchor / C)
  int32_t* sl_slot;        // exclusive prefix of sl_nact
  // forward candidates / items
  int64_t* f_cost;         // [NCF]   cost of candidate (0 = inactive)
  int32_t* f_item;         // [NCF]   candidate id of item i
  int64_t* f_prefix;       // [NCF+1] prefix of item costs in id order
  int32_t* f_sorted;       // [NCF]   item at LPT rank r
  int64_t* f_scost;        // [NCF]   cost of the item at rank r
  int32_t* f_grp;          // [NCF]   worker group of rank r
  int32_t* f_pos;          // [NCF]   queue position of rank r
  int32_t* f_qoff;         // [M+1]
  QEntry* f_queue;         // [NCF*Hkv]
  FwdRec* f_rec;           // [NCF*Hkv] the same entries, decoded
  int64_t* f_load_lpt;     // [M]
  int64_t* f_load_contig;  // [M]
  // backward
  int64_t* b_cost;
  int32_t* b_item;
  int64_t* b_prefix;
  int32_t* b_sorted;
  int64_t* b_scost;
  int32_t* b_grp;
  int32_t* b_pos;
  int32_t* b_qoff;
  QEntry* b_queue;
  BwdRec* b_rec;           // [NCB*Hkv] the same entries, decoded
  int64_t* b_load_lpt;
  int64_t* b_load_contig;
  // [NA] a_j + 1 (end of the visible context) when the mask is inclusive
  int32_t* anchor_end;
  // [NA] start of every block's visible context: the caller's offset o_j
  // with SPLITKV_FLAG_MASK_CONTEXT_OFFSET, else 0
  int32_t* anchor_lo;
  // [3][workers][2] %globaltimer (ns) at the start and the end of every
  // worker's CTA in the latest forward, dQ and dK/dV attention launch
  uint64_t* busy_ns;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Computes offsets (base == nullptr: sizes only). Returns total bytes.
inline size_t plan_layout(const PlanCaps& c, char* base, PlanPtrs* p) {
  size_t off = 0;
  auto take = [&](size_t bytes) -> char* {
    off = align_up(off, 256);
    char* r = base ? base + off : nullptr;
    off += bytes;
    return r;
  };
  PlanPtrs q;
  q.hdr = (PlanHeader*)take(sizeof(PlanHeader));
  q.s_nch = (int32_t*)take(4 * (c.S + 1));
  q.s_nsl = (int32_t*)take(4 * (c.S + 1));
  q.s_nkt = (int32_t*)take(4 * (c.S + 1));
  q.s_cand_off = (int32_t*)take(4 * (c.S + 1));
  q.s_slab_off = (int32_t*)take(4 * (c.S + 1));
  q.s_bcand_off = (int32_t*)take(4 * (c.S + 1));
  q.sl_sample = (int32_t*)take(4 * (c.NSL + 1));
  q.sl_first = (int32_t*)take(4 * (c.NSL + 1));
  q.sl_nblk = (int32_t*)take(4 * (c.NSL + 1));
  q.sl_nact = (int32_t*)take(4 * (c.NSL + 1));
  q.sl_slot = (int32_t*)take(4 * (c.NSL + 1));
  q.f_cost = (int64_t*)take(8 * (c.NCF + 1));
  q.f_item = (int32_t*)take(4 * (c.NCF + 1));
  q.f_prefix = (int64_t*)take(8 * (c.NCF + 1));
  q.f_sorted = (int32_t*)take(4 * (c.NCF + 1));
  q.f_scost = (int64_t*)take(8 * (c.NCF + 1));
  q.f_grp = (int32_t*)take(4 * (c.NCF + 1));
  q.f_pos = (int32_t*)take(4 * (c.NCF + 1));
  q.f_qoff = (int32_t*)take(4 * (c.M + 1));
  q.f_queue = (QEntry*)take(sizeof(QEntry) * (c.NCF * c.Hkv + 1));
  q.f_rec = (FwdRec*)take(sizeof(FwdRec) * (c.NCF * c.Hkv + 1));
  q.f_load_lpt = (int64_t*)take(8 * c.M);
  q.f_load_contig = (int64_t*)take(8 * c.M);
  q.b_cost = (int64_t*)take(8 * (c.NCB + 1));
  q.b_item = (int32_t*)take(4 * (c.NCB + 1));
  q.b_prefix = (int64_t*)take(8 * (c.NCB + 1));
  q.b_sorted = (int32_t*)take(4 * (c.NCB + 1));
  q.b_scost = (int64_t*)take(8 * (c.NCB + 1));
  q.b_grp = (int32_t*)take(4 * (c.NCB + 1));
  q.b_pos = (int32_t*)take(4 * (c.NCB + 1));
  q.b_qoff = (int32_t*)take(4 * (c.M + 1));
  q.b_queue = (QEntry*)take(sizeof(QEntry) * (c.NCB * c.Hkv + 1));
  q.b_rec = (BwdRec*)take(sizeof(BwdRec) * (c.NCB * c.Hkv + 1));
  q.b_load_lpt = (int64_t*)take(8 * c.M);
  q.b_load_contig = (int64_t*)take(8 * c.M);
  q.anchor_end = (int32_t*)take(4 * (c.NA + 1));
  q.anchor_lo = (int32_t*)take(4 * (c.NA + 1));
  q.busy_ns = (uint64_t*)take(16 * 3 * c.M);
  if (p) *p = q;
  return align_up(off, 256);
}

// Work workspace: partial O (or dQ) [slots][d/8][128][8] fp32 (part_off),
// partial lse [slots][128] fp32, dQ of the draft blocks [N_q][Hq][d] fp32, the
// backward row term D [Hq][N_q] fp32, the draft-key P / dS [N_q][Hq][B] and
// the per-(slab, kv head) row table the dK/dV kernel streams with each slab,
// and the task counter of the dK/dV kernel's dQ reduction.
struct WorkPtrs {
  float* part_o;
  float* part_lse;
  float* dq_draft;
  float* dvec;
  float* draft_p;    // [N_q][Hq][B] softmax weight of each draft key
  float* draft_ds;   // [N_q][Hq][B] dS of each draft key
  float* rowinfo;    // [slab][Hkv][4][128]: -LSE*log2(e) (-inf on padding rows), D, and the
                     // row's visible context [lo, end) as int bits
  int* red_next;     // next (slab, kv head) task of the dQ reduction; zeroed by the row-table
                     // kernel before each backward's dQ and dK/dV kernels
};

constexpr int kRowInfoFloats = 4 * kRows;  // one (slab, kv head) record: 2048 bytes

// Offset (in floats) of element (row r, dim x) of partial slot `slot` in
// part_o. A slot's 128 rows x D fp32 are stored as [D/8][128][8]: the eight
// consecutive dims of a row that a 32-byte store writes form one sector, and
// the 32 rows of a warp writing the same 8-dim group fill 1 KB contiguously.
__host__ __device__ inline size_t part_off(size_t slot, int r, int x, int D) {
  return slot * (size_t)kRows * D + ((size_t)(x >> 3) * kRows + r) * 8 + (x & 7);
}

inline size_t work_layout(int64_t slots, int64_t nq, int64_t Hq, int64_t d, int64_t B,
                          int64_t slabs_x_hkv, char* base, WorkPtrs* p) {
  size_t off = 0;
  auto take = [&](size_t bytes) -> char* {
    off = align_up(off, 256);
    char* r = base ? base + off : nullptr;
    off += bytes;
    return r;
  };
  WorkPtrs q;
  q.part_o = (float*)take(sizeof(float) * (size_t)slots * kRows * d);
  q.part_lse = (float*)take(sizeof(float) * (size_t)slots * kRows);
  q.dq_draft = (float*)take(sizeof(float) * (size_t)nq * Hq * d);
  q.dvec = (float*)take(sizeof(float) * (size_t)Hq * nq);
  q.draft_p = (float*)take(sizeof(float) * (size_t)nq * Hq * B);
  q.draft_ds = (float*)take(sizeof(float) * (size_t)nq * Hq * B);
  q.rowinfo = (float*)take(sizeof(float) * (size_t)slabs_x_hkv * kRowInfoFloats);
  q.red_next = (int*)take(sizeof(int));
  if (p) *p = q;
  return align_up(off, 256);
}

// Scalars every kernel needs (passed by value).
struct ProbDev {
  int32_t S, B, Hq, Hkv, group, d, chunk, bps, workers, flags, dtype;
  int64_t T, NA, NQ;
  int32_t max_ctx;
  float scale;
  float scale_log2;  // scale * log2(e)
  uint64_t hash;
  const int32_t* cu_ctx;
  const int32_t* cu_anchor;
  const int32_t* anchors;     // end of each block's visible context (a_j, or a_j + 1)
  const int32_t* anchors_in;  // the caller's anchors (validated by the planner)
  const int32_t* ctx_lo;      // start of each block's visible context (the plan's table)
  const int32_t* ctx_lo_in;   // the caller's offsets (SPLITKV_FLAG_MASK_CONTEXT_OFFSET)
};

}  // namespace skv
