// Device planner: realized-attention costs and LPT assignment.
//
// Cost of a work item = the number of masked (query, key) pairs it covers,
// sum over anchors a_j > start of min(len, a_j - start) * B — the "realized
// attention cost" by which the Split-KV abstract (arXiv:2611.05926) balances
// KV chunks; the rit.work article on Split-KV (paragraph on anchor sampling
// and load imbalance) notes the planner can price every segment in advance
// because it sees all queries, and gives the rule: sort segments from most to
// least expensive, give each to the least-loaded accelerator.
//
// Items are priced per (sample, chunk, slab) — the cost does not depend on
// the kv head — and LPT runs over m/Hkv worker groups. Because the Hkv
// replicas of an item have equal cost and consecutive ids (kv head fastest),
// per-head LPT over m workers puts replica g of every item on worker
// Hkv*G + g, where G is the group that grouped LPT picks; the grouped run is
// therefore bit-identical to the per-head rule, Hkv times cheaper.
//
// Three launches: (1) one CTA validates the metadata, computes per-sample
// and per-slab tables and all candidate costs, and compacts positive-cost
// items; (2) a grid ranks items by (cost desc, id asc) by counting; (3) one
// CTA runs the greedy assignment (one warp per direction) and builds the
// per-worker queues and load tables.
#include "common.cuh"
#include "kernels.h"

namespace skv {

namespace {

// Cost of forward item (sample s, chunk c, slab sigma): the masked pairs of
// the slab's blocks in the chunk, sum over blocks of the overlap of their
// visible context [lo_j, end_j) with the chunk, times B. *ks_out / *ke_out:
// the first and the end of the keys any block of the slab sees in the chunk
// (the kernels compute the 128-key tiles covering [*ks_out, *ke_out)).
__device__ __forceinline__ int64_t fwd_item_cost(const ProbDev& P, int s, int c, int sigma,
                                                 int* ks_out, int* ke_out) {
  const int c0 = P.cu_ctx[s];
  const int L = P.cu_ctx[s + 1] - c0;
  const int a0 = P.cu_anchor[s];
  const int A = P.cu_anchor[s + 1] - a0;
  const int cs = c * P.chunk;
  const int ce = cs + min(P.chunk, L - cs);
  const int first = a0 + sigma * P.bps;
  const int nblk = min(P.bps, A - sigma * P.bps);
  int64_t cost = 0;
  int ks = ce, ke = cs;
  for (int b = 0; b < nblk; ++b) {
    const int lo = max(cs, P.ctx_lo[first + b]);
    const int hi = min(ce, P.anchors[first + b]);
    if (hi > lo) {
      cost += (int64_t)(hi - lo) * P.B;
      ks = min(ks, lo);
      ke = max(ke, hi);
    }
  }
  *ks_out = ks;
  *ke_out = ke;
  return cost;
}

// Cost of backward item (sample s, 128-key tile kt): the masked pairs of all
// of the sample's blocks in the tile.
__device__ __forceinline__ int64_t bwd_item_cost(const ProbDev& P, int s, int kt) {
  const int c0 = P.cu_ctx[s];
  const int L = P.cu_ctx[s + 1] - c0;
  const int a0 = P.cu_anchor[s];
  const int a1 = P.cu_anchor[s + 1];
  const int ks = kt * kKeyTile;
  const int ke = ks + min(kKeyTile, L - ks);
  // first anchor > ks (anchors are non-decreasing within the sample)
  int lo = a0, hi = a1;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (P.anchors[mid] > ks) hi = mid; else lo = mid + 1;
  }
  int64_t cost = 0;
  for (int j = lo; j < a1; ++j) {
    const int v = min(ke, P.anchors[j]) - max(ks, P.ctx_lo[j]);
    if (v > 0) cost += (int64_t)v * P.B;
  }
  return cost;
}

// Chunked block scan over an int array producer; writes exclusive prefixes.
template <typename Get, typename Put>
__device__ int64_t scan_array(int n, Get get, Put put, int64_t* ws) {
  int64_t carry = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const int64_t v = i < n ? get(i) : 0;
    int64_t tot;
    const int64_t pre = block_exclusive_scan<int64_t>(v, ws, &tot);
    if (i < n) put(i, carry + pre);
    carry += tot;
  }
  return carry;
}

}  // namespace

__global__ void __launch_bounds__(1024) plan_setup_kernel(ProbDev P, PlanPtrs pp, PlanCaps caps) {
  __shared__ int64_t ws[32];
  __shared__ unsigned long long tiles_acc, dense_acc;
  PlanHeader* H = pp.hdr;
  const int tid = threadIdx.x;
  if (tid == 0) {
    H->magic = kPlanMagic;
    H->status = 0;
    H->workers = P.workers;
    H->groups = P.workers / P.Hkv;
    H->flags = P.flags;
    H->problem_hash = P.hash;
    H->n_slabs = H->n_fwd_cand = H->n_fwd_items = H->n_slot_base = 0;
    H->n_bwd_cand = H->n_bwd_items = 0;
    H->fwd_total_cost = H->bwd_total_cost = H->fwd_tiles = H->dense_tiles = 0;
    H->dbg_count = H->dbg_first = 0;
    tiles_acc = 0;
    dense_acc = 0;
  }
  __syncthreads();
  const int S = P.S;
  // ---- A: validate metadata, per-sample counts -------------------------
  if (tid == 0) {
    if (P.cu_ctx[0] != 0 || P.cu_anchor[0] != 0 || (int64_t)P.cu_ctx[S] != P.T ||
        (int64_t)P.cu_anchor[S] != P.NA)
      latch(H, SPLITKV_EMETA);
  }
  for (int s = tid; s < S; s += blockDim.x) {
    const int L = P.cu_ctx[s + 1] - P.cu_ctx[s];
    const int A = P.cu_anchor[s + 1] - P.cu_anchor[s];
    if (L < 0 || A < 0 || L > P.max_ctx) {
      latch(H, SPLITKV_EMETA);
      continue;
    }
    pp.s_nch[s] = (L + P.chunk - 1) / P.chunk;
    pp.s_nsl[s] = (A + P.bps - 1) / P.bps;
    pp.s_nkt[s] = (L + kKeyTile - 1) / kKeyTile;
    const long long rows = (long long)A * P.B * P.group;
    atomicAdd(&dense_acc, (unsigned long long)(((rows + kRows - 1) / kRows) *
                                               ((L + kKeyTile - 1) / kKeyTile)));
  }
  for (int64_t i = tid; i < P.NA; i += blockDim.x) {
    const int s = seg_of(P.cu_anchor, S, i);
    const int L = P.cu_ctx[s + 1] - P.cu_ctx[s];
    const int a = P.anchors_in[i];
    if (a < 0 || a > L - P.B) latch(H, SPLITKV_EMETA);
    if (i + 1 < P.NA && i + 1 < P.cu_anchor[s + 1] && P.anchors_in[i + 1] < a)
      latch(H, SPLITKV_EMETA);
    // inclusive context [0, a_j]: every later step works with its end a_j + 1
    const int end = (P.flags & SPLITKV_FLAG_MASK_INCLUSIVE) ? a + 1 : a;
    if (P.flags & SPLITKV_FLAG_MASK_INCLUSIVE) pp.anchor_end[i] = end;
    // the start of the block's visible context: its offset, or 0
    const int lo = P.ctx_lo_in ? P.ctx_lo_in[i] : 0;
    if (lo < 0 || lo > end) latch(H, SPLITKV_EMETA);
    pp.anchor_lo[i] = lo;
  }
  __syncthreads();
  if (read_status(H) != 0) return;
  // ---- B: per-sample offsets --------------------------------------------
  const int64_t ncand = scan_array(
      S, [&](int s) { return (int64_t)pp.s_nch[s] * pp.s_nsl[s]; },
      [&](int s, int64_t v) { pp.s_cand_off[s] = (int32_t)v; }, ws);
  const int64_t nslab = scan_array(
      S, [&](int s) { return (int64_t)pp.s_nsl[s]; },
      [&](int s, int64_t v) { pp.s_slab_off[s] = (int32_t)v; }, ws);
  const int64_t nbcand = scan_array(
      S, [&](int s) { return (int64_t)pp.s_nkt[s]; },
      [&](int s, int64_t v) { pp.s_bcand_off[s] = (int32_t)v; }, ws);
  if (tid == 0) {
    if (ncand > caps.NCF || nslab > caps.NSL || nbcand > caps.NCB) latch(H, SPLITKV_ECAPACITY);
    pp.s_cand_off[S] = (int32_t)ncand;
    pp.s_slab_off[S] = (int32_t)nslab;
    pp.s_bcand_off[S] = (int32_t)nbcand;
    H->n_slabs = (int32_t)nslab;
    H->n_fwd_cand = (int32_t)ncand;
    H->n_bwd_cand = (int32_t)nbcand;
  }
  __syncthreads();
  if (read_status(H) != 0) return;
  // ---- C: slab table ------------------------------------------------------
  for (int sg = tid; sg < nslab; sg += blockDim.x) {
    const int s = seg_of(pp.s_slab_off, S, sg);
    const int sigma = sg - pp.s_slab_off[s];
    const int a0 = P.cu_anchor[s];
    const int A = P.cu_anchor[s + 1] - a0;
    const int first = a0 + sigma * P.bps;
    const int nblk = min(P.bps, A - sigma * P.bps);
    const int amax = P.anchors[first + nblk - 1];
    pp.sl_sample[sg] = s;
    pp.sl_first[sg] = first;
    pp.sl_nblk[sg] = nblk;
    pp.sl_nact[sg] = (amax + P.chunk - 1) / P.chunk;
  }
  __syncthreads();
  const int64_t nslot = scan_array(
      (int)nslab, [&](int i) { return (int64_t)pp.sl_nact[i]; },
      [&](int i, int64_t v) { pp.sl_slot[i] = (int32_t)v; }, ws);
  if (tid == 0) {
    pp.sl_slot[nslab] = (int32_t)nslot;
    H->n_slot_base = (int32_t)nslot;
  }
  // ---- D: candidate costs -------------------------------------------------
  unsigned long long my_tiles = 0;  // summed per warp, one shared atomic per warp
  for (int id = tid; id < ncand; id += blockDim.x) {
    const int s = seg_of(pp.s_cand_off, S, id);
    const int local = id - pp.s_cand_off[s];
    const int nsl = pp.s_nsl[s];
    const int c = local / nsl, sigma = local % nsl;
    int ks, ke;
    const int64_t cost = fwd_item_cost(P, s, c, sigma, &ks, &ke);
    pp.f_cost[id] = cost;
    if (cost > 0) {  // tiles from the one holding the first seen key to the last seen key
      const int t0 = (ks - c * P.chunk) / kKeyTile;
      my_tiles += (unsigned long long)((ke - c * P.chunk - t0 * kKeyTile + kKeyTile - 1) / kKeyTile);
    }
  }
  for (int o = 16; o > 0; o >>= 1) my_tiles += __shfl_xor_sync(0xffffffffu, my_tiles, o);
  if ((tid & 31) == 0 && my_tiles) atomicAdd(&tiles_acc, my_tiles);
  for (int id = tid; id < nbcand; id += blockDim.x) {
    const int s = seg_of(pp.s_bcand_off, S, id);
    pp.b_cost[id] = bwd_item_cost(P, s, id - pp.s_bcand_off[s]);
  }
  __syncthreads();
  // ---- E: compaction (id order preserved) ---------------------------------
  for (int kind = 0; kind < 2; ++kind) {
    const int n = kind == 0 ? (int)ncand : (int)nbcand;
    const int64_t* cost = kind == 0 ? pp.f_cost : pp.b_cost;
    int32_t* item = kind == 0 ? pp.f_item : pp.b_item;
    int64_t* prefix = kind == 0 ? pp.f_prefix : pp.b_prefix;
    int64_t carry_n = 0, carry_c = 0;
    for (int base = 0; base < n; base += blockDim.x) {
      const int i = base + tid;
      const int64_t c = i < n ? cost[i] : 0;
      int64_t tn, tc;
      const int64_t pn = block_exclusive_scan<int64_t>(c > 0 ? 1 : 0, ws, &tn);
      const int64_t pc = block_exclusive_scan<int64_t>(c, ws, &tc);
      if (c > 0) {
        item[carry_n + pn] = i;
        prefix[carry_n + pn] = carry_c + pc;
      }
      carry_n += tn;
      carry_c += tc;
    }
    if (tid == 0) {
      prefix[carry_n] = carry_c;
      if (kind == 0) {
        H->n_fwd_items = (int32_t)carry_n;
        H->fwd_total_cost = carry_c;
      } else {
        H->n_bwd_items = (int32_t)carry_n;
        H->bwd_total_cost = carry_c;
      }
    }
    // the rank kernel accumulates each item's rank here (the LPT overwrites it)
    int32_t* racc = kind == 0 ? pp.f_pos : pp.b_pos;
    for (int64_t x = tid; x < carry_n; x += blockDim.x) racc[x] = 0;
    __syncthreads();
  }
  if (tid == 0) {
    H->fwd_tiles = (int64_t)tiles_acc;
    H->dense_tiles = (int64_t)dense_acc;
  }
}

// Rank of item i = #{j : cost_j > cost_i or (cost_j == cost_i and j < i)}.
// Keys are unique, so the ranks form the permutation of the sort
// (cost desc, id asc); items are in id order after compaction. CTA (x, kind,
// z) counts for its 256 items over the z-th of kRankSlices slices of j and
// adds its counts to the items' accumulators (zeroed by the setup kernel):
// integer sums, so the order of the additions does not matter.
constexpr int kRankSlices = 8;

__global__ void __launch_bounds__(256) plan_rank_kernel(PlanPtrs pp) {
  __shared__ int64_t tile[1024];
  const PlanHeader* H = pp.hdr;
  if (read_status(H) != 0) return;
  const int kind = blockIdx.y;
  const int n = kind == 0 ? H->n_fwd_items : H->n_bwd_items;
  const int64_t* cost = kind == 0 ? pp.f_cost : pp.b_cost;
  const int32_t* item = kind == 0 ? pp.f_item : pp.b_item;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if ((int)(blockIdx.x * blockDim.x) >= n) return;  // whole CTA idle
  const int per = (n + (int)gridDim.z - 1) / (int)gridDim.z;
  const int jb = (int)blockIdx.z * per, je = min(n, jb + per);
  if (jb >= je) return;  // CTA-uniform
  const int64_t ci = i < n ? cost[item[i]] : 0;
  int rank = 0;
  for (int j0 = jb; j0 < je; j0 += 1024) {
    __syncthreads();
    for (int t = threadIdx.x; t < 1024; t += blockDim.x)
      tile[t] = (j0 + t < je) ? cost[item[j0 + t]] : INT64_MIN;
    __syncthreads();
    const int lim = min(1024, je - j0);
    for (int t = 0; t < lim; ++t) {
      const int64_t cj = tile[t];
      rank += (cj > ci) | ((cj == ci) & (j0 + t < i));
    }
  }
  if (i < n && rank > 0) atomicAdd((kind == 0 ? pp.f_pos : pp.b_pos) + i, rank);
}

namespace {

// Greedy LPT over the worker groups for one direction, run by one warp.
// Lane l owns groups l, l+32, ... (at most kMaxGroupsPerLane each).
//
// Runs of equal cost (most items are whole chunks of full slabs, so most
// share one cost) are dealt in one step. Write group g's load as
// base + q_g c + rho_g (base = the least load, 0 <= rho_g < c): its i-th
// next item would be picked at load base + (q_g + i) c + rho_g, so LPT's
// picks for k items of cost c go level by level (level j: every group with
// q_g <= j still taking items), and inside a level by (rho_g, g) — the
// least-loaded-first, lowest-id-on-ties order, the same in every level. The
// run's last level J and each group's count follow from counting, and the
// item of run rank t goes to the slot of rank t in that order (one warp step
// per level): exactly the one-at-a-time greedy result, without its serial
// chain.
constexpr int kLptBatch = 48;  // shorter runs go one item at a time

__device__ void lpt_warp(int n, int G, const int64_t* scost, int32_t* grp, int32_t* pos,
                         int64_t* gload, int32_t* gcount, const PlanHeader* H) {
  const int lane = threadIdx.x & 31;
  // Fast path: one group per lane and 32-bit keys. While items are dealt
  // most expensive first to the least-loaded group, max load - min load
  // never exceeds the largest cost, so (load - running minimum) * 32 + group
  // fits 32 bits when that cost is < 2^26, and a single warp min-reduction
  // finds the least-loaded group with the lowest id.
  if (G <= 32 && (n == 0 || scost[0] < (1LL << 26))) {
    // rel = this lane's load minus the running minimum base (< 2^26)
    uint32_t rel = 0;
    int64_t base = 0;
    int32_t cnt = 0;
    int r = 0;
    // costs [w0, w0 + 32), one per lane (-1 past the end: costs are
    // positive), refilled by one coalesced load when r leaves the window, so
    // that finding a run costs a shuffle and a ballot, not two dependent
    // loads
    int w0 = 0;
    int64_t win = lane < n ? scost[lane] : -1;
    while (r < n) {
      if (r >= w0 + 32) {
        w0 = r;
        win = w0 + lane < n ? scost[w0 + lane] : -1;
      }
      const int64_t c64 = __shfl_sync(0xffffffffu, win, r - w0);
      int e;  // end of the run of items of cost c64
      const unsigned diff =
          __ballot_sync(0xffffffffu, lane > r - w0 && win != c64);
      if (diff) {
        e = w0 + __ffs(diff) - 1;
      } else {  // the run reaches past the window: scan on in global memory
        e = w0 + 32;
        for (;;) {
          const int i = e + lane;
          const unsigned d2 = __ballot_sync(0xffffffffu, i >= n || scost[i] != c64);
          if (d2) {
            e += __ffs(d2) - 1;
            break;
          }
          e += 32;
        }
      }
      const uint32_t c = (uint32_t)c64;
      const int k = e - r;
      if (k < kLptBatch) {
        // one item at a time: the least-loaded group (lowest id on ties) takes it
        for (int t = r; t < e; ++t) {
          const uint32_t key = lane < G ? (rel << 5) | (uint32_t)lane : 0xffffffffu;
          const uint32_t m = __reduce_min_sync(0xffffffffu, key);
          const bool take = (int)(m & 31u) == lane;
          if (take) {
            grp[t] = lane;
            pos[t] = cnt;
          }
          rel = rel - (m >> 5) + (take ? c : 0u);
          cnt += take ? 1 : 0;
          base += (int64_t)(m >> 5);
        }
      } else {
        const bool act = lane < G;
        const int q = act ? (int)(rel / c) : 0x3fffffff;   // level of this group's first pick
        const uint32_t rho = rel % c;
        // J = the smallest level with sum_g max(0, J - q_g + 1) >= k
        int lo = 0, hi = k / G + 1 + (int)__reduce_max_sync(0xffffffffu, act ? (uint32_t)q : 0u);
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          const uint32_t have = __reduce_add_sync(0xffffffffu, act && q <= mid ? (uint32_t)(mid - q + 1) : 0u);
          if ((int)have >= k) hi = mid; else lo = mid + 1;
        }
        const int J = lo;
        const int below = (int)__reduce_add_sync(0xffffffffu, act && q < J ? (uint32_t)(J - q) : 0u);
        // rank of this group in the in-level order (rho, g)
        int ord = 0;
        for (int o = 0; o < G; ++o) {
          const uint32_t ro = __shfl_sync(0xffffffffu, rho, o);
          ord += (ro < rho || (ro == rho && o < lane)) ? 1 : 0;
        }
        // in level J, the first (k - below) groups in that order that reach it
        const bool inJ = act && q <= J;
        const unsigned inJmask = __ballot_sync(0xffffffffu, inJ);
        int before = 0;  // groups of level J ahead of this one in the order
        for (int o = 0; o < G; ++o) {
          const int oo = __shfl_sync(0xffffffffu, ord, o);
          before += (((inJmask >> o) & 1u) && oo < ord) ? 1 : 0;
        }
        const int take = !act ? 0 : (q < J ? J - q : 0) + (inJ && before < k - below ? 1 : 0);
        // the picks, level by level: the groups active at level j (those
        // with q_g <= j < q_g + take_g) take the next ranks of the run, in the
        // in-level order; the set is a bit mask over order positions (G <= 32)
        const int jmin =
            (int)__reduce_min_sync(0xffffffffu, act && take > 0 ? (uint32_t)q : 0x7fffffffu);
        int rk0 = r;
        for (int j = jmin; j <= J; ++j) {
          const bool on = act && take > 0 && q <= j && j < q + take;
          const uint32_t mask = __reduce_or_sync(0xffffffffu, on ? (1u << ord) : 0u);
          if (on) {
            const int rk = rk0 + __popc(mask & ((1u << ord) - 1u));
            if (SKV_OK(rk >= r && rk < e, H, kDbgPlanScatter, rk)) {
              grp[rk] = lane;
              pos[rk] = cnt + (j - q);
            }
          }
          rk0 += __popc(mask);
        }
        // new loads (64-bit: a long run can add more than 2^32), renormalised
        // to the least one; the spread stays below the largest cost (< 2^26)
        const uint64_t nrel = act ? (uint64_t)rel + (uint64_t)take * c : ~0ull;
        uint64_t mn = nrel;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const uint64_t x = __shfl_xor_sync(0xffffffffu, mn, o);
          mn = x < mn ? x : mn;
        }
        rel = act ? (uint32_t)(nrel - mn) : 0u;
        base += (int64_t)mn;
        cnt += take;
      }
      r = e;
    }
    if (lane < G) {
      gload[lane] = base + (int64_t)rel;
      gcount[lane] = cnt;
    }
    return;
  }
  int64_t load[kMaxGroupsPerLane];
  int32_t cnt[kMaxGroupsPerLane];
#pragma unroll
  for (int k = 0; k < kMaxGroupsPerLane; ++k) {
    load[k] = 0;
    cnt[k] = 0;
  }
  for (int r0 = 0; r0 < n; r0 += 32) {
    const int64_t mine = (r0 + lane < n) ? scost[r0 + lane] : 0;
    const int lim = min(32, n - r0);
    for (int t = 0; t < lim; ++t) {
      const int64_t c = __shfl_sync(0xffffffffu, mine, t);
      int64_t bl = INT64_MAX;
      int bg = INT32_MAX;
#pragma unroll
      for (int k = 0; k < kMaxGroupsPerLane; ++k) {
        const int gid = lane + 32 * k;
        if (gid < G && load[k] < bl) {  // ascending gid within the lane
          bl = load[k];
          bg = gid;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const int64_t ol = __shfl_xor_sync(0xffffffffu, bl, o);
        const int og = __shfl_xor_sync(0xffffffffu, bg, o);
        if (ol < bl || (ol == bl && og < bg)) {
          bl = ol;
          bg = og;
        }
      }
      if ((bg & 31) == lane) {
        const int kk = bg >> 5;
#pragma unroll
        for (int k = 0; k < kMaxGroupsPerLane; ++k) {
          if (k == kk) {
            grp[r0 + t] = bg;
            pos[r0 + t] = cnt[k];
            cnt[k] += 1;
            load[k] += c;
          }
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kMaxGroupsPerLane; ++k) {
    const int gid = lane + 32 * k;
    if (gid < G) {
      gload[gid] = load[k];
      gcount[gid] = cnt[k];
    }
  }
}

__device__ __forceinline__ QEntry decode_fwd(const ProbDev& P, const PlanPtrs& pp, int cand,
                                             int g) {
  const int s = seg_of(pp.s_cand_off, P.S, cand);
  const int local = cand - pp.s_cand_off[s];
  const int nsl = pp.s_nsl[s];
  QEntry e;
  e.s = s;
  e.c = local / nsl;
  e.slab = pp.s_slab_off[s] + local % nsl;
  e.g = g;
  return e;
}

// The decoded form of forward entry e (see FwdRec): the 128-key tiles of
// the chunk from the one holding the first key any block of the slab sees to
// the last such key; cs / row0 name the first computed tile.
__device__ __forceinline__ FwdRec fwd_rec(const ProbDev& P, const PlanPtrs& pp, const QEntry& e) {
  FwdRec R;
  R.first = pp.sl_first[e.slab];
  R.nblk = pp.sl_nblk[e.slab];
  const int c0 = P.cu_ctx[e.s];
  int ks, ke;
  fwd_item_cost(P, e.s, e.c, e.slab - pp.s_slab_off[e.s], &ks, &ke);
  const int t0 = (ks - e.c * P.chunk) / kKeyTile;
  R.cs = e.c * P.chunk + t0 * kKeyTile;
  R.ntiles = (ke - R.cs + kKeyTile - 1) / kKeyTile;
  R.row0 = c0 + R.cs;
  R.n0 = R.first * P.B;
  R.g = e.g;
  R.slot = (pp.sl_slot[e.slab] + e.c) * P.Hkv + e.g;
  return R;
}

// The decoded form of backward entry e (see BwdRec): the slabs that see the
// key tile start at the first one whose last visible key lies beyond the
// tile start (anchors, hence slabs' last anchors, rise within a sample).
__device__ __forceinline__ BwdRec bwd_rec(const ProbDev& P, const PlanPtrs& pp, const QEntry& e) {
  BwdRec R;
  R.s = e.s;
  R.g = e.g;
  R.c0 = P.cu_ctx[e.s];
  R.L = P.cu_ctx[e.s + 1] - R.c0;
  R.ks0 = e.c * kKeyTile;
  const int sl0 = pp.s_slab_off[e.s], sl1 = pp.s_slab_off[e.s + 1];
  int lo = sl0, hi = sl1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (P.anchors[pp.sl_first[mid] + pp.sl_nblk[mid] - 1] > R.ks0) hi = mid; else lo = mid + 1;
  }
  R.sl_lo = lo;
  R.sl_hi = sl1;
  R.pad = 0;
  return R;
}

__device__ __forceinline__ QEntry decode_bwd(const ProbDev& P, const PlanPtrs& pp, int cand,
                                             int g) {
  const int s = seg_of(pp.s_bcand_off, P.S, cand);
  QEntry e;
  e.s = s;
  e.c = cand - pp.s_bcand_off[s];
  e.slab = 0;
  e.g = g;
  return e;
}

}  // namespace

__global__ void __launch_bounds__(1024) plan_assign_kernel(ProbDev P, PlanPtrs pp) {
  __shared__ int64_t ws[32];
  __shared__ int64_t gload[2][32 * kMaxGroupsPerLane];
  __shared__ int32_t gcount[2][32 * kMaxGroupsPerLane];
  const PlanHeader* H = pp.hdr;
  if (read_status(H) != 0) return;
  const int tid = threadIdx.x;
  const int m = P.workers, Hkv = P.Hkv, G = m / Hkv;
  const bool contiguous = (P.flags & SPLITKV_FLAG_CONTIGUOUS) != 0;
  const int warp = tid >> 5;
  // the sort order from the ranks the rank kernel accumulated in f_pos / b_pos
  for (int kind = 0; kind < 2; ++kind) {
    const int n = kind == 0 ? H->n_fwd_items : H->n_bwd_items;
    const int32_t* racc = kind == 0 ? pp.f_pos : pp.b_pos;
    const int64_t* cost = kind == 0 ? pp.f_cost : pp.b_cost;
    const int32_t* item = kind == 0 ? pp.f_item : pp.b_item;
    int32_t* sorted = kind == 0 ? pp.f_sorted : pp.b_sorted;
    int64_t* scost = kind == 0 ? pp.f_scost : pp.b_scost;
    for (int i = tid; i < n; i += blockDim.x) {
      const int r = racc[i];
      if (SKV_OK(r >= 0 && r < n, H, kDbgPlanScatter, r)) {
        sorted[r] = i;
        scost[r] = cost[item[i]];
      }
    }
  }
  __syncthreads();  // the LPT reads the sorted costs and overwrites f_pos / b_pos
  if (warp < 2) {
    const int n = warp == 0 ? H->n_fwd_items : H->n_bwd_items;
    lpt_warp(n, G, warp == 0 ? pp.f_scost : pp.b_scost, warp == 0 ? pp.f_grp : pp.b_grp,
             warp == 0 ? pp.f_pos : pp.b_pos, gload[warp], gcount[warp], H);
  }
  __syncthreads();
  for (int kind = 0; kind < 2; ++kind) {
    const int n = kind == 0 ? H->n_fwd_items : H->n_bwd_items;
    const int64_t N = (int64_t)n * Hkv;  // per-head items
    const int64_t* cost = kind == 0 ? pp.f_cost : pp.b_cost;
    const int32_t* item = kind == 0 ? pp.f_item : pp.b_item;
    const int64_t* prefix = kind == 0 ? pp.f_prefix : pp.b_prefix;
    int32_t* qoff = kind == 0 ? pp.f_qoff : pp.b_qoff;
    int64_t* load_lpt = kind == 0 ? pp.f_load_lpt : pp.b_load_lpt;
    int64_t* load_contig = kind == 0 ? pp.f_load_contig : pp.b_load_contig;
    // Per-head cost prefix F(x) over the per-head items in id order.
    auto F = [&](int64_t x) -> int64_t {
      const int64_t b = x / Hkv, r = x % Hkv;
      int64_t v = prefix[b] * Hkv;
      if (r) v += r * cost[item[b]];
      return v;
    };
    for (int w = tid; w < m; w += blockDim.x) {
      load_lpt[w] = gload[kind][w / Hkv];
      const int64_t lo = (int64_t)w * N / m, hi = (int64_t)(w + 1) * N / m;
      load_contig[w] = F(hi) - F(lo);
    }
    if (!contiguous) {
      const int64_t tot = scan_array(
          m, [&](int w) { return (int64_t)gcount[kind][w / Hkv]; },
          [&](int w, int64_t v) { qoff[w] = (int32_t)v; }, ws);
      if (tid == 0) qoff[m] = (int32_t)tot;
    } else {
      for (int w = tid; w <= m; w += blockDim.x) qoff[w] = (int32_t)((int64_t)w * N / m);
    }
    __syncthreads();
  }
}

// Queue entries and decoded records at the positions the assignment chose:
// one thread per candidate (LPT: its Hkv replicas go to the same position of
// the Hkv workers of its group) or per per-head item (contiguous), over a
// grid, since every entry is independent. blockIdx.y is the direction.
__global__ void __launch_bounds__(256) plan_queue_kernel(ProbDev P, PlanPtrs pp) {
  const PlanHeader* H = pp.hdr;
  if (read_status(H) != 0) return;
  const int kind = blockIdx.y;
  const int Hkv = P.Hkv;
  const int n = kind == 0 ? H->n_fwd_items : H->n_bwd_items;
  const int32_t* item = kind == 0 ? pp.f_item : pp.b_item;
  QEntry* queue = kind == 0 ? pp.f_queue : pp.b_queue;
  const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  if ((P.flags & SPLITKV_FLAG_CONTIGUOUS) == 0) {
    const int32_t* qoff = kind == 0 ? pp.f_qoff : pp.b_qoff;
    const int32_t* sorted = kind == 0 ? pp.f_sorted : pp.b_sorted;
    const int32_t* grp = kind == 0 ? pp.f_grp : pp.b_grp;
    const int32_t* pos = kind == 0 ? pp.f_pos : pp.b_pos;
    for (int64_t r = first; r < n; r += stride) {
      const int cand = item[sorted[r]];
      const int Gr = grp[r], p = pos[r];
      // the record of replica g differs from replica 0's only in g (and slot)
      QEntry e = kind == 0 ? decode_fwd(P, pp, cand, 0) : decode_bwd(P, pp, cand, 0);
      FwdRec fr;
      BwdRec br;
      if (kind == 0) fr = fwd_rec(P, pp, e); else br = bwd_rec(P, pp, e);
      for (int g = 0; g < Hkv; ++g) {
        const int at = qoff[Gr * Hkv + g] + p;
        if (!SKV_OK(at >= 0 && at < (int64_t)n * Hkv, H, kDbgPlanScatter, at)) continue;
        e.g = g;
        queue[at] = e;
        if (kind == 0) {
          fr.g = g;
          pp.f_rec[at] = fr;
          ++fr.slot;
        } else {
          br.g = g;
          pp.b_rec[at] = br;
        }
      }
    }
  } else {
    const int64_t N = (int64_t)n * Hkv;  // per-head items, in id order
    for (int64_t x = first; x < N; x += stride) {
      const int cand = item[x / Hkv];
      const int g = (int)(x % Hkv);
      queue[x] = kind == 0 ? decode_fwd(P, pp, cand, g) : decode_bwd(P, pp, cand, g);
      if (kind == 0) pp.f_rec[x] = fwd_rec(P, pp, queue[x]);
      else pp.b_rec[x] = bwd_rec(P, pp, queue[x]);
    }
  }
}

}  // namespace skv

namespace skv {

cudaError_t launch_plan(const ProbDev& P, const PlanPtrs& pp, const PlanCaps& caps,
                        cudaStream_t st) {
  plan_setup_kernel<<<1, 1024, 0, st>>>(P, pp, caps);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int64_t maxn = caps.NCF > caps.NCB ? caps.NCF : caps.NCB;
  dim3 grid((unsigned)((maxn + 255) / 256 > 0 ? (maxn + 255) / 256 : 1), 2);
  plan_rank_kernel<<<dim3(grid.x, 2, kRankSlices), 256, 0, st>>>(pp);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  plan_assign_kernel<<<1, 1024, 0, st>>>(P, pp);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  plan_queue_kernel<<<grid, 256, 0, st>>>(P, pp);
  return cudaGetLastError();
}

}  // namespace skv
