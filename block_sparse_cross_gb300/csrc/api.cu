// C ABI of the library: argument validation, workspace carving and the
// launch sequence of each pass. See include/splitkv.h for the contract.
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <initializer_list>
#include <mutex>
#include <vector>

#include "kernels.h"

using namespace skv;

namespace {

constexpr int kKnownFlags = SPLITKV_FLAG_CUDA_CORE | SPLITKV_FLAG_CONTIGUOUS |
                            SPLITKV_FLAG_MASK_INCLUSIVE | SPLITKV_FLAG_MASK_CAUSAL_BLOCK |
                            SPLITKV_FLAG_MASK_CONTEXT_OFFSET;

int check_problem(const splitkv_problem* p) {
  if (!p) return SPLITKV_EINVAL;
  if (p->num_samples < 1 || !p->cu_ctx || !p->cu_anchor) return SPLITKV_EINVAL;
  if (p->total_anchors > 0 && !p->anchors) return SPLITKV_EINVAL;
  if ((p->flags & SPLITKV_FLAG_MASK_CONTEXT_OFFSET) && p->total_anchors > 0 && !p->ctx_lo)
    return SPLITKV_EINVAL;
  if (p->total_ctx < 0 || p->total_anchors < 0 || p->max_ctx < 0) return SPLITKV_EINVAL;
  if (p->B < 1 || p->Hq < 1 || p->Hkv < 1 || p->chunk < 1 || p->num_workers < 0)
    return SPLITKV_EINVAL;
  if (!(p->scale > 0.f) || !isfinite(p->scale)) return SPLITKV_EINVAL;
  if (p->flags & ~kKnownFlags) return SPLITKV_EINVAL;
  if (p->Hq % p->Hkv) return SPLITKV_EUNSUPPORTED;
  const int group = p->Hq / p->Hkv;
  if ((int64_t)p->B * group > kRows || kRows % (p->B * group)) return SPLITKV_EUNSUPPORTED;
  if (p->d != 64 && p->d != 128) return SPLITKV_EUNSUPPORTED;
  if (p->chunk % kKeyTile) return SPLITKV_EUNSUPPORTED;
  if (p->dtype != SPLITKV_BF16 && p->dtype != SPLITKV_FP32) return SPLITKV_EUNSUPPORTED;
  // int32 indexing of rows, keys and anchors on the device
  if (p->total_ctx >= (1LL << 31) - kKeyTile || p->total_anchors * p->B >= (1LL << 31) ||
      p->max_ctx >= (1 << 30))
    return SPLITKV_EUNSUPPORTED;
  if (p->num_workers > 0) {
    if (p->num_workers % p->Hkv || p->num_workers > kMaxWorkers ||
        p->num_workers / p->Hkv > 32 * kMaxGroupsPerLane)
      return SPLITKV_EUNSUPPORTED;
  }
  return SPLITKV_OK;
}

int resolve_workers(const splitkv_problem* p, int* m) {
  if (p->num_workers > 0) {
    *m = p->num_workers;
    return SPLITKV_OK;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPLITKV_EDEVICE;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SPLITKV_EDEVICE;
  int w = sms / p->Hkv * p->Hkv;
  if (w < p->Hkv) w = p->Hkv;
  const int cap = std::min(kMaxWorkers, 32 * kMaxGroupsPerLane * p->Hkv) / p->Hkv * p->Hkv;
  *m = std::min(w, cap);
  return SPLITKV_OK;
}

PlanCaps caps_of(const splitkv_problem* p, int m) {
  PlanCaps c;
  const int64_t group = p->Hq / p->Hkv;
  const int64_t bps = kRows / (p->B * group);
  c.S = p->num_samples;
  c.NA = p->total_anchors;
  c.NSL = p->total_anchors == 0 ? 0
                                : std::min<int64_t>(p->total_anchors,
                                                    (p->total_anchors + bps - 1) / bps + c.S);
  const int64_t nch = ((int64_t)p->max_ctx + p->chunk - 1) / p->chunk;
  c.NCF = nch * c.NSL;
  c.NCB = (p->total_ctx + kKeyTile - 1) / kKeyTile + c.S;
  c.M = m;
  c.Hkv = p->Hkv;
  return c;
}

uint64_t problem_hash(const splitkv_problem* p, int m) {
  uint64_t h = 1469598103934665603ull;
  auto mix = [&](int64_t v) {
    for (int i = 0; i < 8; ++i) {
      h ^= (uint64_t)((v >> (8 * i)) & 0xff);
      h *= 1099511628211ull;
    }
  };
  uint32_t sbits;
  memcpy(&sbits, &p->scale, 4);
  mix(p->num_samples); mix(p->total_ctx); mix(p->total_anchors); mix(p->max_ctx);
  mix(p->B); mix(p->Hq); mix(p->Hkv); mix(p->d); mix(p->chunk); mix(p->dtype);
  mix(m); mix(sbits);
  mix(p->flags & (SPLITKV_FLAG_CONTIGUOUS | SPLITKV_FLAG_MASK_INCLUSIVE |
                  SPLITKV_FLAG_MASK_CAUSAL_BLOCK | SPLITKV_FLAG_MASK_CONTEXT_OFFSET));
  return h;
}

ProbDev make_dev(const splitkv_problem* p, int m) {
  ProbDev P;
  P.S = p->num_samples;
  P.B = p->B;
  P.Hq = p->Hq;
  P.Hkv = p->Hkv;
  P.group = p->Hq / p->Hkv;
  P.d = p->d;
  P.chunk = p->chunk;
  P.bps = kRows / (p->B * P.group);
  P.workers = m;
  P.flags = p->flags;
  P.dtype = p->dtype;
  P.T = p->total_ctx;
  P.NA = p->total_anchors;
  P.NQ = p->total_anchors * p->B;
  P.max_ctx = p->max_ctx;
  P.scale = p->scale;
  P.scale_log2 = p->scale * 1.4426950408889634f;
  P.hash = problem_hash(p, m);
  P.cu_ctx = p->cu_ctx;
  P.cu_anchor = p->cu_anchor;
  P.anchors = p->anchors;      // replaced by the plan's a_j + 1 table when inclusive
  P.anchors_in = p->anchors;
  P.ctx_lo = nullptr;          // the plan's table (set up in setup())
  P.ctx_lo_in = (p->flags & SPLITKV_FLAG_MASK_CONTEXT_OFFSET) ? p->ctx_lo : nullptr;
  return P;
}

size_t plan_bytes_for(const splitkv_problem* p) {
  // sized for the largest worker count so that the size needs no device query
  return plan_layout(caps_of(p, kMaxWorkers), nullptr, nullptr);
}

size_t work_bytes_for(const splitkv_problem* p) {
  const PlanCaps c = caps_of(p, kMaxWorkers);
  return work_layout(c.NCF * p->Hkv, p->total_anchors * p->B, p->Hq, p->d, p->B,
                     c.NSL * p->Hkv, nullptr, nullptr);
}

struct Ctx {
  ProbDev P;
  PlanCaps caps;
  PlanPtrs pp;
};

int setup(const splitkv_problem* p, const void* plan_ws, Ctx* c) {
  int st = check_problem(p);
  if (st) return st;
  if (!plan_ws) return SPLITKV_EINVAL;
  int m = 0;
  st = resolve_workers(p, &m);
  if (st) return st;
  c->P = make_dev(p, m);
  c->caps = caps_of(p, kMaxWorkers);
  c->caps.M = kMaxWorkers;
  plan_layout(c->caps, (char*)plan_ws, &c->pp);
  // every kernel after the planner's validation reads the end of each
  // block's visible context from P.anchors
  if (p->flags & SPLITKV_FLAG_MASK_INCLUSIVE) c->P.anchors = c->pp.anchor_end;
  c->P.ctx_lo = c->pp.anchor_lo;  // the start of every block's context (0 without offsets)
  return SPLITKV_OK;
}

bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? SPLITKV_OK : SPLITKV_ECUDA; }

bool use_tensor_cores(const ProbDev& P) {
  return P.dtype == SPLITKV_BF16 && !(P.flags & SPLITKV_FLAG_CUDA_CORE);
}

// ---- launch timing --------------------------------------------------------
struct ProfRec {
  int kernel, launches;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof_recs;
std::vector<cudaEvent_t> g_prof_pool;

cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

void prof_clear() {
  for (auto& r : g_prof_recs) {
    g_prof_pool.push_back(r.a);
    g_prof_pool.push_back(r.b);
  }
  g_prof_recs.clear();
}

// Runs a launcher; when timing is on, brackets it with events on `st`.
template <typename F>
cudaError_t timed(int kernel, int launches, cudaStream_t st, F&& f) {
  std::unique_lock<std::mutex> lk(g_prof_mu);
  if (!g_prof_on) {
    lk.unlock();
    return f();
  }
  cudaEvent_t a = prof_event(), b = prof_event();
  cudaEventRecord(a, st);
  const cudaError_t e = f();
  cudaEventRecord(b, st);
  g_prof_recs.push_back({kernel, launches, a, b});
  return e;
}

// ---- projections ------------------------------------------------------------
int check_proj(const splitkv_problem* p, int hidden) {
  const int st = check_problem(p);
  if (st) return st;
  if (hidden <= 0) return SPLITKV_EINVAL;
  if (p->dtype != SPLITKV_BF16 || hidden % 64 || hidden >= (1 << 24)) return SPLITKV_EUNSUPPORTED;
  return SPLITKV_OK;
}

bool all_aligned(std::initializer_list<const void*> ptrs) {
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return false;
  return true;
}

// One-segment product C = A B with the given operand forms.
ProjSpec proj_one(int64_t M, int64_t N, int a_mn, int b_mn, ProjOperand a, ProjOperand b,
                  int64_t b_off, int64_t klen, int out_f32) {
  ProjSpec s;
  memset(&s, 0, sizeof(s));
  s.M = M;
  s.N = N;
  s.a_mn = a_mn;
  s.b_mn = b_mn;
  s.b_off = b_off;
  s.nseg = 1;
  s.a[0] = a;
  s.b[0] = b;
  s.klen[0] = klen;
  s.ksplit = 1;
  s.out_f32 = out_f32;
  return s;
}

void add_seg(ProjSpec* s, ProjOperand a, ProjOperand b, int64_t k0_b, int64_t klen) {
  const int j = s->nseg++;
  s->a[j] = a;
  s->b[j] = b;
  s->k0_b[j] = k0_b;
  s->klen[j] = klen;
}

void add_dst(ProjSpec* s, void* ptr, int col0, int ncols, int64_t ld) {
  ProjDst& d = s->dst[s->ndst++];
  d.ptr = ptr;
  d.col0 = col0;
  d.ncols = ncols;
  d.ld = ld;
}

int run_proj(const ProjSpec* parts, int n, cudaStream_t s) {
  if (n == 0) return SPLITKV_OK;
  return cuda_status(timed(SPLITKV_K_PROJ, 1, s, [&] { return launch_proj(parts, n, s); }));
}

// The per-worker queues the attention kernels walk (LPT or contiguous,
// whichever the plan holds), worker by worker in queue order, each entry
// mapped back to its per-kv-head item id and cost.
int export_queues(const Ctx& c, const PlanHeader& h, bool fwd, int64_t* ids, int64_t* costs,
                  int32_t* worker, int32_t* pos, int64_t capacity, int64_t* count) {
  const int m = c.P.workers, S = c.P.S, Hkv = c.P.Hkv;
  const int ncand = fwd ? h.n_fwd_cand : h.n_bwd_cand;
  std::vector<int32_t> qoff(m + 1), cand_off(S + 1), nsl(S + 1), slab_off(S + 1);
  std::vector<int64_t> cost(ncand > 0 ? ncand : 1);
  cudaError_t e = cudaMemcpy(qoff.data(), fwd ? c.pp.f_qoff : c.pp.b_qoff, 4 * (m + 1),
                             cudaMemcpyDeviceToHost);
  e = e ? e : cudaMemcpy(cand_off.data(), fwd ? c.pp.s_cand_off : c.pp.s_bcand_off, 4 * (S + 1),
                         cudaMemcpyDeviceToHost);
  e = e ? e : cudaMemcpy(nsl.data(), c.pp.s_nsl, 4 * (S + 1), cudaMemcpyDeviceToHost);
  e = e ? e : cudaMemcpy(slab_off.data(), c.pp.s_slab_off, 4 * (S + 1), cudaMemcpyDeviceToHost);
  if (ncand > 0)
    e = e ? e : cudaMemcpy(cost.data(), fwd ? c.pp.f_cost : c.pp.b_cost, 8 * (size_t)ncand,
                           cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return SPLITKV_ECUDA;
  const int64_t n = qoff[m];
  *count = n;
  std::vector<QEntry> q(n > 0 ? n : 1);
  if (n > 0 && cudaMemcpy(q.data(), fwd ? c.pp.f_queue : c.pp.b_queue, sizeof(QEntry) * n,
                          cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPLITKV_ECUDA;
  int64_t k = 0;
  for (int w = 0; w < m; ++w) {
    for (int32_t at = qoff[w]; at < qoff[w + 1]; ++at, ++k) {
      if (k >= capacity) return SPLITKV_OK;
      const QEntry& x = q[at];
      if (x.s < 0 || x.s >= S) return SPLITKV_EINVAL;
      const int64_t cand =
          fwd ? (int64_t)cand_off[x.s] + (int64_t)x.c * nsl[x.s] + (x.slab - slab_off[x.s])
              : (int64_t)cand_off[x.s] + x.c;
      if (cand < 0 || cand >= ncand) return SPLITKV_EINVAL;
      ids[k] = cand * Hkv + x.g;
      costs[k] = cost[cand];
      worker[k] = w;
      pos[k] = at - qoff[w];
    }
  }
  return SPLITKV_OK;
}

}  // namespace

extern "C" {

int splitkv_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (on) prof_clear();
  g_prof_on = on != 0;
  return SPLITKV_OK;
}

int splitkv_profile_read(int32_t* launches, double* total_ms, int n) {
  if (!launches || !total_ms || n < 0) return SPLITKV_EINVAL;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (int i = 0; i < n; ++i) {
    launches[i] = 0;
    total_ms[i] = 0.0;
  }
  for (const auto& r : g_prof_recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return SPLITKV_ECUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return SPLITKV_ECUDA;
    if (r.kernel < n) {
      launches[r.kernel] += r.launches;
      total_ms[r.kernel] += ms;
    }
  }
  return SPLITKV_OK;
}

int splitkv_busy_read(const splitkv_problem* prob, const void* plan_ws, int kernel_id,
                      uint64_t* ns, int capacity, int* workers, splitkv_stream stream) {
  Ctx c;
  const int st = setup(prob, plan_ws, &c);
  if (st) return st;
  int slot;
  switch (kernel_id) {
    case SPLITKV_K_FWD_ATTN: slot = 0; break;
    case SPLITKV_K_BWD_DQ: slot = 1; break;
    case SPLITKV_K_BWD_DKDV: slot = 2; break;
    default: return SPLITKV_EINVAL;
  }
  if (!ns || !workers || capacity < 0) return SPLITKV_EINVAL;
  const int m = c.P.workers;
  *workers = m;
  if (capacity < 2 * m) return SPLITKV_EINVAL;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return SPLITKV_ECUDA;
  return cuda_status(cudaMemcpy(ns, c.pp.busy_ns + (size_t)slot * m * 2, sizeof(uint64_t) * 2 * m,
                                cudaMemcpyDeviceToHost));
}

const char* splitkv_kernel_name(int kernel_id) {
  static const char* names[SPLITKV_NUM_KERNELS] = {
      "plan", "fwd_attention", "merge", "bwd_draft", "bwd_dq", "bwd_dkdv", "dq_reduce",
      "zero_uncovered", "projection"};
  return (kernel_id >= 0 && kernel_id < SPLITKV_NUM_KERNELS) ? names[kernel_id] : "unknown";
}

int splitkv_workspace_size(const splitkv_problem* prob, size_t* plan_bytes, size_t* work_bytes) {
  const int st = check_problem(prob);
  if (st) return st;
  if (!plan_bytes || !work_bytes) return SPLITKV_EINVAL;
  *plan_bytes = plan_bytes_for(prob);
  *work_bytes = work_bytes_for(prob);
  return SPLITKV_OK;
}

int splitkv_resolve_workers(const splitkv_problem* prob, int* workers) {
  const int st = check_problem(prob);
  if (st) return st;
  if (!workers) return SPLITKV_EINVAL;
  return resolve_workers(prob, workers);
}

int splitkv_plan(const splitkv_problem* prob, void* plan_ws, size_t plan_bytes,
                 splitkv_stream stream) {
  Ctx c;
  int st = setup(prob, plan_ws, &c);
  if (st) return st;
  if (plan_bytes < plan_bytes_for(prob)) return SPLITKV_EWORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  return cuda_status(timed(SPLITKV_K_PLAN, 4, s, [&] { return launch_plan(c.P, c.pp, c.caps, s); }));
}

int splitkv_fwd(const splitkv_problem* prob, const void* plan_ws, const void* Q, const void* Kc,
                const void* Vc, const void* Kd, const void* Vd, void* O, float* LSE, void* work,
                size_t work_bytes, splitkv_stream stream) {
  Ctx c;
  int st = setup(prob, plan_ws, &c);
  if (st) return st;
  const bool any_q = prob->total_anchors > 0;
  if (any_q && (!Q || !Kd || !Vd || !O || !LSE || !work)) return SPLITKV_EINVAL;
  if (prob->total_ctx > 0 && (!Kc || !Vc)) return SPLITKV_EINVAL;
  const void* ptrs[] = {Q, Kc, Vc, Kd, Vd, O, LSE, work};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return SPLITKV_EINVAL;
  if (work_bytes < work_bytes_for(prob)) return SPLITKV_EWORKSPACE;
  if (!any_q) return SPLITKV_OK;
  WorkPtrs wk;
  work_layout(c.caps.NCF * prob->Hkv, c.P.NQ, prob->Hq, prob->d, prob->B,
              c.caps.NSL * prob->Hkv, (char*)work, &wk);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = timed(SPLITKV_K_FWD_ATTN, 1, s, [&] {
    return use_tensor_cores(c.P) ? launch_fwd_tc(c.P, c.pp, wk, Q, Kc, Vc, s)
                                 : launch_fwd_simt(c.P, c.pp, wk, Q, Kc, Vc, s);
  });
  if (e != cudaSuccess) return SPLITKV_ECUDA;
  return cuda_status(
      timed(SPLITKV_K_MERGE, 1, s, [&] { return launch_merge(c.P, c.pp, wk, Q, Kd, Vd, O, LSE, s); }));
}

int splitkv_bwd(const splitkv_problem* prob, const void* plan_ws, const void* Q, const void* Kc,
                const void* Vc, const void* Kd, const void* Vd, const void* O, const float* LSE,
                const void* dO, void* dQ, void* dKc, void* dVc, void* dKd, void* dVd, void* work,
                size_t work_bytes, splitkv_stream stream) {
  Ctx c;
  int st = setup(prob, plan_ws, &c);
  if (st) return st;
  const bool any_q = prob->total_anchors > 0;
  if (any_q && (!Q || !Kd || !Vd || !O || !LSE || !dO || !dQ || !dKd || !dVd || !work))
    return SPLITKV_EINVAL;
  if (prob->total_ctx > 0 && (!Kc || !Vc || !dKc || !dVc)) return SPLITKV_EINVAL;
  const void* ptrs[] = {Q, Kc, Vc, Kd, Vd, O, LSE, dO, dQ, dKc, dVc, dKd, dVd, work};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return SPLITKV_EINVAL;
  if (work_bytes < work_bytes_for(prob)) return SPLITKV_EWORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  const bool tc = use_tensor_cores(c.P);
  // The tensor-core dK/dV kernel also sums the dQ partials and zeroes the
  // dK/dV rows of keys no block sees (its reduction warp streams the partials
  // from HBM while the tensor pipe works); otherwise each is a launch of its
  // own.
  const bool fused = tc && any_q && prob->total_ctx > 0 && c.caps.NSL > 0;
  if (prob->total_ctx > 0 && !fused) {
    e = timed(SPLITKV_K_ZERO, 1, s,
              [&] { return launch_zero_uncovered(c.P, c.pp, c.caps.NCB, dKc, dVc, s); });
    if (e != cudaSuccess) return SPLITKV_ECUDA;
  }
  if (!any_q) return SPLITKV_OK;
  WorkPtrs wk;
  work_layout(c.caps.NCF * prob->Hkv, c.P.NQ, prob->Hq, prob->d, prob->B,
              c.caps.NSL * prob->Hkv, (char*)work, &wk);
  e = timed(SPLITKV_K_BWD_DRAFT, bwd_draft_launches(c.P, c.caps.NSL), s, [&] {
    return launch_bwd_draft(c.P, c.pp, wk, Q, Kd, Vd, O, LSE, dO, dKd, dVd, c.caps.NSL, s);
  });
  if (e != cudaSuccess) return SPLITKV_ECUDA;
  e = timed(SPLITKV_K_BWD_DQ, 1, s, [&] {
    return tc ? launch_bwd_dq_tc(c.P, c.pp, wk, Q, Kc, Vc, dO, LSE, s)
              : launch_bwd_dq_simt(c.P, c.pp, wk, Q, Kc, Vc, dO, LSE, s);
  });
  if (e != cudaSuccess) return SPLITKV_ECUDA;
  if (prob->total_ctx > 0) {
    e = timed(SPLITKV_K_BWD_DKDV, 1, s, [&] {
      return tc ? launch_bwd_dkdv_tc(c.P, c.pp, wk, Q, Kc, Vc, dO, LSE, dKc, dVc,
                                     fused ? dQ : nullptr, s)
                : launch_bwd_dkdv_simt(c.P, c.pp, wk, Q, Kc, Vc, dO, LSE, dKc, dVc, s);
    });
    if (e != cudaSuccess) return SPLITKV_ECUDA;
  }
  if (fused) return SPLITKV_OK;
  return cuda_status(
      timed(SPLITKV_K_DQ_REDUCE, 1, s,
            [&] { return launch_dq_reduce(c.P, c.pp, wk, dQ, c.caps.NSL, s); }));
}

int splitkv_device_status(const splitkv_problem* prob, const void* plan_ws, int* status,
                          splitkv_stream stream) {
  Ctx c;
  int st = setup(prob, plan_ws, &c);
  if (st) return st;
  if (!status) return SPLITKV_EINVAL;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return SPLITKV_ECUDA;
  PlanHeader h;
  if (cudaMemcpy(&h, c.pp.hdr, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPLITKV_ECUDA;
  *status = h.magic == kPlanMagic ? h.status : SPLITKV_EPLAN;
  return SPLITKV_OK;
}

int splitkv_plan_stats(const splitkv_problem* prob, const void* plan_ws, splitkv_stats* out,
                       splitkv_stream stream) {
  Ctx c;
  int st = setup(prob, plan_ws, &c);
  if (st) return st;
  if (!out) return SPLITKV_EINVAL;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return SPLITKV_ECUDA;
  PlanHeader h;
  if (cudaMemcpy(&h, c.pp.hdr, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPLITKV_ECUDA;
  memset(out, 0, sizeof(*out));
  out->device_status = h.magic == kPlanMagic ? h.status : SPLITKV_EPLAN;
  out->workers = c.P.workers;
  if (h.magic == kPlanMagic) {
    out->debug_violations = h.dbg_count;
    out->debug_site = (int32_t)((uint64_t)h.dbg_first >> 48);
    out->debug_index = (int64_t)((uint64_t)h.dbg_first & 0xffffffffffffull);
  }
  if (out->device_status != SPLITKV_OK) return SPLITKV_OK;
  const int m = c.P.workers;
  std::vector<int64_t> buf(m);
  auto stats = [&](const int64_t* dev, int64_t* mx, double* imb) -> int {
    if (cudaMemcpy(buf.data(), dev, 8 * m, cudaMemcpyDeviceToHost) != cudaSuccess)
      return SPLITKV_ECUDA;
    int64_t s = 0, x = 0;
    for (int64_t v : buf) {
      s += v;
      x = std::max(x, v);
    }
    *mx = x;
    *imb = s > 0 ? (double)x / ((double)s / m) - 1.0 : 0.0;
    return SPLITKV_OK;
  };
  if ((st = stats(c.pp.f_load_lpt, &out->fwd_lpt_max_load, &out->fwd_lpt_imbalance))) return st;
  if ((st = stats(c.pp.f_load_contig, &out->fwd_contig_max_load, &out->fwd_contig_imbalance)))
    return st;
  if ((st = stats(c.pp.b_load_lpt, &out->bwd_lpt_max_load, &out->bwd_lpt_imbalance))) return st;
  if ((st = stats(c.pp.b_load_contig, &out->bwd_contig_max_load, &out->bwd_contig_imbalance)))
    return st;
  const int64_t Hkv = prob->Hkv;
  out->fwd_items = (int64_t)h.n_fwd_items * Hkv;
  out->bwd_items = (int64_t)h.n_bwd_items * Hkv;
  out->fwd_slots = (int64_t)h.n_slot_base * Hkv;
  out->fwd_total_cost = h.fwd_total_cost * Hkv;
  out->bwd_total_cost = h.bwd_total_cost * Hkv;
  out->fwd_tiles = h.fwd_tiles * Hkv;
  out->dense_tiles = h.dense_tiles * Hkv;
  out->work_bytes_used =
      work_layout(out->fwd_slots, c.P.NQ, prob->Hq, prob->d, prob->B,
                  (int64_t)h.n_slabs * prob->Hkv, nullptr, nullptr);
  return SPLITKV_OK;
}

int splitkv_plan_export(const splitkv_problem* prob, const void* plan_ws, int kind, int64_t* ids,
                        int64_t* costs, int32_t* worker, int32_t* pos, int64_t capacity,
                        int64_t* count, splitkv_stream stream) {
  Ctx c;
  int st = setup(prob, plan_ws, &c);
  if (st) return st;
  if (kind < 0 || kind > 3 || !count || capacity < 0) return SPLITKV_EINVAL;
  if (capacity > 0 && (!ids || !costs || !worker || !pos)) return SPLITKV_EINVAL;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return SPLITKV_ECUDA;
  PlanHeader h;
  if (cudaMemcpy(&h, c.pp.hdr, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPLITKV_ECUDA;
  if (h.magic != kPlanMagic || h.status != SPLITKV_OK) return SPLITKV_EINVAL;
  if (kind >= 2) return export_queues(c, h, kind == 2, ids, costs, worker, pos, capacity, count);
  const int n = kind == 0 ? h.n_fwd_items : h.n_bwd_items;
  const int Hkv = prob->Hkv;
  *count = (int64_t)n * Hkv;
  if (n == 0) return SPLITKV_OK;
  std::vector<int32_t> sorted(n), item(n), grp(n), ps(n);
  std::vector<int64_t> sc(n);
  const bool f = kind == 0;
  cudaError_t e = cudaSuccess;
  e = e ? e : cudaMemcpy(sorted.data(), f ? c.pp.f_sorted : c.pp.b_sorted, 4 * n, cudaMemcpyDeviceToHost);
  e = e ? e : cudaMemcpy(item.data(), f ? c.pp.f_item : c.pp.b_item, 4 * n, cudaMemcpyDeviceToHost);
  e = e ? e : cudaMemcpy(grp.data(), f ? c.pp.f_grp : c.pp.b_grp, 4 * n, cudaMemcpyDeviceToHost);
  e = e ? e : cudaMemcpy(ps.data(), f ? c.pp.f_pos : c.pp.b_pos, 4 * n, cudaMemcpyDeviceToHost);
  e = e ? e : cudaMemcpy(sc.data(), f ? c.pp.f_scost : c.pp.b_scost, 8 * n, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return SPLITKV_ECUDA;
  int64_t k = 0;
  for (int r = 0; r < n; ++r) {
    const int64_t cand = item[sorted[r]];
    for (int g = 0; g < Hkv; ++g, ++k) {
      if (k >= capacity) return SPLITKV_OK;
      ids[k] = cand * Hkv + g;
      costs[k] = sc[r];
      worker[k] = grp[r] * Hkv + g;
      pos[k] = ps[r];
    }
  }
  return SPLITKV_OK;
}

int splitkv_proj_in_fwd(const splitkv_problem* prob, int hidden, const void* Xd, const void* Xc,
                        const void* Wqkv, void* Q, void* Kc, void* Vc, void* Kd, void* Vd,
                        splitkv_stream stream) {
  int st = check_proj(prob, hidden);
  if (st) return st;
  const int64_t NQ = prob->total_anchors * prob->B, T = prob->total_ctx, H = hidden;
  const int qd = prob->Hq * prob->d, kd = prob->Hkv * prob->d;
  const bool draft = NQ > 0, ctx = T > 0 && Xc;
  if (!Wqkv || (draft && (!Xd || !Q || !Kd || !Vd)) || (ctx && (!Kc || !Vc)))
    return SPLITKV_EINVAL;
  if (!all_aligned({Xd, Xc, Wqkv, Q, Kc, Vc, Kd, Vd})) return SPLITKV_EINVAL;
  const ProjOperand W{Wqkv, qd + 2 * kd, H};
  ProjSpec parts[2];
  int n = 0;
  if (draft) {  // [Q | Kd | Vd] = Xd Wqkv^T
    ProjSpec& p = parts[n++];
    p = proj_one(NQ, qd + 2 * kd, 0, 0, {Xd, NQ, H}, W, 0, H, 0);
    add_dst(&p, Q, 0, qd, qd);
    add_dst(&p, Kd, qd, kd, kd);
    add_dst(&p, Vd, qd + kd, kd, kd);
  }
  if (ctx) {  // [Kc | Vc] = Xc Wkv^T: rows [qd, qd + 2 kd) of Wqkv
    ProjSpec& p = parts[n++];
    p = proj_one(T, 2 * kd, 0, 0, {Xc, T, H}, W, qd, H, 0);
    add_dst(&p, Kc, 0, kd, kd);
    add_dst(&p, Vc, kd, kd, kd);
  }
  return run_proj(parts, n, (cudaStream_t)stream);
}

int splitkv_proj_in_bwd(const splitkv_problem* prob, int hidden, const void* Xd, const void* Xc,
                        const void* Wqkv, const void* dQ, const void* dKc, const void* dVc,
                        const void* dKd, const void* dVd, void* dXd, void* dXc, float* dWqkv,
                        splitkv_stream stream) {
  int st = check_proj(prob, hidden);
  if (st) return st;
  const int64_t NQ = prob->total_anchors * prob->B, T = prob->total_ctx, H = hidden;
  const int qd = prob->Hq * prob->d, kd = prob->Hkv * prob->d;
  const bool draft = NQ > 0, ctx = T > 0 && Xc;
  if (!Wqkv || !dWqkv || (draft && (!Xd || !dQ || !dKd || !dVd || !dXd)) ||
      (ctx && (!dKc || !dVc || !dXc)))
    return SPLITKV_EINVAL;
  if (!all_aligned({Xd, Xc, Wqkv, dQ, dKc, dVc, dKd, dVd, dXd, dXc, dWqkv})) return SPLITKV_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  const ProjOperand W{Wqkv, qd + 2 * kd, H};  // read MN-major: [out rows = K][hidden = N]
  // activation gradients (bf16)
  ProjSpec parts[3];
  int n = 0;
  if (draft) {  // dXd = dQ Wq + dKd Wk + dVd Wv
    ProjSpec& p = parts[n++];
    p = proj_one(NQ, H, 0, 1, {dQ, NQ, qd}, W, 0, qd, 0);
    add_seg(&p, {dKd, NQ, kd}, W, qd, kd);
    add_seg(&p, {dVd, NQ, kd}, W, qd + kd, kd);
    add_dst(&p, dXd, 0, (int)H, H);
  }
  if (ctx) {  // dXc = dKc Wk + dVc Wv
    ProjSpec& p = parts[n++];
    p = proj_one(T, H, 0, 1, {dKc, T, kd}, W, 0, kd, 0);
    p.k0_b[0] = qd;
    add_seg(&p, {dVc, T, kd}, W, qd + kd, kd);
    add_dst(&p, dXc, 0, (int)H, H);
  }
  if ((st = run_proj(parts, n, s))) return st;
  // weight gradients (fp32): rows of dWqkv = (dY_part)^T X, summed over the
  // draft rows and then the context rows
  const int64_t kb_ctx = ctx ? (T + 63) / 64 : 0, kb_d = (NQ + 63) / 64;
  const int ksplit = (int)std::min<int64_t>(64, std::max<int64_t>(1, (kb_d + kb_ctx) / 128));
  if (ksplit > 1 || !draft) {  // atomics add into it, or dWq has no terms
    if (cudaMemsetAsync(dWqkv, 0, sizeof(float) * (size_t)(qd + 2 * kd) * H, s) != cudaSuccess)
      return SPLITKV_ECUDA;
  }
  n = 0;
  if (draft) {  // dWq = dQ^T Xd
    ProjSpec& p = parts[n++];
    p = proj_one(qd, H, 1, 1, {dQ, NQ, qd}, {Xd, NQ, H}, 0, NQ, 1);
    add_dst(&p, dWqkv, 0, (int)H, H);
  }
  for (int kv = 0; kv < 2 && (draft || ctx); ++kv) {  // dWk, dWv
    ProjSpec& p = parts[n++];
    memset(&p, 0, sizeof(p));
    p.M = kd;
    p.N = H;
    p.a_mn = p.b_mn = 1;
    p.out_f32 = 1;
    p.ksplit = ksplit;
    if (draft) add_seg(&p, {kv ? dVd : dKd, NQ, kd}, {Xd, NQ, H}, 0, NQ);
    if (ctx) add_seg(&p, {kv ? dVc : dKc, T, kd}, {Xc, T, H}, 0, T);
    add_dst(&p, dWqkv + (size_t)(qd + kv * kd) * H, 0, (int)H, H);
  }
  return run_proj(parts, n, s);
}

int splitkv_proj_out_fwd(const splitkv_problem* prob, int hidden, const void* O, const void* Wo,
                         void* Y, splitkv_stream stream) {
  int st = check_proj(prob, hidden);
  if (st) return st;
  const int64_t NQ = prob->total_anchors * prob->B, H = hidden;
  const int qd = prob->Hq * prob->d;
  if (NQ > 0 && (!O || !Wo || !Y)) return SPLITKV_EINVAL;
  if (!all_aligned({O, Wo, Y})) return SPLITKV_EINVAL;
  if (NQ == 0) return SPLITKV_OK;
  ProjSpec p = proj_one(NQ, H, 0, 0, {O, NQ, qd}, {Wo, H, qd}, 0, qd, 0);
  add_dst(&p, Y, 0, (int)H, H);
  return run_proj(&p, 1, (cudaStream_t)stream);
}

int splitkv_proj_out_bwd(const splitkv_problem* prob, int hidden, const void* O, const void* Wo,
                         const void* dY, void* dO, float* dWo, splitkv_stream stream) {
  int st = check_proj(prob, hidden);
  if (st) return st;
  const int64_t NQ = prob->total_anchors * prob->B, H = hidden;
  const int qd = prob->Hq * prob->d;
  if (!dWo || (NQ > 0 && (!O || !Wo || !dY || !dO))) return SPLITKV_EINVAL;
  if (!all_aligned({O, Wo, dY, dO, dWo})) return SPLITKV_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  if (NQ == 0)
    return cuda_status(cudaMemsetAsync(dWo, 0, sizeof(float) * (size_t)H * qd, s));
  ProjSpec parts[2];
  // dO = dY Wo: Wo read MN-major ([hidden rows = K][Hq d = N])
  parts[0] = proj_one(NQ, qd, 0, 1, {dY, NQ, H}, {Wo, H, qd}, 0, H, 0);
  add_dst(&parts[0], dO, 0, qd, qd);
  // dWo = dY^T O: both MN-major ([N_q rows = K])
  parts[1] = proj_one(H, qd, 1, 1, {dY, NQ, H}, {O, NQ, qd}, 0, NQ, 1);
  add_dst(&parts[1], dWo, 0, qd, qd);
  return run_proj(parts, 2, s);
}

int splitkv_proj_status(int* status, int clear, splitkv_stream stream) {
  if (!status) return SPLITKV_EINVAL;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return SPLITKV_ECUDA;
  return cuda_status(proj_status(status, clear != 0));
}

int splitkv_selftest_wait_timeout(int* status, splitkv_stream stream) {
  if (!status) return SPLITKV_EINVAL;
  return cuda_status(run_wait_probe(status, (cudaStream_t)stream));
}

int splitkv_build_flags(void) {
#ifdef SKV_DEBUG
  return SPLITKV_BUILD_DEBUG;
#else
  return 0;
#endif
}

const char* splitkv_status_string(int status) {
  switch (status) {
    case SPLITKV_OK: return "ok";
    case SPLITKV_EINVAL: return "invalid argument";
    case SPLITKV_EUNSUPPORTED: return "unsupported shape or dtype";
    case SPLITKV_EWORKSPACE: return "workspace too small";
    case SPLITKV_ECUDA: return "CUDA runtime error";
    case SPLITKV_EDEVICE: return "no usable device";
    case SPLITKV_ETIMEOUT: return "device pipeline wait timed out";
    case SPLITKV_EPLAN: return "plan does not match the problem";
    case SPLITKV_EMETA: return "inconsistent cu_ctx / cu_anchor / anchors";
    case SPLITKV_ECAPACITY: return "metadata exceeds the declared sizes";
    default: return "unknown status";
  }
}

}  // extern "C"
