/*
 * splitkv.h — C ABI of the GB300 split-KV block-sparse cross-attention library.
 *
 * What it computes. Exact anchor-masked cross-attention of short draft-query
 * blocks over a long context, forward and backward (Split-KV: Efficient
 * Context Parallelism for Training Diffusion Drafters, arXiv:2611.05926,
 * abstract: anchor sampling builds compact draft queries that cross-attend to
 * a much longer context under a block-sparse mask). For draft block j of
 * sample s with anchor a_j, the B query rows of the block attend to
 *   - the context keys [0, a_j) of sample s (strict prefix), and
 *   - the B keys of the block's own draft tokens (bidirectional),
 * with softmax scale `scale`; query head h reads kv head h / (Hq / Hkv).
 *
 * How. The paper's context-parallel recipe (rit.work article on Split-KV,
 * section "Split-KV двигает запросы, а не ключи и значения": K/V shards stay
 * where they are, every participant sees all queries, computes its local
 * part of attention, the normalisation is reconciled, the result returns to
 * the query owners; the split reproduces the single-device result exactly)
 * is mapped onto the SMs of one GPU: KV chunks are the shards, persistent
 * CTAs are the participants, per-chunk (lse, O) partials are merged exactly
 * by log-sum-exp, and dQ partials are reduced in a fixed order. A planner
 * prices every work item by its realized masked work and assigns items with
 * longest-processing-time-first (abstract; rit.work article, paragraph on
 * anchor sampling and load imbalance).
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers, row-major, contiguous:
 *      Q, O, dO, dQ        [N_q, Hq, d]      dtype     N_q = B * total_anchors
 *      Kc, Vc, dKc, dVc    [T, Hkv, d]       dtype     T = total_ctx
 *      Kd, Vd, dKd, dVd    [N_q, Hkv, d]     dtype     (draft-token keys/values)
 *      LSE                 [Hq, N_q]         float32   natural log of the row's
 *                                                      softmax normaliser
 *    Draft block j (global order over samples) owns query rows [jB, jB+B).
 *    Every pointer must be 16-byte aligned.
 *  - The caller owns every buffer, including both workspaces; the library
 *    never allocates, frees or synchronises device memory, except where a
 *    function says it reads back to the host.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream). The buffers must stay valid until the stream passes
 *    the enqueued work.
 *  - Every function returns a status code (SPLITKV_OK on success) and never
 *    throws or aborts. Host-detectable errors (null pointers, unsupported
 *    shapes, workspace too small) are returned immediately. Errors found on
 *    the device (invalid anchors, a plan that belongs to another problem, a
 *    pipeline wait that timed out) are latched in a status word inside the
 *    plan workspace; kernels that see it set skip their work, and
 *    splitkv_plan_stats() / splitkv_device_status() read it back.
 */
#ifndef SPLITKV_H
#define SPLITKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* splitkv_stream; /* == cudaStream_t */

/* Status codes. */
enum {
  SPLITKV_OK = 0,
  SPLITKV_EINVAL = 1,       /* bad argument: null pointer, negative size, bad metadata */
  SPLITKV_EUNSUPPORTED = 2, /* shape/dtype outside the supported set */
  SPLITKV_EWORKSPACE = 3,   /* a workspace is smaller than splitkv_workspace_size() says */
  SPLITKV_ECUDA = 4,        /* a CUDA runtime call failed */
  SPLITKV_EDEVICE = 5,      /* no usable sm_100-family device */
  SPLITKV_ETIMEOUT = 6,     /* device status: a bounded pipeline wait gave up */
  SPLITKV_EPLAN = 7,        /* device status: plan built for a different problem */
  SPLITKV_EMETA = 8,        /* device status: cu_ctx/cu_anchor/anchors inconsistent */
  SPLITKV_ECAPACITY = 9     /* device status: metadata exceeds the host-declared sizes */
};

/* Compute dtypes (inputs and outputs; accumulation is always fp32). */
enum { SPLITKV_BF16 = 0, SPLITKV_FP32 = 1 };

/* Problem flags. */
enum {
  /* Use the CUDA-core (FMA) attention kernels instead of the tensor-core
   * ones. bf16 problems default to tcgen05 tensor cores; fp32 problems always
   * use the CUDA-core kernels (exact fp32 products). */
  SPLITKV_FLAG_CUDA_CORE = 1,
  /* Execute the naive contiguous assignment (worker w takes items
   * [floor(w n/m), floor((w+1) n/m)) in id order) instead of LPT. */
  SPLITKV_FLAG_CONTIGUOUS = 2,
  /* Mask variants for drafters that share the pattern (the pages name DFlash,
   * Domino and DSpark, rit.work article, section on when the method changes
   * the infrastructure plan, without giving their masks):
   * MASK_INCLUSIVE: block j sees context keys [0, a_j] instead of [0, a_j)
   *   (chunk costs, tile skipping and masks all use a_j + 1);
   * MASK_CAUSAL_BLOCK: query i of a block sees its draft keys t <= i only,
   *   instead of all B;
   * MASK_CONTEXT_OFFSET: block j's context starts at its own offset
   *   o_j = ctx_lo[j] (sample-local): it sees context keys [o_j, a_j)
   *   ([o_j, a_j] with MASK_INCLUSIVE) instead of [0, a_j). Chunk costs, tile
   *   skipping, masks, the merge and the zeroing of unseen keys all use the
   *   range. The flags may be combined. */
  SPLITKV_FLAG_MASK_INCLUSIVE = 4,
  SPLITKV_FLAG_MASK_CAUSAL_BLOCK = 8,
  SPLITKV_FLAG_MASK_CONTEXT_OFFSET = 16
};

/*
 * Problem description. Device pointers: cu_ctx, cu_anchor, anchors. Every
 * other field is a host value.
 *
 *  num_samples   S >= 1 packed samples.
 *  cu_ctx        int32 [S+1] device; cu_ctx[0] = 0, non-decreasing, cu_ctx[S] = total_ctx.
 *                Sample s owns context rows [cu_ctx[s], cu_ctx[s+1]) of Kc/Vc.
 *  cu_anchor     int32 [S+1] device; cu_anchor[0] = 0, non-decreasing,
 *                cu_anchor[S] = total_anchors. Sample s owns draft blocks
 *                [cu_anchor[s], cu_anchor[s+1]).
 *  anchors       int32 [total_anchors] device; sample-local anchor positions,
 *                non-decreasing within a sample, 0 <= a <= L_s - B.
 *  total_ctx     T = cu_ctx[S] (host copy, sizes Kc/Vc).
 *  total_anchors cu_anchor[S] (host copy); N_q = B * total_anchors.
 *  max_ctx       an upper bound on max_s L_s (sizes the plan).
 *  B             draft block size (queries per anchor).
 *  Hq, Hkv       query / kv heads; Hq % Hkv == 0; group = Hq / Hkv.
 *  d             head dim: 64 or 128.
 *  chunk         KV chunk length C (keys) of the split; a multiple of 128.
 *  scale         softmax scale (usually 1/sqrt(d)).
 *  dtype         SPLITKV_BF16 or SPLITKV_FP32.
 *  num_workers   persistent CTAs the plan balances over; 0 = the device's SM
 *                count rounded down to a multiple of Hkv. Must be a multiple
 *                of Hkv and at most 256 * Hkv (and at most 4096).
 *  flags         SPLITKV_FLAG_* bits.
 *  ctx_lo        int32 [total_anchors] device, read only with
 *                SPLITKV_FLAG_MASK_CONTEXT_OFFSET (may be NULL otherwise):
 *                start of each block's visible context, sample-local,
 *                0 <= ctx_lo[j] <= the end of its context (a_j, or a_j + 1
 *                when inclusive; equal to it = no context key). Validated on
 *                the device (SPLITKV_EMETA).
 *
 * Supported set: 128 % (B * group) == 0 (a work item is 128 (query, head)
 * rows = 128 / (B*group) whole draft blocks), d in {64, 128}, dtype bf16 or
 * fp32. Anything else returns SPLITKV_EUNSUPPORTED.
 */
typedef struct splitkv_problem {
  int32_t num_samples;
  const int32_t* cu_ctx;
  const int32_t* cu_anchor;
  const int32_t* anchors;
  int64_t total_ctx;
  int64_t total_anchors;
  int32_t max_ctx;
  int32_t B;
  int32_t Hq;
  int32_t Hkv;
  int32_t d;
  int32_t chunk;
  float scale;
  int32_t dtype;
  int32_t num_workers;
  int32_t flags;
  const int32_t* ctx_lo;
} splitkv_problem;

/* Plan statistics (host struct filled by splitkv_plan_stats). Costs are in
 * masked (query, key) pairs; loads are per persistent CTA. */
typedef struct splitkv_stats {
  int32_t device_status;      /* SPLITKV_OK or the latched device error */
  int32_t workers;            /* persistent CTAs the plan uses */
  int64_t fwd_items;          /* forward items (sample, chunk, slab, kv head), cost > 0 */
  int64_t bwd_items;          /* backward items (sample, 128-key tile, kv head), cost > 0 */
  int64_t fwd_slots;          /* forward/dQ partial slots in use */
  int64_t fwd_total_cost;
  int64_t bwd_total_cost;
  int64_t fwd_lpt_max_load;
  int64_t fwd_contig_max_load;
  int64_t bwd_lpt_max_load;
  int64_t bwd_contig_max_load;
  double fwd_lpt_imbalance;   /* max/mean - 1 over workers */
  double fwd_contig_imbalance;
  double bwd_lpt_imbalance;
  double bwd_contig_imbalance;
  int64_t fwd_tiles;          /* 128x128 (row, key) tiles the forward computes */
  int64_t dense_tiles;        /* tiles of the dense (N_q*group/128) x (L/128) x Hkv grid */
  size_t work_bytes_used;     /* exact bytes of the work workspace this plan needs */
  /* index checks of the debug build (splitkv_build_flags() & SPLITKV_BUILD_DEBUG):
   * failed checks since the plan was built (every kernel that read this plan
   * counts; a failed check skips its access), and the first one's site
   * (1 .. 10, listed in the source) and index; all zero in the release build */
  int64_t debug_violations;
  int32_t debug_site;
  int32_t pad0;
  int64_t debug_index;
} splitkv_stats;

/*
 * splitkv_workspace_size — bytes of the two caller-owned workspaces.
 *   plan_bytes: holds the plan (costs, LPT queues, slab tables, status word);
 *               built by splitkv_plan, read by splitkv_fwd / splitkv_bwd.
 *   work_bytes: fp32 partials of the split (per chunk (lse, O) in the forward,
 *               per chunk dQ and the draft-block terms in the backward) and
 *               the backward's row tables and task counter. This
 *               is an upper bound computed from host scalars; the exact need
 *               of a built plan is splitkv_stats.work_bytes_used.
 * Host-only; no device work. Errors: EINVAL (null), EUNSUPPORTED.
 */
int splitkv_workspace_size(const splitkv_problem* prob, size_t* plan_bytes, size_t* work_bytes);

/*
 * splitkv_plan — build the work plan on the device (no host synchronisation).
 *   Validates the device metadata (latched as SPLITKV_EMETA / ECAPACITY),
 *   prices every forward item (sample s, chunk c, slab of draft blocks, kv
 *   head) and backward item (sample, 128-key tile, kv head) by
 *       cost = sum over anchors a_j > start of min(len, a_j - start) * B
 *   (the chunk's realized masked work, Split-KV abstract), drops cost-0
 *   items, sorts by (cost desc, item id asc) and assigns greedily to the
 *   least-loaded worker (ties: lowest worker id) — LPT as the rit.work
 *   article describes it. The plan depends only on the metadata; one plan
 *   serves every layer that shares the mask.
 *   plan_ws: device buffer of at least plan_bytes (splitkv_workspace_size).
 * Errors: EINVAL, EUNSUPPORTED, EWORKSPACE, EDEVICE, ECUDA.
 */
int splitkv_plan(const splitkv_problem* prob, void* plan_ws, size_t plan_bytes,
                 splitkv_stream stream);

/*
 * splitkv_fwd — forward pass. Writes O (dtype) and LSE (fp32, natural log).
 *   Persistent CTAs walk their LPT queues; each item computes the online-
 *   softmax partial (lse, O) of 128 query rows over one KV chunk ("local
 *   part", rit.work article, Split-KV section); a merge kernel then adds the
 *   draft-block partial and combines all partials of a row exactly by
 *   log-sum-exp in ascending chunk order ("reconcile the normalisation").
 *   work: device buffer of at least work_bytes. prob must be the problem the
 *   plan was built for (checked on the device -> SPLITKV_EPLAN).
 * Errors: EINVAL, EUNSUPPORTED, EWORKSPACE, ECUDA.
 */
int splitkv_fwd(const splitkv_problem* prob, const void* plan_ws,
                const void* Q, const void* Kc, const void* Vc, const void* Kd, const void* Vd,
                void* O, float* LSE, void* work, size_t work_bytes, splitkv_stream stream);

/*
 * splitkv_bwd — backward pass of loss = sum(dO * O).
 *   Inputs are the forward's inputs plus its outputs O and LSE and the
 *   upstream gradient dO. Writes dQ, dKc, dVc, dKd, dVd (dtype; every row is
 *   written, context rows no block sees get zero). dK/dV of a context key
 *   are produced by the one CTA that owns its 128-key tile (kept local, as
 *   the rit.work article's Split-KV section keeps K/V gradients with their
 *   shard); dQ is produced per (chunk, item) as an fp32 partial and reduced
 *   in ascending chunk order (deterministic, no atomics).
 * Errors: EINVAL, EUNSUPPORTED, EWORKSPACE, ECUDA.
 */
int splitkv_bwd(const splitkv_problem* prob, const void* plan_ws,
                const void* Q, const void* Kc, const void* Vc, const void* Kd, const void* Vd,
                const void* O, const float* LSE, const void* dO,
                void* dQ, void* dKc, void* dVc, void* dKd, void* dVd,
                void* work, size_t work_bytes, splitkv_stream stream);

/*
 * splitkv_plan_stats — SYNCHRONISES `stream`, then reads the plan back and
 *   fills *out: item counts, LPT and contiguous per-worker imbalance, skip
 *   accounting and the latched device status.
 * Errors: EINVAL, ECUDA.
 */
int splitkv_plan_stats(const splitkv_problem* prob, const void* plan_ws, splitkv_stats* out,
                       splitkv_stream stream);

/*
 * splitkv_plan_export — SYNCHRONISES `stream` and copies the plan to host
 *   arrays, for verification against an independent implementation.
 *   kind 0 = forward items, 1 = backward items: the LPT result. For every
 *     item of positive cost, in LPT order (cost desc, id asc).
 *   kind 2 = forward queues, 3 = backward queues: the queues the attention
 *     kernels actually walk (the LPT queues, or the contiguous ranges of a
 *     plan built with SPLITKV_FLAG_CONTIGUOUS), worker 0's queue first, each
 *     queue in the order its CTA runs it.
 *   Each entry i receives
 *     ids[i]    per-kv-head item id (forward: ((sample, chunk, slab) index) *
 *               Hkv + kv head; backward: ((sample, key tile) index) * Hkv + kv head)
 *     costs[i]  its cost
 *     worker[i] the persistent CTA it is assigned to
 *     pos[i]    its position in that CTA's queue
 *   capacity: length of each host array; *count receives the entry count
 *   (nothing is written past capacity).
 * Errors: EINVAL (also for a plan whose device status is not SPLITKV_OK),
 * ECUDA.
 */
int splitkv_plan_export(const splitkv_problem* prob, const void* plan_ws, int kind,
                        int64_t* ids, int64_t* costs, int32_t* worker, int32_t* pos,
                        int64_t capacity, int64_t* count, splitkv_stream stream);

/* splitkv_device_status — SYNCHRONISES `stream`; *status = latched device status. */
int splitkv_device_status(const splitkv_problem* prob, const void* plan_ws, int* status,
                          splitkv_stream stream);

/* splitkv_resolve_workers — the persistent-CTA count a plan for `prob` uses
 * on the current device (host-only apart from a device attribute query). */
int splitkv_resolve_workers(const splitkv_problem* prob, int* workers);

/*
 * splitkv_fwd_noalloc — the forward pass (plan + splitkv_fwd) for callers
 *   that cannot allocate device memory where they call it: code running in
 *   another framework's per-call hook where that framework owns all device
 *   memory and forbids allocation, or services that freeze device allocation
 *   after start-up. The paper has no counterpart; this entry point exists
 *   only for such callers.
 *   Same problem description and the same device tensors as splitkv_fwd
 *   (inputs Q, Kc, Vc, Kd, Vd; outputs O, LSE); no workspaces. The plan and
 *   the forward partials live in one file-scope device array of
 *   SPLITKV_NOALLOC_SCRATCH_BYTES per device, reserved when the library's
 *   device code is loaded and held until the process exits. The library
 *   calls no cudaMalloc / cudaFree and no allocating routine here.
 *   The first call on a device looks up that array's device address
 *   (cudaGetSymbolAddress) with the device current; make that first call
 *   before any stream capture.
 *   Limit: problems whose splitkv_workspace_size() plan_bytes (rounded up to
 *   256) + work_bytes exceed SPLITKV_NOALLOC_SCRATCH_BYTES return
 *   SPLITKV_EWORKSPACE; use splitkv_plan + splitkv_fwd with your own
 *   workspaces for them.
 *   Every call on a device shares the array and leaves its contents behind;
 *   calls whose work overlaps on the GPU (e.g. on two streams) race on it.
 *   Order them on one stream. Errors: as splitkv_plan and splitkv_fwd.
 */
#define SPLITKV_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int splitkv_fwd_noalloc(const splitkv_problem* prob, const void* Q, const void* Kc,
                        const void* Vc, const void* Kd, const void* Vd, void* O, float* LSE,
                        splitkv_stream stream);

/*
 * Launch timing (the library's tracing hook; not thread-safe).
 * splitkv_profile_enable(1) clears earlier records and from then on brackets
 * every kernel launch the library makes with a pair of CUDA events recorded
 * on the launch stream (no synchronisation is added). splitkv_profile_enable(0)
 * stops recording. splitkv_profile_read() waits for the recorded events and
 * returns, per kernel family id (SPLITKV_K_*), the number of kernel launches
 * and their summed device time in milliseconds; arrays have length n (at
 * most SPLITKV_NUM_KERNELS entries are written). Errors: EINVAL, ECUDA.
 */
enum {
  SPLITKV_K_PLAN = 0,        /* planner: setup, rank, assign, queues (4 launches) */
  SPLITKV_K_FWD_ATTN = 1,    /* forward partial attention (persistent) */
  SPLITKV_K_MERGE = 2,       /* draft partial + log-sum-exp merge */
  SPLITKV_K_BWD_DRAFT = 3,   /* D = rowsum(dO*O) + draft-block backward */
  SPLITKV_K_BWD_DQ = 4,      /* dQ chunk partials (persistent) */
  SPLITKV_K_BWD_DKDV = 5,    /* dK/dV of 128-key tiles (persistent); on the
                                tensor-core path it also sums dQ and zeroes
                                the rows of keys no block sees */
  SPLITKV_K_DQ_REDUCE = 6,   /* dQ = scale * sum of partials: a launch of its
                                own on the CUDA-core path or without context
                                keys only */
  SPLITKV_K_ZERO = 7,        /* zero dK/dV rows no block sees: a launch of
                                its own on the CUDA-core path or without
                                anchors only */
  SPLITKV_K_PROJ = 8,        /* projection GEMMs (splitkv_proj_*) */
  SPLITKV_NUM_KERNELS = 9
};
int splitkv_profile_enable(int on);
int splitkv_profile_read(int32_t* launches, double* total_ms, int n);

/*
 * splitkv_busy_read — SYNCHRONISES `stream`. Measured load balance of the
 * persistent attention kernels (the realised counterpart of the planned LPT
 * loads; the paper claims balanced per-participant work, abstract and rit.work
 * article, paragraph on anchor sampling and load imbalance). Every launch of
 * the forward, dQ and dK/dV attention kernels with this plan stamps, per
 * worker CTA, the %globaltimer value (ns) at its start and at its end into
 * the plan workspace; this copies the stamps of the latest launch of
 * `kernel_id` (SPLITKV_K_FWD_ATTN, SPLITKV_K_BWD_DQ or SPLITKV_K_BWD_DKDV)
 * to the host array ns[2*w] = start, ns[2*w+1] = end of worker w.
 *   capacity: length of ns; *workers receives the worker count (nothing is
 *   written to ns unless capacity >= 2 * workers).
 * Stamps of a kernel that has not run with this plan are undefined.
 * Errors: EINVAL (other kernel ids, capacity too small), ECUDA, and the
 * errors of an invalid problem / plan workspace.
 */
int splitkv_busy_read(const splitkv_problem* prob, const void* plan_ws, int kernel_id,
                      uint64_t* ns, int capacity, int* workers, splitkv_stream stream);
/*
 * Projections of the drafter layer around the attention (the fused
 * projection epilogue). The pages name the layer the attention sits in — a
 * diffusion drafter whose draft blocks cross-attend to the target model's
 * context (Split-KV abstract; rit.work article, section on when the method
 * changes the infrastructure plan) — but give no projections. Reading taken:
 * the bias-free linear maps of an attention layer, weights in a linear
 * layer's [out, in] row-major layout, the context keys/values projected by
 * the same Wk, Wv as the draft tokens:
 *     [Q | Kd | Vd] = Xd Wqkv^T      Xd   [N_q, hidden]  draft-token hidden states
 *     [Kc | Vc]     = Xc Wkv^T       Xc   [T, hidden]    context hidden states
 *     Y             = O Wo^T         Wqkv [(Hq + 2 Hkv) d, hidden] = [Wq; Wk; Wv]
 *                                    Wkv  = rows [Hq d, (Hq + 2 Hkv) d) of Wqkv
 *                                    Wo   [hidden, Hq d];   Y, dY [N_q, hidden]
 * Q, Kd, Vd, Kc, Vc, O have the layouts of splitkv_fwd ([rows, heads, d] is
 * [rows, heads * d]). Every product is a tcgen05 GEMM (bf16 in, fp32
 * accumulate) whose epilogue writes those layouts directly: one launch over
 * Wqkv produces Q, Kd and Vd (and Kc, Vc), and the backward sums the three
 * terms dQ Wq + dKd Wk + dVd Wv of dXd in one accumulator.
 * Requirements: the problem passes splitkv_plan's checks (no plan is needed),
 * prob->dtype == SPLITKV_BF16, hidden a positive multiple of 64, all
 * pointers 16-byte aligned. Activations and their gradients are bf16; the
 * weight gradients dWqkv, dWo are fp32 and are overwritten (not accumulated
 * into). dWk, dWv sum over N_q + T rows; when T is large that sum is split
 * into slices added with fp32 atomics, so the last bits of dWqkv's k/v rows
 * can differ between runs; every other output is deterministic.
 * Errors: EINVAL (null or misaligned pointer, hidden <= 0), EUNSUPPORTED
 * (dtype, hidden % 64, the problem's shape), ECUDA. A device pipeline wait
 * that times out stops the kernel and is reported by splitkv_proj_status.
 */
/* Forward of the input projections. Xc may be NULL: the context projection
 * is skipped and Kc, Vc (then allowed NULL) are left untouched. */
int splitkv_proj_in_fwd(const splitkv_problem* prob, int hidden, const void* Xd, const void* Xc,
                        const void* Wqkv, void* Q, void* Kc, void* Vc, void* Kd, void* Vd,
                        splitkv_stream stream);
/* Backward of the input projections: dXd = dQ Wq + dKd Wk + dVd Wv,
 * dXc = dKc Wk + dVc Wv, dWqkv = [dQ^T Xd; dKd^T Xd + dKc^T Xc; dVd^T Xd + dVc^T Xc]
 * (fp32). With Xc NULL the context terms are left out (dXc, dKc, dVc may be
 * NULL). */
int splitkv_proj_in_bwd(const splitkv_problem* prob, int hidden, const void* Xd, const void* Xc,
                        const void* Wqkv, const void* dQ, const void* dKc, const void* dVc,
                        const void* dKd, const void* dVd, void* dXd, void* dXc, float* dWqkv,
                        splitkv_stream stream);
/* Forward of the output projection: Y = O Wo^T. */
int splitkv_proj_out_fwd(const splitkv_problem* prob, int hidden, const void* O, const void* Wo,
                         void* Y, splitkv_stream stream);
/* Backward of the output projection: dO = dY Wo (bf16, the input of
 * splitkv_bwd), dWo = dY^T O (fp32). One launch. */
int splitkv_proj_out_bwd(const splitkv_problem* prob, int hidden, const void* O, const void* Wo,
                         const void* dY, void* dO, float* dWo, splitkv_stream stream);
/* SYNCHRONISES `stream`; *status = the first device error of any projection
 * launch in this process (SPLITKV_OK or SPLITKV_ETIMEOUT); clear != 0 resets
 * it. Errors: EINVAL, ECUDA. */
int splitkv_proj_status(int* status, int clear, splitkv_stream stream);

/*
 * splitkv_selftest_wait_timeout — diagnostic of the device-side failure path.
 *   SYNCHRONISES `stream`. Runs one small kernel whose mbarrier wait nothing
 *   can satisfy, with the same bounded-wait routine every pipeline uses: the
 *   wait gives up after its limit (about 1 s), raises the CTA's abort flag
 *   (a second waiting warp stops on it) and the kernel reports the outcome;
 *   *status = SPLITKV_ETIMEOUT when that happened, SPLITKV_OK if the wait
 *   returned without timing out. The context stays usable.
 * Errors: EINVAL (null status), ECUDA.
 */
int splitkv_selftest_wait_timeout(int* status, splitkv_stream stream);

/*
 * splitkv_build_flags — how this library was compiled: SPLITKV_BUILD_DEBUG
 *   when its kernels check their indices (a debug build, in place of a memory
 *   checker: out-of-range accesses are counted in the plan header, reported
 *   by splitkv_plan_stats, and skipped). Host-only.
 */
#define SPLITKV_BUILD_DEBUG 1
int splitkv_build_flags(void);

/* Name of a kernel family id (never NULL). */
const char* splitkv_kernel_name(int kernel_id);

/* Static description of a status code (never NULL). */
const char* splitkv_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPLITKV_H */
