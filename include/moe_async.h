/*
 * moe_async.h -- C ABI of the asynchronous MoE expert-execution library (GB300, sm_103a).
 *
 * What the library computes.  One or more MoE layers executed asynchronously:
 * routed token vectors arrive in waves tagged (RequestID, LayerID, expert,
 * top-k weight) and are appended to per-expert micro-queues; a scheduling step
 * picks ready queues (most-tokens-first or a minimum batch), gathers each
 * picked queue's tokens into one contiguous batch, runs the expert SwiGLU FFN
 * as a grouped GEMM, and scatters w * E(x) into per-(request, k) combine slots;
 * a token's output y = sum_j w_j E_j(x) is released only once all K results
 * (plus the shared expert's, if any) have landed.
 *   - Metadata, token pool, micro-queues, scheduler, gather + top-k merge:
 *     "SOSP'26 StreamEP" (marsggbo.github.io), sections 3 and 4.
 *   - Minimum-batch streaming of ready tokens (streamFFN) and starting expert
 *     work before every replica's tokens are ready: "CascadeEP: Asynchronous
 *     Expert Execution for MoE Prefill under Attention Imbalance", abstract.
 *   - Readiness published after the payload, exactly-once acceptance, reclaim
 *     after the last read, generation-tagged slots: "asynchronous MoE serving"
 *     notes, sections "recent work that narrows the proposals" (CascadeEP,
 *     Appendix C) and "inferred obligations for a concrete protocol".
 *
 * Conventions for every call.
 *   - Pointers named d_* are DEVICE pointers on the current CUDA device; h_*
 *     are host pointers.  `stream` is a cudaStream_t passed as void* (NULL =
 *     the legacy default stream).  Calls are stream-ordered and asynchronous
 *     unless stated otherwise; a handle must be used from one stream at a time.
 *   - Host-detectable errors (bad arguments) return immediately and launch
 *     nothing.  Errors found on the device (duplicate pair, stale generation,
 *     bucket overflow, out-of-range id) set a sticky device error word; it is
 *     returned by the next synchronising call (moe_async_sync, _wait,
 *     _get_stats) and stays set until moe_async_destroy.
 *   - No call blocks without bound: moe_async_wait is limited by a step count.
 *   - Thread safety: a handle is not thread-safe; distinct handles are.
 *   - Kernels are launched as programmatic dependents of the kernel before them
 *     in the stream (they may start early and wait on the device for it to
 *     finish), so every call still sees all earlier work of the stream; the
 *     caller's own kernels, copies and events order as usual.
 */
#ifndef MOE_ASYNC_H
#define MOE_ASYNC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_async_s* moe_async_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = 1,      /* bad argument (host) or out-of-range id (device)          */
  MOE_ERR_CAPACITY = 2,     /* a per-expert bucket or the ready ring overflowed          */
  MOE_ERR_DUPLICATE = 3,    /* a (slot, k) pair was delivered twice; the copy is dropped */
  MOE_ERR_STALE = 4,        /* a pair carried an out-of-date slot generation; dropped    */
  MOE_ERR_TIMEOUT = 5,      /* moe_async_wait ran out of steps with tokens still open;   */
                            /* or (sticky) a device wait in the tensor-core kernels     */
                            /* exceeded its 2 s bound -- the handle's state is then     */
                            /* undefined and it should be destroyed                     */
  MOE_ERR_CUDA = 6,         /* a CUDA runtime call failed                                */
  MOE_ERR_UNSUPPORTED = 7,  /* shape/dtype combination not supported by the kernels      */
  MOE_ERR_BOUNDS = 8        /* (bounds-checked build only) an index read back from device
                               state was out of range; the access was skipped           */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum {
  MOE_POLICY_MTFS = 0,       /* most tokens first: deepest buckets first (StreamEP, section 4) */
  MOE_POLICY_THRESHOLD = 1,  /* buckets holding >= min_batch tokens; else MTFS fallback         */
  MOE_POLICY_RANKS = 2       /* simulated expert-parallel ranks with work stealing: expert e
                              * belongs to rank e mod max_groups; each rank runs its deepest
                              * bucket; with fallback_groups != 0 a rank owning no non-empty
                              * bucket takes the deepest bucket no rank picked (unstarted work
                              * reassigned to an idle helper: "asynchronous MoE serving" notes,
                              * CascadeEP v1).  Picks are planned in rank order.              */
} moe_policy_kind;

typedef enum {
  MOE_EXPERT_SWIGLU = 0,     /* E(x) = (silu(x W1) * (x W3)) W2                               */
  MOE_EXPERT_IDENTITY = 1    /* E(x) = x; exercises queues/readiness/combine without a GEMM    */
} moe_expert_kind;

typedef struct {
  int32_t num_layers;       /* L >= 1                                                          */
  int32_t num_experts;      /* E routed experts per layer, 1..1024                             */
  int32_t top_k;            /* K, 1..30                                                        */
  int32_t hidden;           /* H, multiple of 8                                                */
  int32_t inter;            /* I, multiple of 16                                               */
  int32_t dtype;            /* moe_dtype of x, weights and y (accumulation is always fp32)     */
  int32_t has_shared;       /* 1: one always-on shared expert per layer, weight 1, I_s == I   */
  int32_t max_slots;        /* combine slots (RequestIDs 0..max_slots-1) per layer             */
  int32_t bucket_capacity;  /* pairs per expert bucket; 0 = max_slots (cannot overflow)        */
  int32_t expert_kind;      /* moe_expert_kind                                                 */
  int32_t trace_capacity;   /* >0: record up to this many (step, layer, expert, count) picks   */
} moe_async_config;

typedef struct {
  int32_t kind;             /* moe_policy_kind                                                 */
  int32_t max_groups;       /* at most this many buckets per step; 0 = no limit;
                             * RANKS: the number of ranks, >= 1                                */
  int32_t min_batch;        /* THRESHOLD: minimum bucket depth to run                          */
  int32_t fallback_groups;  /* THRESHOLD: buckets taken (deepest first) when none qualifies;
                             * RANKS: nonzero = idle ranks steal                               */
} moe_async_policy;

typedef struct {
  int64_t steps;            /* scheduling steps executed                                       */
  int64_t pairs_executed;   /* routed (token, expert) pairs run through an expert              */
  int64_t expert_runs;      /* sum over steps of the number of buckets picked                  */
  int64_t weight_bytes;     /* expert weight bytes streamed, as scheduled (3*H*I*elem per run) */
  int64_t tokens_combined;  /* tokens whose merge completed                                    */
  int64_t duplicates;       /* pairs rejected as duplicates                                    */
  int64_t stale;            /* pairs rejected for a stale generation                           */
  int32_t open_tokens;      /* tokens with >= 1 accepted pair not yet combined (all layers)    */
  int32_t pending_pairs;    /* accepted pairs not yet picked (all layers)                      */
  int32_t ready;            /* combined tokens not yet collected (all layers)                  */
  int32_t error;            /* sticky device error (moe_status)                                */
  int64_t packed_weight_bytes; /* library-owned packed weight copy made at create              */
  int64_t kernel_launches;  /* kernels this handle has launched since create                   */
  int64_t cancelled;        /* requests retired by moe_async_cancel                            */
} moe_async_stats;

/* Kernel kinds timed by moe_async_profile (index into the arrays of moe_async_profile_read). */
typedef enum {
  MOE_KERNEL_ENQUEUE = 0,    /* Receptor: pairs into buckets, token rows into the pool          */
  MOE_KERNEL_SCHEDULE = 1,   /* device-side policy + work list                                  */
  MOE_KERNEL_FFN1 = 2,       /* gather + GEMM1 (gate/up) + SwiGLU   (identity: scatter)         */
  MOE_KERNEL_FFN2 = 3,       /* GEMM2 (down) + scatter of the results + readiness               */
  MOE_KERNEL_COLLECT = 4,    /* top-k merge of ready tokens, rows to the caller, slot reclaim   */
  MOE_KERNEL_TICK = 5,       /* moe_async_tick's control kernel: collect + Receptor + reclaim   */
  MOE_KERNEL_KINDS = 6
} moe_kernel_kind;

/* Create a handle.  Weights are given per layer as arrays of L device pointers:
 *   w1[l], w3[l] : [E, H, I] (expert e computes x @ W1[e]),  w2[l] : [E, I, H]
 *   shared_w1[l], shared_w3[l] : [H, I], shared_w2[l] : [I, H]  (NULL arrays when has_shared = 0)
 * all in cfg->dtype, row-major, contiguous.  The library packs them into its own K-major
 * copy (gate/up rows interleaved) before returning (it synchronises `stream`), so the
 * caller's weight buffers may be freed afterwards.  All state (token pool, buckets, combine
 * slots, outputs, work lists) is allocated here; no later call allocates device memory.
 * Returns MOE_ERR_INVALID / MOE_ERR_UNSUPPORTED for bad configs, MOE_ERR_CUDA on allocation
 * failure (nothing leaks).  *out is set only on MOE_OK. */
moe_status moe_async_create(const moe_async_config* cfg,
                            const void* const* w1, const void* const* w3, const void* const* w2,
                            const void* const* shared_w1, const void* const* shared_w3,
                            const void* const* shared_w2,
                            void* stream, moe_async_t* out);

/* Router: top-K experts per token with renormalised softmax weights.
 * StreamEP section 3 (each token selects its K highest-scoring experts); the rule is softmax
 * over the E logits, keep the K largest, renormalise them to sum to one.  Equal logits go to
 * the lower expert index; k = 0 is the highest score.
 *   d_logits : [T, E] fp32      d_idx : [T, K] int32 (out)      d_w : [T, K] fp32 (out)
 * Stateless (no handle).  1 <= K <= E <= 1024, K <= 32. */
moe_status moe_async_route(const float* d_logits, int32_t T, int32_t E, int32_t K,
                           int32_t* d_idx, float* d_w, void* stream);

/* Receptor: deliver one wave of routed pairs into layer `layer`'s expert queue.
 * StreamEP section 3, steps 1-2: each carried token is stored in the token pool under its
 * combine slot, and each delivered (expert, k, w) pair is appended to that expert's bucket
 * (warp-aggregated atomics).  A token's first accepted pair also enqueues the shared expert.
 *   n        : tokens carried (0 is a no-op)
 *   d_rows   : [n] row of d_x / d_expert / d_w for each carried token; NULL = rows 0..n-1
 *   d_slot   : [n] combine slot (RequestID) per token, < max_slots; NULL = the row index
 *   d_x      : [*, H] token vectors in cfg dtype (row-indexed)
 *   d_expert : [*, K] int32 expert ids (row-indexed), 0 <= id < E
 *   d_w      : [*, K] fp32 routing weights (row-indexed)
 *   d_kmask  : [n] uint32, bit k set = pair k is delivered by this wave; NULL = all K
 *   d_gen    : [n] uint32 expected slot generation; NULL = unchecked.  Mismatch -> the
 *              token's pairs are dropped and MOE_ERR_STALE is latched.
 * A pair already accepted for this slot generation is dropped and MOE_ERR_DUPLICATE latched.
 * The caller's buffers may be reused once the stream reaches this point. */
moe_status moe_async_enqueue(moe_async_t h, int32_t layer, int32_t n,
                             const int32_t* d_rows, const int32_t* d_slot, const void* d_x,
                             const int32_t* d_expert, const float* d_w,
                             const uint32_t* d_kmask, const uint32_t* d_gen, void* stream);

/* One scheduling step of layer `layer`, decided on the device from the bucket depths
 * (no host synchronisation): the policy picks buckets, each picked bucket is drained whole,
 * its tokens are gathered and run through the expert (grouped GEMM over all picks), the
 * results E_k(x) are written to their combine slots in the activation dtype, and every
 * token whose K (+shared) results are now complete is appended to the ready list (its
 * merge runs in moe_async_collect).  A step with nothing to pick launches kernels that exit
 * at once. */
moe_status moe_async_schedule_step(moe_async_t h, int32_t layer, const moe_async_policy* policy,
                                   void* stream);

/* Up to max_steps (>= 1) consecutive scheduling steps of layer `layer` in one device plan,
 * with the same picks, values and emission steps as that many moe_async_schedule_step calls
 * with nothing enqueued between them.  StreamEP section 4 (MTFS) and the CascadeEP abstract
 * (streamFFN): with no arrival between steps the queue depths only shrink, so the picks of
 * consecutive steps are one deepest-first order of the non-empty buckets cut into steps --
 * MTFS max_groups buckets a step (0 = all in one); THRESHOLD up to max_groups buckets of at
 * least min_batch a step while any remain, then fallback_groups a step.  All picked buckets
 * run in one grouped GEMM launch pair, each work item tagged with its step, so a drain of
 * many one-expert fallback steps streams weights on every SM instead of one expert per
 * launch.  The steps counter and the pick trace advance by the steps up to the last
 * non-empty one (a call that finds every bucket empty counts none).  MTFS and THRESHOLD
 * only: RANKS returns MOE_ERR_UNSUPPORTED for max_steps > 1.  Asynchronous, no host
 * synchronisation. */
moe_status moe_async_schedule_steps(moe_async_t h, int32_t layer, const moe_async_policy* policy,
                                    int32_t max_steps, void* stream);

/* One tick of a serving loop: one control launch, then the step's launches (plan, GEMM1,
 * GEMM2).  The control launch runs, side by side, the collect of the tokens that were ready
 * when the call was made (outputs as moe_async_collect, with max_out, d_y_out .. d_n_out and
 * append meaning the same; max_out = 0 collects nothing and d_n_out may then be NULL) and the
 * Receptor for a wave of n arriving tokens (arguments as moe_async_enqueue; n = 0 for none);
 * then one scheduling step runs under `policy` (as moe_async_schedule_step).  StreamEP section 3 (the Receptor feeds the per-expert queues,
 * ready tokens leave after their K results) and section 4 (the scheduler then picks).
 *   Equivalent to moe_async_collect, moe_async_enqueue and moe_async_schedule_step in that
 * order, with one difference: the collected slots are reclaimed after the wave's pairs have
 * been judged, so a pair of this wave for a slot collected by this call is judged against the
 * request it completed (a duplicate) rather than against the slot's next generation.  A
 * caller learns which slots are free only from a collect's outputs, so it never assigns a new
 * request to a slot collected by the same call.
 *   Asynchronous, no host synchronisation.  Errors as the three calls; MOE_ERR_INVALID for a
 * bad argument of any of them. */
moe_status moe_async_tick(moe_async_t h, int32_t layer, int32_t n, const int32_t* d_rows, const int32_t* d_slot,
                          const void* d_x, const int32_t* d_expert, const float* d_w, const uint32_t* d_kmask,
                          const uint32_t* d_gen, const moe_async_policy* policy, int32_t max_out, void* d_y_out,
                          int32_t* d_slot_out, uint32_t* d_gen_out, uint32_t* d_step_out, int32_t* d_n_out,
                          int32_t append, void* stream);

/* Collect ready tokens of layer `layer` in completion order, each merged on the way out:
 * y = sum_k w_k E_k(x) in fp32, ascending k (k = K is the shared expert, weight 1), each
 * product and sum rounded (no fused multiply-add), stored in the cfg dtype:
 *   d_y_out    : [max_out, H] cfg dtype     d_slot_out : [max_out] int32
 *   d_gen_out  : [max_out] uint32 (generation the result belongs to; may be NULL)
 *   d_step_out : [max_out] uint32 (emission step: the scheduling step, counted from 1 over
 *                the handle's life, in which the token's last result landed; may be NULL)
 *   d_n_out    : [1] int32 on the device
 *   append = 0 : rows are written from index 0 and *d_n_out = number written (<= max_out)
 *   append = 1 : rows are written from index *d_n_out (read on the device) and *d_n_out is
 *                advanced by the number written (total <= max_out), so a caller can collect
 *                after every step into one buffer without reading anything back
 * Each collected slot is reclaimed (its generation advances) after its output row is copied,
 * so it may carry a new request from then on. */
moe_status moe_async_collect(moe_async_t h, int32_t layer, int32_t max_out, void* d_y_out,
                             int32_t* d_slot_out, uint32_t* d_gen_out, uint32_t* d_step_out,
                             int32_t* d_n_out, int32_t append, void* stream);

/* Cancel the current request of each slot in d_slots[0..n) (int32, device) of `layer`.
 * "asynchronous MoE serving" notes: an abandoned operation retires its buffer until a quiescent
 * point, and output readiness is tracked separately from buffer reclamation (CascadeEP).  The
 * slot is retired: later pairs for it are dropped on arrival, pairs already queued still run
 * but their results are neither merged nor published, and the slot is freed (generation
 * advanced, reusable) when its last queued result has landed -- at once if nothing is queued.
 * Free slots and slots whose output is already merged are left unchanged.  Not available on a
 * handle running the streaming runtime (MOE_ERR_UNSUPPORTED). */
moe_status moe_async_cancel(moe_async_t h, int32_t layer, int32_t n, const int32_t* d_slots,
                            void* stream);

/* Run scheduling steps of `layer` under `policy` until no token of the handle is open
 * (accepted but not yet combined, in any layer); at most max_steps steps.  Under MTFS and
 * THRESHOLD the layer's queued buckets are drained as one plan of consecutive steps
 * (moe_async_schedule_steps), re-planned while the last plan left buckets behind.  Once the
 * queues are empty while tokens are still open, and under RANKS, single steps run: between
 * reads of the device counters as many as the layer's queues certainly still need (each step
 * drains its picks whole and takes at most max_groups buckets under RANKS), else
 * `check_every` steps.  Synchronises `stream`.  Returns MOE_ERR_TIMEOUT when tokens are still open after
 * max_steps (e.g. a withheld pair), else the sticky device error. */
moe_status moe_async_wait(moe_async_t h, int32_t layer, const moe_async_policy* policy,
                          int32_t max_steps, int32_t check_every, void* stream);

/* Synchronise `stream` and return the sticky device error (MOE_OK if none). */
moe_status moe_async_sync(moe_async_t h, void* stream);

/* Synchronise `stream` and copy the counters into *h_stats. */
moe_status moe_async_get_stats(moe_async_t h, void* stream, moe_async_stats* h_stats);

/* Synchronise and copy the pick trace: h_buf receives up to cap records of 4 int32
 * (step, layer, expert, count) in step order, *h_n the number of records written. */
moe_status moe_async_get_trace(moe_async_t h, void* stream, int32_t* h_buf, int32_t cap,
                               int32_t* h_n);

/* Synchronise and copy layer `layer`'s queue contents: h_depth[b] (b < E + has_shared) gets
 * bucket b's depth, and h_records the pending records of every bucket in bucket order, each
 * as (slot, k) int32 pairs (bucket-internal order is arrival order, which concurrent appends
 * make nondeterministic).  cap = capacity of h_records in pairs; *h_n = pairs written. */
moe_status moe_async_snapshot(moe_async_t h, int32_t layer, void* stream, int32_t* h_depth,
                              int32_t* h_records, int32_t cap, int32_t* h_n);

/* ---- Streaming multi-layer decode on the 2L micro-queues --------------------------------
 * "SOSP'26 StreamEP" section 3: each layer has an attention queue and an expert queue; a
 * request's token is served by its layer's attention stage, routed, dispatched to the expert
 * queue, merged back and queued for the next layer's attention -- each request advances at
 * its own pace, with no barrier across requests.  Section 4: one queue is served per
 * scheduling decision, the one holding the most tokens (MTFS; equal counts -> lower layer,
 * attention before expert).  The attention stage is a stub: a = RMSNorm(x) P_l (eps 1e-6,
 * no gain), x^(n+1) = MoE_l(a) with l = n mod L.  All state lives on the device and one
 * scheduling decision ("tick") runs as a CUDA graph with no host round trip. */
typedef enum {
  MOE_STREAM_MTFS = 0,      /* most tokens first (StreamEP section 4)                             */
  MOE_STREAM_FLFS = 1,      /* first layer first: earliest non-empty queue of the chain           */
  MOE_STREAM_DEFRAG = 2,    /* S(s) = Q(s) + sum_{j=1..W} decay^j [Q(s_j) + H(s_j)] (section 4)   */
  MOE_STREAM_BARRIER = 3,   /* synchronous baseline: nothing served while a dispatch is in flight */
  MOE_STREAM_DEFRAG_SRC = 4 /* the same score as section 4 describes the source implementation:
                               H(s) = average of s's depth snapshots over the last history_window
                               ticks, lookahead continued cyclically along the chain              */
} moe_stream_policy;

typedef struct {
  int32_t num_requests;     /* R <= max_slots; request r uses combine slot r in every layer    */
  int32_t max_steps;        /* steps per request at most (history depth)                       */
  int32_t stop_combines;    /* attention queues are closed once this many merges are done      */
  int32_t policy;           /* moe_stream_policy                                               */
  int32_t defrag_window;    /* DEFRAG(_SRC): W, queues looked ahead along att_0, exp_0, att_1, ... */
  int32_t history_window;   /* DEFRAG: H(s) = tokens drained from s over the last N ticks, <=16;
                               DEFRAG_SRC: the window of depth snapshots H(s) averages         */
  double defrag_decay;      /* DEFRAG: decay per lookahead step (scores in fp64)               */
} moe_stream_config;

/* Set up the streaming runtime on a bf16 SwiGLU handle (its merges then feed the runtime,
 * not the collect ring).  Synchronises `stream`.
 *   d_proj[l]   : [H, H] bf16 projection of layer l's attention stub (x @ P); packed, may be freed
 *   d_x0        : [R, H] bf16 initial states (copied into the history)
 *   d_logits    : [R, max_steps, E] fp32 router logits of (request, step)   (borrowed)
 *   d_delay     : [R, max_steps] int32 dispatch delay in ticks, >= 1       (borrowed)
 *   d_admit     : [R] int32 tick at which each request enters layer 0's attention queue
 *                 (<= 0: at the start); NULL = every request at the start   (borrowed)
 *   d_history   : [R, max_steps + 1, H] bf16 out: x^(n) of every request, x^(0) at n = 0
 *   d_done_tick : [R, max_steps + 1] int32 out: tick at which step n completed (-1 = not)
 * Requests admitted later join the attention queue at the start of their tick, after that
 * tick's dispatches are delivered; while attention is open, requests still to be admitted
 * keep the stream running (idle ticks).  MOE_ERR_UNSUPPORTED for fp32 or identity handles or
 * more than 8 layers. */
moe_status moe_async_stream_setup(moe_async_t h, const moe_stream_config* sc,
                                  const void* const* d_proj, const void* d_x0,
                                  const float* d_logits, const int32_t* d_delay,
                                  const int32_t* d_admit, void* d_history, int32_t* d_done_tick,
                                  void* stream);

/* Queue occupancy of the streaming runtime so far (for latency studies; StreamEP section 4:
 * queue depths are what the scheduler acts on).  Depths are in tokens (requests), seen at
 * each tick's decision after that tick's arrivals and admissions. */
typedef struct {
  int32_t ticks;                 /* ticks run                                                    */
  int32_t combined;              /* merges completed (token-layer steps)                         */
  int32_t peak_transit;          /* most requests in transit (dispatched, not yet arrived)       */
  int32_t peak_bucket;           /* deepest expert bucket at the moment its layer was served     */
  int32_t num_queues;            /* 2L: the queues below in chain order att_0, exp_0, att_1, ... */
  int32_t peak_queue[16];        /* deepest each queue was at a decision (closed attention: 0)   */
  int64_t occupancy_sum[16];     /* each queue's depth summed over the ticks (mean = / ticks)    */
} moe_stream_stats;

/* Synchronise `stream` and read the streaming runtime's occupancy figures. */
moe_status moe_async_stream_stats(moe_async_t h, void* stream, moe_stream_stats* out);

/* Run ticks until nothing is left (no dispatch in transit, expert queues empty, attention
 * queues closed or empty), reading the control block every `check_every` ticks; at most
 * max_ticks ticks (then MOE_ERR_TIMEOUT).  Synchronises; *h_ticks = ticks run,
 * *h_combined = merges completed. */
moe_status moe_async_stream_run(moe_async_t h, int32_t max_ticks, int32_t check_every,
                                int32_t* h_ticks, int32_t* h_combined, void* stream);

/* Synchronise and copy the tick trace: 4 int32 per tick (tick, kind, layer, count), kind
 * 1 = attention queue, 2 = expert queue, 0 = idle (only dispatches in transit). */
moe_status moe_async_stream_trace(moe_async_t h, void* stream, int32_t* h_buf, int32_t cap,
                                  int32_t* h_n);

/* Per-kernel timing (tracing).  enable = 1 brackets every later kernel launch of the handle
 * with a pair of CUDA events on its stream (up to 65536 launches are kept); enable = 0 stops.
 * Host-side events only: no device memory is allocated. */
moe_status moe_async_profile(moe_async_t h, int32_t enable);

/* Synchronise `stream`, then for each kernel kind k < n_kinds add the summed event time of its
 * recorded launches to h_ms[k] (milliseconds) and their number to h_launches[k]; the record
 * is cleared afterwards. */
moe_status moe_async_profile_read(moe_async_t h, void* stream, double* h_ms, int64_t* h_launches,
                                  int32_t n_kinds);

/* Free every device allocation of the handle.  Synchronises `stream` first. */
moe_status moe_async_destroy(moe_async_t h, void* stream);

/* One routed MoE layer forward that allocates no device memory.  The pages have no
 * counterpart: this is for callers that cannot call cudaMalloc where they run the layer
 * (a memory pool owns the device, an allocation-free runtime, a plugin that is handed only
 * its input and output buffers).
 *   y[t] = sum_{k=0..K-1, ascending} w[t,k] * E_{expert[t,k]}(x[t]),
 *   E(x) = (silu(x W1) * (x W3)) W2, fp32 accumulation, no shared expert.
 *   d_x [T,H], d_y [T,H] in dtype (moe_dtype); d_expert [T,K] int32 in [0,E); d_w [T,K]
 *   fp32; d_w1, d_w3 [E,H,I] and d_w2 [E,I,H] in dtype -- the caller's own weight layout,
 *   no packing.  All device pointers, all caller-owned.
 * Expert ids outside [0,E) contribute nothing, silently: unlike moe_async_enqueue, which
 * latches MOE_ERR_INVALID in its handle's sticky error, this call has no handle to hold an
 * error, and the ids live in device memory where the host cannot check them without a sync.
 * Scratch: a fixed 16 MiB array compiled into the library (held on every GPU that loads
 * it, until the process exits) holds the T*K*I fp32 SwiGLU activations, so T*K*I*4 bytes
 * may not exceed 16 MiB: larger calls return MOE_ERR_CAPACITY and launch nothing.  Every
 * call looks up the array's device address in the current context (no allocation); the
 * first call in a context may load the library's device code, so make it before any stream
 * capture.  Work: each (token, k) pair reads its expert's W1 and W3 columns on its own (no
 * weight reuse between pairs of one expert), so this path is far slower than the grouped
 * GEMMs of the handle-based calls.  Every call shares the one array and each call
 * overwrites every element it reads, so nothing has to be cleared, but calls whose kernels
 * overlap on the GPU (different streams, or different host threads) race on it: order them.
 * Calls no cudaMalloc/cudaFree.  Asynchronous on `stream`. */
moe_status moe_async_forward_noalloc(int32_t T, int32_t E, int32_t K, int32_t H, int32_t I,
                                     int32_t dtype, const void* d_x, const int32_t* d_expert,
                                     const float* d_w, const void* d_w1, const void* d_w3,
                                     const void* d_w2, void* d_y, void* stream);

/* Bounds-checked build (libmoe_async_debug.so, compiled with MOE_DEBUG_BOUNDS): every bucket,
 * slot and k index the kernels read back from device state is checked before use, and an
 * index out of range latches MOE_ERR_BOUNDS (the access is skipped, the scheduler halts).  This
 * call appends the raw value `record` (slot << 5 | k, unchecked) to bucket `bucket` of `layer`,
 * so a test can plant an out-of-range record and see it rejected without touching memory
 * out of range.  Release builds return MOE_ERR_UNSUPPORTED and write nothing.  Asynchronous. */
moe_status moe_async_debug_append_record(moe_async_t h, int32_t layer, int32_t bucket, int32_t record,
                                        void* stream);

/* 1 if the kernels can write `n` bytes at host address `p` directly (pinned host memory
 * mapped into the device's address space at the same address), else 0.  A caller may then
 * pass such a buffer as a collect output (d_y_out, d_slot_out, ...), so each merged row goes
 * to host memory as it is produced instead of by a copy after the step.  Host-side query, no
 * device work. */
int32_t moe_async_host_writable(const void* p, int64_t n);

/* Human-readable name of a status code (static string). */
const char* moe_async_status_string(moe_status s);

#ifdef __cplusplus
}
#endif
#endif /* MOE_ASYNC_H */
