// Internal declarations of the asynchronous MoE expert-execution library.
//
// Device-side state of one handle (all of it allocated once by moe_async_create):
//
//   per layer l (LayerView):
//     pool     [S, H]          token pool, one row per combine slot (StreamEP section 3: the
//                              Receptor puts each arriving token into a pool)
//     wtab     [S, KS]         top-k weight of each accepted (slot, k); KS = K + has_shared
//     enq_mask [S]             bit k set = pair k accepted for the slot's current generation
//     done     [S]             result parts landed (target = KS * parts_per_pair)
//     gen      [S]             slot generation (advanced when the output is collected)
//     emit_step[S]             scheduling step in which the slot's last result landed
//     slotbuf  [S, KS, H]      expert results E_k(x) in the layer's activation dtype, one row
//                              per (slot, k), as a result row returns to the token's home
//     y        [S, H]          merged output sum_k wtab[slot][k] * slotbuf[slot][k] (fp32,
//                              ascending k)
//     records  [NB, cap] i32   per-expert micro-queue (ring) of (slot << 5 | k); NB = E + has_shared
//     head/tail [NB] u32       monotonic ring counters; depth = tail - head
//     ready    [S] + ready_ht  ring of combined slots awaiting collection
//     w13      [NB, 2I, H]     packed gate/up weights, K-major, gate/up rows interleaved by 16
//     w2       [NB, H, I]      packed down weights, K-major
//   shared by all layers (one step in flight per handle):
//     plan     StepPlan        work list written by the scheduling kernel
//     h        [S*KS, I]       SwiGLU activations of the step's gathered rows
//     counters DevCounters     statistics, sticky error, pick trace
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include "../../include/moe_async.h"

namespace moe {

constexpr int kMaxExperts = 1024;
constexpr int kMaxBuckets = kMaxExperts + 1;
constexpr int kKShift = 5;            // record = slot << 5 | k
constexpr int kKMask = 31;
constexpr uint32_t kRetired = 1u << 31;   // enq_mask flag: the slot's request was cancelled

struct WorkItem {
  int32_t expert;     // bucket id (E = shared expert)
  uint32_t head;      // ring position of the first record
  int32_t count;      // records taken (whole bucket)
  int32_t row_base;   // first row of this item in the step's gathered batch (h rows)
  int32_t t1_base;    // first GEMM1 tile of this item
  int32_t t2_base;    // first GEMM2 tile of this item
  int32_t step;       // scheduling step this item belongs to (a plan may hold several steps)
};

struct StepPlan {
  int32_t layer;
  int32_t n_work;
  int32_t n_tiles1;
  int32_t n_tiles2;
  int32_t rows;
  int32_t pad[3];
  WorkItem items[kMaxBuckets];
};

struct DevCounters {
  unsigned long long steps, pairs_executed, expert_runs, weight_bytes, tokens_combined;
  unsigned long long duplicates, stale, cancelled;
  int32_t open_tokens, pending_pairs, ready;
  uint32_t error;
  int32_t trace_n;
  // after the last scheduling step: its layer, the non-empty buckets it left, and how many
  // of those hold at least the policy's min_batch (the host's drain loop sizes its next
  // batch of steps from these)
  int32_t plan_layer, nonempty_left, elig_left;
};

struct LayerView {
  void* pool;
  float* wtab;
  uint32_t* enq_mask;
  uint32_t* done;       // [S] feature slices merged (target = parts)
  uint32_t* done_part;  // [S][parts] results landed per feature slice (target = KS)
  uint32_t* landed;     // [S] results landed over all slices (for retirement)
  uint32_t* gen;
  uint32_t* emit_step;  // [S] largest step among the slot's landed results (its emission step)
  void* slotbuf;        // [S][KS][H] in the layer dtype: E_k(x), unweighted
  void* y;
  int32_t* records;
  uint32_t* head;
  uint32_t* tail;
  int32_t* ready;
  uint32_t* ready_ht;   // [0] = head (collected up to), [1] = tail (appended up to),
                        // [2] = blocks of the running collect that have finished
  const void* w13;
  const void* w2;
};

struct Dims {
  int32_t E, K, KS, NB, H, I, S, cap;
  int32_t dtype;        // moe_dtype
  int32_t has_shared;
  int32_t expert_kind;
};

constexpr int kMaxLayers = 8;

// Control block of the streaming multi-layer runtime (one per handle, device memory).
struct StreamCtl {
  int32_t tick;                     // logical clock (one scheduling decision per tick)
  int32_t combined;                 // merges completed (token-layer steps)
  int32_t pick_kind;                // 0 none, 1 attention queue, 2 expert queue
  int32_t pick_layer;
  int32_t att_count;                // requests in the current attention batch
  int32_t att_tiles;                // projection GEMM tiles of that batch
  int32_t in_transit;               // dispatched requests whose pairs have not arrived
  int32_t done;                     // 1 once nothing is left to do
  int32_t exp_tokens[kMaxLayers];   // tokens whose pairs wait in layer l's expert queue
  int32_t pad[4];
  int32_t drained[16][2 * kMaxLayers];   // tokens drained per queue, ring over the last ticks
  int32_t snap[16][2 * kMaxLayers];      // depth of each queue at the decision, ring over the last ticks
  int32_t snap_n;                        // snapshots recorded so far
  int32_t to_admit;                      // requests whose admission tick has not come yet
  int32_t peak_transit;                  // most requests in transit at a decision
  int32_t peak_bucket;                   // deepest expert bucket when its layer was served
  int32_t peak_q[2 * kMaxLayers];        // deepest each queue was at a decision
  long long occ_sum[2 * kMaxLayers];     // sum over ticks of each queue's depth at the decision
};

constexpr int kMaxHistoryWindow = 16;

// Device pointers of the streaming runtime, passed by value to its kernels.
//   req_n[r]            completed layer-steps of request r (its state is x^(req_n))
//   arr_tick[r]         tick at which r's dispatched pairs arrive (-1: none in transit)
//   att_ring[l][R] + att_ht[l][2]   attention queue of layer l (ring of request ids)
//   route_idx/route_w   [R][K] routing of r's current step
//   logits [R][n_max][E], delay [R][n_max]   per-(request, step) inputs
//   hist [R][n_max+1][H]   x^(n) of every request; hist[r][0] = x^(0)
//   done_tick [R][n_max+1] tick at which step n completed
//   att_batch / att_scale / att_rowptr [R]   the current attention batch
struct StreamDev {
  StreamCtl* ctl;
  int32_t R, n_max, stop, L;
  int32_t policy, window, hist_window;   // moe_stream_policy and its DEFRAG parameters
  double decay;
  int32_t* req_n;
  int32_t* arr_tick;
  int32_t* att_ring;
  uint32_t* att_ht;
  int32_t* route_idx;
  float* route_w;
  const float* logits;
  const int32_t* delay;
  const int32_t* admit;                  // [R] admission tick of each request (null: all at 0)
  void* hist;
  int32_t* done_tick;
  int32_t* att_batch;
  float* att_scale;
  const void** att_rowptr;
};

// Tile geometry of the FFN kernels in use; the scheduler counts tiles with it and the
// merge target is KS * parts_per_pair (GEMM2 tiles covering H for one token).
struct TileGeom {
  int32_t bn1;          // tokens per GEMM1 tile
  int32_t bm1;          // packed W13 rows per GEMM1 tile
  int32_t bn2;          // tokens per GEMM2 tile
  int32_t bm2;          // H rows per GEMM2 tile
  int32_t bnw;          // tokens per tile of a wide item (0: no wide tiles)
  int32_t wide_min1;    // GEMM1 (and the attention stub): an item of at least this many
  int32_t wide_min2;    //   tokens is cut into wide tiles; GEMM2: the same
};

// Tokens per tile of an item of `count` tokens (bn: the narrow width of the GEMM, wide_min
// its wide threshold).
__host__ __device__ __forceinline__ int tile_tokens(const TileGeom& g, int count, int bn, int wide_min) {
  return (g.bnw > 0 && count >= wide_min) ? g.bnw : bn;
}

}  // namespace moe

struct moe_async_s {
  moe_async_config cfg;
  moe::Dims dims;
  moe::TileGeom geom;
  int32_t parts_per_pair;
  int32_t num_sms;
  int32_t device;
  bool use_tc;                      // bf16 SwiGLU on the tcgen05 kernels
  moe::LayerView* layers;           // host array [L]
  moe::StepPlan* plan;              // device
  void* h;                          // device [S*KS, I]
  moe::DevCounters* counters;       // device
  int4* trace;                      // device [trace_capacity]
  moe::DevCounters* host_counters;  // pinned
  int64_t packed_bytes;
  int64_t launches;                 // kernels launched (host count)
  void* tc_state;                   // tensor maps etc. of the tcgen05 path (device)
  void* prof;                       // per-launch CUDA event pairs while profiling
  void* stream_state;               // streaming multi-layer runtime (moe_async_stream_*)
};

namespace moe {

// ------------------------------------------------------------ device helpers

__device__ __forceinline__ void set_error(DevCounters* c, uint32_t code) {
  atomicCAS(&c->error, 0u, code);
}

__device__ __forceinline__ float silu_f(float a) { return a / (1.0f + __expf(-a)); }

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// One 16-byte vector of slot-row elements (8 bf16 or 4 fp32), widened to fp32 and back.
template <typename T> struct Vec {
  static constexpr int N = 16 / (int)sizeof(T);
};
template <typename T> __device__ __forceinline__ void unpack16(const uint4& u, float (&v)[Vec<T>::N]);
template <> __device__ __forceinline__ void unpack16<float>(const uint4& u, float (&v)[4]) {
  v[0] = __uint_as_float(u.x);
  v[1] = __uint_as_float(u.y);
  v[2] = __uint_as_float(u.z);
  v[3] = __uint_as_float(u.w);
}
template <> __device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4& u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {                     // a bf16 is the top half of an fp32
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
template <typename T> __device__ __forceinline__ uint4 pack16(const float (&v)[Vec<T>::N]);
template <> __device__ __forceinline__ uint4 pack16<float>(const float (&v)[4]) {
  return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
}
template <> __device__ __forceinline__ uint4 pack16<__nv_bfloat16>(const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// The top-k merge of one 16-byte vector of features: a = sum_k w_k * E_k over the slot's KS
// result rows `src` (row stride H) in ascending k, each product and sum rounded in fp32 (no
// fused multiply-add), so the value depends only on the results and weights.  G rows' loads
// are in flight at a time.
template <typename T, int G = 8>
__device__ __forceinline__ void merge_vec(const T* src, const float* wk, int KS, int H, float (&a)[Vec<T>::N]) {
  constexpr int N = Vec<T>::N;
  for (int k0 = 0; k0 < KS; k0 += G) {
    uint4 b[G];
#pragma unroll
    for (int u = 0; u < G; ++u)
      if (k0 + u < KS) b[u] = __ldcg(reinterpret_cast<const uint4*>(src + (size_t)(k0 + u) * H));
#pragma unroll
    for (int u = 0; u < G; ++u) {
      if (k0 + u < KS) {
        const float w = __ldg(wk + k0 + u);
        float v[N];
        unpack16<T>(b[u], v);
#pragma unroll
        for (int i = 0; i < N; ++i) {
          const float p = __fmul_rn(w, v[i]);
          a[i] = k0 + u == 0 ? p : __fadd_rn(a[i], p);
        }
      }
    }
  }
}

// Locate the work item owning global tile `t` (items' bases are ascending).
__device__ __forceinline__ int find_item(const StepPlan* p, int t, bool second) {
  int lo = 0, hi = p->n_work - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    int b = second ? p->items[mid].t2_base : p->items[mid].t1_base;
    if (b <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Top-K of one row of E <= 1024 logits by one warp: (logit desc, index asc); then
// w_k = exp(z_k - m) / sum_{j in top K} exp(z_j - m) with m the largest kept logit, which
// equals softmax over all E renormalised over the top K (the full denominator cancels).
// Lane 0 writes idx[0..K) and w[0..K).
__device__ inline void warp_topk(const float* __restrict__ row, int E, int K, int lane,
                                 int32_t* __restrict__ idx, float* __restrict__ wout) {
  float v[32];
  const int per = (E + 31) / 32;
  for (int i = 0; i < 32; ++i) {
    const int e = lane + 32 * i;
    v[i] = (i < per && e < E) ? row[e] : -INFINITY;
  }
  uint32_t taken = 0;
  float selv[32];
  int seli[32];
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = 0; i < per; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !(taken >> i & 1u)) {
        if (bi == 0x7fffffff || v[i] > bv || (v[i] == bv && e < bi)) { bv = v[i]; bi = e; }
      }
    }
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) { bv = ov; bi = oi; }
    }
    if ((bi & 31) == lane && bi != 0x7fffffff) taken |= 1u << (bi >> 5);
    selv[k] = bv;
    seli[k] = bi;
  }
  if (lane == 0) {
    const float m = selv[0];
    float den = 0.f;
    for (int k = 0; k < K; ++k) den += expf(selv[k] - m);
    for (int k = 0; k < K; ++k) {
      idx[k] = seli[k];
      wout[k] = expf(selv[k] - m) / den;
    }
  }
}

__device__ __forceinline__ int32_t record_at(const LayerView& L, const Dims& d, int e, uint32_t pos) {
  return L.records[(size_t)e * d.cap + (pos % (uint32_t)d.cap)];
}

// Bounds-checked build (MOE_DEBUG_BOUNDS): every bucket, slot and k index read back from
// device state is checked before it is used; an index out of range latches MOE_ERR_BOUNDS
// and the access is skipped -- the stand-in for a memory checker.  Release builds compile
// the checks out.
#ifdef MOE_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif

// A queued record (slot << 5 | k) of bucket e.  In a bounds-checked build a bucket id outside
// [0, NB), a slot outside [0, S) or a k outside [0, KS) latches MOE_ERR_BOUNDS and reads as
// -1, which every consumer treats as an absent row: nothing gathered, nothing written.
__device__ __forceinline__ int32_t record_checked(const LayerView& L, const Dims& d, DevCounters* C, int e,
                                                  uint32_t pos) {
  if (kDebugBounds && (e < 0 || e >= d.NB)) {
    set_error(C, MOE_ERR_BOUNDS);
    return -1;
  }
  const int32_t r = record_at(L, d, e, pos);
  if (kDebugBounds && (r < 0 || (r >> kKShift) >= d.S || (r & kKMask) >= d.KS)) {
    set_error(C, MOE_ERR_BOUNDS);
    return -1;
  }
  return r;
}

// Streaming runtime: request r finished its step at `layer` (its merged output is already in
// hist[r][n+1]).  Advance its step count, record the tick, reclaim its slot in this layer,
// and queue it for the next layer's attention stage unless it reached its last step.
__device__ __forceinline__ void stream_complete(const LayerView& L, DevCounters* C, const StreamDev& sd,
                                                int layer, int r) {
  const int n = sd.req_n[r] + 1;
  sd.req_n[r] = n;
  sd.done_tick[(size_t)r * (sd.n_max + 1) + n] = sd.ctl->tick;
  L.enq_mask[r] = 0u;
  L.done[r] = 0u;
  L.landed[r] = 0u;
  L.emit_step[r] = 0u;
  L.gen[r] = L.gen[r] + 1u;
  atomicAdd(&sd.ctl->combined, 1);
  atomicSub(&C->open_tokens, 1);
  atomicAdd(&C->tokens_combined, 1ull);
  if (n < sd.n_max) {
    const int l2 = (layer + 1) % sd.L;
    const uint32_t pos = atomicAdd(&sd.att_ht[2 * l2 + 1], 1u);
    sd.att_ring[(size_t)l2 * sd.R + (pos % (uint32_t)sd.R)] = r;
  }
}

// Free a slot: clear every per-request counter and advance its generation.
__device__ __forceinline__ void reclaim_slot(const LayerView& L, int parts, int slot) {
  for (int p = 0; p < parts; ++p) L.done_part[(size_t)slot * parts + p] = 0u;
  L.done[slot] = 0u;
  L.landed[slot] = 0u;
  L.enq_mask[slot] = 0u;
  L.emit_step[slot] = 0u;
  L.gen[slot] = L.gen[slot] + 1u;
}

// A cancelled (retired) slot is freed only when every result it accepted has landed: until
// then records of its request may still sit in the queues ("retire until quiescent").
__device__ __forceinline__ bool retired_quiescent(uint32_t mask, uint32_t landed, int parts) {
  return (mask & kRetired) && landed == (uint32_t)__popc(mask & ~kRetired) * (uint32_t)parts;
}

__device__ __forceinline__ void publish_ready(const LayerView& L, const Dims& d, DevCounters* C, int slot) {
  __threadfence();
  uint32_t pos = atomicAdd(&L.ready_ht[1], 1u);
  L.ready[pos % (uint32_t)d.S] = slot;
  atomicAdd(&C->ready, 1);
  atomicSub(&C->open_tokens, 1);
  atomicAdd(&C->tokens_combined, 1ull);
}

struct CtaBarrier {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// Landing of one tile's results and the merges it completes.  Called by the `nthr`
// threads that wrote slotbuf rows for the tile's tokens (slots[0..nj)), after those
// writes.  Each token's landing count is bumped once per (tile, token) with release
// ordering (fence, then atomic); the tile that brings a token to `target` parts performs
// its merge (acquire fence, then reads through L2) and publishes it on the ready ring
// ("inferred obligations": readiness only after the payload is visible).  `bar` is a
// barrier over exactly these threads; `fin` is scratch of >= nj ints visible to them.
//
// The merge is split by feature slice: a tile covering features [f0, f0 + fcount) (slice
// `part` of `parts`) counts, per token, the results landed in that slice; the tile that
// completes a slice (all KS results) sums that slice (ascending k) into y, and the slice
// merges are counted per token in turn -- the last one publishes the token.  So the merge
// work of a token is spread over the CTAs of its slices instead of falling on one.
// `step` is the scheduling step of the tile's work item: a token's emission step is the
// largest step among its results (a plan may hold several consecutive steps).
template <typename T, typename Bar>
__device__ void land_and_merge(const LayerView& L, const Dims& d, DevCounters* C,
                               const int* slots, int nj, int part, int parts, int f0, int fcount,
                               int tid, int nthr, int* fin, Bar bar, int step,
                               const StreamDev* sd = nullptr, int layer = 0) {
  __threadfence();
  bar();
  for (int j = tid; j < nj; j += nthr) {
    const int slot = slots[j];
    if (kDebugBounds && (slot < 0 || slot >= d.S)) {     // an absent row (bounds-checked build)
      fin[j] = 0;
      continue;
    }
    const uint32_t mask = L.enq_mask[slot];              // stable during a step
    if (!sd) atomicMax(&L.emit_step[slot], (uint32_t)step);
    const uint32_t old = atomicAdd(&L.done_part[(size_t)slot * parts + part], 1u);
    const uint32_t landed = atomicAdd(&L.landed[slot], 1u) + 1u;
    fin[j] = (old + 1u == (uint32_t)d.KS) && !(mask & kRetired);
    if (old + 1u > (uint32_t)d.KS) set_error(C, MOE_ERR_DUPLICATE);
    if (retired_quiescent(mask, landed, parts)) reclaim_slot(L, parts, slot);   // last landing
  }
  __threadfence();
  bar();
  // the merge of every finished token's slice: (token, one 16-byte vector of features) items
  // spread over the group (H % 8 == 0 and f0 a multiple of 8 keep every item aligned)
  constexpr int N = Vec<T>::N;
  const int fend = min(f0 + fcount, d.H);
  const int nvec = (fend - f0) / N;
  const int total = nj * nvec;
  const T* rows = static_cast<const T*>(L.slotbuf);
  for (int w = tid; w < total; w += nthr) {
    const int j = w / nvec;
    if (!fin[j]) continue;
    const int slot = slots[j];
    const int f = f0 + N * (w - j * nvec);
    float a[N];
    merge_vec<T>(rows + (size_t)slot * d.KS * d.H + f, L.wtab + (size_t)slot * d.KS, d.KS, d.H, a);
    const uint4 o = pack16<T>(a);
    *reinterpret_cast<uint4*>(static_cast<T*>(L.y) + (size_t)slot * d.H + f) = o;
    if (sd)                                          // req_n is stable until the last slice
      *reinterpret_cast<uint4*>(static_cast<T*>(sd->hist) + ((size_t)slot * (sd->n_max + 1) + sd->req_n[slot] + 1) * d.H + f) = o;
  }
  __threadfence();
  bar();
  for (int j = tid; j < nj; j += nthr) {
    if (fin[j]) {
      const uint32_t old = atomicAdd(&L.done[slots[j]], 1u);
      if (old + 1u == (uint32_t)parts) {             // every slice merged: publish
        if (sd) {
          for (int p = 0; p < parts; ++p) L.done_part[(size_t)slots[j] * parts + p] = 0u;
          stream_complete(L, C, *sd, layer, slots[j]);
        } else {
          publish_ready(L, d, C, slots[j]);
        }
      }
    }
  }
  bar();
}

// Landing of one tile's results when the merge is left to the collect kernel (the per-layer
// path).  Called by the `nthr` threads of the tile's epilogue after its slotbuf writes.  Each
// token's landing count is bumped once per (tile, token); the tile that brings it to KS x parts
// results (every feature slice of every pair) publishes the token on the ready ring.  No fence
// orders the slotbuf writes before the count: collect, which reads them, runs after this kernel
// has finished.  A retired (cancelled) slot is never published and is freed at its last landing.
template <typename Bar>
__device__ void land_only(const LayerView& L, const Dims& d, DevCounters* C, const int* slots, int nj,
                          int parts, int tid, int nthr, Bar bar, int step) {
  const uint32_t target = (uint32_t)d.KS * (uint32_t)parts;
  for (int j = tid; j < nj; j += nthr) {
    const int slot = slots[j];
    if (kDebugBounds && (slot < 0 || slot >= d.S)) continue;     // an absent row (bounds-checked build)
    const uint32_t mask = L.enq_mask[slot];                      // stable during a step
    atomicMax(&L.emit_step[slot], (uint32_t)step);
    const uint32_t landed = atomicAdd(&L.landed[slot], 1u) + 1u;
    if (mask & kRetired) {
      if (retired_quiescent(mask, landed, parts)) reclaim_slot(L, parts, slot);   // last landing
    } else if (landed == target) {
      L.done[slot] = (uint32_t)parts;                            // complete: too late to cancel
      publish_ready(L, d, C, slot);
    } else if (landed > target) {
      set_error(C, MOE_ERR_DUPLICATE);
    }
  }
  bar();
}

// The merge of one ready token, y = sum_k w_k * slotbuf[slot][k] in ascending k (fp32, stored
// in the output dtype with round-to-nearest), by `nthr` threads: one 16-byte vector each at a
// time, the loads of up to G result rows in flight at once (G = 16: one round trip for top-8 +
// the shared expert).
template <typename T, int G = 16>
__device__ __forceinline__ void merge_row(const LayerView& L, const Dims& d, int slot, T* __restrict__ y,
                                          int tid, int nthr) {
  constexpr int N = Vec<T>::N;
  const T* src = static_cast<const T*>(L.slotbuf) + (size_t)slot * d.KS * d.H;
  const float* wk = L.wtab + (size_t)slot * d.KS;
  for (int f = N * tid; f < d.H; f += N * nthr) {
    float a[N];
    merge_vec<T, G>(src + f, wk, d.KS, d.H, a);
    *reinterpret_cast<uint4*>(y + f) = pack16<T>(a);
  }
}

// ------------------------------------------------------------ host helpers

#define MOE_CUDA_TRY(expr)                                  \
  do {                                                      \
    cudaError_t _e = (expr);                                \
    if (_e != cudaSuccess) return MOE_ERR_CUDA;             \
  } while (0)

// Launch bookkeeping: every kernel launch of a handle goes between prof_begin and prof_end
// (events only while profiling is on; the launch count always).
void prof_begin(moe_async_s* h, int kind, cudaStream_t s);
void prof_end(moe_async_s* h, int kind, cudaStream_t s);

// FFN launchers (one per kernel family).  They read the step plan written by the
// scheduling kernel and launch persistent grids; they never synchronise.
moe_status launch_ffn_simt(moe_async_s* h, int layer, cudaStream_t s);
moe_status launch_identity(moe_async_s* h, int layer, cudaStream_t s);
moe_status tc_setup(moe_async_s* h);                 // tensor maps for the tcgen05 path
void tc_teardown(moe_async_s* h);
moe_status launch_ffn_tc(moe_async_s* h, int layer, cudaStream_t s);
moe_status tc_stream_setup(moe_async_s* h, const void* const* proj_packed, const StreamDev& sd);
// out[r][c] = in[c][r] for a bf16 [C][R] matrix (K-major packing of a projection).
cudaError_t pack_transpose_bf16(const void* in, void* out, int C, int R, cudaStream_t s);
moe_status launch_att_tc(moe_async_s* h, cudaStream_t s);
void stream_teardown(moe_async_s* h);
TileGeom simt_geom();
TileGeom tc_geom();

}  // namespace moe
