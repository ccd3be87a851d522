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
//     slotbuf  [S, KS, H] f32  weighted expert results w_k * E_k(x), one row per (slot, k)
//     y        [S, H]          merged output sum_k slotbuf[slot][k] (ascending k)
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

struct WorkItem {
  int32_t expert;     // bucket id (E = shared expert)
  uint32_t head;      // ring position of the first record
  int32_t count;      // records taken (whole bucket)
  int32_t row_base;   // first row of this item in the step's gathered batch (h rows)
  int32_t t1_base;    // first GEMM1 tile of this item
  int32_t t2_base;    // first GEMM2 tile of this item
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
  unsigned long long duplicates, stale;
  int32_t open_tokens, pending_pairs, ready;
  uint32_t error;
  int32_t trace_n;
  int32_t pad[3];
};

struct LayerView {
  void* pool;
  float* wtab;
  uint32_t* enq_mask;
  uint32_t* done;
  uint32_t* gen;
  float* slotbuf;
  void* y;
  int32_t* records;
  uint32_t* head;
  uint32_t* tail;
  int32_t* ready;
  uint32_t* ready_ht;   // [0] = head (collected up to), [1] = tail (appended up to)
  const void* w13;
  const void* w2;
};

struct Dims {
  int32_t E, K, KS, NB, H, I, S, cap;
  int32_t dtype;        // moe_dtype
  int32_t has_shared;
  int32_t expert_kind;
};

// Tile geometry of the FFN kernels in use; the scheduler counts tiles with it and the
// merge target is KS * parts_per_pair (GEMM2 tiles covering H for one token).
struct TileGeom {
  int32_t bn1;          // tokens per GEMM1 tile
  int32_t bm1;          // packed W13 rows per GEMM1 tile
  int32_t bn2;          // tokens per GEMM2 tile
  int32_t bm2;          // H rows per GEMM2 tile
};

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

__device__ __forceinline__ int32_t record_at(const LayerView& L, const Dims& d, int e, uint32_t pos) {
  return L.records[(size_t)e * d.cap + (pos % (uint32_t)d.cap)];
}

// Merge of one token whose K (+shared) results have all landed: y[slot] = sum over k in
// ascending order of slotbuf[slot][k] (StreamEP section 3: y = sum_j w_j E_j(x)), then
// publish the slot on the ready ring.  Called by `nthr` threads of one CTA (thread index
// `tid`), all of which must call it; the caller has made the landing visible (fence +
// barrier) before.  Reads of other CTAs' slot rows go through L2 (ld.global.cg).
template <typename T>
__device__ void merge_token(const LayerView& L, const Dims& d, DevCounters* C, int slot,
                            int tid, int nthr) {
  const float* src = L.slotbuf + (size_t)slot * d.KS * d.H;
  T* dst = reinterpret_cast<T*>(L.y) + (size_t)slot * d.H;
  for (int f = tid * 4; f < d.H; f += nthr * 4) {     // H % 8 == 0
    float4 acc = __ldcg(reinterpret_cast<const float4*>(src + f));
    for (int k = 1; k < d.KS; ++k) {
      float4 v = __ldcg(reinterpret_cast<const float4*>(src + (size_t)k * d.H + f));
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    dst[f + 0] = from_f<T>(acc.x);
    dst[f + 1] = from_f<T>(acc.y);
    dst[f + 2] = from_f<T>(acc.z);
    dst[f + 3] = from_f<T>(acc.w);
  }
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
template <typename T, typename Bar>
__device__ void land_and_merge(const LayerView& L, const Dims& d, DevCounters* C,
                               const int* slots, int nj, int target, int tid, int nthr,
                               int* fin, Bar bar) {
  __threadfence();
  bar();
  for (int j = tid; j < nj; j += nthr) {
    const uint32_t old = atomicAdd(&L.done[slots[j]], 1u);
    fin[j] = (old + 1u == (uint32_t)target);
    if (old + 1u > (uint32_t)target) set_error(C, MOE_ERR_DUPLICATE);
  }
  __threadfence();
  bar();
  for (int j = 0; j < nj; ++j) {
    if (fin[j]) {
      merge_token<T>(L, d, C, slots[j], tid, nthr);
      if (tid == 0) publish_ready(L, d, C, slots[j]);
    }
  }
  bar();
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
TileGeom simt_geom();
TileGeom tc_geom();

}  // namespace moe
