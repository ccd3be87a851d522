// C-ABI entry points and the queue-side kernels of the asynchronous MoE library:
// weight packing, router, Receptor (enqueue), scheduler, collect.
// The expert FFN kernels live in moe_ffn_simt.cu (fp32 / identity) and moe_ffn_tc.cu
// (bf16 on tcgen05 tensor cores).
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <new>
#include "moe_plan.cuh"

using namespace moe;

namespace {

// ---------------------------------------------------------------- packing
// out[e][orow(i)][c] = in[e][c][i] for a row-major [E][C][R] input: a batched transpose
// into K-major rows.  `interleave` places source row i at packed row 32*(i/16) + i%16 +
// 16*which (gate rows first, then up rows, in blocks of 16), so a 32-row slice of the
// packed W13 holds gate and up of the same 16 features.
template <typename T>
__global__ void pack_transpose_kernel(const T* __restrict__ in, T* __restrict__ out, int C, int R,
                                      int out_rows, int interleave, int which) {
  __shared__ T tile[32][33];
  const int e = blockIdx.z;
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  const T* src = in + (size_t)e * C * R;
  T* dst = out + (size_t)e * out_rows * C;
  for (int j = threadIdx.y; j < 32; j += blockDim.y) {
    int c = c0 + j, r = r0 + threadIdx.x;
    if (c < C && r < R) tile[j][threadIdx.x] = src[(size_t)c * R + r];
  }
  __syncthreads();
  for (int j = threadIdx.y; j < 32; j += blockDim.y) {
    int r = r0 + j, c = c0 + threadIdx.x;
    if (r < R && c < C) {
      int orow = interleave ? (32 * (r / 16) + (r % 16) + 16 * which) : r;
      dst[(size_t)orow * C + c] = tile[threadIdx.x][j];
    }
  }
}

template <typename T>
cudaError_t pack_one(const void* in, void* out, int nexp, int C, int R, int out_rows, int inter,
                     int which, cudaStream_t s) {
  dim3 grid((C + 31) / 32, (R + 31) / 32, nexp), block(32, 8);
  pack_transpose_kernel<T><<<grid, block, 0, s>>>(static_cast<const T*>(in), static_cast<T*>(out),
                                                   C, R, out_rows, inter, which);
  return cudaGetLastError();
}

}  // namespace

namespace moe {
cudaError_t pack_transpose_bf16(const void* in, void* out, int C, int R, cudaStream_t s) {
  return pack_one<__nv_bfloat16>(in, out, 1, C, R, R, 0, 0, s);
}
}  // namespace moe

namespace {

// ----------------------------------------------------------------- router
// One warp per token (warp_topk): top-K by (logit desc, index asc), renormalised softmax.
__global__ void route_kernel(const float* __restrict__ logits, int T, int E, int K,
                             int32_t* __restrict__ idx, float* __restrict__ wout) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  warp_topk(logits + (size_t)t * E, E, K, lane, idx + (size_t)t * K, wout + (size_t)t * K);
}

// --------------------------------------------------------------- Receptor
constexpr int kCopyDepth = 16;         // 16-byte loads in flight per lane in the pool copy

// One warp takes `tpw` whole tokens at a time (tpw * KS <= 32): lane l handles pair k = l % KS
// of token l / KS (k == K is the shared expert).  Once a pair's acceptance is known, the warp
// copies into pool[slot] (16-byte vectors) the row of each of its tokens that had at least
// one pair accepted by this call: a stale, retired or duplicate delivery leaves the pool row
// of the slot's current request untouched ("asynchronous MoE serving" notes, inferred
// obligations: accept exactly the selected contributions).  Then the appends, with
// warp-aggregated atomics: lanes bound for the same bucket elect a leader that reserves all
// of their positions with one atomicAdd on the bucket tail.

// The Receptor's work for warp `gw` of `nwarps` (whole tokens, `tpw` a warp at a time).
template <typename T>
__device__ __forceinline__ void enqueue_warps(const LayerView& L, const Dims& d, DevCounters* C, int n, int tpw,
                                              const int32_t* __restrict__ rows, const int32_t* __restrict__ slots,
                                              const T* __restrict__ x, const int32_t* __restrict__ expert,
                                              const float* __restrict__ w, const uint32_t* __restrict__ kmask,
                                              const uint32_t* __restrict__ gens, long long gw, long long nwarps) {
  const int lane = threadIdx.x & 31;
  const int jl = lane / d.KS;              // this lane's token within the warp's group
  const int k = lane % d.KS;
  const uint32_t kbits = (1u << d.KS) - 1u;  // KS <= 31
  constexpr int V = 16 / sizeof(T);
  const int chunks = d.H / V;
  for (long long g0 = gw * tpw; g0 < n; g0 += nwarps * tpw) {
    int key = -1 - lane;          // unique key for lanes with nothing to append
    int slot = -1, row = -1;
    uint32_t head_e = 0;
    bool accepted = false;
    if (jl < tpw && g0 + jl < n) {
      const int i = (int)(g0 + jl);
      row = rows ? rows[i] : i;
      slot = slots ? slots[i] : row;
      bool ok = true;
      if (slot < 0 || slot >= d.S || row < 0) { set_error(C, MOE_ERR_INVALID); ok = false; }
      if (ok && gens && L.gen[slot] != gens[i]) {
        if (k == 0) { set_error(C, MOE_ERR_STALE); atomicAdd(&C->stale, 1ull); }
        ok = false;
      }
      if (ok && k < d.K && kmask && !((kmask[i] >> k) & 1u)) ok = false;
      int e = d.E;
      float wk = 1.0f;                       // the shared expert's weight
      if (ok && k < d.K) {
        e = expert[(size_t)row * d.K + k];
        wk = w[(size_t)row * d.K + k];
        if (e < 0 || e >= d.E) { set_error(C, MOE_ERR_INVALID); ok = false; }
      }
      // the bucket's head, read with the mask (its loads overlap the atomics below); the
      // scheduler, the only writer of heads, is ordered after this kernel in the stream
      if (ok) head_e = L.head[e];
      if (ok && (L.enq_mask[slot] & kRetired)) ok = false;   // late pair of a cancelled request
      if (ok) {
        const uint32_t bit = 1u << k;
        const uint32_t old = atomicOr(&L.enq_mask[slot], bit);
        if (old & bit) {
          if (k < d.K) { set_error(C, MOE_ERR_DUPLICATE); atomicAdd(&C->duplicates, 1ull); }
          ok = false;            // shared expert: already enqueued by an earlier wave
        } else {
          if (old == 0u) atomicAdd(&C->open_tokens, 1);
          L.wtab[(size_t)slot * d.KS + k] = wk;
          key = e;
          accepted = true;
        }
      }
    }
    // token rows -> pool, only for tokens with a pair accepted here (warp-uniform loop); the
    // copies are issued before the bucket appends so their loads overlap the atomics' trips
    const uint32_t acc = __ballot_sync(0xffffffffu, accepted);
    for (int j = 0; j < tpw; ++j) {
      if (!((acc >> (j * d.KS)) & kbits)) continue;
      const int row_j = __shfl_sync(0xffffffffu, row, j * d.KS);
      const int slot_j = __shfl_sync(0xffffffffu, slot, j * d.KS);
      const int4* src = reinterpret_cast<const int4*>(x + (size_t)row_j * d.H);
      int4* dst = reinterpret_cast<int4*>(static_cast<T*>(L.pool) + (size_t)slot_j * d.H);
      for (int c = lane; c < chunks; c += 32 * kCopyDepth) {   // kCopyDepth loads in flight
        int4 v[kCopyDepth];
#pragma unroll
        for (int u = 0; u < kCopyDepth; ++u)
          if (c + 32 * u < chunks) v[u] = __ldg(src + c + 32 * u);
#pragma unroll
        for (int u = 0; u < kCopyDepth; ++u)
          if (c + 32 * u < chunks) dst[c + 32 * u] = v[u];
      }
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    if (key >= 0) {
      const int leader = __ffs(peers) - 1;
      const uint32_t cnt = __popc(peers);
      uint32_t pos0 = 0;
      if (lane == leader) {
        pos0 = atomicAdd(&L.tail[key], cnt);
        atomicAdd(&C->pending_pairs, (int)cnt);
      }
      pos0 = __shfl_sync(peers, pos0, leader);
      const uint32_t pos = pos0 + __popc(peers & ((1u << lane) - 1u));
      if (pos - head_e >= (uint32_t)d.cap) {
        set_error(C, MOE_ERR_CAPACITY);
      } else {
        L.records[(size_t)key * d.cap + (pos % (uint32_t)d.cap)] = (slot << kKShift) | k;
      }
    }
  }
}

template <typename T>
__global__ void enqueue_kernel(LayerView L, Dims d, DevCounters* C, int n, int tpw,
                               const int32_t* __restrict__ rows, const int32_t* __restrict__ slots,
                               const T* __restrict__ x, const int32_t* __restrict__ expert,
                               const float* __restrict__ w, const uint32_t* __restrict__ kmask,
                               const uint32_t* __restrict__ gens) {
  // launched as a programmatic dependent of the kernel before it (e.g. the previous collect):
  // wait for it, then let the scheduler start; the scheduler waits for this kernel
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  enqueue_warps<T>(L, d, C, n, tpw, rows, slots, x, expert, w, kmask, gens, gw, nwarps);
}

// -------------------------------------------------------------- scheduler
__global__ void __launch_bounds__(1024) schedule_kernel(LayerView L, Dims d, StepPlan* P,
                                                        DevCounters* C, moe_async_policy pol,
                                                        TileGeom g, int layer, int trace_cap,
                                                        int4* trace, long long weight_bytes_per_run,
                                                        int max_steps) {
  __shared__ PlanScratch sc;
  // launched as a programmatic dependent of the kernel before it (the last enqueue or
  // GEMM2): wait for it, then let GEMM1 start; GEMM1 waits for this plan
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  plan_layer(L, d, P, C, pol, g, layer, trace_cap, trace, weight_bytes_per_run, (int)C->steps + 1, true, sc,
             max_steps);
}

// ---------------------------------------------------------------- collect
// Copy ready rows (in completion order) to the caller, then reclaim each slot: clear its
// accepted mask and landing count and advance its generation, after the row was read.  G result
// rows' loads in flight per merged vector: 16 when a token has more than 8 results (one round
// trip for top-8 + the shared expert), else 8 (half the registers).  Measured on GB300 (pairs/s,
// same box): DeepSeek-wide layer 3.823 M -> 3.851 M with 16 (collect 0.140 -> 0.132 ms a pass);
// top-4 Zipf prefill 4.88 M -> 4.84 M with 16 (collect 0.138 -> 0.152 ms), hence 8 there.
template <typename T, int G>
__global__ void collect_kernel(LayerView L, Dims d, DevCounters* C, int max_out, T* __restrict__ y_out,
                               int32_t* __restrict__ slot_out, uint32_t* __restrict__ gen_out,
                               uint32_t* __restrict__ step_out, int32_t* __restrict__ n_io, int append,
                               int parts) {
  asm volatile("griddepcontrol.wait;" ::: "memory");   // launched as a dependent of GEMM2
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t rh = L.ready_ht[0], rt = L.ready_ht[1];
  const int base = append ? *n_io : 0;
  const int n = max(0, min((int)(rt - rh), max_out - base));
  for (int i = blockIdx.x; i < n; i += gridDim.x) {
    const int slot = L.ready[(rh + (uint32_t)i) % (uint32_t)d.S];
    if (kDebugBounds && (slot < 0 || slot >= d.S)) {             // bounds-checked build
      if (threadIdx.x == 0) set_error(C, MOE_ERR_BOUNDS);
      continue;
    }
    // the top-k merge of the ready token: y = sum_k w_k E_k(x) over its KS results, ascending k
    merge_row<T, G>(L, d, slot, y_out + (size_t)(base + i) * d.H, threadIdx.x, blockDim.x);
    for (int p = threadIdx.x; p < parts; p += blockDim.x) L.done_part[(size_t)slot * parts + p] = 0u;
    __syncthreads();
    if (threadIdx.x == 0) {
      slot_out[base + i] = slot;
      if (gen_out) gen_out[base + i] = L.gen[slot];
      if (step_out) step_out[base + i] = L.emit_step[slot];
      L.enq_mask[slot] = 0u;
      L.done[slot] = 0u;
      L.landed[slot] = 0u;
      L.emit_step[slot] = 0u;
      L.gen[slot] = L.gen[slot] + 1u;
    }
  }
  // the block that finishes last (every block has read the ring and the caller's count by
  // then) advances the ring head and writes the count
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&L.ready_ht[2], 1u) == gridDim.x - 1) {
      L.ready_ht[2] = 0u;
      L.ready_ht[0] = rh + (uint32_t)n;
      C->ready -= n;
      *n_io = base + n;
    }
  }
}

// ------------------------------------------------------------------ tick
// The control launch of a scheduling tick (moe_async_tick).  Blocks [0, n_enq) run the
// Receptor on the arriving wave while the others merge and copy out the tokens that were
// ready when the call was made (as collect_kernel does, with the same outputs).  The block
// that finishes last -- once every pair of the wave is accepted or rejected and every
// collected row has been read -- reclaims the collected slots and advances the ready ring;
// the scheduling kernel launched next plans the step.  Measured on GB300 against the three
// separate calls (pairs/s, same box): DeepSeek-wide layer 3.870 M vs 3.869 M, decode 194.5 K
// vs 194.2 K, Zipf prefill 4.86 M vs 4.90 M.  Planning in that last block instead was 0.5%
// slower on the DeepSeek-wide layer: it kept the step's GEMM1 CTAs, which each need an SM's
// whole shared memory, off the SMs until the whole launch had ended.
// Threads a block.  Measured on GB300 with the planner in the last block (pairs/s,
// DeepSeek-wide layer / Zipf prefill): 128 -- 3.62 M / 4.69 M; 256 -- 3.67 M / 4.71 M; 512 --
// 3.70 M / 4.71 M.
#ifndef MOE_TICK_THREADS
#define MOE_TICK_THREADS 512
#endif
constexpr int kTickThreads = MOE_TICK_THREADS;

template <typename T>
__global__ void __launch_bounds__(kTickThreads) tick_kernel(
    LayerView L, Dims d, DevCounters* C, int n, int tpw, int n_enq, const int32_t* __restrict__ rows,
    const int32_t* __restrict__ slots,
    const T* __restrict__ x, const int32_t* __restrict__ expert, const float* __restrict__ w,
    const uint32_t* __restrict__ kmask, const uint32_t* __restrict__ gens,
    int max_out, T* __restrict__ y_out, int32_t* __restrict__ slot_out, uint32_t* __restrict__ gen_out,
    uint32_t* __restrict__ step_out, int32_t* __restrict__ n_io, int append, int parts) {
  __shared__ int last;
  // a programmatic dependent of the previous step's GEMM2: wait for it, then let the
  // scheduling kernel start
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t rh = L.ready_ht[0], rt = L.ready_ht[1];
  const int base = (max_out > 0 && append) ? *n_io : 0;
  const int nc = max_out > 0 ? max(0, min((int)(rt - rh), max_out - base)) : 0;
  if ((int)blockIdx.x < n_enq) {
    const long long nwarps = (long long)n_enq * (blockDim.x >> 5);
    const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    enqueue_warps<T>(L, d, C, n, tpw, rows, slots, x, expert, w, kmask, gens, gw, nwarps);
  } else {
    const int cb = (int)blockIdx.x - n_enq, ncb = (int)gridDim.x - n_enq;
    for (int i = cb; i < nc; i += ncb) {
      const int slot = L.ready[(rh + (uint32_t)i) % (uint32_t)d.S];
      if (kDebugBounds && (slot < 0 || slot >= d.S)) {           // bounds-checked build
        if (threadIdx.x == 0) set_error(C, MOE_ERR_BOUNDS);
        continue;
      }
      merge_row<T, 8>(L, d, slot, y_out + (size_t)(base + i) * d.H, threadIdx.x, blockDim.x);
      if (threadIdx.x == 0) {
        slot_out[base + i] = slot;
        if (gen_out) gen_out[base + i] = L.gen[slot];
        if (step_out) step_out[base + i] = L.emit_step[slot];
      }
    }
  }
  // every thread's appends and reads are ordered before the block's arrival
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&L.ready_ht[2], 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int i = threadIdx.x; i < nc; i += blockDim.x) {             // reclaim the collected slots
    const int slot = L.ready[(rh + (uint32_t)i) % (uint32_t)d.S];
    if (kDebugBounds && (slot < 0 || slot >= d.S)) continue;
    for (int q = 0; q < parts; ++q) L.done_part[(size_t)slot * parts + q] = 0u;
    L.enq_mask[slot] = 0u;
    L.done[slot] = 0u;
    L.landed[slot] = 0u;
    L.emit_step[slot] = 0u;
    L.gen[slot] = L.gen[slot] + 1u;
  }
  if (threadIdx.x == 0) {
    L.ready_ht[2] = 0u;
    L.ready_ht[0] = rh + (uint32_t)nc;
    C->ready -= nc;
    if (max_out > 0) *n_io = base + nc;
  }
}

// ----------------------------------------------------------- cancellation
// Retire the current request of each listed slot ("asynchronous MoE serving" notes: an
// abandoned operation retires its buffer until a quiescent point; CascadeEP: readiness is
// tracked apart from reclamation).  A retired slot accepts no more pairs, is never merged
// or published, and is freed -- generation advanced -- when its last accepted result has
// landed (at once if none is queued).  Free slots and already merged ones are left alone.
__global__ void cancel_kernel(LayerView L, Dims d, DevCounters* C, int n, const int32_t* __restrict__ slots,
                              int parts) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int slot = slots[i];
    if (slot < 0 || slot >= d.S) { set_error(C, MOE_ERR_INVALID); continue; }
    if (L.done[slot] == (uint32_t)parts) continue;              // merged already: too late
    uint32_t old = L.enq_mask[slot];
    bool mine = false;
    while (old != 0u && !(old & kRetired)) {                      // duplicates in the list: one wins
      const uint32_t prev = atomicCAS(&L.enq_mask[slot], old, old | kRetired);
      if (prev == old) { mine = true; break; }
      old = prev;
    }
    if (!mine) continue;
    atomicSub(&C->open_tokens, 1);
    atomicAdd(&C->cancelled, 1ull);
    if (retired_quiescent(old | kRetired, L.landed[slot], parts)) reclaim_slot(L, parts, slot);
  }
}

// Bounds-checked build only: append a raw record to bucket b (a test plants an out-of-range
// record this way and checks that the kernels reject it).
__global__ void debug_append_kernel(LayerView L, Dims d, DevCounters* C, int b, int32_t rec) {
  const uint32_t pos = L.tail[b];
  if (pos - L.head[b] >= (uint32_t)d.cap) {
    set_error(C, MOE_ERR_CAPACITY);
    return;
  }
  L.records[(size_t)b * d.cap + (pos % (uint32_t)d.cap)] = rec;
  L.tail[b] = pos + 1u;
  C->pending_pairs += 1;
}

// -------------------------------------------------------------- utilities

// Launch as a programmatic dependent of the previous kernel in the stream: the kernel may
// start before that one finishes and orders itself with griddepcontrol.wait.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Collect CTAs per SM (each merges whole tokens, 256 threads): fewer blocks end sooner (each
// takes part in the last-block count); measured (collect ms per pass, Zipf prefill /
// DeepSeek-wide layer): 8 -- 0.160 / 0.197, 4 -- 0.148 / 0.196, 2 -- 0.139 / 0.196, 1 --
// 0.169 / 0.271.
#ifndef MOE_COLLECT_CTAS_PER_SM
#define MOE_COLLECT_CTAS_PER_SM 2
#endif
constexpr int kCollectCtasPerSm = MOE_COLLECT_CTAS_PER_SM;

// Receptor tokens per warp: one while the wave fits in one round of 16 warps per SM (each warp
// then copies one row), more for large waves; whole tokens per warp, tpw * KS <= 32.
int enqueue_tpw(const moe_async_s* h, long long n) {
  const int tpw_max = 32 / h->dims.KS;
  const long long warps_one_round = (long long)h->num_sms * 16;
  return (int)std::min<long long>(tpw_max, std::max<long long>(1, (n + warps_one_round - 1) / warps_one_round));
}

bool valid_policy(const moe_async_policy* policy, int max_steps) {
  if (!policy || max_steps < 1) return false;
  if (policy->kind != MOE_POLICY_MTFS && policy->kind != MOE_POLICY_THRESHOLD && policy->kind != MOE_POLICY_RANKS)
    return false;
  if (policy->max_groups < 0 || policy->min_batch < 0 || policy->fallback_groups < 0) return false;
  if (policy->kind == MOE_POLICY_RANKS && policy->max_groups < 1) return false;
  return true;
}

bool valid_stream_layer(moe_async_t h, int layer) {
  return h && layer >= 0 && layer < h->cfg.num_layers;
}

size_t elem_size(int dtype) { return dtype == MOE_BF16 ? 2 : 4; }

void prof_free(moe_async_s* h);

void free_handle(moe_async_s* h) {
  if (!h) return;
  prof_free(h);
  if (h->stream_state) stream_teardown(h);
  if (h->tc_state) tc_teardown(h);
  if (h->layers) {
    for (int l = 0; l < h->cfg.num_layers; ++l) {
      LayerView& L = h->layers[l];
      void* ptrs[] = {L.pool, L.wtab, L.enq_mask, L.done, L.done_part, L.landed, L.gen, L.emit_step, L.slotbuf, L.y,
                      L.records,
                      L.head, L.tail, L.ready, L.ready_ht, const_cast<void*>(L.w13),
                      const_cast<void*>(L.w2)};
      for (void* p : ptrs) if (p) cudaFree(p);
    }
    delete[] h->layers;
  }
  if (h->plan) cudaFree(h->plan);
  if (h->h) cudaFree(h->h);
  if (h->counters) cudaFree(h->counters);
  if (h->trace) cudaFree(h->trace);
  if (h->host_counters) cudaFreeHost(h->host_counters);
  delete h;
}

template <typename P>
cudaError_t dalloc(P** p, size_t bytes) {
  void* q = nullptr;
  cudaError_t e = cudaMalloc(&q, bytes ? bytes : 16);
  *p = static_cast<P*>(q);
  return e;
}

moe_status read_counters(moe_async_t h, cudaStream_t s) {
  MOE_CUDA_TRY(cudaMemcpyAsync(h->host_counters, h->counters, sizeof(DevCounters),
                               cudaMemcpyDeviceToHost, s));
  MOE_CUDA_TRY(cudaStreamSynchronize(s));
  return MOE_OK;
}

struct ProfState {
  static constexpr int kCap = 65536;
  bool on = false;
  int n = 0;
  cudaEvent_t ev[2 * kCap];
  int kind[kCap];
  int created = 0;                 // events created so far (lazily)
};

void prof_free(moe_async_s* h) {
  ProfState* p = static_cast<ProfState*>(h->prof);
  if (!p) return;
  for (int i = 0; i < p->created; ++i) cudaEventDestroy(p->ev[i]);
  delete p;
  h->prof = nullptr;
}

}  // namespace

namespace moe {

void prof_begin(moe_async_s* h, int kind, cudaStream_t s) {
  h->launches += 1;
  ProfState* p = static_cast<ProfState*>(h->prof);
  if (!p || !p->on || p->n >= ProfState::kCap) return;
  const int i = p->n;
  while (p->created < 2 * i + 2) {
    if (cudaEventCreate(&p->ev[p->created]) != cudaSuccess) { p->on = false; return; }
    ++p->created;
  }
  p->kind[i] = kind;
  cudaEventRecord(p->ev[2 * i], s);
}

void prof_end(moe_async_s* h, int kind, cudaStream_t s) {
  (void)kind;
  ProfState* p = static_cast<ProfState*>(h->prof);
  if (!p || !p->on || p->n >= ProfState::kCap) return;
  if (p->created < 2 * p->n + 2) return;
  cudaEventRecord(p->ev[2 * p->n + 1], s);
  p->n += 1;
}

}  // namespace moe

// ====================================================================== C ABI

extern "C" {

int32_t moe_async_host_writable(const void* p, int64_t n) {
  if (!p || n < 0) return 0;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();                          // an unregistered pointer: clear, answer no
    return 0;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer != p) return 0;
  cudaPointerAttributes b;                       // the last byte lies in the same allocation
  if (n > 0 && (cudaPointerGetAttributes(&b, static_cast<const char*>(p) + (n - 1)) != cudaSuccess ||
                b.type != cudaMemoryTypeHost)) {
    cudaGetLastError();
    return 0;
  }
  return 1;
}

const char* moe_async_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID: return "invalid argument";
    case MOE_ERR_CAPACITY: return "capacity exceeded";
    case MOE_ERR_DUPLICATE: return "duplicate pair";
    case MOE_ERR_STALE: return "stale slot generation";
    case MOE_ERR_TIMEOUT: return "timeout: tokens still open";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_BOUNDS: return "index out of range (bounds-checked build)";
  }
  return "unknown status";
}

moe_status moe_async_create(const moe_async_config* cfg, const void* const* w1,
                            const void* const* w3, const void* const* w2,
                            const void* const* sw1, const void* const* sw3,
                            const void* const* sw2, void* stream, moe_async_t* out) {
  if (!cfg || !out) return MOE_ERR_INVALID;
  const moe_async_config c = *cfg;
  if (c.num_layers < 1 || c.num_experts < 1 || c.num_experts > kMaxExperts || c.top_k < 1 ||
      c.top_k > c.num_experts || c.top_k + (c.has_shared ? 1 : 0) > 31 || c.hidden < 8 ||
      c.hidden % 8 || c.inter < 16 || c.inter % 16 || c.max_slots < 1 ||
      c.max_slots > (1 << 25) || c.bucket_capacity < 0 ||
      (c.dtype != MOE_F32 && c.dtype != MOE_BF16) ||
      (c.expert_kind != MOE_EXPERT_SWIGLU && c.expert_kind != MOE_EXPERT_IDENTITY) ||
      c.trace_capacity < 0)
    return MOE_ERR_INVALID;
  const bool swiglu = c.expert_kind == MOE_EXPERT_SWIGLU;
  if (swiglu && (!w1 || !w3 || !w2)) return MOE_ERR_INVALID;
  if (swiglu && c.has_shared && (!sw1 || !sw3 || !sw2)) return MOE_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  moe_async_s* h = new (std::nothrow) moe_async_s();
  if (!h) return MOE_ERR_CUDA;
  std::memset(static_cast<void*>(h), 0, sizeof(*h));
  h->cfg = c;
  Dims& d = h->dims;
  d.E = c.num_experts;
  d.K = c.top_k;
  d.KS = c.top_k + (c.has_shared ? 1 : 0);
  d.NB = c.num_experts + (c.has_shared ? 1 : 0);
  d.H = c.hidden;
  d.I = c.inter;
  d.S = c.max_slots;
  d.cap = c.bucket_capacity > 0 ? c.bucket_capacity : c.max_slots;
  d.dtype = c.dtype;
  d.has_shared = c.has_shared ? 1 : 0;
  d.expert_kind = c.expert_kind;
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
    free_handle(h);
    return MOE_ERR_CUDA;
  }
  h->use_tc = swiglu && c.dtype == MOE_BF16;
  h->geom = h->use_tc ? tc_geom() : simt_geom();
  if (!swiglu) h->geom = TileGeom{16, 2 * c.inter, 16, c.hidden, 0, 0, 0};
  h->parts_per_pair = (d.H + h->geom.bm2 - 1) / h->geom.bm2;

  const size_t es = elem_size(c.dtype);
  const size_t S = (size_t)d.S, H = (size_t)d.H, I = (size_t)d.I, KS = (size_t)d.KS;
  h->layers = new (std::nothrow) LayerView[c.num_layers];
  if (!h->layers) { free_handle(h); return MOE_ERR_CUDA; }
  std::memset(static_cast<void*>(h->layers), 0, sizeof(LayerView) * c.num_layers);
  bool ok = true;
  for (int l = 0; l < c.num_layers && ok; ++l) {
    LayerView& L = h->layers[l];
    ok = ok && dalloc(&L.pool, S * H * es) == cudaSuccess;
    ok = ok && dalloc(&L.wtab, S * KS * 4) == cudaSuccess;
    ok = ok && dalloc(&L.enq_mask, S * 4) == cudaSuccess;
    ok = ok && dalloc(&L.done, S * 4) == cudaSuccess;
    ok = ok && dalloc(&L.done_part, S * (size_t)h->parts_per_pair * 4) == cudaSuccess;
    ok = ok && dalloc(&L.landed, S * 4) == cudaSuccess;
    ok = ok && dalloc(&L.gen, S * 4) == cudaSuccess;
    ok = ok && dalloc(&L.emit_step, S * 4) == cudaSuccess;
    ok = ok && dalloc(&L.slotbuf, S * KS * H * es) == cudaSuccess;   // result rows in the layer dtype
    ok = ok && dalloc(&L.y, S * H * es) == cudaSuccess;
    ok = ok && dalloc(&L.records, (size_t)d.NB * d.cap * 4) == cudaSuccess;
    ok = ok && dalloc(&L.head, (size_t)d.NB * 4) == cudaSuccess;
    ok = ok && dalloc(&L.tail, (size_t)d.NB * 4) == cudaSuccess;
    ok = ok && dalloc(&L.ready, S * 4) == cudaSuccess;
    ok = ok && dalloc(&L.ready_ht, 4 * 4) == cudaSuccess;
    if (ok && swiglu) {
      void* p13 = nullptr;
      void* p2 = nullptr;
      ok = ok && dalloc(&p13, (size_t)d.NB * 2 * I * H * es) == cudaSuccess;
      L.w13 = p13;
      ok = ok && dalloc(&p2, (size_t)d.NB * H * I * es) == cudaSuccess;
      L.w2 = p2;
      h->packed_bytes += (int64_t)((size_t)d.NB * 3 * I * H * es);
    }
    if (ok) {
      ok = cudaMemsetAsync(L.enq_mask, 0, S * 4, s) == cudaSuccess &&
           cudaMemsetAsync(L.done, 0, S * 4, s) == cudaSuccess &&
           cudaMemsetAsync(L.done_part, 0, S * (size_t)h->parts_per_pair * 4, s) == cudaSuccess &&
           cudaMemsetAsync(L.landed, 0, S * 4, s) == cudaSuccess &&
           cudaMemsetAsync(L.gen, 0, S * 4, s) == cudaSuccess &&
           cudaMemsetAsync(L.emit_step, 0, S * 4, s) == cudaSuccess &&
           cudaMemsetAsync(L.head, 0, (size_t)d.NB * 4, s) == cudaSuccess &&
           cudaMemsetAsync(L.tail, 0, (size_t)d.NB * 4, s) == cudaSuccess &&
           cudaMemsetAsync(L.ready_ht, 0, 16, s) == cudaSuccess &&
           cudaMemsetAsync(L.records, 0, (size_t)d.NB * d.cap * 4, s) == cudaSuccess &&
           cudaMemsetAsync(L.slotbuf, 0, S * KS * H * es, s) == cudaSuccess;
    }
    if (ok && swiglu) {
      // W1 [E,H,I] -> packed rows 32*(i/16) + i%16 ; W3 -> same + 16 ; W2 [E,I,H] -> [E,H,I]
      void* p13 = const_cast<void*>(L.w13);
      void* p2 = const_cast<void*>(L.w2);
      const int E = d.E, Hh = d.H, Ii = d.I;
      auto pk = [&](const void* in, void* outp, int nexp, int C, int R, int orows, int il, int which) {
        return c.dtype == MOE_BF16
                   ? pack_one<__nv_bfloat16>(in, outp, nexp, C, R, orows, il, which, s)
                   : pack_one<float>(in, outp, nexp, C, R, orows, il, which, s);
      };
      ok = ok && pk(w1[l], p13, E, Hh, Ii, 2 * Ii, 1, 0) == cudaSuccess;
      ok = ok && pk(w3[l], p13, E, Hh, Ii, 2 * Ii, 1, 1) == cudaSuccess;
      ok = ok && pk(w2[l], p2, E, Ii, Hh, Hh, 0, 0) == cudaSuccess;
      if (ok && c.has_shared) {
        char* s13 = static_cast<char*>(p13) + (size_t)E * 2 * I * H * es;
        char* s2 = static_cast<char*>(p2) + (size_t)E * H * I * es;
        ok = ok && pk(sw1[l], s13, 1, Hh, Ii, 2 * Ii, 1, 0) == cudaSuccess;
        ok = ok && pk(sw3[l], s13, 1, Hh, Ii, 2 * Ii, 1, 1) == cudaSuccess;
        ok = ok && pk(sw2[l], s2, 1, Ii, Hh, Hh, 0, 0) == cudaSuccess;
      }
    }
  }
  ok = ok && dalloc(&h->plan, sizeof(StepPlan)) == cudaSuccess;
  ok = ok && dalloc(&h->h, S * KS * I * es) == cudaSuccess;
  ok = ok && dalloc(&h->counters, sizeof(DevCounters)) == cudaSuccess;
  ok = ok && cudaMemsetAsync(h->plan, 0, sizeof(StepPlan), s) == cudaSuccess;
  ok = ok && cudaMemsetAsync(h->counters, 0, sizeof(DevCounters), s) == cudaSuccess;
  if (ok && c.trace_capacity > 0) ok = dalloc(&h->trace, (size_t)c.trace_capacity * sizeof(int4)) == cudaSuccess;
  if (ok) ok = cudaMallocHost(reinterpret_cast<void**>(&h->host_counters), sizeof(DevCounters)) == cudaSuccess;
  if (!ok) { cudaStreamSynchronize(s); free_handle(h); return MOE_ERR_CUDA; }
  if (h->use_tc) {
    moe_status st = tc_setup(h);
    if (st != MOE_OK) { cudaStreamSynchronize(s); free_handle(h); return st; }
  }
  if (cudaStreamSynchronize(s) != cudaSuccess) { free_handle(h); return MOE_ERR_CUDA; }
  *out = h;
  return MOE_OK;
}

moe_status moe_async_route(const float* d_logits, int32_t T, int32_t E, int32_t K, int32_t* d_idx,
                           float* d_w, void* stream) {
  if (T < 0 || E < 1 || E > kMaxExperts || K < 1 || K > E || K > 32) return MOE_ERR_INVALID;
  if (T == 0) return MOE_OK;
  if (!d_logits || !d_idx || !d_w) return MOE_ERR_INVALID;
  const int wpb = 8;
  route_kernel<<<(T + wpb - 1) / wpb, 32 * wpb, 0, static_cast<cudaStream_t>(stream)>>>(d_logits, T, E, K, d_idx, d_w);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_async_enqueue(moe_async_t h, int32_t layer, int32_t n, const int32_t* d_rows,
                             const int32_t* d_slot, const void* d_x, const int32_t* d_expert,
                             const float* d_w, const uint32_t* d_kmask, const uint32_t* d_gen,
                             void* stream) {
  if (!valid_stream_layer(h, layer) || n < 0) return MOE_ERR_INVALID;
  if (n == 0) return MOE_OK;
  if (!d_x || !d_expert || !d_w) return MOE_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(d_x) % 16) return MOE_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Dims& d = h->dims;
  const int tpw = enqueue_tpw(h, n);
  // two warps a block, so a wave of a few hundred tokens spreads over every SM
  const long long warps = (n + tpw - 1) / tpw;
  const int grid = (int)std::max<long long>(1, std::min<long long>((warps + 1) / 2, (long long)h->num_sms * 32));
  prof_begin(h, MOE_KERNEL_ENQUEUE, s);
  cudaError_t e;
  if (d.dtype == MOE_BF16)
    e = launch_dependent(enqueue_kernel<__nv_bfloat16>, dim3(grid), dim3(64), s, h->layers[layer], d, h->counters,
                         (int)n, tpw, d_rows, d_slot, static_cast<const __nv_bfloat16*>(d_x), d_expert, d_w, d_kmask,
                         d_gen);
  else
    e = launch_dependent(enqueue_kernel<float>, dim3(grid), dim3(64), s, h->layers[layer], d, h->counters, (int)n,
                         tpw, d_rows, d_slot, static_cast<const float*>(d_x), d_expert, d_w, d_kmask, d_gen);
  prof_end(h, MOE_KERNEL_ENQUEUE, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

static moe_status launch_ffn(moe_async_t h, int32_t layer, cudaStream_t s) {
  if (h->cfg.expert_kind == MOE_EXPERT_IDENTITY) return launch_identity(h, layer, s);
  if (h->use_tc) return launch_ffn_tc(h, layer, s);
  return launch_ffn_simt(h, layer, s);
}

moe_status schedule_impl(moe_async_t h, int32_t layer, const moe_async_policy* policy, int32_t max_steps,
                         void* stream) {
  if (!valid_stream_layer(h, layer) || !valid_policy(policy, max_steps)) return MOE_ERR_INVALID;
  if (policy->kind == MOE_POLICY_RANKS && max_steps > 1) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Dims& d = h->dims;
  const long long wbytes = h->cfg.expert_kind == MOE_EXPERT_SWIGLU
                               ? 3ll * d.H * d.I * (long long)elem_size(d.dtype) : 0ll;
  prof_begin(h, MOE_KERNEL_SCHEDULE, s);
  const cudaError_t e = launch_dependent(schedule_kernel, dim3(1), dim3(1024), s, h->layers[layer], d, h->plan,
                                         h->counters, *policy, h->geom, (int)layer, (int)h->cfg.trace_capacity,
                                         h->trace, wbytes, (int)max_steps);
  prof_end(h, MOE_KERNEL_SCHEDULE, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return launch_ffn(h, layer, s);
}

moe_status moe_async_schedule_step(moe_async_t h, int32_t layer, const moe_async_policy* policy,
                                   void* stream) {
  return schedule_impl(h, layer, policy, 1, stream);
}

moe_status moe_async_schedule_steps(moe_async_t h, int32_t layer, const moe_async_policy* policy,
                                    int32_t max_steps, void* stream) {
  return schedule_impl(h, layer, policy, max_steps, stream);
}

moe_status moe_async_tick(moe_async_t h, int32_t layer, int32_t n, const int32_t* d_rows, const int32_t* d_slot,
                          const void* d_x, const int32_t* d_expert, const float* d_w, const uint32_t* d_kmask,
                          const uint32_t* d_gen, const moe_async_policy* policy, int32_t max_out, void* d_y_out,
                          int32_t* d_slot_out, uint32_t* d_gen_out, uint32_t* d_step_out, int32_t* d_n_out,
                          int32_t append, void* stream) {
  if (!valid_stream_layer(h, layer) || n < 0 || max_out < 0 || !valid_policy(policy, 1)) return MOE_ERR_INVALID;
  if (n > 0 && (!d_x || !d_expert || !d_w || reinterpret_cast<uintptr_t>(d_x) % 16)) return MOE_ERR_INVALID;
  if (max_out > 0 && (!d_y_out || !d_slot_out || !d_n_out || reinterpret_cast<uintptr_t>(d_y_out) % 16))
    return MOE_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Dims& d = h->dims;
  const int tpw = n > 0 ? enqueue_tpw(h, n) : 1;
  const long long warps = n > 0 ? ((long long)n + tpw - 1) / tpw : 0;
  const int per_block = kTickThreads / 32;
  const int n_enq = (int)std::min<long long>((warps + per_block - 1) / per_block, (long long)h->num_sms * 8);
  // every block resident at once (512 threads an SM): the last one to finish reclaims the
  // collected slots, so a second round of blocks would delay it
  const int resident = h->num_sms * (512 / kTickThreads);
  const int n_col = max_out > 0 ? std::max(1, std::min(max_out, resident - n_enq)) : 0;
  const int grid = std::max(1, n_enq + n_col);
  prof_begin(h, MOE_KERNEL_TICK, s);
  cudaError_t e;
  if (d.dtype == MOE_BF16)
    e = launch_dependent(tick_kernel<__nv_bfloat16>, dim3(grid), dim3(kTickThreads), s, h->layers[layer], d,
                         h->counters, (int)n, tpw, n_enq, d_rows, d_slot, static_cast<const __nv_bfloat16*>(d_x),
                         d_expert, d_w, d_kmask, d_gen, (int)max_out, static_cast<__nv_bfloat16*>(d_y_out), d_slot_out,
                         d_gen_out, d_step_out, d_n_out, (int)append, h->parts_per_pair);
  else
    e = launch_dependent(tick_kernel<float>, dim3(grid), dim3(kTickThreads), s, h->layers[layer], d, h->counters,
                         (int)n, tpw, n_enq, d_rows, d_slot, static_cast<const float*>(d_x), d_expert, d_w, d_kmask,
                         d_gen, (int)max_out, static_cast<float*>(d_y_out), d_slot_out, d_gen_out, d_step_out, d_n_out,
                         (int)append, h->parts_per_pair);
  prof_end(h, MOE_KERNEL_TICK, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return schedule_impl(h, layer, policy, 1, stream);   // the step: plan, GEMM1, GEMM2
}

moe_status moe_async_collect(moe_async_t h, int32_t layer, int32_t max_out, void* d_y_out,
                             int32_t* d_slot_out, uint32_t* d_gen_out, uint32_t* d_step_out,
                             int32_t* d_n_out, int32_t append, void* stream) {
  if (!valid_stream_layer(h, layer) || max_out < 0 || !d_n_out) return MOE_ERR_INVALID;
  if (max_out > 0 && (!d_y_out || !d_slot_out)) return MOE_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(d_y_out) % 16) return MOE_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Dims& d = h->dims;
  const int grid = std::max(1, std::min(max_out, h->num_sms * kCollectCtasPerSm));
  prof_begin(h, MOE_KERNEL_COLLECT, s);
  cudaError_t e;
  const bool wide = d.KS > 8;
  if (d.dtype == MOE_BF16)
    e = launch_dependent(wide ? collect_kernel<__nv_bfloat16, 16> : collect_kernel<__nv_bfloat16, 8>, dim3(grid),
                         dim3(256), s, h->layers[layer], d, h->counters, (int)max_out,
                         static_cast<__nv_bfloat16*>(d_y_out), d_slot_out, d_gen_out, d_step_out, d_n_out,
                         (int)append, h->parts_per_pair);
  else
    e = launch_dependent(wide ? collect_kernel<float, 16> : collect_kernel<float, 8>, dim3(grid), dim3(256), s,
                         h->layers[layer], d, h->counters, (int)max_out, static_cast<float*>(d_y_out), d_slot_out,
                         d_gen_out, d_step_out, d_n_out, (int)append, h->parts_per_pair);
  prof_end(h, MOE_KERNEL_COLLECT, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_async_sync(moe_async_t h, void* stream) {
  if (!h) return MOE_ERR_INVALID;
  moe_status st = read_counters(h, static_cast<cudaStream_t>(stream));
  if (st != MOE_OK) return st;
  return static_cast<moe_status>(h->host_counters->error);
}

// Steps the layer's queues need at least before they are empty, when nothing new arrives:
// every step drains its picks whole, and takes at most max_groups (MTFS), R (RANKS) or, once
// no bucket reaches min_batch, fallback_groups (THRESHOLD) buckets.  0 = no useful bound.
int drain_steps_lower_bound(const DevCounters& c, int layer, const moe_async_policy& pol) {
  if (c.plan_layer != layer || c.nonempty_left <= 0) return 0;
  int per_step = 0;
  if (pol.kind == MOE_POLICY_MTFS) per_step = pol.max_groups;
  else if (pol.kind == MOE_POLICY_RANKS) per_step = pol.max_groups;
  else if (pol.kind == MOE_POLICY_THRESHOLD && c.elig_left == 0)
    per_step = pol.fallback_groups > 0 ? pol.fallback_groups : 1;
  return per_step > 0 ? (c.nonempty_left + per_step - 1) / per_step : 0;
}

moe_status moe_async_wait(moe_async_t h, int32_t layer, const moe_async_policy* policy,
                          int32_t max_steps, int32_t check_every, void* stream) {
  if (!valid_stream_layer(h, layer) || !policy || max_steps < 0) return MOE_ERR_INVALID;
  if (check_every < 1) check_every = 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // MTFS and THRESHOLD drains run as one plan of consecutive steps while buckets are left
  // (nothing arrives during the wait, so the picks are those of single steps); once the
  // queues are empty and tokens are still open (a pair that has not arrived), or under
  // RANKS, single steps are run, check_every (or the steps the queues certainly need) at a time
  const bool fusable = policy->kind == MOE_POLICY_MTFS || policy->kind == MOE_POLICY_THRESHOLD;
  int64_t steps = 0;
  unsigned long long seen = 0;
  for (int iter = 0;; ++iter) {
    moe_status st = read_counters(h, s);
    if (st != MOE_OK) return st;
    const DevCounters& c = *h->host_counters;
    if (iter > 0) steps += (int64_t)(c.steps - seen);
    seen = c.steps;
    if (c.error) return static_cast<moe_status>(c.error);
    if (c.open_tokens == 0) return MOE_OK;
    if (steps >= max_steps) return MOE_ERR_TIMEOUT;
    const int64_t left = (int64_t)max_steps - steps;
    // the first plan is always tried (it counts no step if the queues are empty); later ones
    // only while the last plan of this layer left buckets behind
    const bool queues_left = iter == 0 || (c.plan_layer == layer && c.nonempty_left > 0);
    if (fusable && queues_left) {
      st = schedule_impl(h, layer, policy, (int32_t)left, stream);
      if (st != MOE_OK) return st;
      continue;
    }
    // run as many steps as the queues certainly need before reading the counters again
    // (fewer host round trips in long drains), else check_every
    const int need = drain_steps_lower_bound(c, layer, *policy);
    const int64_t batch = std::min<int64_t>(need > 0 ? need : check_every, left);
    for (int64_t i = 0; i < batch; ++i) {
      st = moe_async_schedule_step(h, layer, policy, stream);
      if (st != MOE_OK) return st;
    }
  }
}

moe_status moe_async_get_stats(moe_async_t h, void* stream, moe_async_stats* out) {
  if (!h || !out) return MOE_ERR_INVALID;
  moe_status st = read_counters(h, static_cast<cudaStream_t>(stream));
  if (st != MOE_OK) return st;
  const DevCounters& c = *h->host_counters;
  out->steps = (int64_t)c.steps;
  out->pairs_executed = (int64_t)c.pairs_executed;
  out->expert_runs = (int64_t)c.expert_runs;
  out->weight_bytes = (int64_t)c.weight_bytes;
  out->tokens_combined = (int64_t)c.tokens_combined;
  out->duplicates = (int64_t)c.duplicates;
  out->stale = (int64_t)c.stale;
  out->cancelled = (int64_t)c.cancelled;
  out->open_tokens = c.open_tokens;
  out->pending_pairs = c.pending_pairs;
  out->ready = c.ready;
  out->error = (int32_t)c.error;
  out->packed_weight_bytes = h->packed_bytes;
  out->kernel_launches = h->launches;
  return MOE_OK;
}

moe_status moe_async_profile(moe_async_t h, int32_t enable) {
  if (!h) return MOE_ERR_INVALID;
  ProfState* p = static_cast<ProfState*>(h->prof);
  if (enable && !p) {
    p = new (std::nothrow) ProfState();
    if (!p) return MOE_ERR_CUDA;
    h->prof = p;
  }
  if (p) p->on = enable != 0;
  return MOE_OK;
}

moe_status moe_async_profile_read(moe_async_t h, void* stream, double* h_ms, int64_t* h_launches,
                                  int32_t n_kinds) {
  if (!h || n_kinds < 0 || (n_kinds > 0 && (!h_ms || !h_launches))) return MOE_ERR_INVALID;
  MOE_CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  ProfState* p = static_cast<ProfState*>(h->prof);
  if (!p) return MOE_OK;
  for (int i = 0; i < p->n; ++i) {
    const int k = p->kind[i];
    if (k < 0 || k >= n_kinds) continue;
    float ms = 0.f;
    MOE_CUDA_TRY(cudaEventElapsedTime(&ms, p->ev[2 * i], p->ev[2 * i + 1]));
    h_ms[k] += ms;
    h_launches[k] += 1;
  }
  p->n = 0;
  return MOE_OK;
}

moe_status moe_async_get_trace(moe_async_t h, void* stream, int32_t* h_buf, int32_t cap, int32_t* h_n) {
  if (!h || !h_n || cap < 0 || (cap > 0 && !h_buf)) return MOE_ERR_INVALID;
  moe_status st = read_counters(h, static_cast<cudaStream_t>(stream));
  if (st != MOE_OK) return st;
  int n = std::min(h->host_counters->trace_n, h->cfg.trace_capacity);
  n = std::min(n, cap);
  if (n > 0) MOE_CUDA_TRY(cudaMemcpy(h_buf, h->trace, (size_t)n * sizeof(int4), cudaMemcpyDeviceToHost));
  *h_n = n;
  return MOE_OK;
}

moe_status moe_async_snapshot(moe_async_t h, int32_t layer, void* stream, int32_t* h_depth,
                              int32_t* h_records, int32_t cap, int32_t* h_n) {
  if (!valid_stream_layer(h, layer) || !h_depth || !h_n || cap < 0 || (cap > 0 && !h_records))
    return MOE_ERR_INVALID;
  MOE_CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  const Dims& d = h->dims;
  const LayerView& L = h->layers[layer];
  uint32_t* head = static_cast<uint32_t*>(std::malloc((size_t)d.NB * 4));
  uint32_t* tail = static_cast<uint32_t*>(std::malloc((size_t)d.NB * 4));
  int32_t* recs = static_cast<int32_t*>(std::malloc((size_t)d.NB * d.cap * 4));
  moe_status st = MOE_OK;
  if (!head || !tail || !recs) st = MOE_ERR_CUDA;
  if (st == MOE_OK && (cudaMemcpy(head, L.head, (size_t)d.NB * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
                       cudaMemcpy(tail, L.tail, (size_t)d.NB * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
                       cudaMemcpy(recs, L.records, (size_t)d.NB * d.cap * 4, cudaMemcpyDeviceToHost) != cudaSuccess))
    st = MOE_ERR_CUDA;
  int n = 0;
  if (st == MOE_OK) {
    for (int b = 0; b < d.NB; ++b) {
      const uint32_t dep = tail[b] - head[b];
      h_depth[b] = (int32_t)dep;
      for (uint32_t j = 0; j < dep && j < (uint32_t)d.cap; ++j) {
        if (n >= cap) { st = MOE_ERR_CAPACITY; break; }
        const int32_t r = recs[(size_t)b * d.cap + ((head[b] + j) % (uint32_t)d.cap)];
        h_records[2 * n] = r >> kKShift;
        h_records[2 * n + 1] = r & kKMask;
        ++n;
      }
    }
  }
  *h_n = n;
  std::free(head);
  std::free(tail);
  std::free(recs);
  return st;
}

moe_status moe_async_cancel(moe_async_t h, int32_t layer, int32_t n, const int32_t* d_slots, void* stream) {
  if (!valid_stream_layer(h, layer) || n < 0) return MOE_ERR_INVALID;
  if (h->stream_state) return MOE_ERR_UNSUPPORTED;
  if (n == 0) return MOE_OK;
  if (!d_slots) return MOE_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  prof_begin(h, MOE_KERNEL_ENQUEUE, s);
  cancel_kernel<<<(n + 255) / 256, 256, 0, s>>>(h->layers[layer], h->dims, h->counters, n, d_slots,
                                                h->parts_per_pair);
  prof_end(h, MOE_KERNEL_ENQUEUE, s);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_async_debug_append_record(moe_async_t h, int32_t layer, int32_t bucket, int32_t record,
                                        void* stream) {
  if (!kDebugBounds) return MOE_ERR_UNSUPPORTED;          // release builds: no raw record writes
  if (!valid_stream_layer(h, layer) || bucket < 0 || bucket >= h->dims.NB) return MOE_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  debug_append_kernel<<<1, 1, 0, s>>>(h->layers[layer], h->dims, h->counters, (int)bucket, record);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_async_destroy(moe_async_t h, void* stream) {
  if (!h) return MOE_ERR_INVALID;
  cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  free_handle(h);
  return MOE_OK;
}

}  // extern "C"
