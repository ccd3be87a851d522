// Streaming multi-layer decode on the 2L micro-queues, resident on the device.
//
// "SOSP'26 StreamEP" section 3: every layer has an attention queue and an expert queue; a
// request's token is served by its layer's attention stage, routed (top-K), dispatched to
// the expert queue, merged back on its home, and enters the next layer's attention queue;
// layers advance per request with no global barrier.  Section 4: the scheduler serves the
// queue holding the most tokens (MTFS).
//
// One tick = one scheduling decision, executed by a fixed sequence of kernels that a CUDA
// graph replays every tick (no host round trip):
//   stream_tick_kernel  (1 CTA)  stop check, tick++, deliver the dispatches due this tick
//                                into their layer's per-expert buckets, pick one of the 2L
//                                queues (most tokens; tie -> lower layer, attention before
//                                expert; attention queues closed once `stop` merges are
//                                done), then plan it: an attention batch, or the layer's
//                                bucket work list (every non-empty bucket)
//   att_prep_kernel              per batch row: its state row x^(n) and RMSNorm scale
//   ffn_tc_kernel<ATT>           a = s * (x P_l) on tcgen05 -> the layer's token pool
//   att_route_kernel             top-K of the (request, step) logits; dispatch: arrival tick
//                                = now + delay(request, step)
//   ffn_tc_kernel<GEMM1/GEMM2>   the expert FFN; each completed merge advances its request
//                                (history row, done tick) and queues its next attention
// Kernels whose queue was not picked exit at once.
#include <algorithm>
#include <cstring>
#include <new>
#include "moe_plan.cuh"

namespace moe {
namespace {

constexpr int kStreamTraceCap = 1 << 18;

struct StreamState {
  StreamDev sd;
  moe_stream_config cfg;
  int4* trace;                     // (tick, kind, layer, count)
  int32_t* trace_n;
  void* proj_packed[kMaxLayers];
  cudaStream_t cap_stream;
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  StreamCtl* host_ctl;             // pinned
};

struct TickArgs {
  StreamDev sd;
  LayerView views[kMaxLayers];
  Dims d;
  DevCounters* C;
  StepPlan* P;
  TileGeom g;
  int4* trace;
  int32_t* trace_n;
  long long wbytes;
};

__global__ void __launch_bounds__(1024) stream_tick_kernel(const __grid_constant__ TickArgs a) {
  __shared__ PlanScratch sc;
  __shared__ int s_kind, s_layer, s_busy, s_tick;
  const StreamDev& sd = a.sd;
  StreamCtl* ctl = sd.ctl;
  const int tid = threadIdx.x;
  const int Lc = sd.L;
  if (tid == 0) {
    int busy = ctl->in_transit > 0;
    const bool allow_att = ctl->combined < sd.stop;
    for (int l = 0; l < Lc; ++l) {
      if (ctl->exp_tokens[l] > 0) busy = 1;
      if (allow_att && sd.att_ht[2 * l + 1] != sd.att_ht[2 * l]) busy = 1;
    }
    if (allow_att && ctl->to_admit > 0) busy = 1;
    if (ctl->done) busy = 0;
    s_busy = busy;
    s_tick = ctl->tick + (busy ? 1 : 0);
  }
  __syncthreads();
  const int tick = s_tick;
  if (s_busy) {
    // deliver the dispatches that arrive this tick
    for (int r = tid; r < sd.R; r += blockDim.x) {
      if (sd.arr_tick[r] != tick) continue;
      const int l = sd.req_n[r] % Lc;
      const LayerView& L = a.views[l];
      for (int k = 0; k < a.d.K; ++k) {
        const int e = sd.route_idx[(size_t)r * a.d.K + k];
        atomicOr(&L.enq_mask[r], 1u << k);
        L.wtab[(size_t)r * a.d.KS + k] = sd.route_w[(size_t)r * a.d.K + k];
        const uint32_t pos = atomicAdd(&L.tail[e], 1u);
        L.records[(size_t)e * a.d.cap + (pos % (uint32_t)a.d.cap)] = (r << kKShift) | k;
      }
      sd.arr_tick[r] = -1;
      atomicAdd(&ctl->exp_tokens[l], 1);
      atomicSub(&ctl->in_transit, 1);
      atomicAdd(&a.C->open_tokens, 1);
      atomicAdd(&a.C->pending_pairs, a.d.K);
    }
    // requests whose admission tick it is join layer 0's attention queue
    if (sd.admit) {
      for (int r = tid; r < sd.R; r += blockDim.x) {
        if (sd.admit[r] != tick) continue;
        const uint32_t pos = atomicAdd(&sd.att_ht[1], 1u);
        sd.att_ring[pos % (uint32_t)sd.R] = r;
        atomicSub(&ctl->to_admit, 1);
      }
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    int kind = 0, layer = 0;
    if (s_busy) {
      // the 2L queues in chain order att_0, exp_0, att_1, exp_1, ... (tokens; closed
      // attention queues count as empty)
      const bool allow_att = ctl->combined < sd.stop;
      int Q[2 * kMaxLayers];
      for (int l = 0; l < Lc; ++l) {
        Q[2 * l] = allow_att ? (int)(sd.att_ht[2 * l + 1] - sd.att_ht[2 * l]) : 0;
        Q[2 * l + 1] = ctl->exp_tokens[l];
      }
      const int nq = 2 * Lc;
      for (int q = 0; q < nq; ++q) {                  // occupancy seen at this decision
        ctl->peak_q[q] = max(ctl->peak_q[q], Q[q]);
        ctl->occ_sum[q] += Q[q];
      }
      ctl->peak_transit = max(ctl->peak_transit, ctl->in_transit);
      int pick = -1;
      if (sd.policy == MOE_STREAM_FLFS ||
          (sd.policy == MOE_STREAM_BARRIER && ctl->in_transit == 0)) {
        for (int q = 0; q < nq && pick < 0; ++q)
          if (Q[q] > 0) pick = q;
      } else if (sd.policy == MOE_STREAM_DEFRAG) {
        int Hd[2 * kMaxLayers];
        const int hw = min(sd.hist_window, kMaxHistoryWindow);
        for (int q = 0; q < nq; ++q) {
          int h = 0;
          for (int i = 0; i < hw; ++i) h += ctl->drained[i][q];
          Hd[q] = h;
        }
        double best_s = 0.0;
        for (int q = 0; q < nq; ++q) {
          if (Q[q] <= 0) continue;
          double s = (double)Q[q], dj = 1.0;
          for (int j = 1; j <= sd.window && q + j < nq; ++j) {
            dj = dj * sd.decay;
            s += dj * (double)(Q[q + j] + Hd[q + j]);
          }
          if (pick < 0 || s > best_s) { pick = q; best_s = s; }
        }
      } else if (sd.policy == MOE_STREAM_DEFRAG_SRC) {
        // H(s) = mean of s's depth snapshots over the window of earlier ticks (those recorded);
        // the lookahead wraps from the last expert queue to att_0.  IEEE round-to-nearest
        // double ops without contraction, so scores equal a plain float64 evaluation.
        const int hw = min(sd.hist_window, kMaxHistoryWindow);
        const int nv = min(ctl->snap_n, hw);
        double Hd[2 * kMaxLayers];
        for (int q = 0; q < nq; ++q) {
          int h = 0;
          for (int i = 0; i < hw; ++i) h += ctl->snap[i][q];    // unrecorded rows are zero
          Hd[q] = nv > 0 ? __ddiv_rn((double)h, (double)nv) : 0.0;
        }
        double best_s = 0.0;
        for (int q = 0; q < nq; ++q) {
          if (Q[q] <= 0) continue;
          double s = (double)Q[q], dj = 1.0;
          for (int j = 1; j <= sd.window; ++j) {
            const int qj = (q + j) % nq;
            dj = __dmul_rn(dj, sd.decay);
            s = __dadd_rn(s, __dmul_rn(dj, __dadd_rn((double)Q[qj], Hd[qj])));
          }
          if (pick < 0 || s > best_s) { pick = q; best_s = s; }
        }
      } else if (sd.policy == MOE_STREAM_MTFS) {
        int best = 0;
        for (int q = 0; q < nq; ++q)
          if (Q[q] > best) { best = Q[q]; pick = q; }
      }
      if (pick >= 0) { kind = 1 + (pick & 1); layer = pick >> 1; }
      if (sd.hist_window > 0) {                       // this decision's depths, for H(s) later
        const int hw = min(sd.hist_window, kMaxHistoryWindow);
        int* row = ctl->snap[tick % hw];
        for (int q = 0; q < 2 * kMaxLayers; ++q) row[q] = q < nq ? Q[q] : 0;
        ctl->snap_n = min(ctl->snap_n + 1, hw);
      }
    } else {
      ctl->done = 1;
    }
    s_kind = kind;
    s_layer = layer;
  }
  __syncthreads();
  const int kind = s_kind, layer = s_layer;
  moe_async_policy all{MOE_POLICY_MTFS, 0, 0, 1};
  plan_layer(a.views[kind == 2 ? layer : 0], a.d, a.P, a.C, all, a.g, kind == 2 ? layer : 0, 0, nullptr,
             a.wbytes, tick, kind == 2, sc);
  if (tid == 0 && kind == 2) {                        // the deepest bucket of the served queue
    int mb = 0;
    for (int b = 0; b < a.d.NB; ++b) mb = max(mb, sc.depth[b]);
    ctl->peak_bucket = max(ctl->peak_bucket, mb);
  }
  int cnt = 0;
  if (kind == 1) {
    const uint32_t hd = sd.att_ht[2 * layer], tl = sd.att_ht[2 * layer + 1];
    cnt = (int)(tl - hd);
    for (int i = tid; i < cnt; i += blockDim.x)
      sd.att_batch[i] = sd.att_ring[(size_t)layer * sd.R + ((hd + (uint32_t)i) % (uint32_t)sd.R)];
  } else if (kind == 2) {
    cnt = ctl->exp_tokens[layer];
  }
  __syncthreads();
  if (tid == 0) {
    if (kind == 1) {
      sd.att_ht[2 * layer] += (uint32_t)cnt;
      ctl->att_count = cnt;
      const int wt = tile_tokens(a.g, cnt, a.g.bn1, a.g.wide_min1);
      ctl->att_tiles = ((cnt + wt - 1) / wt) * ((a.d.H + a.g.bm2 - 1) / a.g.bm2);
    } else {
      ctl->att_count = 0;
      ctl->att_tiles = 0;
    }
    if (kind == 2) ctl->exp_tokens[layer] = 0;
    ctl->pick_kind = kind;
    ctl->pick_layer = layer;
    ctl->tick = tick;
    if (s_busy && sd.hist_window > 0) {               // this tick's drain, for H(s)
      int* row = ctl->drained[tick % min(sd.hist_window, kMaxHistoryWindow)];
      for (int q = 0; q < 2 * kMaxLayers; ++q) row[q] = 0;
      if (kind) row[2 * layer + (kind - 1)] = cnt;
    }
    if (s_busy) {
      const int ti = atomicAdd(a.trace_n, 1);
      if (ti < kStreamTraceCap) a.trace[ti] = make_int4(tick, kind, kind ? layer : -1, cnt);
    }
  }
}

// Attention batch rows: the state row x^(n) of each request and its RMSNorm scale
// s = 1 / sqrt(mean(x^2) + 1e-6) (one warp per row, fp32 sum of squares).
__global__ void att_prep_kernel(StreamDev sd, int H) {
  const StreamCtl* ctl = sd.ctl;
  if (ctl->pick_kind != 1) return;
  const int lane = threadIdx.x & 31;
  const int cnt = ctl->att_count;
  for (int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < cnt; i += gridDim.x * (blockDim.x >> 5)) {
    const int r = sd.att_batch[i];
    const int n = sd.req_n[r];
    const __nv_bfloat16* row = static_cast<const __nv_bfloat16*>(sd.hist) + ((size_t)r * (sd.n_max + 1) + n) * H;
    float ss = 0.f;
    for (int c = lane; c < H; c += 32) {
      const float v = __bfloat162float(row[c]);
      ss = fmaf(v, v, ss);
    }
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) {
      sd.att_rowptr[i] = row;
      sd.att_scale[i] = rsqrtf(ss / (float)H + 1e-6f);
    }
  }
}

// Routing of the attention batch (one warp per request) and dispatch: the request's K pairs
// arrive at its layer's expert queue `delay(r, n)` ticks from now.
__global__ void att_route_kernel(StreamDev sd, int E, int K) {
  StreamCtl* ctl = sd.ctl;
  if (ctl->pick_kind != 1) return;
  const int lane = threadIdx.x & 31;
  const int cnt = ctl->att_count;
  const int tick = ctl->tick;
  for (int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < cnt; i += gridDim.x * (blockDim.x >> 5)) {
    const int r = sd.att_batch[i];
    const int n = sd.req_n[r];
    warp_topk(sd.logits + ((size_t)r * sd.n_max + n) * E, E, K, lane, sd.route_idx + (size_t)r * K,
              sd.route_w + (size_t)r * K);
    if (lane == 0) {
      sd.arr_tick[r] = tick + max(1, sd.delay[(size_t)r * sd.n_max + n]);
      atomicAdd(&ctl->in_transit, 1);
    }
  }
}

__global__ void stream_init_kernel(StreamDev sd) {
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < sd.R; r += gridDim.x * blockDim.x) {
    sd.req_n[r] = 0;
    sd.arr_tick[r] = -1;
    if (!sd.admit) sd.att_ring[r] = r;      // every request starts in layer 0's attention queue
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    uint32_t n0 = (uint32_t)sd.R;
    if (sd.admit) {                         // those admitted at tick 0, in request order
      n0 = 0u;
      int later = 0;
      for (int r = 0; r < sd.R; ++r) {
        if (sd.admit[r] <= 0) sd.att_ring[n0++] = r;
        else ++later;
      }
      sd.ctl->to_admit = later;
    }
    for (int l = 0; l < sd.L; ++l) {
      sd.att_ht[2 * l] = 0u;
      sd.att_ht[2 * l + 1] = l == 0 ? n0 : 0u;
    }
  }
}

cudaError_t enqueue_tick(moe_async_s* h, StreamState* st, const TickArgs& ta, cudaStream_t s) {
  stream_tick_kernel<<<1, 1024, 0, s>>>(ta);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int rows_grid = (st->sd.R + 7) / 8;
  att_prep_kernel<<<rows_grid, 256, 0, s>>>(st->sd, h->dims.H);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (launch_att_tc(h, s) != MOE_OK) return cudaErrorLaunchFailure;
  att_route_kernel<<<rows_grid, 256, 0, s>>>(st->sd, h->dims.E, h->dims.K);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (launch_ffn_tc(h, 0, s) != MOE_OK) return cudaErrorLaunchFailure;
  return cudaSuccess;
}

template <typename P>
cudaError_t salloc(P** p, size_t bytes) {
  void* q = nullptr;
  cudaError_t e = cudaMalloc(&q, bytes ? bytes : 16);
  *p = static_cast<P*>(q);
  return e;
}

}  // namespace

void stream_teardown(moe_async_s* h) {
  StreamState* st = static_cast<StreamState*>(h->stream_state);
  if (!st) return;
  if (st->exec) cudaGraphExecDestroy(st->exec);
  if (st->graph) cudaGraphDestroy(st->graph);
  if (st->cap_stream) cudaStreamDestroy(st->cap_stream);
  void* ptrs[] = {st->sd.ctl, st->sd.req_n, st->sd.arr_tick, st->sd.att_ring, st->sd.att_ht, st->sd.route_idx,
                  st->sd.route_w, st->sd.att_batch, st->sd.att_scale, (void*)st->sd.att_rowptr, st->trace,
                  st->trace_n};
  for (void* p : ptrs) if (p) cudaFree(p);
  for (int l = 0; l < kMaxLayers; ++l) if (st->proj_packed[l]) cudaFree(st->proj_packed[l]);
  if (st->host_ctl) cudaFreeHost(st->host_ctl);
  delete st;
  h->stream_state = nullptr;
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_async_stream_setup(moe_async_t h, const moe_stream_config* sc,
                                             const void* const* d_proj, const void* d_x0,
                                             const float* d_logits, const int32_t* d_delay,
                                             const int32_t* d_admit, void* d_history,
                                             int32_t* d_done_tick, void* stream) {
  if (!h || !sc || !d_proj || !d_x0 || !d_logits || !d_delay || !d_history || !d_done_tick)
    return MOE_ERR_INVALID;
  if (!h->use_tc || h->cfg.num_layers > kMaxLayers) return MOE_ERR_UNSUPPORTED;
  if (sc->num_requests < 1 || sc->num_requests > h->dims.S || sc->max_steps < 1 || sc->stop_combines < 0 ||
      sc->policy < MOE_STREAM_MTFS || sc->policy > MOE_STREAM_DEFRAG_SRC || sc->defrag_window < 0 ||
      sc->history_window < 0 || sc->history_window > kMaxHistoryWindow || !(sc->defrag_decay == sc->defrag_decay))
    return MOE_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (h->stream_state) stream_teardown(h);
  StreamState* st = new (std::nothrow) StreamState();
  if (!st) return MOE_ERR_CUDA;
  std::memset(static_cast<void*>(st), 0, sizeof(StreamState));
  h->stream_state = st;
  st->cfg = *sc;
  const int R = sc->num_requests, L = h->cfg.num_layers, K = h->dims.K, H = h->dims.H;
  StreamDev& sd = st->sd;
  sd.R = R;
  sd.n_max = sc->max_steps;
  sd.stop = sc->stop_combines;
  sd.L = L;
  sd.policy = sc->policy;
  sd.window = sc->defrag_window;
  sd.hist_window = sc->history_window;
  sd.decay = sc->defrag_decay;
  sd.logits = d_logits;
  sd.delay = d_delay;
  sd.admit = d_admit;
  sd.hist = d_history;
  sd.done_tick = d_done_tick;
  bool ok = salloc(&sd.ctl, sizeof(StreamCtl)) == cudaSuccess &&
            salloc(&sd.req_n, (size_t)R * 4) == cudaSuccess &&
            salloc(&sd.arr_tick, (size_t)R * 4) == cudaSuccess &&
            salloc(&sd.att_ring, (size_t)L * R * 4) == cudaSuccess &&
            salloc(&sd.att_ht, (size_t)2 * L * 4) == cudaSuccess &&
            salloc(&sd.route_idx, (size_t)R * K * 4) == cudaSuccess &&
            salloc(&sd.route_w, (size_t)R * K * 4) == cudaSuccess &&
            salloc(&sd.att_batch, (size_t)R * 4) == cudaSuccess &&
            salloc(&sd.att_scale, (size_t)R * 4) == cudaSuccess &&
            salloc(&sd.att_rowptr, (size_t)R * sizeof(void*)) == cudaSuccess &&
            salloc(&st->trace, (size_t)kStreamTraceCap * sizeof(int4)) == cudaSuccess &&
            salloc(&st->trace_n, 4) == cudaSuccess &&
            cudaMallocHost(reinterpret_cast<void**>(&st->host_ctl), sizeof(StreamCtl)) == cudaSuccess;
  for (int l = 0; l < L && ok; ++l) {
    ok = salloc(&st->proj_packed[l], (size_t)H * H * 2) == cudaSuccess &&
         pack_transpose_bf16(d_proj[l], st->proj_packed[l], H, H, s) == cudaSuccess;
  }
  ok = ok && cudaMemsetAsync(sd.ctl, 0, sizeof(StreamCtl), s) == cudaSuccess &&
       cudaMemsetAsync(st->trace_n, 0, 4, s) == cudaSuccess &&
       cudaMemsetAsync(d_done_tick, 0xFF, (size_t)R * (sd.n_max + 1) * 4, s) == cudaSuccess &&
       cudaMemcpy2DAsync(d_history, (size_t)(sd.n_max + 1) * H * 2, d_x0, (size_t)H * 2, (size_t)H * 2, R,
                         cudaMemcpyDeviceToDevice, s) == cudaSuccess;
  if (ok) {
    stream_init_kernel<<<(R + 255) / 256, 256, 0, s>>>(sd);
    ok = cudaGetLastError() == cudaSuccess;
  }
  ok = ok && tc_stream_setup(h, const_cast<const void* const*>(st->proj_packed), sd) == MOE_OK;
  // one tick as a CUDA graph, captured on a library-owned stream
  TickArgs ta;
  std::memset(static_cast<void*>(&ta), 0, sizeof(ta));
  ta.sd = sd;
  for (int l = 0; l < L; ++l) ta.views[l] = h->layers[l];
  ta.d = h->dims;
  ta.C = h->counters;
  ta.P = h->plan;
  ta.g = h->geom;
  ta.trace = st->trace;
  ta.trace_n = st->trace_n;
  ta.wbytes = 3ll * h->dims.H * h->dims.I * 2;
  ok = ok && cudaStreamSynchronize(s) == cudaSuccess &&
       cudaStreamCreateWithFlags(&st->cap_stream, cudaStreamNonBlocking) == cudaSuccess;
  if (ok) {
    void* saved_prof = h->prof;
    h->prof = nullptr;                                   // no event brackets inside the graph
    ok = cudaStreamBeginCapture(st->cap_stream, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
    const bool launched = ok && enqueue_tick(h, st, ta, st->cap_stream) == cudaSuccess;
    ok = cudaStreamEndCapture(st->cap_stream, &st->graph) == cudaSuccess && launched && ok;
    h->prof = saved_prof;
    ok = ok && cudaGraphInstantiate(&st->exec, st->graph, 0) == cudaSuccess;
  }
  if (!ok) {
    stream_teardown(h);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

extern "C" moe_status moe_async_stream_run(moe_async_t h, int32_t max_ticks, int32_t check_every,
                                           int32_t* h_ticks, int32_t* h_combined, void* stream) {
  if (!h || max_ticks < 0) return MOE_ERR_INVALID;
  StreamState* st = static_cast<StreamState*>(h->stream_state);
  if (!st) return MOE_ERR_INVALID;
  if (check_every < 1) check_every = 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int launched = 0;
  for (;;) {
    MOE_CUDA_TRY(cudaMemcpyAsync(st->host_ctl, st->sd.ctl, sizeof(StreamCtl), cudaMemcpyDeviceToHost, s));
    MOE_CUDA_TRY(cudaStreamSynchronize(s));
    if (h_ticks) *h_ticks = st->host_ctl->tick;
    if (h_combined) *h_combined = st->host_ctl->combined;
    if (st->host_ctl->done) break;
    if (launched >= max_ticks) return MOE_ERR_TIMEOUT;
    for (int i = 0; i < check_every && launched < max_ticks; ++i, ++launched) {
      MOE_CUDA_TRY(cudaGraphLaunch(st->exec, s));
      h->launches += 6;
    }
  }
  moe_status dev = moe_async_sync(h, stream);
  return dev;
}

extern "C" moe_status moe_async_stream_stats(moe_async_t h, void* stream, moe_stream_stats* out) {
  if (!h || !out) return MOE_ERR_INVALID;
  StreamState* st = static_cast<StreamState*>(h->stream_state);
  if (!st) return MOE_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MOE_CUDA_TRY(cudaMemcpyAsync(st->host_ctl, st->sd.ctl, sizeof(StreamCtl), cudaMemcpyDeviceToHost, s));
  MOE_CUDA_TRY(cudaStreamSynchronize(s));
  const StreamCtl& c = *st->host_ctl;
  std::memset(static_cast<void*>(out), 0, sizeof(*out));
  out->ticks = c.tick;
  out->combined = c.combined;
  out->peak_transit = c.peak_transit;
  out->peak_bucket = c.peak_bucket;
  out->num_queues = 2 * st->sd.L;
  for (int q = 0; q < 2 * st->sd.L; ++q) {
    out->peak_queue[q] = c.peak_q[q];
    out->occupancy_sum[q] = c.occ_sum[q];
  }
  return MOE_OK;
}

extern "C" moe_status moe_async_stream_trace(moe_async_t h, void* stream, int32_t* h_buf, int32_t cap,
                                             int32_t* h_n) {
  if (!h || !h_n || cap < 0 || (cap > 0 && !h_buf)) return MOE_ERR_INVALID;
  StreamState* st = static_cast<StreamState*>(h->stream_state);
  if (!st) return MOE_ERR_INVALID;
  MOE_CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  int32_t n = 0;
  MOE_CUDA_TRY(cudaMemcpy(&n, st->trace_n, 4, cudaMemcpyDeviceToHost));
  n = std::min(std::min(n, kStreamTraceCap), cap);
  if (n > 0) MOE_CUDA_TRY(cudaMemcpy(h_buf, st->trace, (size_t)n * sizeof(int4), cudaMemcpyDeviceToHost));
  *h_n = n;
  return MOE_OK;
}
