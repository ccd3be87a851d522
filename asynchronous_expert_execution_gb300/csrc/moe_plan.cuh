// Device-side scheduling of one layer's micro-queues: reads every bucket depth, applies the
// pick policy and writes the step's work list (StepPlan).  Kept apart from the FFN kernels'
// header: only the scheduling and streaming kernels compile it.
#pragma once
#include "moe_internal.cuh"

namespace moe {

// One CTA (blockDim multiple of 32, >= 32).  Reads every bucket depth of the layer,
// applies the policy, drains the picked buckets whole (head += depth) and writes the work
// list the FFN kernels consume.  MTFS (StreamEP section 4): deepest first, equal depth ->
// lower bucket id.  THRESHOLD (streamFFN reading): buckets with depth >= min_batch, deepest
// first; if none, MTFS over non-empty buckets limited to fallback_groups.  RANKS (simulated
// expert-parallel ranks, R = max_groups): each rank drains its deepest bucket; with
// fallback_groups != 0 each idle rank then takes the deepest bucket no rank picked.  With
// enabled = false the plan is written empty and nothing is drained or counted.
//
// Several steps at once (max_steps > 1, MTFS and THRESHOLD): with nothing arriving between
// them, consecutive steps pick the non-empty buckets in one fixed order -- deepest first,
// which puts every bucket of at least min_batch ahead of the rest -- so step s takes a
// closed-form range of that order: MTFS G buckets a step (G = max_groups, 0 = all);
// THRESHOLD up to max_groups eligible buckets a step while any remain, then
// fallback_groups a step.  Each work item carries its step; the plan holds the steps up to
// the last non-empty one (at most max_steps), and only those are counted.
struct PlanScratch {
  // deepest-first sort keys: depth in the high word, the complement of the bucket id in the
  // low word (equal depth -> lower id first), 0 for an empty bucket; padded to whole pairs
  alignas(16) unsigned long long key[kMaxBuckets + 1];
  int depth[kMaxBuckets];
  uint32_t head[kMaxBuckets];     // queue heads read with the depths
  int order[kMaxBuckets];
  int pick[kMaxBuckets];          // RANKS: each rank's bucket (-1: none)
  unsigned char taken[kMaxBuckets];
  unsigned long long wmax[32];     // per-warp maxima (few picks)
  int n_elig, n_nonempty, n_picks, trace0;
};

// Plans with at most this many picks (MTFS / THRESHOLD) take them by rounds of a block-wide
// maximum over the keys instead of ranking every bucket.
constexpr int kFewPicks = 4;

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, off);
    v = o > v ? o : v;
  }
  return v;
}

// Threads that rank one bucket together (a power of 2 dividing the warp): each scans an
// interleaved share of the key pairs and the group adds its counts.  Chosen to minimise
// rounds x (pairs a thread scans + the shuffle levels) for nb buckets and nt threads.
__device__ __forceinline__ int rank_group(int nb, int nt) {
  const int pairs = (nb + 1) >> 1;       // nb <= kMaxBuckets, nt <= 1024: int arithmetic
  int best = 1, best_cost = -1;
  for (int per = 1, lv = 0; per <= 32; per <<= 1, ++lv) {
    const int rounds = (nb * per + nt - 1) / nt;
    const int cost = rounds * (((pairs + per - 1) >> lv) + 2 * lv);
    if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = per; }
  }
  return best;
}

// Step (0-based, within this plan) of the r-th bucket in the deepest-first order.
__device__ __forceinline__ int pick_step(const moe_async_policy& pol, int n_elig, int r) {
  if (pol.kind == MOE_POLICY_MTFS) return pol.max_groups > 0 ? r / pol.max_groups : 0;
  if (pol.kind != MOE_POLICY_THRESHOLD) return 0;
  const int ge = pol.max_groups, fb = pol.fallback_groups > 0 ? pol.fallback_groups : 1;
  if (r < n_elig) return ge > 0 ? r / ge : 0;
  const int elig_steps = n_elig > 0 ? (ge > 0 ? (n_elig + ge - 1) / ge : 1) : 0;
  return elig_steps + (r - n_elig) / fb;
}

// Buckets the first `max_steps` steps take out of `n_all` non-empty ones (n_elig of them
// eligible under THRESHOLD), in the deepest-first order.
__device__ __forceinline__ int picks_within(const moe_async_policy& pol, int n_all, int n_elig, int max_steps) {
  const long long ms = max_steps;
  if (pol.kind == MOE_POLICY_MTFS)
    return pol.max_groups > 0 ? (int)min((long long)n_all, (long long)pol.max_groups * ms) : n_all;
  const int ge = pol.max_groups, fb = pol.fallback_groups > 0 ? pol.fallback_groups : 1;
  if (n_elig > 0) {
    const int elig_steps = ge > 0 ? (n_elig + ge - 1) / ge : 1;
    if (ms <= elig_steps) return ge > 0 ? (int)min((long long)n_elig, (long long)ge * ms) : n_elig;
    return (int)min((long long)n_all, (long long)n_elig + (long long)fb * (ms - elig_steps));
  }
  return (int)min((long long)n_all, (long long)fb * ms);
}

__device__ inline void plan_layer(const LayerView& L, const Dims& d, StepPlan* P, DevCounters* C,
                                  const moe_async_policy& pol, const TileGeom& g, int layer,
                                  int trace_cap, int4* trace, long long weight_bytes_per_run,
                                  int trace_step, bool enabled, PlanScratch& sc, int max_steps = 1) {
  int* depth = sc.depth;
  int* order = sc.order;
  const int tid = threadIdx.x, nt = blockDim.x;
  if (tid == 0) { sc.n_elig = 0; sc.n_nonempty = 0; }
  __syncthreads();
  // After an overflow or an out-of-range id the queues no longer describe valid pairs:
  // stop executing (the sticky error is reported to the host).  Read with the depths.
  const uint32_t err = *(volatile uint32_t*)&C->error;
  const int nkey = (d.NB + 1) & ~1;
  int my_nonempty = 0, my_elig = 0;
  for (int b = tid; b < nkey; b += nt) {
    unsigned long long key = 0ull;
    if (b < d.NB) {
      const uint32_t hd = L.head[b];
      const int dep = enabled ? min((int)(L.tail[b] - hd), d.cap) : 0;
      sc.head[b] = hd;
      depth[b] = dep;
      if (dep > 0) {
        key = ((unsigned long long)(uint32_t)dep << 32) | (0xffffffffu - (uint32_t)b);
        ++my_nonempty;
        if (pol.kind != MOE_POLICY_THRESHOLD || dep >= pol.min_batch) ++my_elig;
      }
    }
    sc.key[b] = key;
  }
  my_nonempty = __reduce_add_sync(0xffffffffu, my_nonempty);
  my_elig = __reduce_add_sync(0xffffffffu, my_elig);
  if ((tid & 31) == 0) {
    if (my_nonempty) atomicAdd(&sc.n_nonempty, my_nonempty);
    if (my_elig) atomicAdd(&sc.n_elig, my_elig);
  }
  __syncthreads();
  const int n_elig = sc.n_elig, n_nonempty = sc.n_nonempty;
  const bool halted = err == MOE_ERR_CAPACITY || err == MOE_ERR_INVALID || err == MOE_ERR_BOUNDS;
  // MTFS / THRESHOLD: the picks are a prefix of the deepest-first order of every non-empty
  // bucket; RANKS ranks the non-empty buckets too (its stealers take from that order)
  const bool ranks = pol.kind == MOE_POLICY_RANKS;
  int n = halted ? 0 : (ranks ? n_nonempty : picks_within(pol, n_nonempty, n_elig, max(max_steps, 1)));
  // the trace entries of the picks are reserved while the buckets are ranked (RANKS knows
  // its pick count only after the ranking)
  const bool want_trace = trace && trace_cap > 0;
  int trace0 = 0;                       // its value is first used after the ranking
  if (tid == 0 && want_trace && !ranks && n > 0) trace0 = atomicAdd(&C->trace_n, n);
  if (!ranks && n <= kFewPicks) {
    // pick r is the largest key left: a block-wide maximum, then that bucket leaves the keys
    const int lane = tid & 31, warp = tid >> 5;
    for (int r = 0; r < n; ++r) {
      unsigned long long m = 0ull;
      for (int b = tid; b < nkey; b += nt) m = sc.key[b] > m ? sc.key[b] : m;
      m = warp_max_u64(m);
      if (lane == 0) sc.wmax[warp] = m;
      __syncthreads();
      if (warp == 0) {
        m = warp_max_u64(lane < (nt >> 5) ? sc.wmax[lane] : 0ull);
        if (lane == 0 && m != 0ull) {
          const int b = (int)(0xffffffffu - (uint32_t)m);
          order[r] = b;
          sc.key[b] = 0ull;
        }
      }
      __syncthreads();
    }
  } else {
    // rank of every non-empty bucket in the deepest-first order = the keys above its own
    const int per = rank_group(d.NB, nt);
    const ulonglong2* k2 = reinterpret_cast<const ulonglong2*>(sc.key);
    const int pairs = nkey >> 1;
    for (int base = 0; base < d.NB * per; base += nt) {     // the same trips for every thread
      const int idx = base + tid, b = idx / per, part = idx - b * per;
      const unsigned long long kb = b < d.NB ? sc.key[b] : 0ull;
      int r = 0;
      if (kb != 0ull)
        for (int c = part; c < pairs; c += per) {
          const ulonglong2 v = k2[c];
          r += (int)(v.x > kb) + (int)(v.y > kb);
        }
      for (int off = per >> 1; off > 0; off >>= 1) r += __shfl_down_sync(0xffffffffu, r, off, per);
      if (part == 0 && kb != 0ull && r < n) order[r] = b;
    }
  }
  if (tid == 0) sc.trace0 = trace0;
  __syncthreads();
  if (pol.kind == MOE_POLICY_RANKS) {
    // simulated expert-parallel ranks: bucket b belongs to rank b mod R; each rank runs its
    // deepest bucket (equal depth -> lower id); then each rank that owns no non-empty bucket
    // takes, in rank order, the deepest bucket no rank has picked (order[] holds every
    // non-empty bucket deepest first); the work list is the picks in rank order
    const int R = min(max(pol.max_groups, 1), kMaxBuckets);
    for (int r = tid; r < R; r += nt) {
      int best = -1;
      for (int b = r; b < d.NB; b += R)
        if (depth[b] > 0 && (best < 0 || depth[b] > depth[best])) best = b;
      sc.pick[r] = best;
    }
    for (int b = tid; b < d.NB; b += nt) sc.taken[b] = 0;
    __syncthreads();
    if (tid == 0) {
      for (int r = 0; r < R; ++r)
        if (sc.pick[r] >= 0) sc.taken[sc.pick[r]] = 1;
      int q = 0, m = 0;
      for (int r = 0; r < R; ++r) {
        if (sc.pick[r] < 0 && pol.fallback_groups != 0) {
          while (q < n && sc.taken[order[q]]) ++q;
          if (q < n) {
            sc.pick[r] = order[q];
            sc.taken[order[q]] = 1;
          }
        }
        if (sc.pick[r] >= 0) sc.pick[m++] = sc.pick[r];   // compact in rank order (m <= r)
      }
      for (int i = 0; i < m; ++i) order[i] = sc.pick[i];
      sc.n_picks = halted ? 0 : m;
    }
    __syncthreads();
    n = sc.n_picks;
  }
  if (tid < 32) {
    const int lane = tid;
    int row_run = 0, t1_run = 0, t2_run = 0;
    const int ft1 = (2 * d.I + g.bm1 - 1) / g.bm1;
    const int ft2 = (d.H + g.bm2 - 1) / g.bm2;
    // trace entries of the n picks, in pick order, reserved at once
    int ti0 = 0;
    if (want_trace && n > 0) {
      if (ranks) {
        if (lane == 0) ti0 = atomicAdd(&C->trace_n, n);
        ti0 = __shfl_sync(0xffffffffu, ti0, 0);
      } else {
        ti0 = sc.trace0;
      }
    }
    for (int c0 = 0; c0 < n; c0 += 32) {
      const int r = c0 + lane;
      int b = 0, cnt = 0, t1 = 0, t2 = 0;
      if (r < n) {
        b = order[r];
        cnt = depth[b];
        const int w1 = tile_tokens(g, cnt, g.bn1, g.wide_min1), w2 = tile_tokens(g, cnt, g.bn2, g.wide_min2);
        t1 = ((cnt + w1 - 1) / w1) * ft1;
        t2 = ((cnt + w2 - 1) / w2) * ft2;
      }
      int s_cnt = cnt, s_t1 = t1, s_t2 = t2;      // inclusive prefix sums within the chunk
      for (int off = 1; off < 32; off <<= 1) {
        int a = __shfl_up_sync(0xffffffffu, s_cnt, off);
        int b1 = __shfl_up_sync(0xffffffffu, s_t1, off);
        int b2 = __shfl_up_sync(0xffffffffu, s_t2, off);
        if (lane >= off) { s_cnt += a; s_t1 += b1; s_t2 += b2; }
      }
      if (r < n) {
        WorkItem it;
        it.expert = b;
        it.head = sc.head[b];
        it.count = cnt;
        it.row_base = row_run + s_cnt - cnt;
        it.t1_base = t1_run + s_t1 - t1;
        it.t2_base = t2_run + s_t2 - t2;
        it.step = trace_step + (ranks ? 0 : pick_step(pol, n_elig, r));
        P->items[r] = it;
        L.head[b] = it.head + (uint32_t)cnt;
        if (trace && trace_cap > 0 && ti0 + r < trace_cap) trace[ti0 + r] = make_int4(it.step, layer, b, cnt);
      }
      row_run += __shfl_sync(0xffffffffu, s_cnt, 31);
      t1_run += __shfl_sync(0xffffffffu, s_t1, 31);
      t2_run += __shfl_sync(0xffffffffu, s_t2, 31);
    }
    if (kDebugBounds && lane == 0 && row_run > d.S * d.KS) {     // the step's rows overflow h
      set_error(C, MOE_ERR_BOUNDS);
      n = 0;
      row_run = t1_run = t2_run = 0;
    }
    if (lane == 0) {
      P->layer = layer;
      P->n_work = n;
      P->n_tiles1 = t1_run;
      P->n_tiles2 = t2_run;
      P->rows = row_run;
      if (!enabled) return;
      C->plan_layer = layer;
      C->nonempty_left = n_nonempty - n;          // every pick is a non-empty bucket, drained whole
      C->elig_left = (pol.kind == MOE_POLICY_THRESHOLD && n_elig > n) ? n_elig - n : 0;
      // one step is always counted (an empty step too); a plan of several steps counts the
      // steps up to its last non-empty one
      const int steps_run = max_steps <= 1 ? 1 : (n > 0 ? pick_step(pol, n_elig, n - 1) + 1 : 0);
      // reductions without a returned value: no round trip on the planner's path
      atomicAdd(&C->steps, (unsigned long long)steps_run);
      atomicAdd(&C->pairs_executed, (unsigned long long)row_run);
      atomicAdd(&C->expert_runs, (unsigned long long)n);
      atomicAdd(&C->weight_bytes, (unsigned long long)n * (unsigned long long)weight_bytes_per_run);
      atomicSub(&C->pending_pairs, row_run);
    }
  }
}

}  // namespace moe
