// Expert FFN for bf16 on the 5th-generation tensor cores: tcgen05.mma with TMEM accumulators,
// weights streamed by TMA, gathered token rows by cp.async.
//
// Swap-AB grouped GEMM.  Each tile computes D[128 x N] = A[128 x K] * B[N x K]^T where
//   A = 128 rows of an expert's packed weights (K-major, 128B-swizzled, loaded by TMA), and
//   B = N gathered token rows of the step's batch for that expert (K-major, 128B swizzle
//       applied by the loader), N <= 32 for a small item and <= 128 for a large one,
// so a decode batch of a few tokens per expert still fills the 128-row MMA with weights and
// the kernel streams each picked expert's weights once per token tile.
//   GEMM1: A = W13 (gate/up rows interleaved in blocks of 16), K = H, B = pool rows of the
//          tokens in the expert's bucket (the gather of StreamEP section 3, step 4, fused into
//          the operand load); epilogue: h = silu(gate) * up, stored bf16.
//   GEMM2: A = W2^T, K = I, B = the expert's h rows; epilogue: slotbuf[slot][k] = o (bf16,
//          the activation dtype), then readiness counting; the top-k merge
//          y = sum_k w_k o_k (fp32, ascending k) runs in the collect kernel (or, in the
//          streaming runtime, in this epilogue).
// K may be cut into fixed chunks whose partials are added in chunk order; a launch with few
// tiles spreads a tile's chunks over CTAs (see Unit).  Units are handed out dynamically: a
// CTA claims its next unit from a per-launch counter as it finishes issuing the previous
// one, so SMs that stream faster take more of the launch.
//
// Warp roles (256 threads, one persistent CTA per SM):
//   warp 0  lane 0: TMA producer for A (the weights); claims the units and passes their
//                   indices to the other roles through a ring in shared memory
//   warps 1, 3: cp.async producers for B: the gathered pool rows (GEMM1, attention projection)
//               or the item's contiguous h rows (GEMM2, after GEMM1 has finished)
//   warp 2  lane 0: MMA issuer; warp 2 allocates / frees TMEM
//   warps 4-7: epilogue (TMEM lanes 32*(warp-4) ..), kAccBufs accumulator buffers
// Every wait is bounded in time; a timeout latches MOE_ERR_TIMEOUT, stops all roles, and the
// CTA still frees its TMEM before exiting.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cstring>
#include <new>
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;              // MMA M (weight rows per tile)
constexpr int kBK = 64;               // K per k-block (one 128-byte swizzle atom)
// Pipeline stages fill the shared memory left over (kStage bytes each) and a tile moves as
// many k-blocks a stage as fit (at most MOE_TC_KPS_MAX): a stage's fixed cost (barrier round
// trip, TMA issue, MMA commit) is paid once per stage.  Measured on GB300 with an MMA
// consumer: a lone SM streams 36 / 53 / 69 GB/s with 16 / 32 / 64 KB weight stages, and 152
// SMs 5.3 / 6.1 TB/s with 16 / 32 KB stages.  With 3 stages of 73 KB a 32-token tile moves 3
// k-blocks, a 16-token one 4, a wide tile of up to 64 tokens 3 and a wider one 2 (against 2
// for every wide tile in 64 KB stages: DeepSeek-wide layer +1.7%, Zipf prefill +1.9%).
#ifndef MOE_TC_KPS_MAX
#define MOE_TC_KPS_MAX 8
#endif
constexpr int kKpsMax = MOE_TC_KPS_MAX;
#ifndef MOE_TC_STAGES
#define MOE_TC_STAGES 3
#endif
constexpr int kStagesCfg = MOE_TC_STAGES;   // pipeline stages of the shared-memory ring
// Wide tiles: an item with at least MOE_TC_WIDE_MIN1 (GEMM1, attention stub) or
// MOE_TC_WIDE_MIN2 (GEMM2) tokens is cut into MOE_TC_BNW-token tiles, so its weight rows are
// read once per BNW tokens and each MMA is wide enough for the tensor pipe (measured: 46
// cycles per 128 x N x 16 MMA for N <= 64, 64 for N = 128, 128 for N = 256).  Measured on
// GB300 (pairs/s, Zipf prefill / DeepSeek-wide layer): one threshold for both GEMMs of 128
// -- 3.48 M / 1.17 M; 64 -- 3.66 M / 1.28 M; 33 -- 3.76 M / 1.24 M, when every one-expert
// step of the DeepSeek-wide layer was its own launch (its 63-token items then ran GEMM2 on
// half as many CTAs).  Since those steps drain as one plan, GEMM2 gains from 33 as well:
// 64 -> 33 gives 2.54 M -> 2.71 M and 3.83 M -> 3.86 M, decode unchanged.  0 turns wide
// tiles off.
#ifndef MOE_TC_BNW
#define MOE_TC_BNW 128
#endif
#ifndef MOE_TC_WIDE_MIN1
#define MOE_TC_WIDE_MIN1 33
#endif
#ifndef MOE_TC_WIDE_MIN2
#define MOE_TC_WIDE_MIN2 33
#endif
// TMEM accumulator buffers (each BNW columns): the MMA may run this many units' chunks ahead of
// the epilogue, which absorbs epilogues made slow by the merges some tiles complete.
#ifndef MOE_TC_ACC
#define MOE_TC_ACC 4
#endif
constexpr int kAccBufs = MOE_TC_ACC;
constexpr int kWideMin1 = MOE_TC_WIDE_MIN1, kWideMin2 = MOE_TC_WIDE_MIN2;
constexpr int kThreads = 256;
constexpr int kMaxChunks = 4;          // most K chunks of a contraction
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s per wait

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on a phase parity.  Returns false (and raises the CTA abort flag and the
// sticky device error) when the phase does not complete within the limit, or when another
// role already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          DevCounters* C) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      set_error(C, MOE_ERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

// Bring a tensor map's descriptor on chip ahead of its first TMA.
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
// The executing thread's prior cp.async copies trigger one arrive on `bar` when they complete
// (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 16 consecutive fp32 columns of the accumulator; the wait is tied to the
// registers so no use can be scheduled before it.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15])::"memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Named barrier over the 128 epilogue threads with an AND-reduction of a predicate, so a
// decision taken after a bounded wait is uniform across the group.
__device__ __forceinline__ bool epi_bar_and(bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)pred)
      : "memory");
  return out != 0;
}

struct EpiBarrier {
  __device__ __forceinline__ void operator()() const { asm volatile("bar.sync 1, 128;" ::: "memory"); }
};

// tcgen05 shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row groups
// 1024 bytes apart (SBO), descriptor version 1 (bit 46).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)(16u >> 4) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, N and M encoded.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ----------------------------------------------------------------- tile decoding

enum : int { kModeGemm1 = 0, kModeGemm2 = 1, kModeAtt = 2 };

// Everything a launch needs, for every layer: the layer a tile belongs to is read on the
// device (the step plan, or the streaming runtime's pick), so one launch serves any layer.
struct TcParams {
  CUtensorMap mapA[kMaxLayers];     // GEMM1: packed W13, GEMM2: packed W2^T, ATT: packed P^T
  LayerView views[kMaxLayers];
  Dims d;
  DevCounters* C;
  const StepPlan* P;
  __nv_bfloat16* hbuf;
  int parts;                        // feature slices per token (GEMM2 tiles covering H)
  int stream_on;                    // GEMM2 merges feed the streaming runtime
  StreamDev sd;
  // K is cut into `nchunk` fixed chunks; each chunk's product starts from a zero accumulator
  // and the chunk partials are added in ascending chunk order, so a result never depends on
  // whether a tile's chunks ran on one CTA or on several (split steps).
  int nchunk;
  int split_cap;                    // most tiles a launch may split (workspace capacity)
  float* ws;                        // [split_cap][nchunk][BNW / 4][128] float4 chunk partials
  int* cnt;                         // [split_cap] arrivals per split tile (zero between launches)
  // dynamic unit assignment: [0] units claimed beyond the first round, [1] CTAs that have
  // finished; both zero between launches (the last CTA to finish resets them)
  int* unit_ctr;
};

// A unit of work: one tile and a range of its K chunks [c0, c1).  The first n_whole tiles of a
// launch are one unit each (all chunks); each later tile is split into one unit per chunk
// (n_whole is 0 or the launch's tile count).
struct Unit {
  int t, c0, c1;
  bool split;
};

__device__ __forceinline__ Unit unit_of(int u, int n_whole, int nchunk) {
  Unit x;
  if (u < n_whole) {
    x.t = u;
    x.c0 = 0;
    x.c1 = nchunk;
    x.split = false;
  } else {
    const int v = u - n_whole;
    x.t = n_whole + v / nchunk;
    x.c0 = v % nchunk;
    x.c1 = x.c0 + 1;
    x.split = true;
  }
  return x;
}

// Dynamic unit assignment.  A CTA's first unit is its own index; each later one is claimed
// from the launch's counter when the weight producer has issued the previous unit's last
// stage, so a CTA that streams faster takes more units and the launch ends evenly.  The
// producer hands the indices, in order, to the other roles through a ring in shared memory:
// -1 ends a CTA's sequence.
constexpr int kUnitQ = 16;                // ring depth: above the most units a reader can lag
constexpr uint32_t kUnitReaders = 7;      // the two B warps, the MMA thread, four epilogue warps

struct UnitRing {
  int* q;
  uint64_t* full;
  uint64_t* empty;
};

__device__ __forceinline__ bool ring_put(const UnitRing& r, uint32_t& i, int u, volatile int* abort_flag,
                                         DevCounters* C) {
  const int s = (int)(i % kUnitQ);
  const uint32_t ph = (i / kUnitQ) & 1u;
  ++i;
  if (!mbar_wait(&r.empty[s], ph ^ 1u, abort_flag, C)) return false;
  r.q[s] = u;
  mbar_arrive(&r.full[s]);                  // release: the index is visible to the readers
  return true;
}

// The next unit for one thread (the MMA issuer); -1 at the end or after an abort.
__device__ __forceinline__ int ring_get(const UnitRing& r, uint32_t& i, volatile int* abort_flag, DevCounters* C) {
  const int s = (int)(i % kUnitQ);
  const uint32_t ph = (i / kUnitQ) & 1u;
  ++i;
  if (!mbar_wait(&r.full[s], ph, abort_flag, C)) return -1;
  const int u = *reinterpret_cast<volatile int*>(&r.q[s]);
  mbar_arrive(&r.empty[s]);
  return u;
}

// The next unit for every lane of a warp (one arrival per warp, after all lanes have read).
__device__ __forceinline__ int ring_get_warp(const UnitRing& r, uint32_t& i, int lane, volatile int* abort_flag,
                                             DevCounters* C) {
  const int s = (int)(i % kUnitQ);
  const uint32_t ph = (i / kUnitQ) & 1u;
  ++i;
  const bool ok = mbar_wait(&r.full[s], ph, abort_flag, C);
  const int u = ok ? *reinterpret_cast<volatile int*>(&r.q[s]) : -1;
  const bool all_ok = __all_sync(0xffffffffu, ok);
  if (all_ok && lane == 0) mbar_arrive(&r.empty[s]);
  return all_ok ? u : -1;
}

// Called once per CTA by one thread after every role has stopped: the last CTA of the launch
// puts the counters back to zero for the next launch of these parameters.
__device__ __forceinline__ void unit_ctr_exit(int* ctr) {
  __threadfence();
  if (atomicAdd(&ctr[1], 1) == (int)gridDim.x - 1) {
    ctr[0] = 0;
    ctr[1] = 0;
  }
}

// first k-block of chunk c (chunk c covers [chunk_kb(c), chunk_kb(c + 1))): the even cut,
// rounded to a multiple of 6 k-blocks so chunks hold whole stages of both tile widths
__device__ __forceinline__ int chunk_kb(int c, int nk, int nchunk) {
  if (c >= nchunk) return nk;
  const int e = (int)(((long long)c * nk) / nchunk);
  return min(nk, (e + 3) / 6 * 6);
}

// A stage holds kps k-blocks of a tile: A sub-blocks (16 KB each) from the stage base, then
// B sub-blocks (nmma x 128 B each).  The stages take the dynamic shared memory that the
// barriers, the per-unit arrays and the item table leave (227 KB a CTA, 1 KB of alignment
// slack), in whole KB.
template <int BN, int BNW, int STAGES>
struct SmemLayout {
  static constexpr int kA1 = kBM * kBK * 2;                  // 16 KB: one k-block of A
  static constexpr int kNumBars = 2 * STAGES + 2 * kAccBufs;
  static constexpr int kTail = kNumBars * 8 + 8 + 15 + 4 * BNW * 4 + 16 + 7 + 2 * kUnitQ * 8 + kUnitQ * 4 +
                               kMaxBuckets * 4;              // everything after the stages (upper bound)
  static constexpr int kStage = ((227 * 1024 - 1024 - kTail) / STAGES) & ~1023;
  static_assert(kStage >= kA1 + BNW * kBK * 2, "a stage must hold one k-block of the widest tile");
  static constexpr int kOffBar = STAGES * kStage;
  static constexpr int kOffTmem = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmem + 4;
  static constexpr int kOffSlot = (kOffAbort + 4 + 15) & ~15;
  static constexpr int kOffK = kOffSlot + BNW * 4;
  static constexpr int kOffFin = kOffK + BNW * 4;
  static constexpr int kOffW = kOffFin + BNW * 4;
  static constexpr int kOffFlag = kOffW + BNW * 4;
  static constexpr int kOffRingBar = (kOffFlag + 16 + 7) & ~7;
  static constexpr int kOffRing = kOffRingBar + 2 * kUnitQ * 8;
  static constexpr int kOffTb = kOffRing + kUnitQ * 4;
  static constexpr int kBytes = kOffTb + kMaxBuckets * 4;
  static constexpr int kAlloc = kBytes + 1024;               // room to align the base to 1024
  static_assert(kAlloc <= 227 * 1024, "dynamic shared memory of a CTA: at most 227 KB");
};

struct Tile {
  int expert;
  int step;     // scheduling step of the work item
  uint32_t head;
  int row_base;
  int fti;      // feature (A-row) tile
  int j0;       // first token of the tile within the item
  int nj;       // valid tokens
  int nmma;     // MMA N (multiple of 16, >= nj)
  int bn;       // tile width: narrow or wide
  int kps;      // k-blocks per pipeline stage for this tile width
  int bstride;  // bytes between the B sub-blocks of a stage (nmma rows of 128 B)
  bool single;  // the item has one token tile: its A rows are read once
};

// tb = the step's first-tile indices of the work items, staged in shared memory
template <int BN, int BNW, int MODE>
__device__ __forceinline__ Tile decode_tile(const TcParams& p, const int* tb, int t) {
  Tile tl;
  int local, count;
  if (MODE == kModeAtt) {
    count = p.sd.ctl->att_count;
    local = t;
    tl.expert = 0;
    tl.step = 0;
    tl.head = 0;
    tl.row_base = 0;
  } else {
    const StepPlan* P = p.P;
    int lo = 0, hi = P->n_work - 1;                 // last item whose first tile is <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tb[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const WorkItem it = P->items[lo];
    local = t - (MODE == kModeGemm2 ? it.t2_base : it.t1_base);
    count = it.count;
    tl.expert = it.expert;
    tl.step = it.step;
    tl.head = it.head;
    tl.row_base = it.row_base;
  }
  // the planner applies the same rule
  const bool wide = BNW > BN && count >= (MODE == kModeGemm2 ? kWideMin2 : kWideMin1);
  tl.bn = wide ? BNW : BN;
  const int ntt = (count + tl.bn - 1) / tl.bn;
  tl.single = ntt <= 1;
  tl.fti = local / ntt;
  tl.j0 = (local % ntt) * tl.bn;
  tl.nj = min(tl.bn, count - tl.j0);
  tl.nmma = min(tl.bn, max(16, (tl.nj + 15) & ~15));
  tl.bstride = tl.nmma * kBK * 2;
  // as many k-blocks as a stage holds, up to kKpsMax
  using SL = SmemLayout<BN, BNW, kStagesCfg>;
  tl.kps = max(1, min(kKpsMax, SL::kStage / (SL::kA1 + tl.bstride)));
  return tl;
}


// ------------------------------------------------------------------ the kernel

template <int BN, int BNW, int STAGES, int MODE>
__global__ void __launch_bounds__(kThreads, 1) ffn_tc_kernel(const __grid_constant__ TcParams p) {
  using SL = SmemLayout<BN, BNW, STAGES>;
  constexpr uint32_t kTmemCols = kAccBufs * BNW;   // accumulator buffers of the wider width
  static_assert(kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM columns: a power of 2, at most 512");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SL::kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = bars + 2 * STAGES + kAccBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SL::kOffTmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SL::kOffAbort);
  int* slot_s = reinterpret_cast<int*>(smem + SL::kOffSlot);
  int* k_s = reinterpret_cast<int*>(smem + SL::kOffK);
  int* fin = reinterpret_cast<int*>(smem + SL::kOffFin);
  float* w_s = reinterpret_cast<float*>(smem + SL::kOffW);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + SL::kOffFlag);
  int* tb_s = reinterpret_cast<int*>(smem + SL::kOffTb);
  uint64_t* ring_bars = reinterpret_cast<uint64_t*>(smem + SL::kOffRingBar);
  const UnitRing ring{reinterpret_cast<int*>(smem + SL::kOffRing), ring_bars, ring_bars + kUnitQ};

  const Dims& d = p.d;
  DevCounters* C = p.C;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Programmatic dependent launch: GEMM1 may start while the scheduling kernel runs and waits
  // here for its plan; it then lets GEMM2 start on SMs as they free up.  (A no-op when the
  // kernel was launched without a programmatic dependency.)
  // barriers and TMEM do not depend on the plan: GEMM1 sets them up before it waits for it
  auto setup = [&]() {
    if (threadIdx.x == 0) {
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(&full[s], 1 + 64);    // the A producer's expect_tx arrive + 64 cp.async B lanes
        mbar_init(&empty[s], 1);        // tcgen05.commit
      }
      for (int b = 0; b < kAccBufs; ++b) {
        mbar_init(&tfull[b], 1);        // tcgen05.commit after the tile's last MMA
        mbar_init(&tempty[b], 4);       // one arrive per epilogue warp
      }
      for (int i = 0; i < kUnitQ; ++i) {
        mbar_init(&ring.full[i], 1);              // the weight producer
        mbar_init(&ring.empty[i], kUnitReaders);  // every reader role
      }
      *abort_flag = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 2) {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
  };
  if (MODE == kModeGemm1) {
    setup();
    griddep_wait();
    griddep_launch_dependents();
  }
  // GEMM2: the collect launched after it may start and wait (GEMM2 itself waits for GEMM1
  // before reading h, so its completion implies GEMM1's)
  if (MODE == kModeGemm2) griddep_launch_dependents();
  int n_tiles, layer;
  if (MODE == kModeAtt) {
    const bool picked = p.sd.ctl->pick_kind == 1;
    n_tiles = picked ? p.sd.ctl->att_tiles : 0;
    layer = picked ? p.sd.ctl->pick_layer : 0;
  } else {
    n_tiles = MODE == kModeGemm2 ? p.P->n_tiles2 : p.P->n_tiles1;
    layer = p.P->layer;
  }
  if (layer < 0 || layer >= kMaxLayers) n_tiles = 0;
  const LayerView& L = p.views[layer < 0 || layer >= kMaxLayers ? 0 : layer];
  const CUtensorMap* tmA = &p.mapA[layer < 0 || layer >= kMaxLayers ? 0 : layer];
  const int Kdim = MODE == kModeGemm2 ? d.I : d.H;
  const int nk = (Kdim + kBK - 1) / kBK;
  // A launch with few tiles for the grid splits every tile into its K chunks (one unit each)
  // when that shortens the launch: a single SM streams weights far below the HBM rate, so a
  // lone expert needs many SMs.  Every role derives the same split from the plan.  (Splitting
  // only the last, partial round's tiles was measured too: with the 45-k-block GPT-OSS
  // contractions cut in 2 for it, decode lost 0.4% and prefill 1.5%.)
  const int nchunk = p.nchunk;
  int n_whole = n_tiles;
  if (nchunk > 1 && n_tiles <= p.split_cap) {
    const int G = (int)gridDim.x;
    const long long whole = (long long)((n_tiles + G - 1) / G) * nchunk;   // in chunk times
    const long long split = ((long long)n_tiles * nchunk + G - 1) / G;
    if (split < whole) n_whole = 0;
  }
  const int n_units = n_whole + (n_tiles - n_whole) * nchunk;
  if ((int)blockIdx.x >= n_units) {              // no work for this CTA: skip the rest of the set-up
    // every CTA of a programmatic dependent waits for its predecessor before it ends, so this
    // launch's completion implies GEMM1's even when it has no work
    if (MODE == kModeGemm2) griddep_wait();
    if (MODE == kModeGemm1) {                   // give back the TMEM taken before the plan
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (warp == 2) {
        __syncwarp();
        tmem_dealloc(*tmem_slot, kTmemCols);
      }
    }
    if (threadIdx.x == 0) unit_ctr_exit(p.unit_ctr);
    return;
  }

  if (threadIdx.x == 0) prefetch_tmap(tmA);     // descriptors load while the CTA sets up
  if (MODE != kModeGemm1) setup();
  if (MODE != kModeAtt) {                       // item lookups then search shared memory
    const int nw = min(p.P->n_work, kMaxBuckets);
    for (int i = threadIdx.x; i < nw; i += blockDim.x)
      tb_s[i] = MODE == kModeGemm2 ? p.P->items[i].t2_base : p.P->items[i].t1_base;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ A producer: TMA of weight tiles
    if (lane == 0) {
      // weights read by one token tile only are streamed with L2 evict-first; tiles whose A
      // rows are shared by several token tiles (a popular expert) keep the normal policy so
      // the concurrent readers hit L2
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_reuse = policy_evict_normal();
      uint32_t it = 0;
      bool ok = true;
      // GEMM2 runs as a programmatic dependent of GEMM1: its weights do not depend on GEMM1,
      // so this producer streams W2 at once; the B warps wait for GEMM1 before the h rows.
      uint32_t qi = 0;
      for (int u = blockIdx.x; ok;) {
        if (!(ok = ring_put(ring, qi, u, abort_flag, C)) || u < 0) break;
        const Unit un = unit_of(u, n_whole, nchunk);
        const Tile tl = decode_tile<BN, BNW, MODE>(p, tb_s, un.t);
        const uint64_t pol = tl.single ? pol_stream : pol_reuse;
        for (int c = un.c0; c < un.c1 && ok; ++c) {
          const int kb1 = chunk_kb(c + 1, nk, nchunk);
          for (int kbs = chunk_kb(c, nk, nchunk); kbs < kb1; kbs += tl.kps, ++it) {
            const int nv = min(tl.kps, kb1 - kbs);
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1u;
            if (!(ok = mbar_wait(&empty[s], ph ^ 1u, abort_flag, C))) break;
            const uint32_t a_s = smem_u32(smem + s * SL::kStage);
            mbar_arrive_expect_tx(&full[s], nv * SL::kA1);
            for (int j = 0; j < nv; ++j)
              tma_load_3d(a_s + j * SL::kA1, tmA, &full[s], (kbs + j) * kBK, tl.fti * kBM, tl.expert, pol);
          }
        }
        if (!ok) break;
        const int nxt = (int)gridDim.x + atomicAdd(&p.unit_ctr[0], 1);   // claimed now, streamed next
        u = nxt < n_units ? nxt : -1;
      }
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------- B producer (two warps): gathered rows via cp.async
    // Lane l of B warp wi copies the 16-byte chunk c = l % 8 of rows 4 wi + l / 8 + 8 i of every
    // k-block (i < BNW / 8): its rows, its chunk and its swizzled destination offset are fixed
    // for a tile, so each lane looks its rows' source addresses up once per tile and a k-block
    // is just its copies (measured: the copy issue loop, not DRAM, had set the pace of wide tiles).
    const int wi = warp == 1 ? 0 : 1;               // each warp copies half of every stage
    constexpr int kRowsPerLane = BNW / 8;
    const int c8 = lane & 7;
    const int rbase = (lane >> 3) + 4 * wi;
    const uint32_t dst_off = (uint32_t)(rbase * 128 + ((c8 ^ (rbase & 7)) << 4));
    const char* pool = static_cast<const char*>(L.pool);
    // GEMM2: the h rows are GEMM1's output -- wait for it (the weight producer does not)
    if (MODE == kModeGemm2) griddep_wait();
    uint32_t it = 0, qi = 0;
    bool ok = true;
    for (int u = ring_get_warp(ring, qi, lane, abort_flag, C); u >= 0 && ok;
         u = ring_get_warp(ring, qi, lane, abort_flag, C)) {
      const Unit un = unit_of(u, n_whole, nchunk);
      const Tile tl = decode_tile<BN, BNW, MODE>(p, tb_s, un.t);
      const char* srow[kRowsPerLane];
#pragma unroll
      for (int i = 0; i < kRowsPerLane; ++i) {
        const int r = rbase + 8 * i;
        const char* rp = nullptr;
        if (r < tl.nj) {
          if (MODE == kModeAtt) {
            rp = static_cast<const char*>(p.sd.att_rowptr[tl.j0 + r]);
          } else if (MODE == kModeGemm2) {
            rp = reinterpret_cast<const char*>(p.hbuf) + (size_t)(tl.row_base + tl.j0 + r) * d.I * 2;
          } else {
            const int rec = record_checked(L, d, C, tl.expert, tl.head + tl.j0 + r);
            rp = rec >= 0 ? pool + (size_t)(rec >> kKShift) * d.H * 2 : nullptr;
          }
        }
        srow[i] = rp;
      }
      for (int ch = un.c0; ch < un.c1 && ok; ++ch) {
        const int kb1 = chunk_kb(ch + 1, nk, nchunk);
        for (int kbs = chunk_kb(ch, nk, nchunk); kbs < kb1; kbs += tl.kps, ++it) {
          const int nv = min(tl.kps, kb1 - kbs);
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          const bool w_ok = mbar_wait(&empty[s], ph ^ 1u, abort_flag, C);
          if (!(ok = __all_sync(0xffffffffu, w_ok))) break;
          const uint32_t b_s = smem_u32(smem + s * SL::kStage) + tl.kps * SL::kA1;
          for (int j = 0; j < nv; ++j) {
            const uint32_t bs = b_s + j * tl.bstride + dst_off;
            const int col = (kbs + j) * kBK + c8 * 8;
            const bool colok = col < Kdim;
#pragma unroll
            for (int i = 0; i < kRowsPerLane; ++i) {
              if (rbase + 8 * i < tl.nmma) {
                const bool valid = srow[i] != nullptr && colok;
                cp_async16(bs + i * 1024, valid ? static_cast<const void*>(srow[i] + (size_t)col * 2)
                                                : static_cast<const void*>(pool),
                           valid ? 16u : 0u);
              }
            }
          }
          // each lane's copies arrive on the stage barrier when they complete -- no waiting
          // here, so the producer runs a full ring ahead; the consumer issues the generic ->
          // async proxy fence after it observes the barrier
          cp_async_arrive_noinc(&full[s]);
        }
      }
    }
    cp_async_wait<0>();
  } else if (warp == 2) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, acc_i = 0, qi = 0;
      bool ok = true;
      for (int u = ring_get(ring, qi, abort_flag, C); u >= 0 && ok; u = ring_get(ring, qi, abort_flag, C)) {
        const Unit un = unit_of(u, n_whole, nchunk);
        const Tile tl = decode_tile<BN, BNW, MODE>(p, tb_s, un.t);
        const uint32_t idesc = idesc_bf16(kBM, tl.nmma);
        // one accumulator buffer per chunk, in rotation, so the epilogue drains earlier chunks
        // while later ones accumulate
        for (int c = un.c0; c < un.c1 && ok; ++c, ++acc_i) {
          const int buf = acc_i % kAccBufs;
          const uint32_t tph = (acc_i / kAccBufs) & 1u;
          if (!(ok = mbar_wait(&tempty[buf], tph ^ 1u, abort_flag, C))) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BNW);
          const int kb0 = chunk_kb(c, nk, nchunk), kb1 = chunk_kb(c + 1, nk, nchunk);
          for (int kbs = kb0; kbs < kb1; kbs += tl.kps, ++it) {
            const int nv = min(tl.kps, kb1 - kbs);
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1u;
            if (!(ok = mbar_wait(&full[s], ph, abort_flag, C))) break;
            tc_fence_after();
            fence_proxy_async();                      // B came through cp.async (generic proxy)
            const uint32_t a_s = smem_u32(smem + s * SL::kStage);
            for (int j = 0; j < nv; ++j) {
              const uint32_t a0 = a_s + j * SL::kA1;
              const uint32_t b0 = a_s + tl.kps * SL::kA1 + j * tl.bstride;
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k)
                mma_bf16(d_tmem, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), idesc,
                         (kbs + j != kb0) || (k != 0));
            }
            mma_commit(&empty[s]);
          }
          if (ok) mma_commit(&tfull[buf]);
        }
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp - 4;                       // TMEM lane quarter
    const int et = threadIdx.x - 128;             // 0..127
    const int row = 32 * q + lane;                // accumulator row (A row of the tile)
    uint32_t acc_i = 0, qi = 0;
    for (int u = ring_get_warp(ring, qi, lane, abort_flag, C); u >= 0; u = ring_get_warp(ring, qi, lane, abort_flag, C)) {
      const Unit un = unit_of(u, n_whole, nchunk);
      const Tile tl = decode_tile<BN, BNW, MODE>(p, tb_s, un.t);
      if (MODE == kModeGemm2) {
        for (int j = et; j < tl.nj; j += 128) {
          const int rec = record_checked(L, d, C, tl.expert, tl.head + tl.j0 + j);
          slot_s[j] = rec >= 0 ? rec >> kKShift : -1;
          k_s[j] = rec >= 0 ? rec & kKMask : 0;
        }
      } else if (MODE == kModeAtt) {
        for (int j = et; j < tl.nj; j += 128) {
          slot_s[j] = p.sd.att_batch[tl.j0 + j];
          w_s[j] = p.sd.att_scale[tl.j0 + j];
        }
      }
      // chunk partials, added in ascending chunk order as each accumulator completes
      float acc[BNW];
      bool ok = true;
      for (int c = un.c0; c < un.c1; ++c, ++acc_i) {
        const int buf = acc_i % kAccBufs;
        const uint32_t tph = (acc_i / kAccBufs) & 1u;
        const bool w_ok = mbar_wait(&tfull[buf], tph, abort_flag, C);
        if (!(ok = epi_bar_and(w_ok))) break;
        tc_fence_after();
        const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BNW);
#pragma unroll
        for (int c0 = 0; c0 < BNW; c0 += 16) {
          if (c0 < tl.nj) {
            float v[16];
            tmem_ld16(tbase + c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[c0 + j] = c == un.c0 ? v[j] : acc[c0 + j] + v[j];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
      }
      if (!ok) break;
      if (un.split) {
        // this unit holds one chunk of the tile: publish its partial; the unit that arrives
        // last adds all partials of the tile in chunk order and runs the epilogue
        // partials as [chunk][column / 4][row] float4 groups: a warp's 32 rows store (and the
        // fold later loads) 512 contiguous bytes per instruction
        const int st = un.t - n_whole;              // split tiles: [0, split_cap)
        float4* wt = reinterpret_cast<float4*>(p.ws + (size_t)st * nchunk * BNW * kBM);
#pragma unroll
        for (int c0 = 0; c0 < BNW; c0 += 16) {
          if (c0 < tl.nj) {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              __stcg(wt + ((size_t)un.c0 * (BNW / 4) + (c0 + j) / 4) * kBM + row,
                     make_float4(acc[c0 + j], acc[c0 + j + 1], acc[c0 + j + 2], acc[c0 + j + 3]));
          }
        }
        __threadfence();
        EpiBarrier{}();
        if (et == 0) {
          const int old = atomicAdd(p.cnt + st, 1);
          const int last = old == nchunk - 1;
          if (last) p.cnt[st] = 0;                // every arrival of this launch is in
          *last_flag = last;
        }
        EpiBarrier{}();
        if (!*last_flag) continue;
        __threadfence();
        // 12 columns of every chunk in flight at once (a group may read workspace columns past
        // nj that no unit wrote this launch: in bounds, and their sums are never stored), then
        // the adds in ascending chunk order
#pragma unroll
        for (int c0 = 0; c0 < BNW; c0 += 12) {
          if (c0 < tl.nj) {
            float4 v[kMaxChunks][3];
#pragma unroll
            for (int c = 0; c < kMaxChunks; ++c) {
              if (c < nchunk) {
#pragma unroll
                for (int j = 0; j < 3; ++j)
                  if (c0 + 4 * j < BNW) v[c][j] = __ldcg(wt + ((size_t)c * (BNW / 4) + c0 / 4 + j) * kBM + row);
              }
            }
#pragma unroll
            for (int j = 0; j < 3; ++j) {
              if (c0 + 4 * j >= BNW) continue;
              float4 a = v[0][j];
#pragma unroll
              for (int c = 1; c < kMaxChunks; ++c) {
                if (c < nchunk) {
                  a.x += v[c][j].x;
                  a.y += v[c][j].y;
                  a.z += v[c][j].z;
                  a.w += v[c][j].w;
                }
              }
              acc[c0 + 4 * j] = a.x;
              acc[c0 + 4 * j + 1] = a.y;
              acc[c0 + 4 * j + 2] = a.z;
              acc[c0 + 4 * j + 3] = a.w;
            }
          }
        }
      }
      if (MODE == kModeGemm1) {
        const int f = tl.fti * (kBM / 2) + 16 * q + (lane & 15);       // feature of this lane pair
        const bool lo = lane < 16;
#pragma unroll
        for (int c0 = 0; c0 < BNW; c0 += 16) {
          if (c0 < tl.nj) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float send = lo ? acc[c0 + 8 + j] : acc[c0 + j];
              const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
              const int col = c0 + (lo ? j : 8 + j);
              const float g = lo ? acc[c0 + j] : recv;
              const float uu = lo ? recv : acc[c0 + 8 + j];
              if (col < tl.nj && f < d.I)
                p.hbuf[(size_t)(tl.row_base + tl.j0 + col) * d.I + f] = __float2bfloat16_rn(silu_f(g) * uu);
            }
          }
        }
      } else if (MODE == kModeGemm2) {
        // E_k(x) rounded to bf16 (the activation dtype); the merge applies the top-k weight
        const int f = tl.fti * kBM + row;                               // output feature of H
        __nv_bfloat16* rows = static_cast<__nv_bfloat16*>(L.slotbuf);
        if (f < d.H) {
#pragma unroll
          for (int c0 = 0; c0 < BNW; c0 += 16) {
            if (c0 < tl.nj) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int col = c0 + j;
                if (col < tl.nj && (!kDebugBounds || slot_s[col] >= 0))
                  rows[((size_t)slot_s[col] * d.KS + k_s[col]) * d.H + f] = __float2bfloat16_rn(acc[col]);
              }
            }
          }
        }
      } else {
        // attention stub: a = RMSNorm(x) P = s * (x P), written to the token pool of the layer
        const int f = tl.fti * kBM + row;
        __nv_bfloat16* pool = static_cast<__nv_bfloat16*>(L.pool);
        if (f < d.H) {
#pragma unroll
          for (int c0 = 0; c0 < BNW; c0 += 16) {
            if (c0 < tl.nj) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int col = c0 + j;
                if (col < tl.nj) pool[(size_t)slot_s[col] * d.H + f] = __float2bfloat16_rn(w_s[col] * acc[col]);
              }
            }
          }
        }
      }
      if (MODE == kModeGemm2 && p.stream_on)        // streaming runtime: merge in place (its
        land_and_merge<__nv_bfloat16>(L, d, C, slot_s, tl.nj, tl.fti, p.parts, tl.fti * kBM, kBM, et, 128, fin,
                                      EpiBarrier{}, tl.step, &p.sd, layer);   // next tick reads it)
      else if (MODE == kModeGemm2)                   // per-layer path: collect merges ready tokens
        land_only(L, d, C, slot_s, tl.nj, p.parts, et, 128, EpiBarrier{}, tl.step);
      else
        asm volatile("bar.sync 1, 128;" ::: "memory");   // slot_s / w_s / last_flag reused by the next unit
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) unit_ctr_exit(p.unit_ctr);
  if (warp == 2) {
    __syncwarp();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side

struct TcState {
  TcParams gemm1, gemm2, att;       // parameter blocks (tensor maps of every layer)
  bool att_ready;
  int* unit_ctr;                    // two counters per parameter block, zeroed once
  void* split_buf[2];               // GEMM1 / GEMM2 chunk-partial workspace + arrival counters
};

// Token-tile width and pipeline depth.  Measured on GB300 (bench c2/c3/c4, pairs/s): 32-token
// tiles suit decode and steps with few experts (more CTAs per expert); prefill with very
// popular experts prefers wider tiles (64: c3 +9%, c2 -1.7%, c4 -22%).  Earlier stage sweeps
// (k-blocks x stages, same tile): 1 x 10 -- c2 176.5 K, c3 2.61 M, c4 1.08 M; 2 x 5 -- 179.1 K,
// 2.79 M, 1.15 M; 3 x 3 -- 181.8 K, 2.92 M, 1.19 M; 4 x 2 -- 175.3 K, 2.91 M, 1.18 M.
#ifndef MOE_TC_BN
#define MOE_TC_BN 32
#endif
constexpr int kBN = MOE_TC_BN;
constexpr int kBNW = kWideMin1 > 0 && kWideMin2 > 0 && MOE_TC_BNW > MOE_TC_BN ? MOE_TC_BNW : MOE_TC_BN;
constexpr int kStages = kStagesCfg;

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 3-D map over packed weights [NB][rows][K] (bf16, K contiguous), box 64 x 128 x 1, 128B swizzle,
// zero fill outside the tensor (ragged K and ragged row tails).
bool encode_weights(CUtensorMap* m, const void* base, int K, int rows, int nb) {
  auto fn = get_encode();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)nb};
  cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)K * 2 * rows};
  cuuint32_t box[3] = {kBK, kBM, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, int BNW, int STAGES, int MODE>
cudaError_t set_attrs() {
  using SL = SmemLayout<BN, BNW, STAGES>;
  return cudaFuncSetAttribute(ffn_tc_kernel<BN, BNW, STAGES, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              SL::kAlloc);
}

// GEMM1 and GEMM2 are launched as programmatic dependents of the kernel before them (PDL):
// their CTAs may start early and order themselves with griddepcontrol.wait.
template <int BN, int BNW, int STAGES, int MODE>
cudaError_t launch_one(moe_async_s* h, const TcParams& prm, cudaStream_t s) {
  using SL = SmemLayout<BN, BNW, STAGES>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(h->num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SL::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = MODE == kModeAtt ? 0 : 1;
  return cudaLaunchKernelEx(&cfg, ffn_tc_kernel<BN, BNW, STAGES, MODE>, prm);
}

void fill_common(moe_async_s* h, TcParams& p) {
  for (int l = 0; l < h->cfg.num_layers; ++l) p.views[l] = h->layers[l];
  p.d = h->dims;
  p.C = h->counters;
  p.P = h->plan;
  p.hbuf = static_cast<__nv_bfloat16*>(h->h);
  p.parts = h->parts_per_pair;
  p.stream_on = 0;
  p.nchunk = 1;
  p.split_cap = 0;
  p.ws = nullptr;
  p.cnt = nullptr;
  p.unit_ctr = nullptr;
}

// K chunks for a contraction of nk k-blocks: 1, 2 or 4 chunks of at least MOE_SPLIT_MIN_KB
// k-blocks each, so a chunk's partial (BN x 128 fp32) stays small next to the weight bytes
// the chunk streams.  Measured on GB300 (pairs/s): 24 leaves the GPT-OSS shapes (45 k-blocks)
// whole and cuts the 7168-deep GEMM1 of the DeepSeek-wide layer in 4 -- c4 +15%; 16 also
// cuts the GPT-OSS GEMMs in 2, which costs decode 0.5% and prefill 1.2%.
#ifndef MOE_SPLIT_MIN_KB
#define MOE_SPLIT_MIN_KB 24
#endif
int chunks_for(int nk) {
  const int q = nk / MOE_SPLIT_MIN_KB;
  return q >= kMaxChunks ? kMaxChunks : q >= 2 ? 2 : 1;
}

// Workspace for launches that split tiles over their K chunks: up to two tiles per SM.
cudaError_t setup_split(moe_async_s* h, TcParams& p, int K, void** buf) {
  const int nk = (K + kBK - 1) / kBK;
  p.nchunk = chunks_for(nk);
  if (p.nchunk == 1) return cudaSuccess;
  p.split_cap = 2 * h->num_sms;
  const size_t ws_bytes = (size_t)p.split_cap * p.nchunk * kBNW * kBM * sizeof(float);
  const size_t cnt_bytes = (size_t)p.split_cap * sizeof(int);
  cudaError_t e = cudaMalloc(buf, ws_bytes + cnt_bytes);
  if (e != cudaSuccess) return e;
  p.ws = static_cast<float*>(*buf);
  p.cnt = reinterpret_cast<int*>(static_cast<char*>(*buf) + ws_bytes);
  return cudaMemset(p.cnt, 0, cnt_bytes);
}

}  // namespace

TileGeom tc_geom() { return TileGeom{kBN, kBM, kBN, kBM, kBNW > kBN ? kBNW : 0, kWideMin1, kWideMin2}; }

moe_status tc_setup(moe_async_s* h) {
  if (h->cfg.num_layers > kMaxLayers) return MOE_ERR_UNSUPPORTED;
  // dynamic shared memory limits, set once per handle outside any stream capture
  if (set_attrs<kBN, kBNW, kStages, kModeGemm1>() != cudaSuccess ||
      set_attrs<kBN, kBNW, kStages, kModeGemm2>() != cudaSuccess ||
      set_attrs<kBN, kBNW, kStages, kModeAtt>() != cudaSuccess)
    return MOE_ERR_CUDA;
  TcState* st = new (std::nothrow) TcState();
  if (!st) return MOE_ERR_CUDA;
  std::memset(static_cast<void*>(st), 0, sizeof(TcState));
  const Dims& d = h->dims;
  fill_common(h, st->gemm1);
  fill_common(h, st->gemm2);
  for (int l = 0; l < h->cfg.num_layers; ++l) {
    if (!encode_weights(&st->gemm1.mapA[l], h->layers[l].w13, d.H, 2 * d.I, d.NB) ||
        !encode_weights(&st->gemm2.mapA[l], h->layers[l].w2, d.I, d.H, d.NB)) {
      delete st;
      return MOE_ERR_CUDA;
    }
  }
  h->tc_state = st;
  if (cudaMalloc(&st->unit_ctr, 6 * sizeof(int)) != cudaSuccess) {
    st->unit_ctr = nullptr;
    tc_teardown(h);
    return MOE_ERR_CUDA;
  }
  st->gemm1.unit_ctr = st->unit_ctr;
  st->gemm2.unit_ctr = st->unit_ctr + 2;
  if (cudaMemset(st->unit_ctr, 0, 6 * sizeof(int)) != cudaSuccess ||
      setup_split(h, st->gemm1, d.H, &st->split_buf[0]) != cudaSuccess ||
      setup_split(h, st->gemm2, d.I, &st->split_buf[1]) != cudaSuccess) {
    tc_teardown(h);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

void tc_teardown(moe_async_s* h) {
  TcState* st = static_cast<TcState*>(h->tc_state);
  if (st) {
    for (void* b : st->split_buf)
      if (b) cudaFree(b);
    if (st->unit_ctr) cudaFree(st->unit_ctr);
  }
  delete st;
  h->tc_state = nullptr;
}

moe_status launch_ffn_tc(moe_async_s* h, int layer, cudaStream_t s) {
  (void)layer;                                     // the plan carries the layer
  TcState* st = static_cast<TcState*>(h->tc_state);
  if (!st) return MOE_ERR_INVALID;
  prof_begin(h, MOE_KERNEL_FFN1, s);
  cudaError_t e = launch_one<kBN, kBNW, kStages, kModeGemm1>(h, st->gemm1, s);
  prof_end(h, MOE_KERNEL_FFN1, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  prof_begin(h, MOE_KERNEL_FFN2, s);
  e = launch_one<kBN, kBNW, kStages, kModeGemm2>(h, st->gemm2, s);
  prof_end(h, MOE_KERNEL_FFN2, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Streaming runtime: attach the attention-stub projections (packed P^T per layer) and the
// stream state; GEMM2 merges then feed the streaming runtime.
moe_status tc_stream_setup(moe_async_s* h, const void* const* proj_packed, const StreamDev& sd) {
  TcState* st = static_cast<TcState*>(h->tc_state);
  if (!st) return MOE_ERR_UNSUPPORTED;
  fill_common(h, st->att);
  st->att.unit_ctr = st->unit_ctr + 4;
  for (int l = 0; l < h->cfg.num_layers; ++l)
    if (!encode_weights(&st->att.mapA[l], proj_packed[l], h->dims.H, h->dims.H, 1)) return MOE_ERR_CUDA;
  st->att.sd = sd;
  st->att.stream_on = 1;
  st->gemm2.sd = sd;
  st->gemm2.stream_on = 1;
  st->att_ready = true;
  return MOE_OK;
}

moe_status launch_att_tc(moe_async_s* h, cudaStream_t s) {
  TcState* st = static_cast<TcState*>(h->tc_state);
  if (!st || !st->att_ready) return MOE_ERR_INVALID;
  return launch_one<kBN, kBNW, kStages, kModeAtt>(h, st->att, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
