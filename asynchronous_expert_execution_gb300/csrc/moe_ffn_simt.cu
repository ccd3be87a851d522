// Expert FFN on CUDA cores: the fp32 path (fp32 FMA throughout, so results meet a 1e-5
// relative bound that tf32 tensor cores cannot) and the identity-expert test mode.
//
// Both consume the step plan written by the scheduling kernel: a list of picked buckets,
// each drained whole, whose tokens form one contiguous batch (StreamEP section 3, step 4:
// scattered inputs are reorganised into a contiguous batch before expert compute).  The
// gather is fused into GEMM1's operand load (token rows read from the pool by the slot
// stored in each queue record); GEMM2's epilogue writes each result row E_k(x) and counts
// the token's landings, and the top-k merge y = sum_k w_k E_k(x) runs in collect.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kBF = 32;    // GEMM1 features per tile (64 packed gate/up rows)
constexpr int kBT = 16;    // tokens per tile
constexpr int kKC = 32;    // reduction chunk
constexpr int kBH = 64;    // GEMM2 output features (of H) per tile

// GEMM1 + SwiGLU: h[row, f] = silu(sum_c x[c] W1[c, f]) * (sum_c x[c] W3[c, f]) for the
// tile's 16 gathered tokens and 32 features.  Packed W13 row of gate feature f is
// 32*(f/16) + f%16, its up row 16 further.
template <typename T>
__global__ void __launch_bounds__(256) ffn1_simt_kernel(LayerView L, Dims d, DevCounters* C,
                                                        const StepPlan* __restrict__ P, T* __restrict__ hbuf) {
  __shared__ float xs[kBT][kKC + 1];
  __shared__ float gs[kBF][kKC + 1];
  __shared__ float us[kBF][kKC + 1];
  __shared__ int slot_s[kBT];
  const int tid = threadIdx.x;
  const int n_tiles = P->n_tiles1;
  const int ftiles = (d.I + kBF - 1) / kBF;
  const T* pool = static_cast<const T*>(L.pool);
  const T* w13 = static_cast<const T*>(L.w13);
  for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const WorkItem it = P->items[find_item(P, t, false)];
    const int local = t - it.t1_base;
    const int ntt = (it.count + kBT - 1) / kBT;
    const int fti = local / ntt, tti = local % ntt;
    (void)ftiles;
    const int f0 = fti * kBF, j0 = tti * kBT;
    const int nj = min(kBT, it.count - j0);
    if (tid < kBT) {
      const int rec = tid < nj ? record_checked(L, d, C, it.expert, it.head + j0 + tid) : -1;
      slot_s[tid] = rec >= 0 ? rec >> kKShift : -1;
    }
    __syncthreads();
    const int tx = tid & 31, ty = tid >> 5;
    float g0 = 0.f, g1 = 0.f, u0 = 0.f, u1 = 0.f;
    const size_t ebase = (size_t)it.expert * 2 * d.I;
    for (int k0 = 0; k0 < d.H; k0 += kKC) {
      for (int q = tid; q < kBT * kKC; q += 256) {
        const int r = q / kKC, c = q % kKC;
        const int sl = slot_s[r];
        xs[r][c] = (sl >= 0 && k0 + c < d.H) ? to_f(pool[(size_t)sl * d.H + k0 + c]) : 0.f;
      }
      for (int q = tid; q < kBF * kKC; q += 256) {
        const int r = q / kKC, c = q % kKC;
        const int f = f0 + r;
        float gv = 0.f, uv = 0.f;
        if (f < d.I && k0 + c < d.H) {
          const size_t grow = ebase + 32 * (f / 16) + (f % 16);
          gv = to_f(w13[grow * d.H + k0 + c]);
          uv = to_f(w13[(grow + 16) * d.H + k0 + c]);
        }
        gs[r][c] = gv;
        us[r][c] = uv;
      }
      __syncthreads();
#pragma unroll 8
      for (int c = 0; c < kKC; ++c) {
        const float gw = gs[tx][c], uw = us[tx][c];
        const float xa = xs[ty][c], xb = xs[ty + 8][c];
        g0 = fmaf(gw, xa, g0);
        u0 = fmaf(uw, xa, u0);
        g1 = fmaf(gw, xb, g1);
        u1 = fmaf(uw, xb, u1);
      }
      __syncthreads();
    }
    const int f = f0 + tx;
    if (f < d.I) {
      if (ty < nj) hbuf[(size_t)(it.row_base + j0 + ty) * d.I + f] = from_f<T>(silu_f(g0) * u0);
      if (ty + 8 < nj) hbuf[(size_t)(it.row_base + j0 + ty + 8) * d.I + f] = from_f<T>(silu_f(g1) * u1);
    }
    __syncthreads();
  }
}

// GEMM2 + scatter + landing: o[f] = sum_i h[i] W2[i, f] for 64 features of H and 16 tokens;
// slotbuf[slot][k][f] = o[f] (the layer dtype); the merge applies the top-k weights.
template <typename T>
__global__ void __launch_bounds__(256) ffn2_simt_kernel(LayerView L, Dims d, DevCounters* C,
                                                        const StepPlan* __restrict__ P,
                                                        const T* __restrict__ hbuf, int parts) {
  __shared__ float hs[kBT][kKC + 1];
  __shared__ float ws[kBH][kKC + 1];
  __shared__ int slot_s[kBT], k_s[kBT];
  const int tid = threadIdx.x;
  const int n_tiles = P->n_tiles2;
  const T* w2 = static_cast<const T*>(L.w2);
  T* rows = static_cast<T*>(L.slotbuf);
  for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const WorkItem it = P->items[find_item(P, t, true)];
    const int local = t - it.t2_base;
    const int ntt = (it.count + kBT - 1) / kBT;
    const int fti = local / ntt, tti = local % ntt;
    const int f0 = fti * kBH, j0 = tti * kBT;
    const int nj = min(kBT, it.count - j0);
    if (tid < kBT) {
      int sl = -1, kk = 0;
      if (tid < nj) {
        const int rec = record_checked(L, d, C, it.expert, it.head + j0 + tid);
        if (rec >= 0) {
          sl = rec >> kKShift;
          kk = rec & kKMask;
        }
      }
      slot_s[tid] = sl; k_s[tid] = kk;
    }
    __syncthreads();
    const int tx = tid & 63, ty = tid >> 6;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const size_t ebase = (size_t)it.expert * d.H;
    for (int k0 = 0; k0 < d.I; k0 += kKC) {
      for (int q = tid; q < kBT * kKC; q += 256) {
        const int r = q / kKC, c = q % kKC;
        hs[r][c] = (r < nj && k0 + c < d.I) ? to_f(hbuf[(size_t)(it.row_base + j0 + r) * d.I + k0 + c]) : 0.f;
      }
      for (int q = tid; q < kBH * kKC; q += 256) {
        const int r = q / kKC, c = q % kKC;
        const int f = f0 + r;
        ws[r][c] = (f < d.H && k0 + c < d.I) ? to_f(w2[(ebase + f) * d.I + k0 + c]) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int c = 0; c < kKC; ++c) {
        const float wv = ws[tx][c];
#pragma unroll
        for (int m = 0; m < 4; ++m) acc[m] = fmaf(wv, hs[ty + 4 * m][c], acc[m]);
      }
      __syncthreads();
    }
    const int f = f0 + tx;
    if (f < d.H) {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int j = ty + 4 * m;
        if (j < nj && (!kDebugBounds || slot_s[j] >= 0))
          rows[((size_t)slot_s[j] * d.KS + k_s[j]) * d.H + f] = from_f<T>(acc[m]);
      }
    }
    land_only(L, d, C, slot_s, nj, parts, tid, 256, CtaBarrier{}, it.step);
  }
}

// Identity experts: slotbuf[slot][k] = x (one part per pair), then landing.
template <typename T>
__global__ void __launch_bounds__(256) identity_kernel(LayerView L, Dims d, DevCounters* C,
                                                       const StepPlan* __restrict__ P) {
  __shared__ int slot_s[kBT], k_s[kBT];
  const int tid = threadIdx.x;
  const int n_tiles = P->n_tiles2;
  const T* pool = static_cast<const T*>(L.pool);
  for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const WorkItem it = P->items[find_item(P, t, true)];
    const int j0 = (t - it.t2_base) * kBT;
    const int nj = min(kBT, it.count - j0);
    if (tid < kBT) {
      int sl = -1, kk = 0;
      if (tid < nj) {
        const int rec = record_checked(L, d, C, it.expert, it.head + j0 + tid);
        if (rec >= 0) {
          sl = rec >> kKShift;
          kk = rec & kKMask;
        }
      }
      slot_s[tid] = sl; k_s[tid] = kk;
    }
    __syncthreads();
    for (int j = 0; j < nj; ++j) {
      if (kDebugBounds && slot_s[j] < 0) continue;
      const T* src = pool + (size_t)slot_s[j] * d.H;
      T* dst = static_cast<T*>(L.slotbuf) + ((size_t)slot_s[j] * d.KS + k_s[j]) * d.H;
      for (int f = tid; f < d.H; f += 256) dst[f] = src[f];
    }
    land_only(L, d, C, slot_s, nj, 1, tid, 256, CtaBarrier{}, it.step);
  }
}

}  // namespace

TileGeom simt_geom() { return TileGeom{kBT, 2 * kBF, kBT, kBH, 0, 0, 0}; }

moe_status launch_ffn_simt(moe_async_s* h, int layer, cudaStream_t s) {
  const Dims& d = h->dims;
  const LayerView& L = h->layers[layer];
  const int grid = h->num_sms * 4;
  const int parts = h->parts_per_pair;
  prof_begin(h, MOE_KERNEL_FFN1, s);
  if (d.dtype == MOE_BF16)
    ffn1_simt_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(L, d, h->counters, h->plan, static_cast<__nv_bfloat16*>(h->h));
  else
    ffn1_simt_kernel<float><<<grid, 256, 0, s>>>(L, d, h->counters, h->plan, static_cast<float*>(h->h));
  prof_end(h, MOE_KERNEL_FFN1, s);
  prof_begin(h, MOE_KERNEL_FFN2, s);
  if (d.dtype == MOE_BF16)
    ffn2_simt_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(L, d, h->counters, h->plan,
                                                          static_cast<const __nv_bfloat16*>(h->h), parts);
  else
    ffn2_simt_kernel<float><<<grid, 256, 0, s>>>(L, d, h->counters, h->plan,
                                                  static_cast<const float*>(h->h), parts);
  prof_end(h, MOE_KERNEL_FFN2, s);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_identity(moe_async_s* h, int layer, cudaStream_t s) {
  const Dims& d = h->dims;
  const int grid = h->num_sms * 4;
  prof_begin(h, MOE_KERNEL_FFN1, s);
  if (d.dtype == MOE_BF16)
    identity_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(h->layers[layer], d, h->counters, h->plan);
  else
    identity_kernel<float><<<grid, 256, 0, s>>>(h->layers[layer], d, h->counters, h->plan);
  prof_end(h, MOE_KERNEL_FFN1, s);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
