// moe_async_forward_noalloc: one routed MoE layer forward that allocates no device memory.
//
// Who needs it: callers that cannot call cudaMalloc at the point they run the layer -- code
// running while a memory pool owns the whole device, allocation-free real-time or embedded
// runtimes, plugins handed only input/output buffers by a host framework.  The regular path
// (moe_async_create ...) allocates its pool, queues and combine slots up front; this entry
// point instead uses one fixed scratch array compiled into the library.
//
// What it computes: y[t] = sum over k = 0..K-1 (ascending) of w[t,k] * E_{e[t,k]}(x[t]) with
// SwiGLU experts E(x) = (silu(x W1) * (x W3)) W2, i.e. the same merged output as the
// asynchronous path for the same routed batch (no shared expert here).  Two kernels, both on
// CUDA cores with fp32 accumulation: the first writes the SwiGLU activations h of every
// (token, k) pair into the scratch array, the second reads them back for the down
// projection and the weighted merge.
#include <algorithm>
#include "moe_internal.cuh"

namespace moe {
namespace {

// Scratch: h[T*K][I] fp32.  16 MiB, resident on every GPU that loads the library until exit.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

// Device address of the scratch array in the current context.  The array's name is only a
// host-side stand-in, so the address is looked up with cudaGetSymbolAddress -- on every call:
// the lookup is a host-side table read, and a cached address would go stale when the module
// is loaded again at another address (after cudaDeviceReset, or under another context made
// current by the caller).  The first lookup in a context may load the module; that first
// call belongs before any stream capture.
cudaError_t noalloc_scratch(float** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = static_cast<float*>(p);
  return cudaSuccess;
}

template <typename T>
__global__ void noalloc_h_kernel(int npairs, int K, int E, int H, int I, const T* __restrict__ x,
                                 const int32_t* __restrict__ expert, const T* __restrict__ w1,
                                 const T* __restrict__ w3, float* __restrict__ h) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= I) return;
  for (int p = blockIdx.y; p < npairs; p += gridDim.y) {
    const int e = expert[p];
    float g = 0.f, u = 0.f;
    if (e >= 0 && e < E) {
      const T* xr = x + (size_t)(p / K) * H;
      const T* a = w1 + (size_t)e * H * I + i;
      const T* b = w3 + (size_t)e * H * I + i;
      for (int c = 0; c < H; ++c) {
        const float xv = to_f(xr[c]);
        g = fmaf(xv, to_f(a[(size_t)c * I]), g);
        u = fmaf(xv, to_f(b[(size_t)c * I]), u);
      }
    }
    h[(size_t)p * I + i] = silu_f(g) * u;     // every element written: nothing starts at zero
  }
}

template <typename T>
__global__ void noalloc_y_kernel(int T_, int K, int E, int H, int I, const int32_t* __restrict__ expert,
                                 const float* __restrict__ wts, const T* __restrict__ w2,
                                 const float* __restrict__ h, T* __restrict__ y) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= H) return;
  for (int t = blockIdx.y; t < T_; t += gridDim.y) {
    float acc = 0.f;
    for (int k = 0; k < K; ++k) {
      const int p = t * K + k;
      const int e = expert[p];
      if (e < 0 || e >= E) continue;
      const float* hr = h + (size_t)p * I;
      const T* b = w2 + (size_t)e * I * H + j;
      float o = 0.f;
      for (int i = 0; i < I; ++i) o = fmaf(hr[i], to_f(b[(size_t)i * H]), o);
      acc += wts[p] * o;
    }
    y[(size_t)t * H + j] = from_f<T>(acc);
  }
}

template <typename T>
cudaError_t noalloc_launch(int T_, int E, int K, int H, int I, const void* x, const int32_t* expert,
                           const float* w, const void* w1, const void* w3, const void* w2, void* y,
                           float* scratch, cudaStream_t s) {
  const int npairs = T_ * K;
  dim3 g1((I + 127) / 128, (unsigned)std::min(npairs, 65535));
  noalloc_h_kernel<T><<<g1, 128, 0, s>>>(npairs, K, E, H, I, static_cast<const T*>(x), expert,
                                         static_cast<const T*>(w1), static_cast<const T*>(w3), scratch);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g2((H + 127) / 128, (unsigned)std::min(T_, 65535));
  noalloc_y_kernel<T><<<g2, 128, 0, s>>>(T_, K, E, H, I, expert, w, static_cast<const T*>(w2), scratch,
                                         static_cast<T*>(y));
  return cudaGetLastError();
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_async_forward_noalloc(int32_t T, int32_t E, int32_t K, int32_t H, int32_t I,
                                                int32_t dtype, const void* d_x, const int32_t* d_expert,
                                                const float* d_w, const void* d_w1, const void* d_w3,
                                                const void* d_w2, void* d_y, void* stream) {
  using namespace moe;
  if (T < 0 || E < 1 || K < 1 || K > E || H < 1 || I < 1 || (dtype != MOE_F32 && dtype != MOE_BF16))
    return MOE_ERR_INVALID;
  if (T == 0) return MOE_OK;
  if (!d_x || !d_expert || !d_w || !d_w1 || !d_w3 || !d_w2 || !d_y) return MOE_ERR_INVALID;
  if ((size_t)T * (size_t)K * (size_t)I * sizeof(float) > kNoAllocScratchBytes) return MOE_ERR_CAPACITY;
  float* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e =
      dtype == MOE_BF16
          ? noalloc_launch<__nv_bfloat16>(T, E, K, H, I, d_x, d_expert, d_w, d_w1, d_w3, d_w2, d_y, scratch, s)
          : noalloc_launch<float>(T, E, K, H, I, d_x, d_expert, d_w, d_w1, d_w3, d_w2, d_y, scratch, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
