// Elementwise feature-map kernels for the backward pass with a feature map.
//
// Causal linear attention ("Transformers are RNNs") feeds the causal product
// phi(q) and phi(k) with phi(x) = elu(x) + 1 (x + 1 for x > 0, e^x
// otherwise).  The forward pass applies phi inside the product kernels; the
// backward pass runs the product backward on phi(q), phi(k) written by
// feature_map_launch, then turns dL/dphi into dL/dx with feature_grad_launch:
//     dL/dx = dL/dphi * phi'(x),   phi'(x) = 1 for x > 0, e^x otherwise.
// Both are single sweeps over contiguous tensors: 16-byte accesses, a grid
// of a few CTAs per SM striding over the elements.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cp_internal.h"

namespace cp {
namespace {

constexpr int kFeatThreads = 256;

__device__ __forceinline__ float phi(float x) { return x > 0.f ? x + 1.f : expf(x); }
__device__ __forceinline__ float dphi(float x) { return x > 0.f ? 1.f : expf(x); }

// one 16-byte chunk: 8 bf16 or 4 f32 values
template <typename T>
struct Chunk;
template <>
struct Chunk<__nv_bfloat16> {
  static constexpr int kN = 8;
  static __device__ __forceinline__ void load(const void* p, int64_t c, float* f) {
    const uint4 w = __ldg(static_cast<const uint4*>(p) + c);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = __uint_as_float(u[j] << 16);
      f[2 * j + 1] = __uint_as_float(u[j] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ void load_rw(const void* p, int64_t c, float* f) {
    const uint4 w = static_cast<const uint4*>(p)[c];
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = __uint_as_float(u[j] << 16);
      f[2 * j + 1] = __uint_as_float(u[j] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ void store(void* p, int64_t c, const float* f) {
    uint4 w;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
    static_cast<uint4*>(p)[c] = w;
  }
  static __device__ __forceinline__ float elem(const void* p, int64_t i) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  }
  static __device__ __forceinline__ void set(void* p, int64_t i, float x) {
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
  }
};
template <>
struct Chunk<__half> {
  static constexpr int kN = 8;
  static __device__ __forceinline__ void from_word(const uint4& w, float* f) {
    const __half2* h = reinterpret_cast<const __half2*>(&w);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 t = __half22float2(h[j]);
      f[2 * j] = t.x;
      f[2 * j + 1] = t.y;
    }
  }
  static __device__ __forceinline__ void load(const void* p, int64_t c, float* f) {
    from_word(__ldg(static_cast<const uint4*>(p) + c), f);
  }
  static __device__ __forceinline__ void load_rw(const void* p, int64_t c, float* f) {
    from_word(static_cast<const uint4*>(p)[c], f);
  }
  static __device__ __forceinline__ void store(void* p, int64_t c, const float* f) {
    uint4 w;
    __half2* h = reinterpret_cast<__half2*>(&w);
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = __floats2half2_rn(f[2 * j], f[2 * j + 1]);
    static_cast<uint4*>(p)[c] = w;
  }
  static __device__ __forceinline__ float elem(const void* p, int64_t i) {
    return __half2float(static_cast<const __half*>(p)[i]);
  }
  static __device__ __forceinline__ void set(void* p, int64_t i, float x) {
    static_cast<__half*>(p)[i] = __float2half_rn(x);
  }
};

template <>
struct Chunk<float> {
  static constexpr int kN = 4;
  static __device__ __forceinline__ void load(const void* p, int64_t c, float* f) {
    const float4 w = __ldg(static_cast<const float4*>(p) + c);
    f[0] = w.x;
    f[1] = w.y;
    f[2] = w.z;
    f[3] = w.w;
  }
  static __device__ __forceinline__ void load_rw(const void* p, int64_t c, float* f) {
    const float4 w = static_cast<const float4*>(p)[c];
    f[0] = w.x;
    f[1] = w.y;
    f[2] = w.z;
    f[3] = w.w;
  }
  static __device__ __forceinline__ void store(void* p, int64_t c, const float* f) {
    static_cast<float4*>(p)[c] = make_float4(f[0], f[1], f[2], f[3]);
  }
  static __device__ __forceinline__ float elem(const void* p, int64_t i) {
    return static_cast<const float*>(p)[i];
  }
  static __device__ __forceinline__ void set(void* p, int64_t i, float x) {
    static_cast<float*>(p)[i] = x;
  }
};

// GRAD = false: y = phi(x).  GRAD = true: y *= phi'(x) (y read and written).
template <typename T, bool GRAD>
__global__ void __launch_bounds__(kFeatThreads) feature_kernel(const void* x, void* y, int64_t n) {
  using C = Chunk<T>;
  const int64_t n_chunks = n / C::kN;
  const int64_t stride = (int64_t)gridDim.x * kFeatThreads;
  for (int64_t c = (int64_t)blockIdx.x * kFeatThreads + threadIdx.x; c < n_chunks; c += stride) {
    float f[C::kN], o[C::kN];
    C::load(x, c, f);
    if (GRAD) C::load_rw(y, c, o);
#pragma unroll
    for (int j = 0; j < C::kN; ++j) o[j] = GRAD ? o[j] * dphi(f[j]) : phi(f[j]);
    C::store(y, c, o);
  }
  // the tail that does not fill a chunk
  for (int64_t i = n_chunks * C::kN + (int64_t)blockIdx.x * kFeatThreads + threadIdx.x; i < n;
       i += stride) {
    const float f = C::elem(x, i);
    C::set(y, i, GRAD ? C::elem(y, i) * dphi(f) : phi(f));
  }
}

template <bool GRAD>
cudaError_t feature_run(const void* x, void* y, int64_t n, cp_dtype_t dtype, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  int dev = 0, n_sm = kPlanSMs;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  const int64_t per = dtype == CP_DTYPE_F32 ? 4 : 8;
  const int64_t want = (n / per + kFeatThreads - 1) / kFeatThreads;
  const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, 8LL * n_sm));
  if (dtype == CP_DTYPE_BF16)
    feature_kernel<__nv_bfloat16, GRAD><<<grid, kFeatThreads, 0, st>>>(x, y, n);
  else if (dtype == CP_DTYPE_F16)
    feature_kernel<__half, GRAD><<<grid, kFeatThreads, 0, st>>>(x, y, n);
  else
    feature_kernel<float, GRAD><<<grid, kFeatThreads, 0, st>>>(x, y, n);
  return cudaGetLastError();
}

}  // namespace

cudaError_t feature_map_launch(int feature, const void* x, void* y, int64_t n, cp_dtype_t dtype,
                               cudaStream_t stream) {
  if (feature != CP_FEATURE_ELU1) return cudaErrorInvalidValue;
  return feature_run<false>(x, y, n, dtype, stream);
}

cudaError_t feature_grad_launch(int feature, const void* x, void* g, int64_t n,
                                cp_dtype_t dtype, cudaStream_t stream) {
  if (feature != CP_FEATURE_ELU1) return cudaErrorInvalidValue;
  return feature_run<true>(x, g, n, dtype, stream);
}

}  // namespace cp
