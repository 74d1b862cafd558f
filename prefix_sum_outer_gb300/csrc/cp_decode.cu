// One decoding step of the recurrence for every (b, h): with the state S
// (fp32, D x M) carried between calls,
//     S <- S + k v^T,    out = S^T q        (the readout after the update),
// the loop body of triton-lang/triton issue #217 applied to a single row.
// The step is bound by the state's traffic (8 D M bytes per problem, read
// and written once): one CTA per problem streams its rows with consecutive
// threads on consecutive columns, so every state row moves in whole sectors.
// When M is a multiple of 4 the state moves in 16-byte accesses.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cp_internal.h"

namespace cp {
namespace {

constexpr int kDecThreads = 256;

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }

template <typename T>
__global__ void __launch_bounds__(kDecThreads)
    decode_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                  T* __restrict__ out, float* __restrict__ state, int D, int M) {
  extern __shared__ float sm[];
  float* qs = sm;          // [D]
  float* ks = qs + D;      // [D]
  float* vs = ks + D;      // [M]
  float* part = vs + M;    // [groups][M] partial readouts
  const int64_t p = blockIdx.x;
  for (int i = threadIdx.x; i < D; i += kDecThreads) {
    qs[i] = to_f32(q[p * D + i]);
    ks[i] = to_f32(k[p * D + i]);
  }
  for (int i = threadIdx.x; i < M; i += kDecThreads) vs[i] = to_f32(v[p * M + i]);
  __syncthreads();
  // thread -> (column m, row group g), rows g, g + groups, ...  (M <= 256)
  const int groups = kDecThreads / M;
  const int m = threadIdx.x % M, g = threadIdx.x / M;
  float* S = state + p * D * M;
  if (g < groups) {
    const float vm = vs[m];
    float acc = 0.f;
#pragma unroll 4
    for (int d = g; d < D; d += groups) {
      const float s = fmaf(ks[d], vm, S[(int64_t)d * M + m]);
      S[(int64_t)d * M + m] = s;
      acc = fmaf(qs[d], s, acc);
    }
    part[g * M + m] = acc;
  }
  __syncthreads();
  // fixed-order sum of the row groups' partial readouts
  for (int mm = threadIdx.x; mm < M; mm += kDecThreads) {
    float o = 0.f;
    for (int gg = 0; gg < groups; ++gg) o += part[gg * M + mm];
    out[p * M + mm] = from_f32<T>(o);
  }
}

// The same step with 16-byte state accesses (M % 4 == 0): a thread owns four
// consecutive columns of a row group and issues the loads of four rows
// before using them, so a CTA keeps its whole state tile in flight.
// STREAM: a state larger than half the L2 cannot stay there until the next
// step, so it is read and written with the evict-first (streaming) hints
// (B=512 H=16 D=M=64, 128 MiB of state: 48.1 against 43.6 us per step).
template <bool STREAM>
__device__ __forceinline__ float4 ld_state(const float4* p) {
  if constexpr (STREAM) return __ldcs(p);
  return *p;
}
template <bool STREAM>
__device__ __forceinline__ void st_state(float4* p, float4 v) {
  if constexpr (STREAM)
    __stcs(p, v);
  else
    *p = v;
}

template <typename T, bool STREAM>
__global__ void __launch_bounds__(kDecThreads)
    decode_kernel_v4(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     T* __restrict__ out, float* __restrict__ state, int D, int M) {
  extern __shared__ float sm[];
  float* qs = sm;          // [D]
  float* ks = qs + D;      // [D]
  float* vs = ks + D;      // [M]
  float* part = vs + M;    // [groups][M]
  const int64_t p = blockIdx.x;
  const int c4 = M / 4;                  // float4 columns
  const int groups = kDecThreads / c4;   // row groups (>= 4)
  const int cq = threadIdx.x % c4, g = threadIdx.x / c4;
  float4* S4 = reinterpret_cast<float4*>(state + p * D * M);
  // the first four rows' state loads do not depend on q, k, v: they go out
  // before the staging below, so the two latencies overlap
  float4 st[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int d = g + u * groups;
    if (g < groups && d < D) st[u] = ld_state<STREAM>(&S4[(int64_t)d * c4 + cq]);
  }
  for (int i = threadIdx.x; i < D; i += kDecThreads) {
    qs[i] = to_f32(q[p * D + i]);
    ks[i] = to_f32(k[p * D + i]);
  }
  for (int i = threadIdx.x; i < M; i += kDecThreads) vs[i] = to_f32(v[p * M + i]);
  __syncthreads();
  if (g < groups) {
    const float4 vm = make_float4(vs[4 * cq], vs[4 * cq + 1], vs[4 * cq + 2], vs[4 * cq + 3]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int d0 = g; d0 < D; d0 += 4 * groups) {
      if (d0 != g) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int d = d0 + u * groups;
          if (d < D) st[u] = ld_state<STREAM>(&S4[(int64_t)d * c4 + cq]);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int d = d0 + u * groups;
        if (d < D) {
          const float kd = ks[d], qd = qs[d];
          st[u].x = fmaf(kd, vm.x, st[u].x);
          st[u].y = fmaf(kd, vm.y, st[u].y);
          st[u].z = fmaf(kd, vm.z, st[u].z);
          st[u].w = fmaf(kd, vm.w, st[u].w);
          st_state<STREAM>(&S4[(int64_t)d * c4 + cq], st[u]);
          acc.x = fmaf(qd, st[u].x, acc.x);
          acc.y = fmaf(qd, st[u].y, acc.y);
          acc.z = fmaf(qd, st[u].z, acc.z);
          acc.w = fmaf(qd, st[u].w, acc.w);
        }
      }
    }
    float* pr = part + g * M + 4 * cq;
    pr[0] = acc.x;
    pr[1] = acc.y;
    pr[2] = acc.z;
    pr[3] = acc.w;
  }
  __syncthreads();
  // fixed-order sum of the row groups' partial readouts
  for (int mm = threadIdx.x; mm < M; mm += kDecThreads) {
    float o = 0.f;
    for (int gg = 0; gg < groups; ++gg) o += part[gg * M + mm];
    out[p * M + mm] = from_f32<T>(o);
  }
}

template <bool STREAM>
cudaError_t decode_v4(const void* q, const void* k, const void* v, void* out, float* state,
                      int64_t BH, int64_t D, int64_t M, cp_dtype_t dtype, size_t smem,
                      cudaStream_t stream) {
  if (dtype == CP_DTYPE_BF16)
    decode_kernel_v4<__nv_bfloat16, STREAM><<<(unsigned)BH, kDecThreads, smem, stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(v), static_cast<__nv_bfloat16*>(out), state, (int)D,
        (int)M);
  else if (dtype == CP_DTYPE_F16)
    decode_kernel_v4<__half, STREAM><<<(unsigned)BH, kDecThreads, smem, stream>>>(
        static_cast<const __half*>(q), static_cast<const __half*>(k),
        static_cast<const __half*>(v), static_cast<__half*>(out), state, (int)D, (int)M);
  else
    decode_kernel_v4<float, STREAM><<<(unsigned)BH, kDecThreads, smem, stream>>>(
        static_cast<const float*>(q), static_cast<const float*>(k),
        static_cast<const float*>(v), static_cast<float*>(out), state, (int)D, (int)M);
  return cudaGetLastError();
}

}  // namespace

size_t decode_smem_bytes(int64_t D, int64_t M) {
  return sizeof(float) * (size_t)(2 * D + M + (kDecThreads / M) * M);
}

cudaError_t decode_launch(const void* q, const void* k, const void* v, void* out, float* state,
                          int64_t BH, int64_t D, int64_t M, cp_dtype_t dtype,
                          cudaStream_t stream) {
  if (M % 4 == 0) {
    const size_t smem = sizeof(float) * (size_t)(2 * D + M + (kDecThreads / (M / 4)) * M);
    const bool stream_state = (size_t)BH * D * M * sizeof(float) > device_l2_bytes() / 2;
    return stream_state ? decode_v4<true>(q, k, v, out, state, BH, D, M, dtype, smem, stream)
                        : decode_v4<false>(q, k, v, out, state, BH, D, M, dtype, smem, stream);
  }
  const size_t smem = decode_smem_bytes(D, M);
  if (dtype == CP_DTYPE_BF16)
    decode_kernel<__nv_bfloat16><<<(unsigned)BH, kDecThreads, smem, stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(v), static_cast<__nv_bfloat16*>(out), state, (int)D,
        (int)M);
  else if (dtype == CP_DTYPE_F16)
    decode_kernel<__half><<<(unsigned)BH, kDecThreads, smem, stream>>>(
        static_cast<const __half*>(q), static_cast<const __half*>(k),
        static_cast<const __half*>(v), static_cast<__half*>(out), state, (int)D, (int)M);
  else
    decode_kernel<float><<<(unsigned)BH, kDecThreads, smem, stream>>>(
        static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
        static_cast<float*>(out), state, (int)D, (int)M);
  return cudaGetLastError();
}

}  // namespace cp
