// Exclusive scan over segment aggregates, between the two passes of a split
// scan.
//
// A problem whose sequence is split into G segments is scanned in two
// passes: the first writes each segment's own state sum (its aggregate,
// sum of k_j v_j^T over the segment's rows, or q_i g_i^T for a reverse
// scan), the second scans every segment from the state that precedes it.
// This kernel turns the aggregates into those starting states in place:
// slot s becomes the sum of the aggregates before s in scan order
// (s' < s for a forward scan, s' > s for a reverse one).  Each second-pass
// CTA then reads one D x M slot instead of summing up to G - 1 of them on
// its critical path.
//
// triton-lang/triton issue #217 asks for the running state as a parallel
// prefix sum (O(log n) depth) rather than a serial loop; this is that idea
// at the granularity of segments.  The sums run in one fixed order, so the
// result is bitwise reproducible.
#include "cp_internal.h"

namespace cp {
namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 8;  // aggregate loads in flight per thread

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
__device__ __forceinline__ float add4(float a, float b) { return a + b; }

template <typename V>
__device__ __forceinline__ V zero4();
template <>
__device__ __forceinline__ float4 zero4<float4>() {
  return make_float4(0.f, 0.f, 0.f, 0.f);
}
template <>
__device__ __forceinline__ float zero4<float>() {
  return 0.f;
}

// agg: [P][G][Ev] vectors of V.  One thread owns one vector position of one
// problem and walks its G slots in scan order.  The last slot in scan order
// was never written by the first pass (no segment starts after it): it is
// not read, only set to its starting state.
template <typename V>
__global__ void __launch_bounds__(kThreads)
    seg_prefix_kernel(V* __restrict__ agg, int64_t P, int G, int64_t Ev, int reverse) {
  const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  if (i >= P * Ev) return;
  const int64_t p = i / Ev;
  V* col = agg + p * (int64_t)G * Ev + (i - p * Ev);
  V run = zero4<V>();
  for (int o0 = 0; o0 < G; o0 += kBatch) {
    V t[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int o = o0 + u;  // position in scan order
      const int s = reverse ? G - 1 - o : o;
      t[u] = o < G - 1 ? col[(int64_t)s * Ev] : zero4<V>();
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int o = o0 + u;
      if (o < G) {
        const int s = reverse ? G - 1 - o : o;
        col[(int64_t)s * Ev] = run;
        run = add4(run, t[u]);
      }
    }
  }
}

}  // namespace

cudaError_t seg_prefix_launch(float* agg, int64_t P, int G, int64_t E, bool reverse,
                              cudaStream_t stream) {
  if (G <= 1 || P <= 0 || E <= 0) return cudaSuccess;
  const bool vec = (E % 4) == 0 && (reinterpret_cast<uintptr_t>(agg) & 15) == 0;
  const int64_t Ev = vec ? E / 4 : E;
  const int64_t n = P * Ev;
  const unsigned grid = (unsigned)((n + kThreads - 1) / kThreads);
  if (vec)
    seg_prefix_kernel<float4><<<grid, kThreads, 0, stream>>>(reinterpret_cast<float4*>(agg), P,
                                                              G, Ev, reverse ? 1 : 0);
  else
    seg_prefix_kernel<float><<<grid, kThreads, 0, stream>>>(agg, P, G, Ev, reverse ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace cp
