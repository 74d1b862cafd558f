// fp32 causal product on the CUDA cores (FFMA), chunked over the sequence.
//
// TF32 tensor-core rounding (10-bit mantissa) would not hold fp32 accuracy,
// so the fp32 path uses plain fp32 FMA.  fp16 inputs take the same kernel:
// elements are widened to fp32 on load and the outputs rounded to fp16 once.  One CTA owns one (problem,
// value-column block, segment).  It walks its segment in tiles of C rows:
//     P      = Q_t K_t^T, masked to the causal triangle of the tile
//     O_t    = Q_t S + P V_t            (S = state before the tile)
//     S     += K_t^T V_t
// which is the recurrence "state += k v^T; out = state^T q" of
// triton-lang/triton issue #217 regrouped by tiles: within a tile the
// prefix is the masked product, across tiles it is the carried state.
#include <algorithm>

#include <cuda_fp16.h>

#include "cp_internal.h"

namespace cp {
namespace {

constexpr int kC = 32;          // rows per tile
constexpr int kThreads = 256;
constexpr int kMaxMb = 64;

struct SimtArgs {
  const void* q;    // element type T of the kernel
  const void* k;
  const void* v;
  void* out;
  int64_t N;
  int D, M, Mb, n_mb, G, BH;
  int64_t seg_rows;
  int reverse;
  const float* agg_in;  // [P][G][D][Mb] aggregates (pass 2 reads), may be null
  float* agg_out;       // pass 1 writes
  int agg_only;
  // carried state (see Product): [BH] x D x M, element (d, m) at
  // d * st_ld_r + m * st_ld_c; may be null
  const float* state_in;
  float* state_out;
  int64_t st_ld_r, st_ld_c;
  int feature;  // 1: phi(x) = elu(x) + 1 applied to q and k on load
};

__device__ __forceinline__ float elu1(float x) { return x > 0.f ? x + 1.f : expf(x); }

__device__ __forceinline__ float widen(float x) { return x; }
__device__ __forceinline__ float widen(__half x) { return __half2float(x); }
template <typename T>
__device__ __forceinline__ T narrow(float x);
template <>
__device__ __forceinline__ float narrow<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half narrow<__half>(float x) { return __float2half_rn(x); }

template <typename T>
__global__ void __launch_bounds__(kThreads) simt_kernel(SimtArgs a) {
  extern __shared__ float smem[];
  const int D = a.D, Mb = a.Mb;
  const int ldq = D + 1;
  float* Qs = smem;                  // [C][D+1]
  float* Ks = Qs + kC * ldq;         // [C][D+1]
  float* Vs = Ks + kC * ldq;         // [C][Mb]
  float* Ps = Vs + kC * Mb;          // [C][C+1]
  float* Ss = Ps + kC * (kC + 1);    // [D][Mb]

  // block -> (segment, problem, value block); pass 1 skips the one segment
  // whose aggregate nobody reads.
  int idx = blockIdx.x;
  const int mb = idx % a.n_mb;
  idx /= a.n_mb;
  const int bh = idx % a.BH;
  int s = idx / a.BH;
  if (a.agg_only && a.reverse) s += 1;
  const int pidx = bh * a.n_mb + mb;
  const int m0 = mb * Mb;
  const int mw = min(Mb, a.M - m0);  // columns of this block that exist

  const int64_t seg_lo = (int64_t)s * a.seg_rows;
  const int64_t seg_hi = min(a.N, seg_lo + a.seg_rows);
  const int64_t n_rows = seg_hi - seg_lo;
  const int n_t = (int)((n_rows + kC - 1) / kC);

  const T* qb = static_cast<const T*>(a.q) + (int64_t)bh * a.N * D;
  const T* kb = static_cast<const T*>(a.k) + (int64_t)bh * a.N * D;
  const T* vb = static_cast<const T*>(a.v) + (int64_t)bh * a.N * a.M;
  T* ob = static_cast<T*>(a.out) + (int64_t)bh * a.N * a.M;

  // initial state: the carried state plus the aggregates of the segments
  // before this one in scan order
  const float* st_in =
      (!a.agg_only && a.state_in != nullptr) ? a.state_in + (int64_t)bh * D * a.M : nullptr;
  for (int e = threadIdx.x; e < D * Mb; e += kThreads) {
    const int d0 = e / Mb, m_ = e % Mb;
    float acc = (st_in != nullptr && m_ < mw) ? st_in[d0 * a.st_ld_r + (m0 + m_) * a.st_ld_c] : 0.f;
    if (!a.agg_only && a.agg_in != nullptr) {
      const int lo = a.reverse ? s + 1 : 0;
      const int hi = a.reverse ? a.G : s;
      for (int s2 = lo; s2 < hi; ++s2)
        acc += a.agg_in[((int64_t)pidx * a.G + s2) * D * Mb + e];
    }
    Ss[e] = acc;
  }

  for (int it = 0; it < n_t; ++it) {
    const int t = a.reverse ? (n_t - 1 - it) : it;
    const int64_t r0 = seg_lo + (int64_t)t * kC;
    __syncthreads();
    for (int e = threadIdx.x; e < kC * D; e += kThreads) {
      const int r = e / D, d = e % D;
      const int64_t row = r0 + r;
      const bool in = row < seg_hi;
      float kx = in ? widen(kb[row * D + d]) : 0.f;
      if (a.feature && in) kx = elu1(kx);
      Ks[r * ldq + d] = kx;
      if (!a.agg_only) {
        float qx = in ? widen(qb[row * D + d]) : 0.f;
        if (a.feature && in) qx = elu1(qx);
        Qs[r * ldq + d] = qx;
      }
    }
    for (int e = threadIdx.x; e < kC * Mb; e += kThreads) {
      const int r = e / Mb, m = e % Mb;
      const int64_t row = r0 + r;
      Vs[e] = (row < seg_hi && m < mw) ? widen(vb[row * a.M + m0 + m]) : 0.f;
    }
    __syncthreads();
    if (!a.agg_only) {
      // P = Q K^T restricted to the causal triangle of the tile
      for (int e = threadIdx.x; e < kC * kC; e += kThreads) {
        const int i = e / kC, j = e % kC;
        float acc = 0.f;
        const bool keep = a.reverse ? (j >= i) : (j <= i);
        if (keep) {
          const float* qi = Qs + i * ldq;
          const float* kj = Ks + j * ldq;
          for (int d = 0; d < D; ++d) acc = fmaf(qi[d], kj[d], acc);
        }
        Ps[i * (kC + 1) + j] = acc;
      }
      __syncthreads();
      // O = Q S + P V
      for (int e = threadIdx.x; e < kC * Mb; e += kThreads) {
        const int i = e / Mb, m = e % Mb;
        const int64_t row = r0 + i;
        if (row >= seg_hi || m >= mw) continue;
        float acc = 0.f;
        const float* qi = Qs + i * ldq;
        for (int d = 0; d < D; ++d) acc = fmaf(qi[d], Ss[d * Mb + m], acc);
        const float* pi = Ps + i * (kC + 1);
        for (int j = 0; j < kC; ++j) acc = fmaf(pi[j], Vs[j * Mb + m], acc);
        ob[row * a.M + m0 + m] = narrow<T>(acc);
      }
      __syncthreads();
    }
    // S += K^T V
    for (int e = threadIdx.x; e < D * Mb; e += kThreads) {
      const int d = e / Mb, m = e % Mb;
      float acc = Ss[e];
      for (int j = 0; j < kC; ++j) acc = fmaf(Ks[j * ldq + d], Vs[j * Mb + m], acc);
      Ss[e] = acc;
    }
  }
  if (a.agg_only) {
    __syncthreads();
    float* dst = a.agg_out + ((int64_t)pidx * a.G + s) * D * Mb;
    for (int e = threadIdx.x; e < D * Mb; e += kThreads) dst[e] = Ss[e];
  } else if (a.state_out != nullptr && (a.reverse ? s == 0 : s == a.G - 1)) {
    // the last segment in scan order hands on its final state
    __syncthreads();
    float* st = a.state_out + (int64_t)bh * D * a.M;
    for (int e = threadIdx.x; e < D * Mb; e += kThreads) {
      const int d0 = e / Mb, m_ = e % Mb;
      if (m_ < mw) st[d0 * a.st_ld_r + (m0 + m_) * a.st_ld_c] = Ss[e];
    }
  }
}

size_t simt_smem_bytes(int D, int Mb) {
  return sizeof(float) *
         (size_t)(2 * kC * (D + 1) + kC * Mb + kC * (kC + 1) + D * Mb);
}

}  // namespace

SimtPlan simt_plan(int64_t BH, int64_t N, int64_t D, int64_t M) {
  SimtPlan p{};
  p.C = kC;
  p.Mb = (int)std::min<int64_t>(M, kMaxMb);
  p.n_mb = (int)((M + p.Mb - 1) / p.Mb);
  const int64_t problems = BH * p.n_mb;
  const int64_t n_tiles = (N + kC - 1) / kC;
  // aim for about two CTAs per SM; every segment holds at least 4 tiles
  int64_t G = std::max<int64_t>(1, (2 * kPlanSMs) / std::max<int64_t>(problems, 1));
  G = std::min<int64_t>(G, std::max<int64_t>(1, n_tiles / 4));
  const int64_t tiles_per_seg = (n_tiles + G - 1) / std::max<int64_t>(G, 1);
  p.seg_rows = std::max<int64_t>(1, tiles_per_seg) * kC;
  p.G = (int)std::max<int64_t>(1, (N + p.seg_rows - 1) / p.seg_rows);
  p.agg_bytes = p.G > 1 ? sizeof(float) * (size_t)problems * p.G * D * p.Mb : 0;
  return p;
}

cudaError_t simt_launch(const Product& p, const SimtPlan& plan, float* agg, int* status,
                        cudaStream_t stream) {
  (void)status;
  const size_t smem = simt_smem_bytes((int)p.D, plan.Mb);
  auto kern = p.dtype == CP_DTYPE_F16 ? simt_kernel<__half> : simt_kernel<float>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  SimtArgs a{};
  a.q = p.q;
  a.k = p.k;
  a.v = p.v;
  a.out = p.out;
  a.N = p.N;
  a.D = (int)p.D;
  a.M = (int)p.M;
  a.Mb = plan.Mb;
  a.n_mb = plan.n_mb;
  a.G = plan.G;
  a.BH = (int)p.BH;
  a.seg_rows = plan.seg_rows;
  a.reverse = p.reverse ? 1 : 0;
  a.state_in = p.state_in;
  a.state_out = p.state_out;
  a.st_ld_r = p.st_ld_r;
  a.st_ld_c = p.st_ld_c;
  a.feature = p.feature;
  const int64_t problems = p.BH * plan.n_mb;
  if (plan.G > 1) {
    a.agg_only = 1;
    a.agg_out = agg;
    // (the aggregate pass ignores the carried state: agg_only is set)
    kern<<<(unsigned)(problems * (plan.G - 1)), kThreads, smem, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    a.agg_only = 0;
    a.agg_in = agg;
    a.agg_out = nullptr;
  }
  kern<<<(unsigned)(problems * plan.G), kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace cp
