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

constexpr int kThreads = 256;
constexpr int kMaxMb = 64;

struct SimtArgs {
  const void* q;    // element type T of the kernel
  const void* k;
  const void* v;
  void* out;
  int64_t N;
  int D, M, Mb, n_mb, G, BH;
  int C;            // rows per tile (a multiple of 4)
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

__device__ __forceinline__ int round4(int x) { return (x + 3) & ~3; }

// acc[i][j] += sum_{k in [k0, k1)} A[r0 + i][k] * B[k][c0 + j] for a 4 x 4
// block: A and B row-major in shared memory (lda, ldb multiples of 4), k0
// and k1 multiples of 4.  Sixteen FMAs per two 16-byte loads of each
// operand row; the k order is fixed, so results are reproducible.
__device__ __forceinline__ void mm4x4(float (&acc)[4][4], const float* A, int lda,
                                      const float* B, int ldb, int r0, int c0, int k0, int k1) {
  for (int k = k0; k < k1; k += 4) {
    float a[4][4], b[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 t = *reinterpret_cast<const float4*>(A + (r0 + i) * lda + k);
      a[i][0] = t.x;
      a[i][1] = t.y;
      a[i][2] = t.z;
      a[i][3] = t.w;
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float4 t = *reinterpret_cast<const float4*>(B + (k + kk) * ldb + c0);
      b[kk][0] = t.x;
      b[kk][1] = t.y;
      b[kk][2] = t.z;
      b[kk][3] = t.w;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i][kk], b[kk][j], acc[i][j]);
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 4) simt_kernel(SimtArgs a) {
  extern __shared__ __align__(16) float smem[];
  const int D = a.D, Mb = a.Mb, C = a.C;
  const int Dp = round4(D), Mbp = round4(Mb);
  float* Qs = smem;                  // [C][Dp]   q tile, row-major
  float* Kt = Qs + C * Dp;           // [Dp][C]   k tile, transposed
  float* Vs = Kt + Dp * C;           // [C][Mbp]
  float* Ps = Vs + C * Mbp;          // [C][C]    masked Q K^T
  float* Ss = Ps + C * C;            // [Dp][Mbp] state (padding stays zero)
  float* Os = Ss + Dp * Mbp;         // [C][Mbp]  Q S of the tile (phase 1 -> phase 2)

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
  const int n_t = (int)((n_rows + C - 1) / C);

  const T* qb = static_cast<const T*>(a.q) + (int64_t)bh * a.N * D;
  const T* kb = static_cast<const T*>(a.k) + (int64_t)bh * a.N * D;
  const T* vb = static_cast<const T*>(a.v) + (int64_t)bh * a.N * a.M;
  T* ob = static_cast<T*>(a.out) + (int64_t)bh * a.N * a.M;

  // initial state: the carried state plus the aggregates of the segments
  // before this one in scan order
  const float* st_in =
      (!a.agg_only && a.state_in != nullptr) ? a.state_in + (int64_t)bh * D * a.M : nullptr;
  for (int e = threadIdx.x; e < Dp * Mbp; e += kThreads) {
    const int d0 = e / Mbp, m_ = e % Mbp;
    float acc = 0.f;
    if (d0 < D && m_ < mw) {
      if (st_in != nullptr) acc = st_in[d0 * a.st_ld_r + (m0 + m_) * a.st_ld_c];
      // slot s of agg_in: the sum of the preceding segments' aggregates
      if (!a.agg_only && a.agg_in != nullptr && (a.reverse ? s < a.G - 1 : s > 0))
        acc += a.agg_in[((int64_t)pidx * a.G + s) * D * Mb + d0 * Mb + m_];
    }
    Ss[e] = acc;
  }

  const int tc_p = C / 4, tc_o = Mbp / 4;
  for (int it = 0; it < n_t; ++it) {
    const int t = a.reverse ? (n_t - 1 - it) : it;
    const int64_t r0 = seg_lo + (int64_t)t * C;
    __syncthreads();
    // ---- load, as two-dimensional loops (rows by warp, columns by lane: no
    // index division).  q and v rows are read along their columns
    // (coalesced); k is stored transposed with consecutive lanes on
    // consecutive rows, so its shared-memory stores hit distinct banks.
    // Each thread issues all its loads of a row block before storing them.
    {
      const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
      constexpr int kW = kThreads / 32;
      // k: Kt[d][r] for d = warp + kW i, r = lane + 32 j
      for (int d0 = warp; d0 < Dp; d0 += 4 * kW) {
        float r_[4][2];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int d = d0 + u * kW;
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int r = lane + 32 * jj;
            const int64_t row = r0 + r;
            const bool in = d < D && r < C && row < seg_hi;
            float x = in ? widen(kb[row * D + d]) : 0.f;
            if (a.feature && in) x = elu1(x);
            r_[u][jj] = x;
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int d = d0 + u * kW;
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int r = lane + 32 * jj;
            if (d < Dp && r < C) Kt[d * C + r] = r_[u][jj];
          }
        }
      }
      // q: Qs[r][d] and v: Vs[r][m], in 32-column blocks (column lane + 32 cb),
      // four rows r = r1 + kW u of a block in flight per thread
      for (int cb = 0; !a.agg_only && cb * 32 < Dp; ++cb) {
        const int d = lane + 32 * cb;
        for (int r1 = warp; r1 < C; r1 += 4 * kW) {
          float r_[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int r = r1 + u * kW;
            const int64_t row = r0 + r;
            const bool in = r < C && row < seg_hi && d < D;
            float x = in ? widen(qb[row * D + d]) : 0.f;
            if (a.feature && in) x = elu1(x);
            r_[u] = x;
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int r = r1 + u * kW;
            if (r < C && d < Dp) Qs[r * Dp + d] = r_[u];
          }
        }
      }
      for (int cb = 0; cb * 32 < Mbp; ++cb) {
        const int m = lane + 32 * cb;
        for (int r1 = warp; r1 < C; r1 += 4 * kW) {
          float r_[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int r = r1 + u * kW;
            const int64_t row = r0 + r;
            r_[u] = (r < C && row < seg_hi && m < mw) ? widen(vb[row * a.M + m0 + m]) : 0.f;
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int r = r1 + u * kW;
            if (r < C && m < Mbp) Vs[r * Mbp + m] = r_[u];
          }
        }
      }
    }
    __syncthreads();
    // Two compute phases per tile.  Q S reads the state before this tile's
    // update and does not need P, so it runs beside P; P V and the state
    // update touch disjoint data, so they run side by side after it.
    if (!a.agg_only) {
      // ---- phase 1: P = Q K^T on the causal triangle of the tile, and
      // Q S into Os
      const int nP = tc_p * tc_p, nO = tc_p * tc_o;
      for (int tt = threadIdx.x; tt < nP + nO; tt += kThreads) {
        float acc[4][4] = {};
        if (tt < nP) {
          const int i0 = (tt / tc_p) * 4, j0 = (tt % tc_p) * 4;
          const bool none = a.reverse ? (j0 + 3 < i0) : (j0 > i0 + 3);
          if (!none) mm4x4(acc, Qs, Dp, Kt, C, i0, j0, 0, Dp);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const bool keep = a.reverse ? (j0 + j >= i0 + i) : (j0 + j <= i0 + i);
              o[j] = keep ? acc[i][j] : 0.f;
            }
            *reinterpret_cast<float4*>(Ps + (i0 + i) * C + j0) =
                make_float4(o[0], o[1], o[2], o[3]);
          }
        } else {
          const int u = tt - nP;
          const int i0 = (u / tc_o) * 4, c0 = (u % tc_o) * 4;
          mm4x4(acc, Qs, Dp, Ss, Mbp, i0, c0, 0, Dp);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<float4*>(Os + (i0 + i) * Mbp + c0) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
      }
      __syncthreads();
    }
    // ---- phase 2: O = Q S + P V and its store (P is zero outside the
    // triangle: only the columns j a row can see are visited), and
    // S += K^T V
    const int nO2 = a.agg_only ? 0 : tc_p * tc_o;
    const int nS = (Dp / 4) * tc_o;
    for (int tt = threadIdx.x; tt < nO2 + nS; tt += kThreads) {
      float acc[4][4];
      if (tt < nO2) {
        const int i0 = (tt / tc_o) * 4, c0 = (tt % tc_o) * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 t4 = *reinterpret_cast<const float4*>(Os + (i0 + i) * Mbp + c0);
          acc[i][0] = t4.x;
          acc[i][1] = t4.y;
          acc[i][2] = t4.z;
          acc[i][3] = t4.w;
        }
        if (a.reverse)
          mm4x4(acc, Ps, C, Vs, Mbp, i0, c0, i0, C);
        else
          mm4x4(acc, Ps, C, Vs, Mbp, i0, c0, 0, i0 + 4);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int64_t row = r0 + i0 + i;
          if (row >= seg_hi) continue;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (c0 + j < mw) ob[row * a.M + m0 + c0 + j] = narrow<T>(acc[i][j]);
        }
      } else {
        const int u = tt - nO2;
        const int d0 = (u / tc_o) * 4, c0 = (u % tc_o) * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 t4 = *reinterpret_cast<const float4*>(Ss + (d0 + i) * Mbp + c0);
          acc[i][0] = t4.x;
          acc[i][1] = t4.y;
          acc[i][2] = t4.z;
          acc[i][3] = t4.w;
        }
        mm4x4(acc, Kt, C, Vs, Mbp, d0, c0, 0, C);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<float4*>(Ss + (d0 + i) * Mbp + c0) =
              make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      }
    }
  }
  __syncthreads();
  if (a.agg_only) {
    float* dst = a.agg_out + ((int64_t)pidx * a.G + s) * D * Mb;
    for (int e = threadIdx.x; e < D * Mb; e += kThreads) {
      const int d0 = e / Mb, m_ = e % Mb;
      dst[e] = Ss[d0 * Mbp + m_];
    }
  } else if (a.state_out != nullptr && (a.reverse ? s == 0 : s == a.G - 1)) {
    // the last segment in scan order hands on its final state
    float* st = a.state_out + (int64_t)bh * D * a.M;
    for (int e = threadIdx.x; e < D * Mb; e += kThreads) {
      const int d0 = e / Mb, m_ = e % Mb;
      if (m_ < mw) st[d0 * a.st_ld_r + (m0 + m_) * a.st_ld_c] = Ss[d0 * Mbp + m_];
    }
  }
}

// rows per tile: 32 keeps a CTA's shared memory small enough for four CTAs
// per SM at D = M = 64 (and the quadratic in-tile part of the work small);
// a sequence of at most 64 rows with narrow operands is one tile of 64
int simt_rows(int64_t N, int64_t D) { return (N <= 64 && D <= 64) ? 64 : 32; }

size_t simt_smem_bytes(int C_, int D, int Mb) {
  const size_t C = C_, Dp = (D + 3) / 4 * 4, Mbp = (Mb + 3) / 4 * 4;
  return sizeof(float) * (2 * C * Dp + 2 * C * Mbp + C * C + Dp * Mbp);
}

}  // namespace

SimtPlan simt_plan(int64_t BH, int64_t N, int64_t D, int64_t M) {
  SimtPlan p{};
  p.C = simt_rows(N, D);
  p.Mb = (int)std::min<int64_t>(M, kMaxMb);
  p.n_mb = (int)((M + p.Mb - 1) / p.Mb);
  const int64_t problems = BH * p.n_mb;
  const int64_t n_tiles = (N + p.C - 1) / p.C;
  // aim for about four CTAs per SM; every segment holds at least 2 tiles
  int64_t G = std::max<int64_t>(1, (4 * kPlanSMs) / std::max<int64_t>(problems, 1));
  G = std::min<int64_t>(G, std::max<int64_t>(1, n_tiles / 2));
  const int64_t tiles_per_seg = (n_tiles + G - 1) / std::max<int64_t>(G, 1);
  p.seg_rows = std::max<int64_t>(1, tiles_per_seg) * p.C;
  p.G = (int)std::max<int64_t>(1, (N + p.seg_rows - 1) / p.seg_rows);
  p.agg_bytes = p.G > 1 ? sizeof(float) * (size_t)problems * p.G * D * p.Mb : 0;
  return p;
}

cudaError_t simt_launch(const Product& p, const SimtPlan& plan, float* agg, int* status,
                        cudaStream_t stream) {
  (void)status;
  const size_t smem = simt_smem_bytes(plan.C, (int)p.D, plan.Mb);
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
  a.C = plan.C;
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
    // each segment's starting state: one slot per second-pass CTA
    if (e == cudaSuccess)
      e = seg_prefix_launch(agg, problems, plan.G, (int64_t)p.D * plan.Mb, p.reverse, stream);
    if (e != cudaSuccess) return e;
    a.agg_only = 0;
    a.agg_in = agg;
    a.agg_out = nullptr;
  }
  kern<<<(unsigned)(problems * plan.G), kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace cp
