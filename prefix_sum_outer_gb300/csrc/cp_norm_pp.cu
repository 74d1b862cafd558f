// The normaliser of causal linear attention and its backward with one CTA
// per problem (b, h), for rows of D = 64 when there are enough problems to
// keep the HBM busy (at least half as many as SMs).  It serves the calls it
// measured faster in than the look-back kernel (cp_norm.cu), at B=8 H=16
// N=4096 bf16: z of plain rows (39.6 against 47.7 us) and the backward of
// mapped rows (dq + dk 110.8 against 172.5 us); the plain backward (90.3
// against 86.4 us) and z of mapped rows (96.1 against 77.3 us: eight warps
// per SM leave the exponentials' latency exposed) stay on the look-back.
//
//     z_i = q_i . c_i,     c_i = sum_{j<=i} k_j                 (forward)
//     dq_i = g_i c_i,      dk_j = sum_{i>=j} g_i q_i            (backward)
//
// ("Transformers are RNNs", the denominator phi(q_i)^T sum_{j<=i} phi(k_j)
// of causal linear attention; with feature != 0 the rows are raw inputs
// mapped by phi = elu + 1 on load and the gradients are taken through phi'.)
//
// A CTA walks its problem's 128-row tiles in scan order (backwards for dk)
// through a ring of shared-memory stages filled by TMA bulk copies, so no
// CTA waits on another: the scan's carry stays in registers.  Eight warps
// cover a tile: warp w takes the 32 columns 32 (w & 1) + lane and the 32
// rows 32 (w >> 1) + i.  Per tile:
//   1. each lane sums its 32 scanned values (k, or g q for dk) and publishes
//      the sum for its row group;
//   2. each lane forms the running (inclusive) scan of its rows from the
//      carry plus the sums of the row groups before its own, and every lane
//      of a column advances the carry by the four row-group sums in the
//      same order;
//   3. z: the products q_i,c c_i,c of the warp's 32 rows are reduced across
//      its 32 lanes (a transposing butterfly: lane l ends with row l), and
//      the two column halves are added through shared memory;
//      dq, dk: each element is written as it is formed.
// Every sum runs in a fixed order, so results are bitwise reproducible.
// Every wait is bounded; a wait that runs out records CP_ERR_TIMEOUT.
#include <algorithm>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cp_internal.h"
#include "sm103_ptx.cuh"

namespace cp {
namespace {

constexpr int kPpThreads = 256;
constexpr int kPpD = 64;
constexpr int kPpRows = 128;
constexpr int kPpMaxStages = 8;
constexpr uint32_t kPpRingBytes = 192 * 1024;
constexpr int kPpMaxDev = 64;
// shared memory: the stages' barriers, the row-group sums [4][64] and the
// column halves' partial z [2][128] (fp32), then the ring
constexpr int kPpRingOff = 4096;
static_assert(8 * kPpMaxStages + 4 * (4 * kPpD + 2 * kPpRows) <= kPpRingOff, "layout");
enum PpMode : int { kPpZ = 0, kPpDQ = 1, kPpDK = 2 };

template <typename T>
__device__ __forceinline__ float pp_ld(const uint8_t* tile, int e);
template <>
__device__ __forceinline__ float pp_ld<__nv_bfloat16>(const uint8_t* tile, int e) {
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(tile)[e]);
}
template <>
__device__ __forceinline__ float pp_ld<__half>(const uint8_t* tile, int e) {
  return __half2float(reinterpret_cast<const __half*>(tile)[e]);
}
template <>
__device__ __forceinline__ float pp_ld<float>(const uint8_t* tile, int e) {
  return reinterpret_cast<const float*>(tile)[e];
}

template <typename T>
__device__ __forceinline__ void pp_st(void* out, int64_t e, float x);
template <>
__device__ __forceinline__ void pp_st<__nv_bfloat16>(void* out, int64_t e, float x) {
  static_cast<__nv_bfloat16*>(out)[e] = __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ void pp_st<__half>(void* out, int64_t e, float x) {
  static_cast<__half*>(out)[e] = __float2half_rn(x);
}
template <>
__device__ __forceinline__ void pp_st<float>(void* out, int64_t e, float x) {
  static_cast<float*>(out)[e] = x;
}

// rows of a tile that exist, given the rows left from its first
__device__ __forceinline__ int64_t pp_rows(int64_t left) { return left < kPpRows ? left : kPpRows; }

// phi(x) = elu(x) + 1 = e^min(x, 0) + max(x, 0); phi'(x) = e^min(x, 0)
__device__ __forceinline__ float pp_dphi(float x) { return __expf(fminf(x, 0.f)); }
__device__ __forceinline__ float pp_phi(float x) { return pp_dphi(x) + fmaxf(x, 0.f); }

struct PpArgs {
  const void* scan;    // the scanned rows: k (z, dq) or q (dk)
  const void* other;   // z: q; dq, dk with a feature map: the raw rows of the output
  const float* grad_z; // dq, dk: [BH][N]
  float* z;            // z: [BH][N]
  void* out;           // dq or dk, [BH][N][64] in the input dtype
  int64_t N;
  int n_tiles;
  int n_stages;
  uint32_t in_bytes;   // one input's share of a stage
  int* status;
};

template <typename T, int MODE, bool FEAT>
__global__ void __launch_bounds__(kPpThreads, 1) norm_pp_kernel(const PpArgs a) {
  constexpr bool kRev = MODE == kPpDK;
  constexpr bool kTwo = MODE == kPpZ || FEAT;  // a second row stream
  extern __shared__ __align__(128) uint8_t pp_smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(pp_smem);                 // [kPpMaxStages]
  float* part = reinterpret_cast<float*>(pp_smem + 8 * kPpMaxStages);    // [4][64]
  float* zpart = part + 4 * kPpD;                                        // [2][128]
  uint8_t* ring = pp_smem + kPpRingOff;                                  // [S][1 or 2][in_bytes]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int col = 32 * (warp & 1) + lane;
  const int rg = warp >> 1;
  const int64_t bh = blockIdx.x;
  const int S = a.n_stages, nT = a.n_tiles;
  const uint32_t stage_bytes = (kTwo ? 2u : 1u) * a.in_bytes;
  const uint8_t* scan_base = static_cast<const uint8_t*>(a.scan) + bh * a.N * kPpD * sizeof(T);
  const uint8_t* other_base =
      kTwo ? static_cast<const uint8_t*>(a.other) + bh * a.N * kPpD * sizeof(T) : nullptr;

  auto tile_of = [&](int t) { return kRev ? nT - 1 - t : t; };
  auto issue = [&](int t) {
    const int s = t % S;
    const int64_t row0 = (int64_t)tile_of(t) * kPpRows;
    const uint32_t bytes =
        (uint32_t)(pp_rows(a.N - row0) * kPpD * (int64_t)sizeof(T));
    uint8_t* st = ring + (size_t)s * stage_bytes;
    ptx::mbar_arrive_expect_tx(&full[s], (kTwo ? 2u : 1u) * bytes);
    ptx::bulk_load(st, scan_base + row0 * kPpD * sizeof(T), bytes, &full[s]);
    if (kTwo) ptx::bulk_load(st + a.in_bytes, other_base + row0 * kPpD * sizeof(T), bytes, &full[s]);
  };

  if (tid == 0) {
    for (int s = 0; s < S; ++s) ptx::mbar_init(&full[s], 1);
    ptx::fence_mbar_init();
    for (int t = 0; t < min(S, nT); ++t) issue(t);
  }
  __syncthreads();

  float carry = 0.f;  // the scan of everything before this tile, column col
  volatile int never = 0;
  int t = 0;
  for (; t < nT; ++t) {
    const int s = t % S;
    const int64_t row0 = (int64_t)tile_of(t) * kPpRows;
    const int rows = (int)pp_rows(a.N - row0);
    bool ok = ptx::mbar_wait(&full[s], (uint32_t)((t / S) & 1), &never);
    const uint8_t* sc = ring + (size_t)s * stage_bytes;
    const uint8_t* ot = sc + a.in_bytes;
    // g of this lane's row of the group (dq, dk), broadcast row by row
    float g_mine = 0.f;
    if (MODE != kPpZ && 32 * rg + lane < rows)
      g_mine = __ldg(a.grad_z + bh * a.N + row0 + 32 * rg + lane);
    // 1. the lane's scanned values and their sum
    float v[32];
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int r = 32 * rg + i;
      // (selects, not branches: the unrolled loop stays one block)
      const float raw = pp_ld<T>(sc, r * kPpD + col);
      float x = FEAT ? pp_phi(raw) : raw;
      if (MODE == kPpDK) x *= __shfl_sync(0xffffffffu, g_mine, i);
      v[i] = r < rows ? x : 0.f;
    }
    if (kRev) {
#pragma unroll
      for (int i = 31; i >= 0; --i) sum += v[i];
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) sum += v[i];
    }
    part[rg * kPpD + col] = sum;
    // every thread's wait succeeded, or all leave together
    if (!__syncthreads_and(ok)) break;
    // 2. the running scan of the lane's rows, and the carry
    float base = carry;
    if (kRev) {
      for (int r2 = 3; r2 > rg; --r2) base += part[r2 * kPpD + col];
#pragma unroll
      for (int i = 31; i >= 0; --i) {
        base += v[i];
        v[i] = base;
      }
    } else {
      for (int r2 = 0; r2 < rg; ++r2) base += part[r2 * kPpD + col];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        base += v[i];
        v[i] = base;
      }
    }
    if (kRev) {
      for (int r2 = 3; r2 >= 0; --r2) carry += part[r2 * kPpD + col];
    } else {
      for (int r2 = 0; r2 < 4; ++r2) carry += part[r2 * kPpD + col];
    }
    // 3. outputs
    if constexpr (MODE == kPpZ) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int r = 32 * rg + i;
        const float raw = pp_ld<T>(ot, r * kPpD + col);
        const float qx = FEAT ? pp_phi(raw) : raw;
        v[i] = r < rows ? v[i] * qx : 0.f;
      }
      // transposing butterfly: after the round of width w, lane l holds the
      // rows whose bit w matches its own; at the end, row l
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1) {
        const bool upper = (lane & w) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
          const float send = upper ? v[i] : v[i + w];
          const float keep = upper ? v[i + w] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
      }
      zpart[(warp & 1) * kPpRows + 32 * rg + lane] = v[0];
    } else {
      T* out = static_cast<T*>(a.out);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int r = 32 * rg + i;
        float o = v[i];
        if (MODE == kPpDQ) o *= __shfl_sync(0xffffffffu, g_mine, i);
        if (FEAT) o *= pp_dphi(pp_ld<T>(ot, r * kPpD + col));
        if (r < rows) pp_st<T>(out, (bh * a.N + row0 + r) * kPpD + col, o);
      }
    }
    // the stage's reads are done before the copy engine refills it
    ptx::fence_proxy_async_smem();
    __syncthreads();
    if (MODE == kPpZ && tid < rows)
      a.z[bh * a.N + row0 + tid] = zpart[tid] + zpart[kPpRows + tid];
    if (tid == 0 && t + S < nT) issue(t + S);
  }
  if (t < nT) {
    // a wait ran out: record it, and let the copies in flight land before
    // the CTA's memory goes away
    if (tid == 0) {
      if (a.status != nullptr) atomicCAS(a.status, 0, (int)CP_ERR_TIMEOUT);
      for (int j = t; j < min(nT, t + S); ++j)
        ptx::mbar_wait_timeout(&full[j % S], (uint32_t)((j / S) & 1), CP_WAIT_TIMEOUT_NS);
    }
  }
}

template <typename T, int MODE, bool FEAT>
cudaError_t pp_run(PpArgs a, int64_t BH, cudaStream_t st) {
  constexpr bool kTwo = MODE == kPpZ || FEAT;
  a.in_bytes = (uint32_t)(kPpRows * kPpD * sizeof(T));
  const uint32_t stage = (kTwo ? 2u : 1u) * a.in_bytes;
  a.n_stages = (int)std::max<uint32_t>(1u, std::min<uint32_t>(kPpMaxStages, kPpRingBytes / stage));
  const size_t smem = kPpRingOff + (size_t)a.n_stages * stage;
  auto kern = norm_pp_kernel<T, MODE, FEAT>;
  static std::mutex mu;
  static bool opted[kPpMaxDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kPpMaxDev) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!opted[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      opted[dev] = true;
    }
  }
  kern<<<(unsigned)BH, kPpThreads, smem, st>>>(a);
  return cudaGetLastError();
}

// the calls this kernel serves (see the top of the file)
bool pp_mode_served(int mode, bool feat) { return feat ? mode != kPpZ : mode == kPpZ; }

template <typename T>
cudaError_t pp_modes(int mode, bool feat, const PpArgs& a, int64_t BH, cudaStream_t st) {
  if (feat) {
    if (mode == kPpDQ) return pp_run<T, kPpDQ, true>(a, BH, st);
    return pp_run<T, kPpDK, true>(a, BH, st);
  }
  return pp_run<T, kPpZ, false>(a, BH, st);
}

}  // namespace

bool norm_pp_eligible(int mode, int feature, int64_t BH, int64_t N, int64_t D) {
  return pp_mode_served(mode, feature != 0) && D == kPpD && N > 0 &&
         2 * BH >= device_sm_count() && BH < ((int64_t)1 << 31) &&
         (N + kPpRows - 1) / kPpRows < ((int64_t)1 << 31);
}

cudaError_t norm_pp_launch(int mode, const void* q, const void* k, const float* grad_z, float* z,
                           void* out, int64_t BH, int64_t N, cp_dtype_t dtype, int* status,
                           cudaStream_t stream, int feature) {
  if (!pp_mode_served(mode, feature != 0)) return cudaErrorInvalidValue;
  PpArgs a{};
  // z scans k and dots q; dq scans k (raw q for phi'); dk scans g q (raw k
  // for phi')
  a.scan = mode == kPpDK ? q : k;
  a.other = mode == kPpZ ? q : (mode == kPpDQ ? q : k);
  a.grad_z = grad_z;
  a.z = z;
  a.out = out;
  a.N = N;
  a.n_tiles = (int)((N + kPpRows - 1) / kPpRows);
  a.status = status;
  const bool feat = feature != 0;
  if (dtype == CP_DTYPE_BF16) return pp_modes<__nv_bfloat16>(mode, feat, a, BH, stream);
  if (dtype == CP_DTYPE_F16) return pp_modes<__half>(mode, feat, a, BH, stream);
  return pp_modes<float>(mode, feat, a, BH, stream);
}

}  // namespace cp
