// A split forward scan in one launch (the scan step of "Parallel prefix sum"
// on the triton-lang/triton issue #217 pages, with segments as the scanned
// elements): every CTA first sums its own segment (the aggregate-only body),
// publishes that sum, waits until the segments before it in scan order have
// published theirs, forms its prefix from them (all threads, a fixed order:
// the result does not depend on timing) and scans its segment from it.  The
// two-pass form instead ends the aggregate launch, runs a prefix launch over
// the sums and starts a third launch for the scan.
//
// Every CTA must be resident at once (each waits on CTAs with smaller
// indices): the host launches this kernel only when the grid, one CTA per
// SM, fits the device.  Every wait is bounded; a wait that gives up records
// CP_ERR_TIMEOUT and the scan still runs, on whatever it read.  The flags
// are cleared by the host before each launch (stream-ordered, so the launch
// also works inside a CUDA graph).
#include <atomic>

#include "cp_internal.h"
#include "cp_tc_causal.cuh"

namespace cp {
namespace tc {
namespace {

__device__ __forceinline__ void st_release_u32(unsigned int* p, unsigned int v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// CTA (seg, pidx) with work index seg * P + pidx, the order of the other
// launches' grids.
template <int DP, int MB, bool CKPT>
__global__ void __launch_bounds__(kThreads, 1)
    tc_lookback_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o, const ArgsX a) {
  const int P = a.BH * a.n_mb;
  const int work = (int)blockIdx.x;
  const int seg = work / P;
  const int pidx = work - seg * P;
  const bool has_sum = seg < a.G - 1;  // the last segment's sum is never read
  if (has_sum) {
    ArgsX b = a;
    b.agg_in = nullptr;
    b.state_in = nullptr;  // the segment's own sum
    b.state_out = nullptr;
    b.ckpt = nullptr;
    causal_body<DP, MB, true, false, false, false, false, false, false, false, ArgsX>(
        tm_q, tm_k, tm_v, tm_o, b, Phase{work, true, false});
    // every thread's part of the sum is written: publish it
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      st_release_u32(&a.lb_flags[(int64_t)pidx * a.G + seg], 1u);
    }
  }
  if (seg > 0) {
    if (threadIdx.x == 0) {
      const uint64_t t0 = ptx::globaltimer();
      bool ok = true;
      for (int s = 0; s < seg && ok; ++s) {
        const unsigned int* f = &a.lb_flags[(int64_t)pidx * a.G + s];
        // (the status word is not consulted: it keeps an earlier call's
        // error until the caller reads it)
        while (ld_acquire_u32(f) == 0u) {
          if (ptx::globaltimer() - t0 > CP_WAIT_TIMEOUT_NS) {
            if (a.status != nullptr) atomicCAS(a.status, 0, (int)CP_ERR_TIMEOUT);
            ok = false;
            break;
          }
          __nanosleep(128);
        }
      }
      __threadfence();
    }
    __syncthreads();
    // the prefix: the sums of segments 0 .. seg - 1 added in that order, two
    // segments' loads in flight per step
    constexpr int kVec = DP * MB / 4;
    const float4* sums = reinterpret_cast<const float4*>(a.agg_out) + (int64_t)pidx * a.G * kVec;
    float4* pre = reinterpret_cast<float4*>(const_cast<float*>(a.agg_in)) +
                  ((int64_t)pidx * a.G + seg) * kVec;
    for (int i = threadIdx.x; i < kVec; i += kThreads) {
      float4 acc = __ldcg(sums + i);
      int s = 1;
      for (; s + 1 < seg; s += 2) {
        const float4 u = __ldcg(sums + (int64_t)s * kVec + i);
        const float4 w = __ldcg(sums + (int64_t)(s + 1) * kVec + i);
        acc.x += u.x;
        acc.y += u.y;
        acc.z += u.z;
        acc.w += u.w;
        acc.x += w.x;
        acc.y += w.y;
        acc.z += w.z;
        acc.w += w.w;
      }
      if (s < seg) {
        const float4 u = __ldcg(sums + (int64_t)s * kVec + i);
        acc.x += u.x;
        acc.y += u.y;
        acc.z += u.z;
        acc.w += u.w;
      }
      __stcg(pre + i, acc);
    }
    __syncthreads();  // the scan's state group reads the slot
  }
  causal_body<DP, MB, false, false, false, CKPT, false, false, false, false, ArgsX>(
      tm_q, tm_k, tm_v, tm_o, a, Phase{work, !has_sum, true});
}

template <int DP, int MB, bool CKPT>
cudaError_t launch_lb(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                      const CUtensorMap& o, const ArgsX& a, unsigned grid, cudaStream_t st) {
  constexpr int kSmem = Layout<DP, MB, true>::kSmemBytes > Layout<DP, MB, false>::kSmemBytes
                            ? Layout<DP, MB, true>::kSmemBytes
                            : Layout<DP, MB, false>::kSmemBytes;
  static_assert(kSmem <= kSmemLimit, "shared memory overflow");
  auto kern = tc_lookback_kernel<DP, MB, CKPT>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if ((configured.load(std::memory_order_acquire) & bit) == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, q, k, v, o, a);
}

template <int DP, int MB>
cudaError_t launch_lb2(bool ckpt, const CUtensorMap& q, const CUtensorMap& k,
                       const CUtensorMap& v, const CUtensorMap& o, const ArgsX& a, unsigned grid,
                       cudaStream_t st) {
  return ckpt ? launch_lb<DP, MB, true>(q, k, v, o, a, grid, st)
              : launch_lb<DP, MB, false>(q, k, v, o, a, grid, st);
}

}  // namespace

cudaError_t lookback_launch(int DP, int MB, const CUtensorMap& q, const CUtensorMap& k,
                            const CUtensorMap& v, const CUtensorMap& o, const ArgsX& a,
                            unsigned grid, cudaStream_t st) {
  const bool ck = a.ckpt != nullptr;
  if (DP == 64 && MB == 64) return launch_lb2<64, 64>(ck, q, k, v, o, a, grid, st);
  if (DP == 64 && MB == 128) return launch_lb2<64, 128>(ck, q, k, v, o, a, grid, st);
  if (DP == 128 && MB == 64) return launch_lb2<128, 64>(ck, q, k, v, o, a, grid, st);
  if (DP == 128 && MB == 128) return launch_lb2<128, 128>(ck, q, k, v, o, a, grid, st);
  if (DP == 192 && MB == 64) return launch_lb2<192, 64>(ck, q, k, v, o, a, grid, st);
  if (DP == 256 && MB == 64) return launch_lb2<256, 64>(ck, q, k, v, o, a, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace tc
}  // namespace cp
