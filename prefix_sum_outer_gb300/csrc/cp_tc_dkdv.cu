// Backward pass for bf16 with D, M <= 64: dq as one causal-product launch,
// then the fused dk/dv reverse scan (cp_tc_dkdv.cuh), preceded by its
// aggregate pass when the problems are split into segments.
//
// (Running both scans of a problem in one CTA, dk/dv and then dq, was
// measured: no faster than two launches, since each scan's pipeline fill and
// drain stay on the critical path either way.)
#include <algorithm>
#include <atomic>
#include <utility>

#include "cp_internal.h"
#include "cp_tc_dkdv.cuh"

namespace cp {
namespace tc {
namespace {

template <bool STATE_OUT>
__global__ void __launch_bounds__(dkdv::kThreads, 1)
    tc_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                   const __grid_constant__ CUtensorMap tm_dk,
                   const __grid_constant__ CUtensorMap tm_dv, const dkdv::DkdvArgs a) {
  dkdv::dkdv_body<STATE_OUT>(tm_q, tm_k, tm_v, tm_g, tm_dk, tm_dv, a);
}

template <typename Kernel>
cudaError_t set_smem_once(Kernel kern, int bytes, std::atomic<uint64_t>& configured) {
  // the shared-memory opt-in is set once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if ((configured.load(std::memory_order_acquire) & bit) == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_release);
  }
  return cudaSuccess;
}

}  // namespace
}  // namespace tc

bool tc_dkdv_supported(const TcPlan& plan) {
  return plan.ok && plan.DP == tc::dkdv::kW && plan.MB == tc::dkdv::kW && plan.n_mb == 1;
}

namespace {

template <typename... KArgs, typename... Act>
cudaError_t launch_pdl(void (*kern)(KArgs...), unsigned grid, int smem, cudaStream_t stream,
                       Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(tc::dkdv::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Act>(args)...);
}

}  // namespace

cp_status_t tc_bwd_launch(const void* q, const void* k, const void* v, const void* g, void* dq,
                          void* dk, void* dv, const float* state_in,
                          const float* grad_state_out, float* grad_state_in, int64_t BH,
                          int64_t N, int64_t D, int64_t M, const TcPlan& plan, float* agg,
                          int* status, cudaStream_t stream) {
  using namespace tc;
  if (!tc_dkdv_supported(plan)) return CP_ERR_UNSUPPORTED_SHAPE;
  CUtensorMap mq, mk, mv, mg, mdk, mdv;
  if (!make_map(&mq, q, BH, N, D) || !make_map(&mk, k, BH, N, D) || !make_map(&mv, v, BH, N, M) ||
      !make_map(&mg, g, BH, N, M) || !make_map(&mdk, dk, BH, N, D) || !make_map(&mdv, dv, BH, N, M))
    return CP_ERR_UNSUPPORTED_SHAPE;
  dkdv::DkdvArgs a{};
  a.N = N;
  a.n_tiles = plan.n_tiles;
  a.seg_tiles = plan.seg_tiles;
  a.G = plan.G;
  a.BH = (int)BH;
  a.D = (int)D;
  a.M = (int)M;
  a.agg_in = plan.G > 1 ? agg : nullptr;
  a.state_in = grad_state_out;
  a.state_out = grad_state_in;
  a.status = status;
  cudaError_t e;
  // dq_i = sum_{j<=i} (g_i . v_j) k_j: the forward product (g, v, k); then
  // (split problems) the aggregate pass of the state sum q g^T, i.e. of the
  // reverse product with k' = q and v' = g; then the fused dk/dv scan
  Product pq{g, v, k, dq, BH, N, M, D, false};
  // its state is sum v k^T: the transpose of the caller's S_0
  pq.state_in = state_in;
  pq.st_ld_r = 1;
  pq.st_ld_c = M;
  cp_status_t st = tc_launch(pq, tc_plan(BH, N, M, D), agg, status, stream);
  if (st != CP_OK) return st;
  if (plan.G > 1) {
    const Product pa{k, q, g, dv, BH, N, D, M, true};
    st = tc_aggregate(pa, plan, agg, status, stream);
    if (st != CP_OK) return st;
  }
  const unsigned grid = (unsigned)(BH * plan.G);
  if (grad_state_in != nullptr) {
    static std::atomic<uint64_t> configured{0};
    e = set_smem_once(tc_dkdv_kernel<true>, dkdv::kSmemBytes, configured);
    if (e == cudaSuccess)
      e = launch_pdl(tc_dkdv_kernel<true>, grid, dkdv::kSmemBytes, stream, mq, mk, mv, mg, mdk,
                     mdv, a);
  } else {
    static std::atomic<uint64_t> configured{0};
    e = set_smem_once(tc_dkdv_kernel<false>, dkdv::kSmemBytes, configured);
    if (e == cudaSuccess)
      e = launch_pdl(tc_dkdv_kernel<false>, grid, dkdv::kSmemBytes, stream, mq, mk, mv, mg, mdk,
                     mdv, a);
  }
  return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

}  // namespace cp
