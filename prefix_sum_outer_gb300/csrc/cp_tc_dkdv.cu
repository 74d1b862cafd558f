// Backward pass for bf16 with D, M <= 64: the fused dk/dv reverse scan
// (cp_tc_dkdv.cuh) and dq, a forward causal product.
//
// Unsplit problems on fewer problems than SMs run as one launch with a
// static schedule (tc_bwd_kernel): CTA p < BH runs the dk/dv scan of problem
// p, and the SMs that would otherwise idle run dq scans, two each; the
// remaining dq scans follow the dk/dv scan of their own problem on the same
// CTA, whose first tiles that scan has just read.  Per problem the dk/dv
// scan takes about 1.6 times a dq scan, so two dq scans per spare SM keep
// those SMs busy about as long as a dk/dv + dq CTA.  (Cutting the dq scans
// into segments seeded from forward checkpoints, handed out from a ticket
// pool, measured slower: each extra scan start and drain cost about 7 us.)
// Split problems run dq as a product launch (its segments seeded from the
// forward's checkpoints when the caller has them), then the aggregate pass
// and the fused scan.
#include <algorithm>
#include <atomic>
#include <utility>

#include "cp_internal.h"
#include "cp_tc_causal.cuh"
#include "cp_tc_dkdv.cuh"

namespace cp {
namespace tc {
namespace {

template <bool STATE_OUT, bool FEAT>
__global__ void __launch_bounds__(dkdv::kThreads, 1)
    tc_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                   const __grid_constant__ CUtensorMap tm_dk,
                   const __grid_constant__ CUtensorMap tm_dv, const dkdv::DkdvArgs a) {
  dkdv::dkdv_body<STATE_OUT, FEAT>(tm_q, tm_k, tm_v, tm_g, tm_dk, tm_dv, a,
                                   Phase{(int)blockIdx.x, true, true});
}

constexpr int kDqPerSpare = 2;

// CTA c < BH: the dk/dv scan of problem c, then dq of problem c when c <
// n_main_dq.  CTA BH + e: dq of problems n_main_dq + kDqPerSpare * e + j.
// FEAT: q and k are raw rows of phi = elu + 1: the dk/dv scan maps them (see
// dkdv_body), and the dq scan maps its value operand k and multiplies dq by
// phi'(q) read through tm_xq (the raw q; aq.epi_x).
template <bool STATE_OUT, bool FEAT>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                  const __grid_constant__ CUtensorMap tm_dk,
                  const __grid_constant__ CUtensorMap tm_dv,
                  const __grid_constant__ CUtensorMap tm_dq,
                  const __grid_constant__ CUtensorMap tm_xq, const dkdv::DkdvArgs a,
                  const KArgs<FEAT> aq, int n_main_dq) {
  // dq_i = sum_{j<=i} (g_i . v_j) k_j: the forward product (g, v, k)
  auto dq_scan = [&](int p, bool first, bool last) {
    return causal_body<dkdv::kW, dkdv::kW, false, false, false, false, false, false, FEAT, FEAT,
                       KArgs<FEAT>>(tm_g, tm_v, tm_k, tm_dq, aq, Phase{p, first, last}, &tm_xq);
  };
  const int c = (int)blockIdx.x;
  if (c < a.BH) {
    const bool more = c < n_main_dq;
    if (dkdv::dkdv_body<STATE_OUT, FEAT>(tm_q, tm_k, tm_v, tm_g, tm_dk, tm_dv, a,
                                         Phase{c, true, !more}) &&
        more)
      dq_scan(c, false, true);
    return;
  }
  const int p0 = n_main_dq + kDqPerSpare * (c - a.BH);
  const int n = min(kDqPerSpare, a.BH - p0);
  for (int j = 0; j < n; ++j)
    if (!dq_scan(p0 + j, j == 0, j == n - 1)) return;
}

static_assert(dkdv::kThreads == kThreads, "both scans run on the same CTA");
static_assert(dkdv::kSmemBytes == Layout<dkdv::kW, dkdv::kW>::kSmemBytes,
              "both scans use the same shared-memory size");

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

// The backward kernels are launched in plain stream order, not as
// programmatic dependents of the kernel before them: measured on the
// B=8 H=16 N=4096 D=M=64 step, a dependent backward launch saved 2-3 us
// after another backward but cost about 35 us after a forward that writes
// its final state, so the backward waits for its predecessor to complete.
template <typename... KArgs, typename... Act>
cudaError_t launch_bwd(void (*kern)(KArgs...), unsigned grid, int smem, cudaStream_t stream,
                       Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(tc::dkdv::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Act>(args)...);
}

}  // namespace

cp_status_t tc_bwd_launch(const void* q, const void* k, const void* v, const void* g, void* dq,
                          void* dk, void* dv, const float* state_in,
                          const float* grad_state_out, float* grad_state_in, int64_t BH,
                          int64_t N, int64_t D, int64_t M, const TcPlan& plan, float* agg,
                          int* status, const float* ckpt, const CkptPlan& ck,
                          cudaStream_t stream, bool feature) {
  using namespace tc;
  // checkpoints replace the carried S_0 (they already contain it) and need
  // the segment geometry of the dq product
  const bool seeded = ckpt != nullptr && ck.G > 1;
  if (seeded && state_in != nullptr) return CP_ERR_INVALID_ARG;
  // the feature backward (raw q, k) carries no state and takes no checkpoints
  if (feature && (state_in != nullptr || grad_state_out != nullptr || grad_state_in != nullptr ||
                  ckpt != nullptr))
    return CP_ERR_INVALID_ARG;
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
  int dev = 0, n_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return CP_ERR_CUDA;
  if (plan.G == 1 && BH < n_sm && !seeded) {
    // one launch: dk/dv scans on BH CTAs, dq scans on the spare SMs first
    CUtensorMap mdq;
    if (!make_map(&mdq, dq, BH, N, D)) return CP_ERR_UNSUPPORTED_SHAPE;
    ArgsX aq{};
    aq.N = N;
    aq.n_tiles = plan.n_tiles;
    aq.seg_tiles = plan.n_tiles;
    aq.G = 1;
    aq.BH = (int)BH;
    aq.n_mb = 1;
    aq.reverse = 0;
    aq.status = status;
    // the product's state sum v k^T is the transpose of the caller's S_0
    aq.state_in = state_in;
    aq.st_ld_r = 1;
    aq.st_ld_c = M;
    aq.Dr = (int)M;
    aq.Mc = (int)D;
    // the feature backward: dq times phi'(q), the raw q read with q's map
    aq.epi_x = feature ? q : nullptr;
    const int64_t spare = n_sm - BH;
    const int64_t n_spare_dq = std::min<int64_t>(BH, spare * kDqPerSpare);
    const int n_main_dq = (int)(BH - n_spare_dq);
    const unsigned grid = (unsigned)(BH + (n_spare_dq + kDqPerSpare - 1) / kDqPerSpare);
    constexpr int kSmem = dkdv::kSmemBytes;
    const Args aq_plain = aq;
    if (feature) {
      static std::atomic<uint64_t> configured{0};
      e = set_smem_once(tc_bwd_kernel<false, true>, kSmem, configured);
      if (e == cudaSuccess)
        e = launch_bwd(tc_bwd_kernel<false, true>, grid, kSmem, stream, mq, mk, mv, mg, mdk, mdv,
                       mdq, mq, a, aq, n_main_dq);
    } else if (grad_state_in != nullptr) {
      static std::atomic<uint64_t> configured{0};
      e = set_smem_once(tc_bwd_kernel<true, false>, kSmem, configured);
      if (e == cudaSuccess)
        e = launch_bwd(tc_bwd_kernel<true, false>, grid, kSmem, stream, mq, mk, mv, mg, mdk, mdv,
                       mdq, mdq, a, aq_plain, n_main_dq);
    } else {
      static std::atomic<uint64_t> configured{0};
      e = set_smem_once(tc_bwd_kernel<false, false>, kSmem, configured);
      if (e == cudaSuccess)
        e = launch_bwd(tc_bwd_kernel<false, false>, grid, kSmem, stream, mq, mk, mv, mg, mdk, mdv,
                       mdq, mdq, a, aq_plain, n_main_dq);
    }
    return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
  }
  // dq_i = sum_{j<=i} (g_i . v_j) k_j: the forward product (g, v, k); then
  // (split problems) the aggregate pass of the state sum q g^T, i.e. of the
  // reverse product with k' = q and v' = g; then the fused dk/dv scan
  Product pq{g, v, k, dq, BH, N, M, D, false};
  // its state is sum v k^T: the transpose of the caller's S_0
  pq.state_in = state_in;
  pq.st_ld_r = 1;
  pq.st_ld_c = M;
  if (seeded) seed_from_ckpt(pq, ckpt, ck);
  if (feature) {
    // the value operand k mapped on load, dq times phi'(q)
    pq.feature_v = 1;
    pq.epi_x = q;
  }
  cp_status_t st = tc_launch(pq, tc_plan(BH, N, M, D), agg, status, stream);
  if (st != CP_OK) return st;
  if (plan.G > 1) {
    Product pa{k, q, g, dv, BH, N, D, M, true};
    // the segment sums of phi(q) g^T: the aggregate pass maps its K operand
    if (feature) pa.feature = CP_FEATURE_ELU1;
    st = tc_aggregate(pa, plan, agg, status, stream);
    if (st != CP_OK) return st;
  }
  const unsigned grid = (unsigned)(BH * plan.G);
  if (feature) {
    static std::atomic<uint64_t> configured{0};
    e = set_smem_once(tc_dkdv_kernel<false, true>, dkdv::kSmemBytes, configured);
    if (e == cudaSuccess)
      e = launch_bwd(tc_dkdv_kernel<false, true>, grid, dkdv::kSmemBytes, stream, mq, mk, mv, mg,
                     mdk, mdv, a);
  } else if (grad_state_in != nullptr) {
    static std::atomic<uint64_t> configured{0};
    e = set_smem_once(tc_dkdv_kernel<true, false>, dkdv::kSmemBytes, configured);
    if (e == cudaSuccess)
      e = launch_bwd(tc_dkdv_kernel<true, false>, grid, dkdv::kSmemBytes, stream, mq, mk, mv, mg,
                     mdk, mdv, a);
  } else {
    static std::atomic<uint64_t> configured{0};
    e = set_smem_once(tc_dkdv_kernel<false, false>, dkdv::kSmemBytes, configured);
    if (e == cudaSuccess)
      e = launch_bwd(tc_dkdv_kernel<false, false>, grid, dkdv::kSmemBytes, stream, mq, mk, mv, mg,
                     mdk, mdv, a);
  }
  return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

}  // namespace cp
