// bf16 causal product on the 5th-generation tensor cores (sm_103a): the
// product kernel (one CTA = causal_body of cp_tc_causal.cuh) and its host
// side (tile plan, tensor maps, launches).
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <mutex>
#include <type_traits>

#include "cp_internal.h"
#include "cp_tc_causal.cuh"

namespace cp {
namespace tc {

template <int DP, int MB, bool AGG_ONLY, bool STATE_OUT, bool FEAT, bool CKPT, bool SEED,
          bool NORM, bool FEAT_V, bool EPI>
__global__ void __launch_bounds__(kThreads, 1)
    tc_causal_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_o,
                     const __grid_constant__ CUtensorMap tm_x,
                     const KArgs<CKPT || SEED || NORM || EPI> a) {
  causal_body<DP, MB, AGG_ONLY, STATE_OUT, FEAT, CKPT, SEED, NORM, FEAT_V, EPI,
              KArgs<CKPT || SEED || NORM || EPI>>(tm_q, tm_k, tm_v, tm_o, a,
                                                  Phase{(int)blockIdx.x, true, true}, &tm_x);
}

// ------------------------------------------------------------------ host
template <int DP, int MB, bool AGG, bool STATE_OUT = false, bool FEAT = false, bool CKPT = false,
          bool SEED = false, bool NORM = false, bool FEAT_V = false, bool EPI = false>
cudaError_t launch_one(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& o, const ArgsX& ax, unsigned grid, cudaStream_t st,
                       const CUtensorMap* x = nullptr) {
  // the plain kernels get the plain arguments (a copy of the base part)
  const KArgs<CKPT || SEED || NORM || EPI> a = ax;
  using L = Layout<DP, MB, AGG>;
  constexpr int kSmem = L::kSmemBytes + (NORM ? kNormBytes<DP> : 0);
  static_assert(kSmem <= kSmemLimit, "shared memory overflow");
  auto kern = tc_causal_kernel<DP, MB, AGG, STATE_OUT, FEAT, CKPT, SEED, NORM, FEAT_V, EPI>;
  // the shared-memory opt-in is set once per device for each instantiation
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
  // the raw-row map of the derivative epilogue (unused elsewhere)
  return cudaLaunchKernelEx(&cfg, kern, q, k, v, o, x != nullptr ? *x : o, a);
}

// A split scan that runs as one launch (tc_lookback_kernel): when enabled,
// forward, plain or writing checkpoints, and every CTA resident at once (one
// per SM).
bool lookback_eligible(const ArgsX& a, bool feat_v, int64_t grid) {
  if (!lookback_enabled() || a.reverse || a.state_out != nullptr || a.feature || feat_v ||
      a.epi_x != nullptr || a.z != nullptr)
    return false;
  return grid <= device_sm_count();
}

template <int DP, int MB>
cudaError_t launch_pair(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                        const CUtensorMap& o, ArgsX a, const TcPlan& plan, int64_t problems,
                        float* agg, bool agg_only, cudaStream_t st, bool feat_v,
                        const CUtensorMap* x) {
  cudaError_t e = cudaSuccess;
  if (plan.G > 1 && !agg_only && lookback_eligible(a, feat_v, problems * plan.G)) {
    // one launch: each segment's sum, its prefix, its scan (the prefixes and
    // the flags follow the sums)
    const size_t slots = (size_t)problems * plan.G * DP * MB;
    ArgsX b = a;
    b.agg_out = agg;
    b.agg_in = agg + slots;
    b.lb_flags = reinterpret_cast<unsigned int*>(agg + 2 * slots);
    e = cudaMemsetAsync(b.lb_flags, 0, sizeof(unsigned int) * (size_t)problems * plan.G, st);
    if (e != cudaSuccess) return e;
    return lookback_launch(DP, MB, q, k, v, o, b, (unsigned)(problems * plan.G), st);
  }
  if (plan.G > 1) {
    ArgsX b = a;
    b.agg_in = nullptr;
    b.agg_out = agg;
    b.state_in = nullptr;   // aggregates are the segments' own sums
    b.state_out = nullptr;
    const unsigned g1 = (unsigned)(problems * (plan.G - 1));
    e = a.feature ? launch_one<DP, MB, true, false, true>(q, k, v, o, b, g1, st)
        : feat_v  ? launch_one<DP, MB, true, false, false, false, false, false, true>(q, k, v, o,
                                                                                    b, g1, st)
                  : launch_one<DP, MB, true>(q, k, v, o, b, g1, st);
    // each segment's starting state: one slot per second-pass CTA
    if (e == cudaSuccess)
      e = seg_prefix_launch(agg, problems, plan.G, (int64_t)DP * MB, a.reverse != 0, st);
    if (e != cudaSuccess || agg_only) return e;
    a.agg_in = agg;
  } else if (agg_only) {
    return cudaSuccess;
  }
  const unsigned g2 = (unsigned)(problems * plan.G);
  if (feat_v || a.epi_x != nullptr) {
    // a backward product on raw rows: the value map and the derivative
    // epilogue, together and alone
    if (!feat_v || a.epi_x == nullptr || x == nullptr || a.feature || a.state_out != nullptr ||
        a.ckpt != nullptr || a.z != nullptr)
      return cudaErrorInvalidValue;
    return launch_one<DP, MB, false, false, false, false, false, false, true, true>(q, k, v, o, a,
                                                                                  g2, st, x);
  }
  // (a feature map, a carried state, checkpoints and the normaliser are
  // never combined)
  if constexpr (DP == 64 && MB == 64) {
    if (a.z != nullptr) {
      if (plan.G != 1 || a.feature || a.state_out != nullptr || a.state_in != nullptr ||
          a.ckpt != nullptr || a.reverse)
        return cudaErrorInvalidValue;
      return launch_one<DP, MB, false, false, false, false, false, true>(q, k, v, o, a, g2, st);
    }
  }
  if (a.z != nullptr) return cudaErrorInvalidValue;
  if (a.feature) return launch_one<DP, MB, false, false, true>(q, k, v, o, a, g2, st);
  if (a.state_out != nullptr) return launch_one<DP, MB, false, true>(q, k, v, o, a, g2, st);
  if (a.ckpt != nullptr) return launch_one<DP, MB, false, false, false, true>(q, k, v, o, a, g2, st);
  return launch_one<DP, MB, false>(q, k, v, o, a, g2, st);
}

// The scan pass alone, every segment seeded from a precomputed slot
// (checkpoints a forward product left): agg_in holds [P][G][DP][MB] with
// slot s the state before segment s.
template <int DP, int MB>
cudaError_t launch_seeded(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& o, const ArgsX& a, int64_t problems,
                          cudaStream_t st) {
  return launch_one<DP, MB, false, false, false, false, true>(q, k, v, o, a,
                                                             (unsigned)(problems * a.G), st);
}

}  // namespace tc

TcPlan tc_plan(int64_t BH, int64_t N, int64_t D, int64_t M) {
  TcPlan p{};
  p.DP = (int)((D + 63) / 64 * 64);
  const int Mpad = (int)((M + 63) / 64 * 64);
  // widest value block whose tile set fits shared memory and TMEM
  if (p.DP <= 128 && Mpad >= 128)
    p.MB = 128;
  else
    p.MB = 64;
  p.n_mb = (Mpad + p.MB - 1) / p.MB;
  p.n_tiles = (int)((N + tc::kTile - 1) / tc::kTile);
  const int64_t problems = BH * p.n_mb;
  int64_t G = 1;
  if (problems * 4 < (int64_t)kPlanSMs * 3)  // fewer than 3/4 of the SMs busy: split
    G = std::max<int64_t>(1, kPlanSMs / problems);
  G = std::min<int64_t>(G, std::max(1, p.n_tiles));
  p.seg_tiles = (int)((p.n_tiles + G - 1) / G);
  p.G = p.seg_tiles > 0 ? (p.n_tiles + p.seg_tiles - 1) / p.seg_tiles : 1;
  if (p.G < 1) p.G = 1;
  // the segments' sums, then (forward scans in one launch) their prefixes
  // and flags
  p.agg_bytes = p.G > 1 ? 2 * sizeof(float) * (size_t)problems * p.G * p.DP * p.MB +
                              lb_flag_bytes(problems, p.G)
                        : 0;
  // the entry points allow M <= 256; internal products (the gradients of the
  // positive random features, with hi | lo value halves) go to 512
  p.ok = p.DP <= 256 && Mpad <= 512;
  return p;
}

CkptPlan ckpt_plan(int64_t BH, int64_t N, int64_t D, int64_t M) {
  CkptPlan c;
  const TcPlan fp = tc_plan(BH, N, D, M);
  const TcPlan qp = tc_plan(BH, N, M, D);  // the dq product (g, v, k)
  if (!fp.ok || !qp.ok || qp.n_tiles < 2) return c;
  int tiles = 0;
  if (qp.G > 1) {
    // dq is split into segments anyway: the checkpoints replace its
    // segment-sum pass and the prefix between the passes.  (The one-launch
    // backward keeps whole dq scans: measured on B=8 H=16 N=4096 D=M=64, a
    // dq scan cut into 2, 4 or 8 seeded segments made that launch 8, 8 and
    // 31 us slower, each extra scan start and drain costing about 7 us.)
    tiles = qp.seg_tiles;
  }
  if (tiles < 1) return c;
  const int G = (qp.n_tiles + tiles - 1) / tiles;
  if (G < 2) return c;
  c.tiles = tiles;
  c.G = G;
  c.bytes = sizeof(float) * (size_t)BH * (G - 1) * D * M;
  return c;
}

namespace {
cp_status_t tc_run(const Product& p, const TcPlan& plan, float* agg, int* status,
                   cudaStream_t stream, bool agg_only) {
  if (!plan.ok) return CP_ERR_UNSUPPORTED_SHAPE;
  CUtensorMap mq, mk, mv, mo, mx;
  if (!tc::make_map(&mq, p.q, p.BH, p.N, p.D, p.ld_qk) ||
      !tc::make_map(&mk, p.k, p.BH, p.N, p.D, p.ld_qk) ||
      !tc::make_map(&mv, p.v, p.BH, p.N, p.M, p.ld_v) ||
      !tc::make_map(&mo, p.out, p.BH, p.N, p.M, p.ld_o) ||
      (p.epi_x != nullptr && !tc::make_map(&mx, p.epi_x, p.BH, p.N, p.M, p.ld_o)))
    return CP_ERR_UNSUPPORTED_SHAPE;
  tc::ArgsX a{};
  a.N = p.N;
  a.n_tiles = plan.n_tiles;
  a.seg_tiles = plan.seg_tiles;
  a.G = plan.G;
  a.BH = (int)p.BH;
  a.n_mb = plan.n_mb;
  a.reverse = p.reverse ? 1 : 0;
  a.status = status;
  a.state_in = p.state_in;
  a.state_out = p.state_out;
  a.st_ld_r = p.st_ld_r;
  a.st_ld_c = p.st_ld_c;
  a.Dr = (int)p.D;
  a.Mc = (int)p.M;
  a.feature = p.feature;
  a.ckpt = p.ckpt;
  a.ck_tiles = p.ck.tiles;
  a.ck_G = p.ck.G;
  a.z = p.z;
  a.epi_x = p.epi_x;
  const int64_t problems = p.BH * plan.n_mb;
  const bool seeded = p.seed != nullptr;
  if (seeded) {
    // segments each seeded from a precomputed state (read through the
    // carried-state strides; no carried state besides)
    if (agg_only || p.seed_G < 2 || p.seed_tiles < 1 || p.state_in != nullptr || p.feature ||
        p.feature_v || p.epi_x != nullptr ||
        (int64_t)(p.seed_G - 1) * p.seed_tiles >= plan.n_tiles)
      return CP_ERR_INVALID_ARG;
    a.G = p.seed_G;
    a.seg_tiles = p.seed_tiles;
    a.agg_in = nullptr;
    a.seed = p.seed;
    a.seed_bh = p.seed_bh;
    a.seed_seg = p.seed_seg;
    a.seed_seg_off = p.seed_seg_off;
  }
  cudaError_t e;
#define CP_TC_CASE(DP_, MB_)                                                                  \
  if (plan.DP == DP_ && plan.MB == MB_)                                                       \
    e = seeded ? tc::launch_seeded<DP_, MB_>(mq, mk, mv, mo, a, problems, stream)             \
               : tc::launch_pair<DP_, MB_>(mq, mk, mv, mo, a, plan, problems, agg, agg_only,  \
                                           stream, p.feature_v != 0,                          \
                                           p.epi_x != nullptr ? &mx : nullptr);               \
  else
  CP_TC_CASE(64, 64)
  CP_TC_CASE(64, 128)
  CP_TC_CASE(128, 64)
  CP_TC_CASE(128, 128)
  CP_TC_CASE(192, 64)
  CP_TC_CASE(256, 64)
  return CP_ERR_UNSUPPORTED_SHAPE;
#undef CP_TC_CASE
  return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

}  // namespace

cp_status_t tc_launch(const Product& p, const TcPlan& plan, float* agg, int* status,
                      cudaStream_t stream) {
  return tc_run(p, plan, agg, status, stream, false);
}

cp_status_t tc_aggregate(const Product& p, const TcPlan& plan, float* agg, int* status,
                         cudaStream_t stream) {
  return tc_run(p, plan, agg, status, stream, true);
}

}  // namespace cp
