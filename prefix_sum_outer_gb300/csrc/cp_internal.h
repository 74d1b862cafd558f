// Internal interface between the C ABI (cp_api.cu) and the kernels.
//
// Every entry point is reduced to one or more "causal products":
//     out_i = sum_{j in W(i)} (q_i . k_j) v_j,
// with W(i) = {j <= i} (forward order) or {j >= i} (reverse order), over a
// batch of BH independent problems.  The forward pass is one forward-order
// product; the backward pass is three products with permuted operands
// (dq: (g, v, k) forward; dv: (k, q, g) reverse; dk: (v, g, q) reverse).
//
// Each product is computed as a two-pass scan over the sequence:
//   pass 1 (only when a problem is split into G > 1 segments): per-segment
//          state aggregates A_s = sum_{j in segment s} k_j v_j^T (fp32);
//   pass 2: every segment starts from the sum of the aggregates that precede
//          it (in scan order, summed in a fixed order) and streams its tiles,
//          carrying the fp32 state on chip.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/causal_product.h"

namespace cp {

// Planning is a pure function of the problem so that the workspace size is
// known on the host without a device; it assumes the 152 SMs of a GB300.
constexpr int kPlanSMs = 152;
// SMs of the current device (kPlanSMs when there is none)
int device_sm_count();
// L2 bytes of the current device (kPlanL2Bytes, a GB300's, when there is none)
constexpr size_t kPlanL2Bytes = 126u << 20;
size_t device_l2_bytes();
// Split forward scans in one launch (tc_lookback_kernel) instead of three:
// environment variable CP_SPLIT_SCAN=lookback, read at each call.  Off by
// default: measured slower on the 16-problem N = 32768 D = M = 128 forward.
bool lookback_enabled();
// flags of a forward split scan run as one launch, after the segments' sums
inline size_t lb_flag_bytes(int64_t problems, int G) {
  return ((size_t)problems * G * sizeof(unsigned int) + 15) / 16 * 16;
}
constexpr size_t kStatusBytes = 256;

// Checkpoints a bf16 forward product leaves for the backward's dq product:
// the state before every `tiles`-th 128-row tile, G - 1 of them per
// problem, fp32 [BH][G - 1][D][M] (the carried-state layout).  The dq
// product runs in G segments of `tiles` tiles, segment s > 0 seeded from
// checkpoint s.  G < 2: no checkpoints.
struct CkptPlan {
  int tiles = 0;
  int G = 1;
  size_t bytes = 0;
};

struct Product {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  int64_t BH, N, D, M;
  bool reverse;
  // Carried state of the scan (fp32, D x M per problem, may be null): the
  // state before the first row in scan order, and the state after the last.
  // Element (r, c) of problem p sits at p * D * M + r * st_ld_r + c * st_ld_c,
  // so a product whose state is the transpose of the caller's reads it
  // through swapped strides.
  const float* state_in = nullptr;
  float* state_out = nullptr;
  int64_t st_ld_r = 0, st_ld_c = 0;
  // feature map applied to q and k as they are loaded (cp_feature_t)
  int feature = 0;
  // element type of q, k, v and out (the fp32 SIMT path also takes fp16)
  cp_dtype_t dtype = CP_DTYPE_F32;
  // bf16 forward: write checkpoints (ck geometry) into ckpt
  CkptPlan ck;
  float* ckpt = nullptr;
  // bf16: run in seed_G segments of seed_tiles tiles, every segment but the
  // first in scan order starting from a precomputed state (instead of a
  // segment-sum pass): element (r, c) of the start of segment s of problem
  // p at seed[p * seed_bh + (s + seed_seg_off) * seed_seg + r * st_ld_r +
  // c * st_ld_c]; no carried state besides
  const float* seed = nullptr;
  int seed_G = 0, seed_tiles = 0;
  int64_t seed_bh = 0, seed_seg = 0;
  int seed_seg_off = 0;
  // bf16: row pitch (elements) of q, k (ld_qk) and of v, out (ld_v, ld_o);
  // 0: dense rows of D or M elements
  int64_t ld_qk = 0, ld_v = 0, ld_o = 0;
  // bf16 forward of an unsplit problem with D, M <= 64 (tc_norm_fused):
  // also write the normaliser z = q_i . sum_{j<=i} k_j, [BH][N] fp32
  float* z = nullptr;
  // bf16 backward products on raw rows (feature map cp_feature_t): map v by
  // phi as it is loaded (feature_v), and multiply each output element by
  // phi'(x) of the raw rows epi_x ([BH][N][M], the output's shape); used
  // together
  int feature_v = 0;
  const void* epi_x = nullptr;
};

// The dq product (g, v, k) of a backward seeded from a forward's checkpoints
// (fp32 [BH][G - 1][D][M] with D = p.M, M = p.D: checkpoint s is the state
// before segment s, read transposed through the product's strides).
inline void seed_from_ckpt(Product& p, const float* ckpt, const CkptPlan& ck) {
  p.seed = ckpt;
  p.seed_G = ck.G;
  p.seed_tiles = ck.tiles;
  p.seed_bh = (int64_t)(ck.G - 1) * p.D * p.M;
  p.seed_seg = p.D * p.M;
  p.seed_seg_off = -1;
}

// ---- fp32 (SIMT FMA) path, also for fp16 inputs (widened on load)
struct SimtPlan {
  int C;        // rows per tile
  int Mb;       // value columns per CTA
  int n_mb;     // value-column blocks
  int G;        // segments per problem
  int64_t seg_rows;
  size_t agg_bytes;
};
SimtPlan simt_plan(int64_t BH, int64_t N, int64_t D, int64_t M);
cudaError_t simt_launch(const Product& p, const SimtPlan& plan, float* agg, int* status,
                        cudaStream_t stream);

// ---- bf16 (tcgen05 tensor-core) path
struct TcPlan {
  int DP;       // D padded to a multiple of 64
  int MB;       // value columns per CTA (64 or 128)
  int n_mb;     // value-column blocks
  int n_tiles;  // 128-row tiles per problem
  int seg_tiles;
  int G;
  size_t agg_bytes;
  bool ok;
};
TcPlan tc_plan(int64_t BH, int64_t N, int64_t D, int64_t M);
// The forward of this plan can write the normaliser in the same launch
// (Product::z): one 64-column box of q, k and of v, one segment per problem.
inline bool tc_norm_fused(const TcPlan& p) {
  return p.ok && p.DP == 64 && p.MB == 64 && p.n_mb == 1 && p.G == 1;
}
// Checkpoint plan of a bf16 problem (pure host computation, 152-SM part).
CkptPlan ckpt_plan(int64_t BH, int64_t N, int64_t D, int64_t M);
cp_status_t tc_launch(const Product& p, const TcPlan& plan, float* agg, int* status,
                      cudaStream_t stream);
// Only pass 1 of the two-pass scan (a no-op when plan.G == 1).  On return
// agg holds each segment's starting state (seg_prefix_launch has run).
cp_status_t tc_aggregate(const Product& p, const TcPlan& plan, float* agg, int* status,
                         cudaStream_t stream);

// Between the passes of a split scan: agg [P][G][E] fp32 per-segment
// aggregates become, in place, the exclusive prefix in scan order (slot s
// holds the sum of the slots before it: s' < s forward, s' > s reverse).
// The slot last in scan order is only written.  A no-op when G <= 1.
cudaError_t seg_prefix_launch(float* agg, int64_t P, int G, int64_t E, bool reverse,
                              cudaStream_t stream);

// Backward pass for bf16 with D, M <= 64 (tc_dkdv_supported(plan), plan =
// tc_plan(BH, N, D, M)): dq is one product launch; dk and dv share the
// reverse state sum q g^T and are computed in one scan.  With checkpoints
// (ckpt non-null, ck.G > 1, no S_0) the dq scans are segments seeded from
// them (on split problems; the one-launch backward keeps whole dq scans).
bool tc_dkdv_supported(const TcPlan& plan);
// state_in (S_0), grad_state_out (dL/dS_N) and grad_state_in (dL/dS_0) are
// [BH][D][M] fp32 or null.  feature: q and k are raw rows of phi = elu + 1
// (mapped inside the scans; dq and dk are the gradients with respect to the
// raw rows); no state, no checkpoints.
cp_status_t tc_bwd_launch(const void* q, const void* k, const void* v, const void* g, void* dq,
                          void* dk, void* dv, const float* state_in,
                          const float* grad_state_out, float* grad_state_in, int64_t BH,
                          int64_t N, int64_t D, int64_t M, const TcPlan& plan, float* agg,
                          int* status, const float* ckpt, const CkptPlan& ck,
                          cudaStream_t stream, bool feature = false);

// ---- decoding step (SIMT): S += k v^T, out = S^T q for every problem;
// M <= 256
cudaError_t decode_launch(const void* q, const void* k, const void* v, void* out, float* state,
                          int64_t BH, int64_t D, int64_t M, cp_dtype_t dtype, cudaStream_t stream);

// ---- normaliser (SIMT): mode 0: z_i = q_i . sum_{j<=i} k_j (fp32 z);
// mode 1: dq_i = g_i sum_{j<=i} k_j; mode 2: dk_j = sum_{i>=j} g_i q_i
// (dq, dk in the input dtype; g fp32).  `scratch` (256-byte aligned) holds
// norm_scratch_bytes(...); a bounded wait that runs out records
// CP_ERR_TIMEOUT in *status.
// With feature != 0, q and k are raw inputs mapped by phi = elu + 1 (rows of
// 16-byte multiples only: norm_feature_supported).
size_t norm_scratch_bytes(int64_t BH, int64_t N, int64_t D, cp_dtype_t dtype);
bool norm_feature_supported(int64_t D, cp_dtype_t dtype);
// kernels one forward normaliser call (mode 0) launches
int norm_launch_count(int64_t BH, int64_t N, int64_t D, cp_dtype_t dtype);
cudaError_t norm_launch(int mode, const void* q, const void* k, const float* grad_z, float* z,
                        void* out, int64_t BH, int64_t N, int64_t D, cp_dtype_t dtype,
                        void* scratch, int* status, cudaStream_t stream, int feature = 0);

// The normaliser with one CTA per problem (no look-back, no scratch): rows
// of D = 64, at least half as many problems as SMs, and the calls it is
// faster for (z of plain rows; dq and dk of mapped rows).  Modes as for
// norm_launch.
bool norm_pp_eligible(int mode, int feature, int64_t BH, int64_t N, int64_t D);
cudaError_t norm_pp_launch(int mode, const void* q, const void* k, const float* grad_z, float* z,
                           void* out, int64_t BH, int64_t N, cp_dtype_t dtype, int* status,
                           cudaStream_t stream, int feature);

// ---- feature map, elementwise over n elements of `dtype`:
// feature_map: y = phi(x); feature_grad: g *= phi'(x) in place
cudaError_t feature_map_launch(int feature, const void* x, void* y, int64_t n, cp_dtype_t dtype,
                               cudaStream_t stream);
cudaError_t feature_grad_launch(int feature, const void* x, void* g, int64_t n,
                                cp_dtype_t dtype, cudaStream_t stream);

// ---- positive random features (bf16, tensor cores): rows x of R input
// features ([BH][N][R]), one projection W [D][R]; R in 8..64 (multiple of
// 8), D in 64..256 (multiple of 64).
// map:   y = phi(x) = exp(W x - |x|^2 / 2) / sqrt(D): rows of bf16(phi)
//        ([BH][N][D]), or with `lo` rows [bf16(phi) | bf16(phi - bf16(phi))]
//        ([BH][N][2D]).
// chain: dx = sum_d a_d phi_d (w_d - x) for a = dL/dphi given as rows
//        [a_1 | a_2] ([BH][N][2D] bf16, a = a_1 + a_2) and phi the first D
//        columns of rows `phi_pitch` elements apart.
bool favor_supported(int64_t R, int64_t D);
cp_status_t favor_map_launch(const void* x, const void* W, void* y, int64_t BH, int64_t N,
                             int64_t R, int64_t D, bool lo, int* status, cudaStream_t stream);
cp_status_t favor_chain_launch(const void* x, const void* W, const void* a, const void* phi,
                               int64_t phi_pitch, void* dx, int64_t BH, int64_t N, int64_t R,
                               int64_t D, int* status, cudaStream_t stream);

// The feature map fused into the product kernel (D = 128 or 256, value
// blocks of 64 columns): out = causal product of phi(xq), phi(xk), v, with
// phi never leaving the CTA.  Split problems run an aggregate pass (phi(xk)
// only) and the segment prefix first; `agg` holds favor_fused_plan(...).agg_bytes.
struct FavorPlan {
  int n_mb, n_tiles, seg_tiles, G;
  size_t agg_bytes;
};
bool favor_fused_supported(int64_t R, int64_t D);
FavorPlan favor_fused_plan(int64_t BH, int64_t N, int64_t D, int64_t M);
cp_status_t favor_fused_fwd_launch(const void* xq, const void* xk, const void* v, const void* W,
                                   void* out, int64_t BH, int64_t N, int64_t R, int64_t D,
                                   int64_t M, float* agg, int* status, cudaStream_t stream);

// ---- failure-path self-test: records CP_ERR_TIMEOUT after `wait_ns`
cudaError_t selftest_timeout_launch(int* status, uint64_t wait_ns, cudaStream_t stream);

}  // namespace cp
