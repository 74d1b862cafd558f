// C ABI of libcausal_product.so: argument checks, planning, workspace
// carving and the launches of the per-dtype kernels.  See
// include/causal_product.h for the contract.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <cstdint>
#include <mutex>

#include <cuda.h>

#include "cp_internal.h"

namespace cp {

bool lookback_enabled() {
  const char* v = std::getenv("CP_SPLIT_SCAN");
  return v != nullptr && std::strcmp(v, "lookback") == 0;
}

int device_sm_count() {
  int dev = 0, n_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      n_sm <= 0) {
    cudaGetLastError();  // no device here: plan for the 152-SM part
    return kPlanSMs;
  }
  return n_sm;
}

size_t device_l2_bytes() {
  int dev = 0, l2 = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess || l2 <= 0) {
    cudaGetLastError();
    return kPlanL2Bytes;
  }
  return (size_t)l2;
}

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// (a null pointer counts as aligned: optional arguments are checked this way)
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// With no rows, the carried state passes through unchanged (zero when absent).
cp_status_t pass_state(const float* from, float* to, size_t bytes, cudaStream_t stream) {
  if (to == nullptr) return CP_OK;
  const cudaError_t e = from != nullptr
                            ? cudaMemcpyAsync(to, from, bytes, cudaMemcpyDeviceToDevice, stream)
                            : cudaMemsetAsync(to, 0, bytes, stream);
  return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

cp_status_t check_dims(int64_t B, int64_t H, int64_t N, int64_t D, int64_t M, cp_dtype_t dtype) {
  if (B <= 0 || H <= 0 || N < 0) return CP_ERR_INVALID_ARG;
  if (dtype != CP_DTYPE_F32 && dtype != CP_DTYPE_BF16 && dtype != CP_DTYPE_F16)
    return CP_ERR_UNSUPPORTED_DTYPE;
  if (D < 1 || D > 256 || M < 1 || M > 256) return CP_ERR_UNSUPPORTED_SHAPE;
  if (dtype == CP_DTYPE_BF16 && ((D % 8) != 0 || (M % 8) != 0)) return CP_ERR_UNSUPPORTED_SHAPE;
  // index arithmetic inside the kernels uses 32-bit tile and problem counts
  if (B * H > (int64_t)1 << 24 || N > (int64_t)1 << 31) return CP_ERR_UNSUPPORTED_SHAPE;
  return CP_OK;
}

// Aggregate bytes one product of shape (BH, N, D', M') needs.
size_t product_agg_bytes(int64_t BH, int64_t N, int64_t D, int64_t M, cp_dtype_t dtype) {
  if (N == 0) return 0;
  if (dtype != CP_DTYPE_BF16) return simt_plan(BH, N, D, M).agg_bytes;
  return tc_plan(BH, N, D, M).agg_bytes;
}

size_t workspace_bytes(int64_t BH, int64_t N, int64_t D, int64_t M, cp_dtype_t dtype,
                       bool backward) {
  size_t agg = product_agg_bytes(BH, N, D, M, dtype);
  if (backward) {
    // dq: (g, v, k) -> D' = M, M' = D ; dv: (k, q, g) -> D' = D, M' = M ;
    // dk: (v, g, q) -> D' = M, M' = D.  They run one after another on the
    // stream, so they share one aggregate area.
    agg = std::max(agg, product_agg_bytes(BH, N, M, D, dtype));
  }
  return kStatusBytes + round_up(agg);
}

cp_status_t run_product(Product p, cp_dtype_t dtype, float* agg, int* status,
                        cudaStream_t stream) {
  if (dtype != CP_DTYPE_BF16) {
    // fp32, and fp16 widened on load: the SIMT kernel
    p.dtype = dtype;
    const SimtPlan plan = simt_plan(p.BH, p.N, p.D, p.M);
    return simt_launch(p, plan, agg, status, stream) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
  }
  const TcPlan plan = tc_plan(p.BH, p.N, p.D, p.M);
  return tc_launch(p, plan, agg, status, stream);
}

// Scratch for one call: the caller's workspace, or a stream-ordered
// allocation released on the same stream when the call's work is enqueued.
struct Scratch {
  void* base = nullptr;
  bool owned = false;
  cudaStream_t stream = nullptr;
  ~Scratch() {
    if (owned && base != nullptr) cudaFreeAsync(base, stream);
  }
};

cp_status_t acquire(Scratch& s, void* workspace, size_t workspace_bytes, size_t need,
                    cudaStream_t stream) {
  s.stream = stream;
  if (workspace != nullptr) {
    if (workspace_bytes < need) return CP_ERR_WORKSPACE_TOO_SMALL;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return CP_ERR_MISALIGNED;
    s.base = workspace;
    return CP_OK;
  }
  if (cudaMallocAsync(&s.base, need, stream) != cudaSuccess) {
    s.base = nullptr;
    return CP_ERR_CUDA;
  }
  s.owned = true;
  // a fresh allocation starts with a clear status word; a caller's workspace
  // keeps its (sticky) status until causal_product_status() reads it
  if (cudaMemsetAsync(s.base, 0, sizeof(int), stream) != cudaSuccess) return CP_ERR_CUDA;
  return CP_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

cp_status_t check_norm_dims(int64_t B, int64_t H, int64_t N, int64_t D, cp_dtype_t dtype) {
  if (B <= 0 || H <= 0 || N < 0) return CP_ERR_INVALID_ARG;
  if (dtype != CP_DTYPE_F32 && dtype != CP_DTYPE_BF16 && dtype != CP_DTYPE_F16)
    return CP_ERR_UNSUPPORTED_DTYPE;
  if (D < 1 || D > 256) return CP_ERR_UNSUPPORTED_SHAPE;
  // 16-bit rows move in 16-byte vectors
  if (dtype != CP_DTYPE_F32 && (D % 8) != 0) return CP_ERR_UNSUPPORTED_SHAPE;
  if (B * H > (int64_t)1 << 24 || N > (int64_t)1 << 31) return CP_ERR_UNSUPPORTED_SHAPE;
  return CP_OK;
}

// phi(q), phi(k) in the feature backward's workspace, after the backward's area
size_t feature_copy_bytes(int64_t BH, int64_t N, int64_t D, cp_dtype_t dtype) {
  const size_t es = dtype == CP_DTYPE_F32 ? 4 : 2;
  return (size_t)BH * N * D * es;
}

size_t norm_workspace_bytes(int64_t BH, int64_t N, int64_t D, cp_dtype_t dtype) {
  return kStatusBytes + round_up(norm_scratch_bytes(BH, N, D, dtype));
}

// Checkpoint plan of a call (none for fp32 and fp16, or without rows).
CkptPlan call_ckpt_plan(int64_t B, int64_t H, int64_t N, int64_t D, int64_t M,
                        cp_dtype_t dtype) {
  if (dtype != CP_DTYPE_BF16 || N <= 0) return CkptPlan{};
  return ckpt_plan(B * H, N, D, M);
}


}  // namespace
}  // namespace cp

extern "C" {

size_t causal_product_workspace_size(int64_t B, int64_t H, int64_t N, int64_t D, int64_t M,
                                     cp_dtype_t dtype, int backward) {
  if (cp::check_dims(B, H, N, D, M, dtype) != CP_OK) return 0;
  return cp::workspace_bytes(B * H, N, D, M, dtype, backward != 0);
}

int causal_product_launch_count(int64_t B, int64_t H, int64_t N, int64_t D, int64_t M,
                                cp_dtype_t dtype, int backward) {
  if (cp::check_dims(B, H, N, D, M, dtype) != CP_OK) return -1;
  if (N == 0) return 0;
  const int64_t BH = B * H;
  // a split scan is three launches: segment sums, their prefix, the scan; a
  // bf16 forward split scan whose grid fits the device is one
  auto product = [&](int64_t d, int64_t m, bool reverse) {
    if (dtype == CP_DTYPE_BF16) {
      const cp::TcPlan p = cp::tc_plan(BH, N, d, m);
      if (p.G <= 1) return 1;
      return !reverse && cp::lookback_enabled() && BH * p.n_mb * p.G <= cp::device_sm_count()
                 ? 1
                 : 3;
    }
    return cp::simt_plan(BH, N, d, m).G > 1 ? 3 : 1;
  };
  if (backward < 0 || backward > 4) return -1;
  // mode 4: the forward with the normaliser (one launch when fused)
  if (backward == 4) {
    if (dtype == CP_DTYPE_BF16 && cp::tc_norm_fused(cp::tc_plan(BH, N, D, M))) return 1;
    return product(D, M, false) + cp::norm_launch_count(BH, N, D, dtype);
  }
  // modes 2 and 3 are the checkpoint calls (forward and backward); with
  // checkpoints the dq product is one launch, seeded from them
  const bool ckpt = backward >= 2 && cp::call_ckpt_plan(B, H, N, D, M, dtype).G > 1;
  if (backward == 0 || backward == 2) return product(D, M, false);
  const int dq_launches = ckpt ? 1 : product(M, D, false);
  if (dtype == CP_DTYPE_BF16) {
    const cp::TcPlan plan = cp::tc_plan(BH, N, D, M);
    if (cp::tc_dkdv_supported(plan)) {
      if (plan.G == 1 && BH < cp::device_sm_count()) return 1;
      // dq product, the reverse segment sums and their prefix, the dk/dv scan
      return dq_launches + (plan.G > 1 ? 2 : 0) + 1;
    }
  }
  // dq (g, v, k), dv (k, q, g), dk (v, g, q); bf16 dk starts from dv's
  // segment prefixes when dv's scan is split with one value block
  int dk_launches = product(M, D, true);
  if (dtype == CP_DTYPE_BF16) {
    const cp::TcPlan pvp = cp::tc_plan(BH, N, D, M);
    if (pvp.ok && pvp.G > 1 && pvp.n_mb == 1) dk_launches = 1;
  }
  return dq_launches + product(D, M, true) + dk_launches;
}

}  // extern "C"

namespace cp {
namespace {

cp_status_t check_ckpt(const CkptPlan& ck, const void* ckpt, size_t ckpt_bytes) {
  if (ck.G < 2) return CP_OK;
  if (ckpt == nullptr) return CP_ERR_INVALID_ARG;
  if (ckpt_bytes < ck.bytes) return CP_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(ckpt)) return CP_ERR_MISALIGNED;
  return CP_OK;
}

cp_status_t fwd_impl(const void* q, const void* k, const void* v, void* out,
                     const float* state_in, float* state_out, float* ckpt, size_t ckpt_bytes,
                     int64_t B, int64_t H, int64_t N, int64_t D, int64_t M, cp_dtype_t dtype,
                     void* workspace, size_t workspace_bytes, void* stream_, bool use_ckpt) {
  cp_status_t st = cp::check_dims(B, H, N, D, M, dtype);
  if (st != CP_OK) return st;
  const CkptPlan ck = use_ckpt ? call_ckpt_plan(B, H, N, D, M, dtype) : CkptPlan{};
  st = check_ckpt(ck, ckpt, ckpt_bytes);
  if (st != CP_OK) return st;
  // with no rows nothing is read or written but the states
  if (N > 0 && (!q || !k || !v || !out)) return CP_ERR_INVALID_ARG;
  if (!cp::aligned16(q) || !cp::aligned16(k) || !cp::aligned16(v) || !cp::aligned16(out) ||
      !cp::aligned16(state_in) || !cp::aligned16(state_out))
    return CP_ERR_MISALIGNED;
  const size_t es = dtype == CP_DTYPE_F32 ? 4 : 2;
  const int64_t BH = B * H;
  const size_t nqk = (size_t)BH * N * D * es, nv = (size_t)BH * N * M * es;
  const size_t nst = (size_t)BH * D * M * sizeof(float);
  if (cp::overlaps(out, nv, q, nqk) || cp::overlaps(out, nv, k, nqk) ||
      cp::overlaps(out, nv, v, nv) || cp::overlaps(out, nv, state_in, nst))
    return CP_ERR_INVALID_ARG;
  if (cp::overlaps(state_out, nst, q, nqk) || cp::overlaps(state_out, nst, k, nqk) ||
      cp::overlaps(state_out, nst, v, nv) || cp::overlaps(state_out, nst, out, nv) ||
      cp::overlaps(state_out, nst, state_in, nst))
    return CP_ERR_INVALID_ARG;
  if (ck.G > 1) {
    const void* others[4] = {q, k, v, out};
    const size_t sz[4] = {nqk, nqk, nv, nv};
    for (int i = 0; i < 4; ++i)
      if (cp::overlaps(ckpt, ck.bytes, others[i], sz[i])) return CP_ERR_INVALID_ARG;
  }
  const size_t need = cp::workspace_bytes(BH, N, D, M, dtype, false);
  if (workspace != nullptr && workspace_bytes < need) return CP_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (N == 0) return cp::pass_state(state_in, state_out, nst, stream);
  cp::Scratch s;
  st = cp::acquire(s, workspace, workspace_bytes, need, stream);
  if (st != CP_OK) return st;
  int* status = static_cast<int*>(s.base);
  float* agg = reinterpret_cast<float*>(static_cast<char*>(s.base) + cp::kStatusBytes);
  cp::Product p{q, k, v, out, BH, N, D, M, false};
  p.state_in = state_in;
  p.state_out = state_out;
  p.st_ld_r = M;
  p.st_ld_c = 1;
  if (ck.G > 1) {
    p.ck = ck;
    p.ckpt = ckpt;
  }
  return cp::run_product(p, dtype, agg, status, stream);
}

}  // namespace
}  // namespace cp

extern "C" {

cp_status_t causal_product_fwd_state(const void* q, const void* k, const void* v, void* out,
                                     const float* state_in, float* state_out, int64_t B,
                                     int64_t H, int64_t N, int64_t D, int64_t M,
                                     cp_dtype_t dtype, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  return cp::fwd_impl(q, k, v, out, state_in, state_out, nullptr, 0, B, H, N, D, M, dtype,
                      workspace, workspace_bytes, stream, false);
}

size_t causal_product_checkpoint_size(int64_t B, int64_t H, int64_t N, int64_t D, int64_t M,
                                      cp_dtype_t dtype) {
  if (cp::check_dims(B, H, N, D, M, dtype) != CP_OK) return 0;
  return cp::call_ckpt_plan(B, H, N, D, M, dtype).bytes;
}

cp_status_t causal_product_fwd_ckpt(const void* q, const void* k, const void* v, void* out,
                                    float* ckpt, size_t ckpt_bytes, int64_t B, int64_t H,
                                    int64_t N, int64_t D, int64_t M, cp_dtype_t dtype,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  return cp::fwd_impl(q, k, v, out, nullptr, nullptr, ckpt, ckpt_bytes, B, H, N, D, M, dtype,
                      workspace, workspace_bytes, stream, true);
}

size_t causal_product_feature_workspace_size(int64_t B, int64_t H, int64_t N, int64_t D,
                                             int64_t M, cp_dtype_t dtype, int backward) {
  if (cp::check_dims(B, H, N, D, M, dtype) != CP_OK) return 0;
  size_t ws = cp::workspace_bytes(B * H, N, D, M, dtype, backward != 0);
  // bf16 maps inside the product kernels; the others keep phi(q), phi(k)
  if (backward && dtype != CP_DTYPE_BF16)
    ws += 2 * cp::round_up(cp::feature_copy_bytes(B * H, N, D, dtype));
  return ws;
}

cp_status_t causal_product_fwd_feature(const void* q, const void* k, const void* v, void* out,
                                       cp_feature_t feature, int64_t B, int64_t H, int64_t N,
                                       int64_t D, int64_t M, cp_dtype_t dtype, void* workspace,
                                       size_t workspace_bytes, void* stream_) {
  if (feature != CP_FEATURE_NONE && feature != CP_FEATURE_ELU1) return CP_ERR_INVALID_ARG;
  cp_status_t st = cp::check_dims(B, H, N, D, M, dtype);
  if (st != CP_OK) return st;
  if (N > 0 && (!q || !k || !v || !out)) return CP_ERR_INVALID_ARG;
  if (!cp::aligned16(q) || !cp::aligned16(k) || !cp::aligned16(v) || !cp::aligned16(out))
    return CP_ERR_MISALIGNED;
  const size_t es = dtype == CP_DTYPE_F32 ? 4 : 2;
  const int64_t BH = B * H;
  const size_t nqk = (size_t)BH * N * D * es, nv = (size_t)BH * N * M * es;
  if (cp::overlaps(out, nv, q, nqk) || cp::overlaps(out, nv, k, nqk) || cp::overlaps(out, nv, v, nv))
    return CP_ERR_INVALID_ARG;
  const size_t need = cp::workspace_bytes(BH, N, D, M, dtype, false);
  if (workspace != nullptr && workspace_bytes < need) return CP_ERR_WORKSPACE_TOO_SMALL;
  if (N == 0) return CP_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cp::Scratch s;
  st = cp::acquire(s, workspace, workspace_bytes, need, stream);
  if (st != CP_OK) return st;
  int* status = static_cast<int*>(s.base);
  float* agg = reinterpret_cast<float*>(static_cast<char*>(s.base) + cp::kStatusBytes);
  cp::Product p{q, k, v, out, BH, N, D, M, false};
  p.feature = feature;
  return cp::run_product(p, dtype, agg, status, stream);
}

cp_status_t causal_product_bwd_feature(const void* q, const void* k, const void* v,
                                       const void* grad_out, void* grad_q, void* grad_k,
                                       void* grad_v, cp_feature_t feature, int64_t B, int64_t H,
                                       int64_t N, int64_t D, int64_t M, cp_dtype_t dtype,
                                       void* workspace, size_t workspace_bytes, void* stream_) {
  if (feature == CP_FEATURE_NONE)
    return causal_product_bwd(q, k, v, grad_out, grad_q, grad_k, grad_v, B, H, N, D, M, dtype,
                              workspace, workspace_bytes, stream_);
  if (feature != CP_FEATURE_ELU1) return CP_ERR_INVALID_ARG;
  cp_status_t st = cp::check_dims(B, H, N, D, M, dtype);
  if (st != CP_OK) return st;
  if (N > 0 && (!q || !k || !v || !grad_out || !grad_q || !grad_k || !grad_v))
    return CP_ERR_INVALID_ARG;
  const void* ptrs[7] = {q, k, v, grad_out, grad_q, grad_k, grad_v};
  for (const void* p : ptrs)
    if (!cp::aligned16(p)) return CP_ERR_MISALIGNED;
  const int64_t BH = B * H;
  {
    const size_t es = dtype == CP_DTYPE_F32 ? 4 : 2;
    const size_t nqk = (size_t)BH * N * D * es, nv = (size_t)BH * N * M * es;
    const void* ins[4] = {q, k, v, grad_out};
    const size_t in_sz[4] = {nqk, nqk, nv, nv};
    void* outs[3] = {grad_q, grad_k, grad_v};
    const size_t out_sz[3] = {nqk, nqk, nv};
    for (int o = 0; o < 3; ++o) {
      for (int i = 0; i < 4; ++i)
        if (cp::overlaps(outs[o], out_sz[o], ins[i], in_sz[i])) return CP_ERR_INVALID_ARG;
      for (int o2 = o + 1; o2 < 3; ++o2)
        if (cp::overlaps(outs[o], out_sz[o], outs[o2], out_sz[o2])) return CP_ERR_INVALID_ARG;
    }
  }
  const size_t bwd_ws = cp::workspace_bytes(BH, N, D, M, dtype, true);
  const size_t copy =
      dtype == CP_DTYPE_BF16 ? 0 : cp::round_up(cp::feature_copy_bytes(BH, N, D, dtype));
  const size_t need = bwd_ws + 2 * copy;
  if (workspace != nullptr && workspace_bytes < need) return CP_ERR_WORKSPACE_TOO_SMALL;
  if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return CP_ERR_MISALIGNED;
  if (N == 0) return CP_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cp::Scratch s;
  st = cp::acquire(s, workspace, workspace_bytes, need, stream);
  if (st != CP_OK) return st;
  if (dtype == CP_DTYPE_BF16) {
    // Three products on the raw rows, phi applied to the tiles in shared
    // memory and phi' to the outputs before their store, so that neither
    // phi(q), phi(k) nor an unscaled gradient reaches memory:
    //   dq_i = phi'(q_i) * sum_{j<=i} (g_i . v_j) phi(k_j)   product (g, v, phi(k))
    //   dv_j = sum_{i>=j} (phi(k_j) . phi(q_i)) g_i         reverse (phi(k), phi(q), g)
    //   dk_j = phi'(k_j) * sum_{i>=j} (v_j . g_i) phi(q_i)  reverse (v, g, phi(q))
    int* status = static_cast<int*>(s.base);
    float* agg = reinterpret_cast<float*>(static_cast<char*>(s.base) + cp::kStatusBytes);
    // D, M <= 64: dk and dv from one reverse scan that maps q and k (dK
    // times phi'(k) from the mapped K box), dq as below, in one launch on
    // unsplit problems
    const cp::TcPlan plan = cp::tc_plan(BH, N, D, M);
    if (cp::tc_dkdv_supported(plan))
      return cp::tc_bwd_launch(q, k, v, grad_out, grad_q, grad_k, grad_v, nullptr, nullptr,
                               nullptr, BH, N, D, M, plan, agg, status, nullptr, cp::CkptPlan{},
                               stream, true);
    cp::Product pq{grad_out, v, k, grad_q, BH, N, M, D, false};
    pq.feature_v = 1;
    pq.epi_x = q;
    cp::Product pv{k, q, grad_out, grad_v, BH, N, D, M, true};
    pv.feature = feature;
    cp::Product pk{v, grad_out, q, grad_k, BH, N, M, D, true};
    pk.feature_v = 1;
    pk.epi_x = k;
    st = cp::run_product(pq, dtype, agg, status, stream);
    if (st == CP_OK) st = cp::run_product(pv, dtype, agg, status, stream);
    if (st == CP_OK) st = cp::run_product(pk, dtype, agg, status, stream);
    return st;
  }
  char* fq = static_cast<char*>(s.base) + bwd_ws;
  char* fk = fq + copy;
  const int64_t n = BH * N * D;
  if (cp::feature_map_launch(feature, q, fq, n, dtype, stream) != cudaSuccess ||
      cp::feature_map_launch(feature, k, fk, n, dtype, stream) != cudaSuccess)
    return CP_ERR_CUDA;
  // the product backward on phi(q), phi(k)
  st = causal_product_bwd(fq, fk, v, grad_out, grad_q, grad_k, grad_v, B, H, N, D, M, dtype,
                          s.base, bwd_ws, stream_);
  if (st != CP_OK) return st;
  if (cp::feature_grad_launch(feature, q, grad_q, n, dtype, stream) != cudaSuccess ||
      cp::feature_grad_launch(feature, k, grad_k, n, dtype, stream) != cudaSuccess)
    return CP_ERR_CUDA;
  return CP_OK;
}

cp_status_t causal_product_fwd(const void* q, const void* k, const void* v, void* out, int64_t B,
                               int64_t H, int64_t N, int64_t D, int64_t M, cp_dtype_t dtype,
                               void* workspace, size_t workspace_bytes, void* stream) {
  return causal_product_fwd_state(q, k, v, out, nullptr, nullptr, B, H, N, D, M, dtype,
                                  workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace cp {
namespace {

cp_status_t bwd_impl(const void* q, const void* k, const void* v, const void* grad_out,
                     const float* state_in, const float* grad_state_out, const float* ckpt,
                     size_t ckpt_bytes, void* grad_q, void* grad_k, void* grad_v,
                     float* grad_state_in, int64_t B, int64_t H, int64_t N, int64_t D, int64_t M,
                     cp_dtype_t dtype, void* workspace, size_t workspace_bytes, void* stream_,
                     bool use_ckpt) {
  cp_status_t st = cp::check_dims(B, H, N, D, M, dtype);
  if (st != CP_OK) return st;
  const CkptPlan ck = use_ckpt ? call_ckpt_plan(B, H, N, D, M, dtype) : CkptPlan{};
  st = check_ckpt(ck, ckpt, ckpt_bytes);
  if (st != CP_OK) return st;
  if (N > 0 && (!q || !k || !v || !grad_out || !grad_q || !grad_k || !grad_v))
    return CP_ERR_INVALID_ARG;
  const void* ptrs[10] = {q, k, v, grad_out, grad_q, grad_k, grad_v,
                          state_in, grad_state_out, grad_state_in};
  for (const void* p : ptrs)
    if (!cp::aligned16(p)) return CP_ERR_MISALIGNED;
  const size_t es = dtype == CP_DTYPE_F32 ? 4 : 2;
  const int64_t BH = B * H;
  const size_t nqk = (size_t)BH * N * D * es, nv = (size_t)BH * N * M * es;
  const size_t nst = (size_t)BH * D * M * sizeof(float);
  const void* ins[6] = {q, k, v, grad_out, state_in, grad_state_out};
  const size_t in_sz[6] = {nqk, nqk, nv, nv, nst, nst};
  void* outs[4] = {grad_q, grad_k, grad_v, grad_state_in};
  const size_t out_sz[4] = {nqk, nqk, nv, nst};
  for (int o = 0; o < 4; ++o) {
    for (int i = 0; i < 6; ++i)
      if (cp::overlaps(outs[o], out_sz[o], ins[i], in_sz[i])) return CP_ERR_INVALID_ARG;
    for (int o2 = o + 1; o2 < 4; ++o2)
      if (cp::overlaps(outs[o], out_sz[o], outs[o2], out_sz[o2])) return CP_ERR_INVALID_ARG;
  }
  if (ck.G > 1) {
    for (int o = 0; o < 4; ++o)
      if (cp::overlaps(outs[o], out_sz[o], ckpt, ck.bytes)) return CP_ERR_INVALID_ARG;
  }
  const size_t need = cp::workspace_bytes(BH, N, D, M, dtype, true);
  if (workspace != nullptr && workspace_bytes < need) return CP_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  // no rows: dL/dS_0 = dL/dS_N
  if (N == 0) return cp::pass_state(grad_state_out, grad_state_in, nst, stream);
  cp::Scratch s;
  st = cp::acquire(s, workspace, workspace_bytes, need, stream);
  if (st != CP_OK) return st;
  int* status = static_cast<int*>(s.base);
  float* agg = reinterpret_cast<float*>(static_cast<char*>(s.base) + cp::kStatusBytes);
  // dq_i = (S_0 + sum_{j<=i} k_j v_j^T) g_i: the forward product (g, v, k),
  // whose state sum v k^T is the transpose of the caller's S_0
  cp::Product pq{grad_out, v, k, grad_q, BH, N, M, D, false};
  pq.state_in = state_in;
  pq.st_ld_r = 1;
  pq.st_ld_c = M;
  // dv_j = R_j^T k_j with R_j = dS_N + sum_{i>=j} q_i g_i^T: the reverse
  // product (k, q, g) with state R; it also hands on dS_0 = R_0
  cp::Product pv{k, q, grad_out, grad_v, BH, N, D, M, true};
  pv.state_in = grad_state_out;
  pv.state_out = grad_state_in;
  pv.st_ld_r = M;
  pv.st_ld_c = 1;
  // dk_j = R_j v_j: the reverse product (v, g, q), whose state is R^T
  cp::Product pk{v, grad_out, q, grad_k, BH, N, M, D, true};
  pk.state_in = grad_state_out;
  pk.st_ld_r = 1;
  pk.st_ld_c = M;
  if (dtype == CP_DTYPE_BF16) {
    // dv and dk share the reverse state R: one scan over q, k, v, g
    const cp::TcPlan plan = cp::tc_plan(BH, N, D, M);
    if (cp::tc_dkdv_supported(plan))
      return cp::tc_bwd_launch(q, k, v, grad_out, grad_q, grad_k, grad_v, state_in,
                               grad_state_out, grad_state_in, BH, N, D, M, plan, agg, status,
                               ck.G > 1 ? ckpt : nullptr, ck, stream);
    // dq: every segment seeded from the forward's checkpoints
    if (ck.G > 1) cp::seed_from_ckpt(pq, ckpt, ck);
    // dk's reverse state R^T is the transpose of dv's R: when dv's scan is
    // split with one value block, dk's segments start from dv's segment
    // prefixes (left in the aggregate area, read transposed) instead of
    // running a segment-sum pass of their own
    const cp::TcPlan pvp = cp::tc_plan(BH, N, D, M);
    if (pvp.ok && pvp.G > 1 && pvp.n_mb == 1 && grad_state_out == nullptr) {
      pk.seed = agg;
      pk.seed_G = pvp.G;
      pk.seed_tiles = pvp.seg_tiles;
      pk.seed_bh = (int64_t)pvp.G * pvp.DP * pvp.MB;
      pk.seed_seg = (int64_t)pvp.DP * pvp.MB;
      pk.seed_seg_off = 0;
      pk.state_in = nullptr;
      pk.st_ld_r = 1;
      pk.st_ld_c = pvp.MB;
    }
  }
  st = cp::run_product(pq, dtype, agg, status, stream);
  if (st != CP_OK) return st;
  st = cp::run_product(pv, dtype, agg, status, stream);
  if (st == CP_OK) st = cp::run_product(pk, dtype, agg, status, stream);
  return st;
}

}  // namespace
}  // namespace cp

extern "C" {

cp_status_t causal_product_bwd_state(const void* q, const void* k, const void* v,
                                     const void* grad_out, const float* state_in,
                                     const float* grad_state_out, void* grad_q, void* grad_k,
                                     void* grad_v, float* grad_state_in, int64_t B, int64_t H,
                                     int64_t N, int64_t D, int64_t M, cp_dtype_t dtype,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  return cp::bwd_impl(q, k, v, grad_out, state_in, grad_state_out, nullptr, 0, grad_q, grad_k,
                      grad_v, grad_state_in, B, H, N, D, M, dtype, workspace, workspace_bytes,
                      stream, false);
}

cp_status_t causal_product_bwd_ckpt(const void* q, const void* k, const void* v,
                                    const void* grad_out, const float* ckpt, size_t ckpt_bytes,
                                    void* grad_q, void* grad_k, void* grad_v, int64_t B,
                                    int64_t H, int64_t N, int64_t D, int64_t M, cp_dtype_t dtype,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  return cp::bwd_impl(q, k, v, grad_out, nullptr, nullptr, ckpt, ckpt_bytes, grad_q, grad_k,
                      grad_v, nullptr, B, H, N, D, M, dtype, workspace, workspace_bytes, stream,
                      true);
}

cp_status_t causal_product_bwd(const void* q, const void* k, const void* v, const void* grad_out,
                               void* grad_q, void* grad_k, void* grad_v, int64_t B, int64_t H,
                               int64_t N, int64_t D, int64_t M, cp_dtype_t dtype, void* workspace,
                               size_t workspace_bytes, void* stream) {
  return causal_product_bwd_state(q, k, v, grad_out, nullptr, nullptr, grad_q, grad_k, grad_v,
                                  nullptr, B, H, N, D, M, dtype, workspace, workspace_bytes,
                                  stream);
}

cp_status_t causal_product_decode(const void* q, const void* k, const void* v, void* out,
                                  float* state, int64_t B, int64_t H, int64_t D, int64_t M,
                                  cp_dtype_t dtype, void* stream_) {
  cp_status_t st = cp::check_dims(B, H, 1, D, M, dtype);
  if (st != CP_OK) return st;
  if (!q || !k || !v || !out || !state) return CP_ERR_INVALID_ARG;
  if (!cp::aligned16(q) || !cp::aligned16(k) || !cp::aligned16(v) || !cp::aligned16(out) ||
      !cp::aligned16(state))
    return CP_ERR_MISALIGNED;
  const size_t es = dtype == CP_DTYPE_F32 ? 4 : 2;
  const int64_t BH = B * H;
  const size_t nq = (size_t)BH * D * es, nv = (size_t)BH * M * es;
  const size_t nst = (size_t)BH * D * M * sizeof(float);
  const void* ins[3] = {q, k, v};
  const size_t in_sz[3] = {nq, nq, nv};
  for (int i = 0; i < 3; ++i)
    if (cp::overlaps(out, nv, ins[i], in_sz[i]) || cp::overlaps(state, nst, ins[i], in_sz[i]))
      return CP_ERR_INVALID_ARG;
  if (cp::overlaps(out, nv, state, nst)) return CP_ERR_INVALID_ARG;
  return cp::decode_launch(q, k, v, out, state, BH, D, M, dtype,
                           static_cast<cudaStream_t>(stream_)) == cudaSuccess
             ? CP_OK
             : CP_ERR_CUDA;
}

size_t causal_product_normalizer_workspace_size(int64_t B, int64_t H, int64_t N, int64_t D,
                                                cp_dtype_t dtype) {
  if (cp::check_norm_dims(B, H, N, D, dtype) != CP_OK) return 0;
  return cp::norm_workspace_bytes(B * H, N, D, dtype);
}

cp_status_t causal_product_normalizer_feature(const void* q, const void* k, float* z,
                                              cp_feature_t feature, int64_t B, int64_t H,
                                              int64_t N, int64_t D, cp_dtype_t dtype,
                                              void* workspace, size_t workspace_bytes,
                                              void* stream_) {
  if (feature != CP_FEATURE_NONE && feature != CP_FEATURE_ELU1) return CP_ERR_INVALID_ARG;
  cp_status_t st = cp::check_norm_dims(B, H, N, D, dtype);
  if (st != CP_OK) return st;
  if (feature != CP_FEATURE_NONE && !cp::norm_feature_supported(D, dtype))
    return CP_ERR_UNSUPPORTED_SHAPE;
  if (N > 0 && (!q || !k || !z)) return CP_ERR_INVALID_ARG;
  if (!cp::aligned16(q) || !cp::aligned16(k) || !cp::aligned16(z)) return CP_ERR_MISALIGNED;
  const size_t es = dtype == CP_DTYPE_F32 ? 4 : 2;
  const int64_t BH = B * H;
  const size_t nqk = (size_t)BH * N * D * es, nz = (size_t)BH * N * sizeof(float);
  if (cp::overlaps(z, nz, q, nqk) || cp::overlaps(z, nz, k, nqk)) return CP_ERR_INVALID_ARG;
  const size_t need = cp::norm_workspace_bytes(BH, N, D, dtype);
  if (workspace != nullptr && workspace_bytes < need) return CP_ERR_WORKSPACE_TOO_SMALL;
  if (N == 0) return CP_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cp::Scratch s;
  st = cp::acquire(s, workspace, workspace_bytes, need, stream);
  if (st != CP_OK) return st;
  int* status = static_cast<int*>(s.base);
  void* scratch = static_cast<char*>(s.base) + cp::kStatusBytes;
  return cp::norm_launch(0, q, k, nullptr, z, nullptr, BH, N, D, dtype, scratch, status, stream,
                         feature) == cudaSuccess
             ? CP_OK
             : CP_ERR_CUDA;
}

cp_status_t causal_product_normalizer(const void* q, const void* k, float* z, int64_t B, int64_t H,
                                      int64_t N, int64_t D, cp_dtype_t dtype, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  return causal_product_normalizer_feature(q, k, z, CP_FEATURE_NONE, B, H, N, D, dtype, workspace,
                                           workspace_bytes, stream);
}

size_t causal_product_fwd_norm_workspace_size(int64_t B, int64_t H, int64_t N, int64_t D,
                                              int64_t M, cp_dtype_t dtype) {
  if (cp::check_dims(B, H, N, D, M, dtype) != CP_OK ||
      cp::check_norm_dims(B, H, N, D, dtype) != CP_OK)
    return 0;
  // the product and the separate normaliser run one after the other and
  // share the area
  return std::max(cp::workspace_bytes(B * H, N, D, M, dtype, false),
                  cp::norm_workspace_bytes(B * H, N, D, dtype));
}

cp_status_t causal_product_fwd_norm(const void* q, const void* k, const void* v, void* out,
                                    float* z, int64_t B, int64_t H, int64_t N, int64_t D,
                                    int64_t M, cp_dtype_t dtype, void* workspace,
                                    size_t workspace_bytes, void* stream_) {
  cp_status_t st = cp::check_dims(B, H, N, D, M, dtype);
  if (st == CP_OK) st = cp::check_norm_dims(B, H, N, D, dtype);
  if (st != CP_OK) return st;
  if (N > 0 && (!q || !k || !v || !out || !z)) return CP_ERR_INVALID_ARG;
  if (!cp::aligned16(q) || !cp::aligned16(k) || !cp::aligned16(v) || !cp::aligned16(out) ||
      !cp::aligned16(z))
    return CP_ERR_MISALIGNED;
  const size_t es = dtype == CP_DTYPE_F32 ? 4 : 2;
  const int64_t BH = B * H;
  const size_t nqk = (size_t)BH * N * D * es, nv = (size_t)BH * N * M * es;
  const size_t nz = (size_t)BH * N * sizeof(float);
  const void* ins[3] = {q, k, v};
  const size_t in_sz[3] = {nqk, nqk, nv};
  for (int i = 0; i < 3; ++i)
    if (cp::overlaps(out, nv, ins[i], in_sz[i]) || cp::overlaps(z, nz, ins[i], in_sz[i]))
      return CP_ERR_INVALID_ARG;
  if (cp::overlaps(z, nz, out, nv)) return CP_ERR_INVALID_ARG;
  const size_t need = std::max(cp::workspace_bytes(BH, N, D, M, dtype, false),
                               cp::norm_workspace_bytes(BH, N, D, dtype));
  if (workspace != nullptr && workspace_bytes < need) return CP_ERR_WORKSPACE_TOO_SMALL;
  if (N == 0) return CP_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cp::Scratch s;
  st = cp::acquire(s, workspace, workspace_bytes, need, stream);
  if (st != CP_OK) return st;
  int* status = static_cast<int*>(s.base);
  void* scratch = static_cast<char*>(s.base) + cp::kStatusBytes;
  cp::Product p{q, k, v, out, BH, N, D, M, false};
  p.st_ld_r = M;
  p.st_ld_c = 1;
  if (dtype == CP_DTYPE_BF16 && cp::tc_norm_fused(cp::tc_plan(BH, N, D, M))) {
    // one launch: the product kernel also writes z
    p.z = z;
    return cp::run_product(p, dtype, static_cast<float*>(scratch), status, stream);
  }
  st = cp::run_product(p, dtype, static_cast<float*>(scratch), status, stream);
  if (st != CP_OK) return st;
  return cp::norm_launch(0, q, k, nullptr, z, nullptr, BH, N, D, dtype, scratch, status, stream,
                         0) == cudaSuccess
             ? CP_OK
             : CP_ERR_CUDA;
}

cp_status_t causal_product_normalizer_bwd_feature(const void* q, const void* k,
                                                  const float* grad_z, void* grad_q, void* grad_k,
                                                  cp_feature_t feature, int64_t B, int64_t H,
                                                  int64_t N, int64_t D, cp_dtype_t dtype,
                                                  void* workspace, size_t workspace_bytes,
                                                  void* stream_) {
  if (feature != CP_FEATURE_NONE && feature != CP_FEATURE_ELU1) return CP_ERR_INVALID_ARG;
  cp_status_t st = cp::check_norm_dims(B, H, N, D, dtype);
  if (st != CP_OK) return st;
  if (feature != CP_FEATURE_NONE && !cp::norm_feature_supported(D, dtype))
    return CP_ERR_UNSUPPORTED_SHAPE;
  if (N > 0 && (!q || !k || !grad_z || !grad_q || !grad_k)) return CP_ERR_INVALID_ARG;
  const void* ptrs[5] = {q, k, grad_z, grad_q, grad_k};
  for (const void* p : ptrs)
    if (!cp::aligned16(p)) return CP_ERR_MISALIGNED;
  const size_t es = dtype == CP_DTYPE_F32 ? 4 : 2;
  const int64_t BH = B * H;
  const size_t nqk = (size_t)BH * N * D * es, nz = (size_t)BH * N * sizeof(float);
  const void* ins[3] = {q, k, grad_z};
  const size_t in_sz[3] = {nqk, nqk, nz};
  for (int i = 0; i < 3; ++i)
    if (cp::overlaps(grad_q, nqk, ins[i], in_sz[i]) || cp::overlaps(grad_k, nqk, ins[i], in_sz[i]))
      return CP_ERR_INVALID_ARG;
  if (cp::overlaps(grad_q, nqk, grad_k, nqk)) return CP_ERR_INVALID_ARG;
  const size_t need = cp::norm_workspace_bytes(BH, N, D, dtype);
  if (workspace != nullptr && workspace_bytes < need) return CP_ERR_WORKSPACE_TOO_SMALL;
  if (N == 0) return CP_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cp::Scratch s;
  st = cp::acquire(s, workspace, workspace_bytes, need, stream);
  if (st != CP_OK) return st;
  int* status = static_cast<int*>(s.base);
  void* scratch = static_cast<char*>(s.base) + cp::kStatusBytes;
  // dq scans k forwards, dk scans g q backwards; they share the scratch
  // area one after the other on the stream
  if (cp::norm_launch(1, q, k, grad_z, nullptr, grad_q, BH, N, D, dtype, scratch, status, stream,
                      feature) != cudaSuccess)
    return CP_ERR_CUDA;
  return cp::norm_launch(2, q, k, grad_z, nullptr, grad_k, BH, N, D, dtype, scratch, status,
                         stream, feature) == cudaSuccess
             ? CP_OK
             : CP_ERR_CUDA;
}

cp_status_t causal_product_normalizer_bwd(const void* q, const void* k, const float* grad_z,
                                          void* grad_q, void* grad_k, int64_t B, int64_t H,
                                          int64_t N, int64_t D, cp_dtype_t dtype, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  return causal_product_normalizer_bwd_feature(q, k, grad_z, grad_q, grad_k, CP_FEATURE_NONE, B, H,
                                               N, D, dtype, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace cp {
namespace {

cp_status_t check_favor(int64_t B, int64_t H, int64_t N, int64_t R, int64_t D, int64_t M,
                        cp_dtype_t dtype) {
  if (dtype != CP_DTYPE_BF16) return CP_ERR_UNSUPPORTED_DTYPE;
  cp_status_t st = check_dims(B, H, N, D, M, dtype);
  if (st != CP_OK) return st;
  if (!favor_supported(R, D)) return CP_ERR_UNSUPPORTED_SHAPE;
  return CP_OK;
}

// Workspace of the positive-random-feature calls: a header and the segment
// sums of the products, then the features and (backward) their gradients.
// Forward: phi(xq), phi(xk) as bf16 [BH][N][D].  Backward: [hi | lo] rows
// of both features ([BH][N][2D]) and the gradients against them
// ([BH][N][2D]).
size_t favor_feat_bytes(int64_t BH, int64_t N, int64_t D, bool backward) {
  return round_up((size_t)BH * N * D * 2 * (backward ? 2 : 1));
}

size_t favor_agg_bytes(int64_t BH, int64_t N, int64_t D, int64_t M, bool backward) {
  if (!backward)
    return round_up(std::max(tc_plan(BH, N, D, M).agg_bytes,
                             favor_fused_plan(BH, N, D, M).agg_bytes));
  return round_up(std::max(tc_plan(BH, N, M, 2 * D).agg_bytes, tc_plan(BH, N, D, M).agg_bytes));
}

size_t favor_ws_bytes(int64_t BH, int64_t N, int64_t D, int64_t M, bool backward) {
  return kStatusBytes + favor_agg_bytes(BH, N, D, M, backward) +
         (backward ? 4 : 2) * favor_feat_bytes(BH, N, D, backward);
}

}  // namespace
}  // namespace cp

extern "C" {

size_t causal_product_favor_workspace_size(int64_t B, int64_t H, int64_t N, int64_t R, int64_t D,
                                           int64_t M, cp_dtype_t dtype, int backward) {
  if (cp::check_favor(B, H, N, R, D, M, dtype) != CP_OK) return 0;
  return cp::favor_ws_bytes(B * H, N, D, M, backward != 0);
}

cp_status_t causal_product_fwd_favor(const void* xq, const void* xk, const void* v, const void* W,
                                     void* out, int64_t B, int64_t H, int64_t N, int64_t R,
                                     int64_t D, int64_t M, cp_dtype_t dtype, void* workspace,
                                     size_t workspace_bytes, void* stream_) {
  cp_status_t st = cp::check_favor(B, H, N, R, D, M, dtype);
  if (st != CP_OK) return st;
  if (N > 0 && (!xq || !xk || !v || !W || !out)) return CP_ERR_INVALID_ARG;
  const void* ptrs[5] = {xq, xk, v, W, out};
  for (const void* p : ptrs)
    if (!cp::aligned16(p)) return CP_ERR_MISALIGNED;
  const int64_t BH = B * H;
  const size_t nx = (size_t)BH * N * R * 2, nv = (size_t)BH * N * M * 2, nw = (size_t)D * R * 2;
  if (cp::overlaps(out, nv, xq, nx) || cp::overlaps(out, nv, xk, nx) ||
      cp::overlaps(out, nv, v, nv) || cp::overlaps(out, nv, W, nw))
    return CP_ERR_INVALID_ARG;
  const size_t need = cp::favor_ws_bytes(BH, N, D, M, false);
  if (workspace != nullptr && workspace_bytes < need) return CP_ERR_WORKSPACE_TOO_SMALL;
  if (N == 0) return CP_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cp::Scratch s;
  st = cp::acquire(s, workspace, workspace_bytes, need, stream);
  if (st != CP_OK) return st;
  int* status = static_cast<int*>(s.base);
  float* agg = reinterpret_cast<float*>(static_cast<char*>(s.base) + cp::kStatusBytes);
  // D = 128 or 256: the feature map inside the product kernel
  if (cp::favor_fused_supported(R, D))
    return cp::favor_fused_fwd_launch(xq, xk, v, W, out, BH, N, R, D, M, agg, status, stream);
  const size_t feat = cp::favor_feat_bytes(BH, N, D, false);
  char* fq = static_cast<char*>(s.base) + cp::kStatusBytes + cp::favor_agg_bytes(BH, N, D, M, false);
  char* fk = fq + feat;
  st = cp::favor_map_launch(xq, W, fq, BH, N, R, D, false, status, stream);
  if (st == CP_OK) st = cp::favor_map_launch(xk, W, fk, BH, N, R, D, false, status, stream);
  if (st != CP_OK) return st;
  cp::Product p{fq, fk, v, out, BH, N, D, M, false};
  return cp::run_product(p, CP_DTYPE_BF16, agg, status, stream);
}

cp_status_t causal_product_bwd_favor(const void* xq, const void* xk, const void* v, const void* W,
                                     const void* grad_out, void* grad_xq, void* grad_xk,
                                     void* grad_v, int64_t B, int64_t H, int64_t N, int64_t R,
                                     int64_t D, int64_t M, cp_dtype_t dtype, void* workspace,
                                     size_t workspace_bytes, void* stream_) {
  cp_status_t st = cp::check_favor(B, H, N, R, D, M, dtype);
  if (st != CP_OK) return st;
  if (N > 0 && (!xq || !xk || !v || !W || !grad_out || !grad_xq || !grad_xk || !grad_v))
    return CP_ERR_INVALID_ARG;
  const void* ptrs[8] = {xq, xk, v, W, grad_out, grad_xq, grad_xk, grad_v};
  for (const void* p : ptrs)
    if (!cp::aligned16(p)) return CP_ERR_MISALIGNED;
  const int64_t BH = B * H;
  const size_t nx = (size_t)BH * N * R * 2, nv = (size_t)BH * N * M * 2, nw = (size_t)D * R * 2;
  const void* ins[5] = {xq, xk, v, W, grad_out};
  const size_t in_sz[5] = {nx, nx, nv, nw, nv};
  void* outs[3] = {grad_xq, grad_xk, grad_v};
  const size_t out_sz[3] = {nx, nx, nv};
  for (int o = 0; o < 3; ++o) {
    for (int i = 0; i < 5; ++i)
      if (cp::overlaps(outs[o], out_sz[o], ins[i], in_sz[i])) return CP_ERR_INVALID_ARG;
    for (int o2 = o + 1; o2 < 3; ++o2)
      if (cp::overlaps(outs[o], out_sz[o], outs[o2], out_sz[o2])) return CP_ERR_INVALID_ARG;
  }
  const size_t need = cp::favor_ws_bytes(BH, N, D, M, true);
  if (workspace != nullptr && workspace_bytes < need) return CP_ERR_WORKSPACE_TOO_SMALL;
  if (N == 0) return CP_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cp::Scratch s;
  st = cp::acquire(s, workspace, workspace_bytes, need, stream);
  if (st != CP_OK) return st;
  int* status = static_cast<int*>(s.base);
  float* agg = reinterpret_cast<float*>(static_cast<char*>(s.base) + cp::kStatusBytes);
  const size_t feat = cp::favor_feat_bytes(BH, N, D, true);
  char* fq = static_cast<char*>(s.base) + cp::kStatusBytes + cp::favor_agg_bytes(BH, N, D, M, true);
  char* fk = fq + feat;
  char* aq = fk + feat;
  char* ak = aq + feat;
  // Features as [hi | lo] bf16 parts.  The gradient of x flows through
  // differences between the a_d = dL/dphi_d of one row (the common part of
  // a_d multiplies sum_d phi_d, nearly independent of x), so each a is
  // taken against both parts of the other side's features: a bf16 feature
  // alone put up to a quarter of a row's scale into dL/dx on the D = 256
  // workload (emulated on the CPU against the fp64 oracle); hi + lo brings it
  // to the bf16 output floor.
  st = cp::favor_map_launch(xq, W, fq, BH, N, R, D, true, status, stream);
  if (st == CP_OK) st = cp::favor_map_launch(xk, W, fk, BH, N, R, D, true, status, stream);
  if (st != CP_OK) return st;
  // dL/dphi(xq)_i = sum_{j<=i} (g_i . v_j) phi(xk)_j: the forward product
  // (g, v, [hi | lo] of phi(xk)), both halves in one launch
  cp::Product pq{grad_out, v, fk, aq, BH, N, M, 2 * D, false};
  // dL/dphi(xk)_j = sum_{i>=j} (v_j . g_i) phi(xq)_i: the reverse product
  cp::Product pk{v, grad_out, fq, ak, BH, N, M, 2 * D, true};
  // dv_j = sum_{i>=j} (phi(xq)_i . phi(xk)_j) g_i on the hi parts
  cp::Product pv{fk, fq, grad_out, grad_v, BH, N, D, M, true};
  pv.ld_qk = 2 * D;
  st = cp::run_product(pq, CP_DTYPE_BF16, agg, status, stream);
  if (st == CP_OK) st = cp::run_product(pk, CP_DTYPE_BF16, agg, status, stream);
  if (st == CP_OK) st = cp::run_product(pv, CP_DTYPE_BF16, agg, status, stream);
  if (st != CP_OK) return st;
  st = cp::favor_chain_launch(xq, W, aq, fq, 2 * D, grad_xq, BH, N, R, D, status, stream);
  if (st == CP_OK)
    st = cp::favor_chain_launch(xk, W, ak, fk, 2 * D, grad_xk, BH, N, R, D, status, stream);
  return st;
}

cp_status_t causal_product_selftest_timeout(void* workspace, uint64_t wait_ns, void* stream_) {
  if (workspace == nullptr) return CP_ERR_INVALID_ARG;
  if (!cp::aligned16(workspace)) return CP_ERR_MISALIGNED;
  if (wait_ns == 0 || wait_ns > 1000000000ull) return CP_ERR_INVALID_ARG;
  return cp::selftest_timeout_launch(static_cast<int*>(workspace), wait_ns,
                                     static_cast<cudaStream_t>(stream_)) == cudaSuccess
             ? CP_OK
             : CP_ERR_CUDA;
}

cp_status_t causal_product_status(void* workspace, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return CP_ERR_CUDA;
  if (workspace == nullptr) return CP_OK;
  int h = 0;
  if (cudaMemcpy(&h, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CP_ERR_CUDA;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpy(workspace, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return CP_ERR_CUDA;
  }
  return h == 0 ? CP_OK : static_cast<cp_status_t>(h);
}

const char* causal_product_error_string(cp_status_t s) {
  switch (s) {
    case CP_OK: return "CP_OK";
    case CP_ERR_INVALID_ARG: return "CP_ERR_INVALID_ARG: null pointer, bad size or aliasing outputs";
    case CP_ERR_UNSUPPORTED_SHAPE: return "CP_ERR_UNSUPPORTED_SHAPE: D or M outside the supported range";
    case CP_ERR_UNSUPPORTED_DTYPE: return "CP_ERR_UNSUPPORTED_DTYPE";
    case CP_ERR_MISALIGNED: return "CP_ERR_MISALIGNED: pointers must be 16-byte aligned (workspace 256)";
    case CP_ERR_WORKSPACE_TOO_SMALL: return "CP_ERR_WORKSPACE_TOO_SMALL";
    case CP_ERR_CUDA: return "CP_ERR_CUDA: a CUDA call failed";
    case CP_ERR_TIMEOUT: return "CP_ERR_TIMEOUT: a kernel wait expired";
    case CP_ERR_NO_DEVICE: return "CP_ERR_NO_DEVICE";
    case CP_ERR_NOALLOC_LIMIT:
      return "CP_ERR_NOALLOC_LIMIT: the problem needs more scratch than the static array of "
             "causal_product_fwd_noalloc holds";
  }
  return "unknown causal_product status";
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Forward pass without any allocation.  Its scratch is a file-scope device
// array; host code only ever passes the array's device address (looked up
// once per device and context), never the host-side symbol itself.
namespace cp {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[CP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};
// the context the cached address belongs to: after cudaDeviceReset the
// runtime creates a new primary context and loads the module again, so the
// address is looked up afresh
CUcontext g_noalloc_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of the scratch array on the current device.
cp_status_t noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CP_ERR_NO_DEVICE;
  const CtxGetCurrentFn get = ctx_get_current();
  if (get == nullptr) return CP_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return CP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr || ctx == nullptr || g_noalloc_ctx[dev] != ctx) {
    // the lookup makes the device's primary context current (and loads the
    // module into it) when nothing has yet
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return CP_ERR_CUDA;
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return CP_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
    g_noalloc_ctx[dev] = ctx;
  }
  *out = g_noalloc_ptr[dev];
  return CP_OK;
}

}  // namespace
}  // namespace cp

extern "C" cp_status_t causal_product_fwd_noalloc(const void* q, const void* k, const void* v,
                                                  void* out, int64_t B, int64_t H, int64_t N,
                                                  int64_t D, int64_t M, cp_dtype_t dtype,
                                                  void* stream) {
  cp_status_t st = cp::check_dims(B, H, N, D, M, dtype);
  if (st != CP_OK) return st;
  if (cp::workspace_bytes(B * H, N, D, M, dtype, false) > CP_NOALLOC_SCRATCH_BYTES)
    return CP_ERR_NOALLOC_LIMIT;
  if (N == 0) return causal_product_fwd(q, k, v, out, B, H, N, D, M, dtype, nullptr, 0, stream);
  void* scratch = nullptr;
  st = cp::noalloc_scratch(&scratch);
  if (st != CP_OK) return st;
  // The array starts zeroed when the module loads, so its status word starts
  // clear; like a caller's workspace it is sticky until
  // causal_product_noalloc_status reads it.  With a caller-style workspace
  // the forward entry point allocates nothing.
  return causal_product_fwd(q, k, v, out, B, H, N, D, M, dtype, scratch,
                            CP_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" cp_status_t causal_product_noalloc_status(void* stream) {
  void* scratch = nullptr;
  const cp_status_t st = cp::noalloc_scratch(&scratch);
  if (st != CP_OK) return st;
  return causal_product_status(scratch, stream);
}
