// Normaliser of causal linear attention and its backward (SIMT).
//
// The denominator of causal linear attention ("Transformers are RNNs",
// phi(q_i)^T sum_{j<=i} phi(k_j)) is the causal product with a value of 1:
//     z_i = q_i . c_i,           c_i = sum_{j<=i} k_j            (forward)
// and with g = dL/dz
//     dq_i = g_i c_i,            dk_j = sum_{i>=j} g_i q_i        (backward).
// Each is a scan of a D-vector along the sequence, bound by HBM: a row is
// read once and its result written once.
//
// Layout of a CTA over one tile of rows: TPR consecutive lanes share a row
// (each holds K vectors of that row's columns, so a warp reads whole rows),
// and each thread holds RPT consecutive rows in registers.  The scan of a
// tile runs in three levels: sequentially over a thread's own rows, a
// shuffle scan across the row groups of a warp, and the warps' column totals
// combined through shared memory; the carry of everything before the tile
// is added last.
//
// Rows of 16-byte multiples (every bf16 shape, fp32 with D % 4 == 0) take a
// single pass: persistent CTAs take tiles from a ticket counter (tiles of
// all problems interleaved, in scan order), stream them into a ring of
// shared-memory stages with TMA bulk copies, publish each tile's column sum,
// and take the carry from a look-back over the tiles before it: the
// inclusive prefix published W tiles back plus the column sums of the W - 1
// tiles in between, added in that fixed order (so the result does not
// depend on timing).  The published vectors start out as an all-ones NaN
// pattern that fp32 arithmetic never produces, and a reader polls the
// values themselves until none is left (one round trip when they are
// ready; no flags, no fences).  A tile waits only on tiles with smaller
// tickets, which are held by running CTAs, so the scheme cannot deadlock;
// every wait is bounded all the same.  Other fp32 rows use two passes over segments: a
// first pass writes each segment's column sums and every segment starts from
// the fixed-order sum of those before it in scan order.  Either way the
// results are bitwise reproducible.
#include <algorithm>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cp_internal.h"
#include "sm103_ptx.cuh"

namespace cp {
namespace {

constexpr int kNormWarps = 8;
constexpr int kNormThreads = 32 * kNormWarps;
constexpr int kNormMaxD = 256;

enum NormMode : int { kZ = 0, kDQ = 1, kDK = 2 };

struct NormArgs {
  const void* q;
  const void* k;
  const float* grad_z;  // dq, dk: [BH][N]
  float* z;             // z: [BH][N]
  void* out;            // dq or dk, in the input dtype
  int64_t N;
  int D;
  int tpr;              // lanes per row (a power of two <= 32)
  int G;                // segments per problem
  int GL;               // segments this launch covers per problem
  int seg_base;         // first segment this launch covers
  int64_t seg_rows;
  const float* agg_in;  // [BH][G][D] segment column sums (second pass), may be null
  float* agg_out;       // first pass
  int agg_only;
};

// V elements of T moved by one (16-byte, or scalar) access.
template <typename T, int V>
struct VecIO;

template <>
struct VecIO<__nv_bfloat16, 8> {
  using R = uint4;
  static __device__ __forceinline__ R zero() { return make_uint4(0u, 0u, 0u, 0u); }
  static __device__ __forceinline__ R load(const void* p, int64_t e) {
    return __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p) + e));
  }
  static __device__ __forceinline__ R lds(const uint8_t* p, int64_t e) {
    return *reinterpret_cast<const uint4*>(p + e * 2);
  }
  static __device__ __forceinline__ void unpack(const R& r, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 t = __bfloat1622float2(h[j]);
      f[2 * j] = t.x;
      f[2 * j + 1] = t.y;
    }
  }
  // the 8 values as 4 pairs (bf16 -> f32 is a shift of the bit pattern)
  static __device__ __forceinline__ void unpack2(const R& r, float2* f) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      f[j] = make_float2(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xffff0000u));
  }
  static __device__ __forceinline__ void store2(void* p, int64_t e, const float2* f) {
    uint4 r;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(f[j].x, f[j].y);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p) + e) = r;
  }
  static __device__ __forceinline__ void store(void* p, int64_t e, const float* f) {
    uint4 r;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p) + e) = r;
  }
};

template <>
struct VecIO<__half, 8> {
  using R = uint4;
  static __device__ __forceinline__ R zero() { return make_uint4(0u, 0u, 0u, 0u); }
  static __device__ __forceinline__ R lds(const uint8_t* p, int64_t e) {
    return *reinterpret_cast<const uint4*>(p + e * 2);
  }
  static __device__ __forceinline__ void unpack2(const R& r, float2* f) {
    const __half2* h = reinterpret_cast<const __half2*>(&r);
#pragma unroll
    for (int j = 0; j < 4; ++j) f[j] = __half22float2(h[j]);
  }
  static __device__ __forceinline__ void store2(void* p, int64_t e, const float2* f) {
    uint4 r;
    __half2* h = reinterpret_cast<__half2*>(&r);
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = __floats2half2_rn(f[j].x, f[j].y);
    *reinterpret_cast<uint4*>(static_cast<__half*>(p) + e) = r;
  }
};

template <>
struct VecIO<float, 4> {
  using R = float4;
  static __device__ __forceinline__ R zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
  static __device__ __forceinline__ R load(const void* p, int64_t e) {
    return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p) + e));
  }
  static __device__ __forceinline__ R lds(const uint8_t* p, int64_t e) {
    return *reinterpret_cast<const float4*>(p + e * 4);
  }
  static __device__ __forceinline__ void unpack(const R& r, float* f) {
    f[0] = r.x;
    f[1] = r.y;
    f[2] = r.z;
    f[3] = r.w;
  }
  static __device__ __forceinline__ void store(void* p, int64_t e, const float* f) {
    *reinterpret_cast<float4*>(static_cast<float*>(p) + e) = make_float4(f[0], f[1], f[2], f[3]);
  }
  static __device__ __forceinline__ void unpack2(const R& r, float2* f) {
    f[0] = make_float2(r.x, r.y);
    f[1] = make_float2(r.z, r.w);
  }
  static __device__ __forceinline__ void store2(void* p, int64_t e, const float2* f) {
    *reinterpret_cast<float4*>(static_cast<float*>(p) + e) = make_float4(f[0].x, f[0].y, f[1].x, f[1].y);
  }
};

template <>
struct VecIO<float, 1> {
  using R = float;
  static __device__ __forceinline__ R zero() { return 0.f; }
  static __device__ __forceinline__ R load(const void* p, int64_t e) {
    return __ldg(static_cast<const float*>(p) + e);
  }
  static __device__ __forceinline__ void unpack(const R& r, float* f) { f[0] = r; }
  static __device__ __forceinline__ void store(void* p, int64_t e, const float* f) {
    static_cast<float*>(p)[e] = f[0];
  }
};

// T: element type; V: elements per access; K: accesses per thread per row.
template <typename T, int V, int K, int MODE>
__global__ void __launch_bounds__(kNormThreads, 2) norm_kernel(const NormArgs a) {
  constexpr int RPT = 8 / K;  // rows per thread
  constexpr bool kRev = MODE == kDK;
  using IO = VecIO<T, V>;
  using R = typename IO::R;
  __shared__ float carry[kNormMaxD];              // sum of everything before this tile
  __shared__ float wt[kNormWarps][kNormMaxD];     // the warps' column totals
  __shared__ float cw[kNormWarps][kNormMaxD];     // carry into each warp

  const int D = a.D, TPR = a.tpr;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cc = lane & (TPR - 1);  // position within the row
  const int gw = lane / TPR;        // row group within the warp
  const int gpw = 32 / TPR;
  const int tile_rows = RPT * kNormWarps * gpw;
  const int p = blockIdx.x / a.GL;
  const int s = blockIdx.x % a.GL + a.seg_base;
  const int64_t seg_lo = (int64_t)s * a.seg_rows;
  const int64_t seg_hi = min(a.N, seg_lo + a.seg_rows);
  const int64_t base = (int64_t)p * a.N;
  const void* src = MODE == kDK ? a.q : a.k;  // the scanned rows (times g for dk)

  int col[K];
  bool colv[K];
#pragma unroll
  for (int kk = 0; kk < K; ++kk) {
    col[kk] = (cc + kk * TPR) * V;
    colv[kk] = col[kk] < D;
  }

  // initial carry: fixed-order sum of the segments before this one in scan order
  for (int d = threadIdx.x; d < D; d += kNormThreads) {
    float c = 0.f;
    if (!a.agg_only && a.agg_in != nullptr) {
      const int lo = kRev ? s + 1 : 0, hi = kRev ? a.G : s;
      for (int s2 = lo; s2 < hi; ++s2) c += a.agg_in[((int64_t)p * a.G + s2) * D + d];
    }
    carry[d] = c;
  }
  __syncthreads();

  const int n_t = (int)((seg_hi - seg_lo + tile_rows - 1) / tile_rows);
  const int sp0 = (warp * gpw + gw) * RPT;  // this thread's first scan position in a tile
  for (int it = 0; it < n_t; ++it) {
    const int t = kRev ? n_t - 1 - it : it;
    const int64_t lo = seg_lo + (int64_t)t * tile_rows;
    const int64_t hi = min(seg_hi, lo + tile_rows);
    // ---- load this thread's rows (scan order: ascending rows, descending for dk)
    R xs[RPT][K];
    R qs[MODE == kZ ? RPT : 1][K];
    float gz[RPT];
    int64_t rows[RPT];
    bool valid[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      rows[i] = kRev ? hi - 1 - (sp0 + i) : lo + sp0 + i;
      valid[i] = kRev ? rows[i] >= lo : rows[i] < hi;
      const int64_t e0 = (base + rows[i]) * D;
#pragma unroll
      for (int kk = 0; kk < K; ++kk) {
        const bool ok = valid[i] && colv[kk];
        xs[i][kk] = ok ? IO::load(src, e0 + col[kk]) : IO::zero();
        if constexpr (MODE == kZ) qs[i][kk] = ok ? IO::load(a.q, e0 + col[kk]) : IO::zero();
      }
      gz[i] = (MODE != kZ && valid[i]) ? a.grad_z[base + rows[i]] : 0.f;
    }
    // ---- level 1: this thread's rows
    float sum[K][V];
#pragma unroll
    for (int kk = 0; kk < K; ++kk)
#pragma unroll
      for (int v = 0; v < V; ++v) sum[kk][v] = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; ++i)
#pragma unroll
      for (int kk = 0; kk < K; ++kk) {
        float f[V];
        IO::unpack(xs[i][kk], f);
#pragma unroll
        for (int v = 0; v < V; ++v) sum[kk][v] += MODE == kDK ? gz[i] * f[v] : f[v];
      }
    // ---- level 2: inclusive scan across the warp's row groups (same cc)
    for (int o = TPR; o < 32; o <<= 1) {
#pragma unroll
      for (int kk = 0; kk < K; ++kk)
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const float y = __shfl_up_sync(0xffffffffu, sum[kk][v], o);
          if (lane >= o) sum[kk][v] += y;
        }
    }
    float ex[K][V];  // exclusive: the groups before this one
#pragma unroll
    for (int kk = 0; kk < K; ++kk)
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const float y = __shfl_up_sync(0xffffffffu, sum[kk][v], TPR);
        ex[kk][v] = gw == 0 ? 0.f : y;
      }
    if (gw == gpw - 1) {
#pragma unroll
      for (int kk = 0; kk < K; ++kk)
        if (colv[kk])
#pragma unroll
          for (int v = 0; v < V; ++v) wt[warp][col[kk] + v] = sum[kk][v];
    }
    __syncthreads();
    // ---- level 3: carry into each warp, in warp order
    for (int i = threadIdx.x; i < kNormWarps * D; i += kNormThreads) {
      const int w = i / D, d = i - w * D;
      float c = carry[d];
      for (int w2 = 0; w2 < w; ++w2) c += wt[w2][d];
      cw[w][d] = c;
    }
    __syncthreads();
    if (!a.agg_only) {
      float c[K][V];
#pragma unroll
      for (int kk = 0; kk < K; ++kk)
#pragma unroll
        for (int v = 0; v < V; ++v) c[kk][v] = (colv[kk] ? cw[warp][col[kk] + v] : 0.f) + ex[kk][v];
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        float part = 0.f;
        const int64_t e0 = (base + rows[i]) * D;
#pragma unroll
        for (int kk = 0; kk < K; ++kk) {
          float f[V];
          IO::unpack(xs[i][kk], f);
#pragma unroll
          for (int v = 0; v < V; ++v) c[kk][v] += MODE == kDK ? gz[i] * f[v] : f[v];
          if constexpr (MODE == kZ) {
            float qf[V];
            IO::unpack(qs[i][kk], qf);
#pragma unroll
            for (int v = 0; v < V; ++v) part = fmaf(qf[v], c[kk][v], part);
          } else {
            float o[V];
#pragma unroll
            for (int v = 0; v < V; ++v) o[v] = MODE == kDQ ? gz[i] * c[kk][v] : c[kk][v];
            if (valid[i] && colv[kk]) IO::store(a.out, e0 + col[kk], o);
          }
        }
        if constexpr (MODE == kZ) {
          // the row's dot product is spread over its TPR lanes
          for (int o = TPR >> 1; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
          if (valid[i] && (i & (TPR - 1)) == cc) a.z[base + rows[i]] = part;
        }
      }
    }
    // carry past this tile
    for (int d = threadIdx.x; d < D; d += kNormThreads)
      carry[d] = cw[kNormWarps - 1][d] + wt[kNormWarps - 1][d];
    __syncthreads();
  }
  if (a.agg_only) {
    for (int d = threadIdx.x; d < D; d += kNormThreads)
      a.agg_out[((int64_t)p * a.G + s) * D + d] = carry[d];
  }
}

// ---------------------------------------------------------------------------
// Single-pass kernel with look-back (rows of 16-byte multiples).
constexpr int kLbWarps = 4;
constexpr int kLbThreads = 32 * kLbWarps;
constexpr int kLbMaxStages = 8;
constexpr int kLbRowsPerThread = 8;           // divided by K
constexpr uint32_t kLbRingBytes = 32 * 1024;  // shared memory of a CTA's ring
constexpr int kMaxDev = 64;

struct LbArgs {
  const void* q;
  const void* k;
  const float* grad_z;
  float* z;
  void* out;
  int64_t N;
  int D;
  int tpr;
  int BH;
  int T;                  // tiles per problem
  int W;                  // look-back window
  int n_stages;
  uint32_t stage_bytes;   // one ring stage (all inputs of a tile)
  uint32_t in_bytes;      // offset of the second input in a stage
  uint32_t total;         // BH * T tickets (< 2^31)
  float* agg;             // [BH][T][D] column sums of the tiles (scan order)
  float* incl;            // [BH][T][D] inclusive prefixes
  unsigned int* ticket;   // starts at all ones: the first ticket is 0
  int* status;
};

// Not yet published: the fill pattern of the look-back arrays (a NaN that
// no fp32 addition returns; those return the canonical NaN).
constexpr uint32_t kUnset = 0xffffffffu;

__device__ __forceinline__ bool unset(float v) { return __float_as_uint(v) == kUnset; }

// Give up on a poll after the wait limit, or once some CTA recorded an error.
__device__ __forceinline__ bool poll_expired(uint64_t t0, const int* status) {
  if (*reinterpret_cast<const volatile int*>(status) != 0) return true;
  return ptx::globaltimer() - t0 > CP_WAIT_TIMEOUT_NS;
}

__device__ __forceinline__ void lb_record_timeout(int* status, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicCAS(status, 0, (int)CP_ERR_TIMEOUT);
}

// Feature map phi(x) = elu(x) + 1 of causal linear attention on a pair:
// with e = e^min(x, 0), phi(x) = e + max(x, 0) and phi'(x) = e.
__device__ __forceinline__ void elu1_pair(float2 x, float2& phi, float2& dphi) {
  dphi = make_float2(__expf(fminf(x.x, 0.f)), __expf(fminf(x.y, 0.f)));
  phi = __fadd2_rn(dphi, make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)));
}

// FEAT: q and k are raw inputs x mapped by phi on load; dq and dk are then
// taken through phi' (dq = phi'(x_q) g sum phi(k), dk = phi'(x_k) sum g phi(q)),
// so every mode streams both q and k.
template <typename T, int V, int K, int MODE, bool FEAT>
__global__ void __launch_bounds__(kLbThreads, 3) norm_lb_kernel(const LbArgs a) {
  constexpr int RPT = kLbRowsPerThread / K;
  constexpr bool kRev = MODE == kDK;
  constexpr bool kTwo = MODE == kZ || FEAT;  // a second input per tile
  constexpr int kIn = kTwo ? 2 : 1;          // inputs streamed per tile
  constexpr int V2 = V / 2;
  using IO = VecIO<T, V>;
  using R = typename IO::R;
  extern __shared__ __align__(128) uint8_t lsm[];
  __shared__ uint64_t full[kLbMaxStages];
  __shared__ int st_p[kLbMaxStages];  // problem of the stage's tile, -1: no tile
  __shared__ int st_t[kLbMaxStages];  // the tile's index in scan order
  __shared__ int abort_flag;

  const int D = a.D, TPR = a.tpr, S = a.n_stages;
  // after the ring: the warps' column totals, the carry into each warp, the
  // tile's sum and partial sums of the look-back
  float* wt = reinterpret_cast<float*>(lsm + (size_t)S * a.stage_bytes);  // [kLbWarps][D]
  float* cw = wt + kLbWarps * D;                                           // [kLbWarps][D]
  float* tsum = cw + kLbWarps * D;                                         // [D]
  float* part = tsum + D;                                                  // [max(128, D)]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cc = lane & (TPR - 1), gw = lane / TPR, gpw = 32 / TPR;
  const int tile_rows = RPT * kLbWarps * gpw;
  const int sp0 = (warp * gpw + gw) * RPT;
  const void* src = MODE == kDK ? a.q : a.k;
  const void* other = MODE == kDK ? a.k : a.q;  // the second input (z, FEAT)
  // look-back work of this thread: column lb_d of run lb_pt (D <= 128: the
  // runs split the tiles between nparts thread groups; else one run)
  const int nparts = D <= kLbThreads ? kLbThreads / D : 1;
  const int lb_pt = D <= kLbThreads ? tid / D : 0;
  const int lb_d = D <= kLbThreads ? tid - lb_pt * D : tid;

  int col[K];
  bool colv[K];
#pragma unroll
  for (int kk = 0; kk < K; ++kk) {
    col[kk] = (cc + kk * TPR) * V;
    colv[kk] = col[kk] < D;
  }

  // thread 0: take ticket x into stage s and start its copies
  auto issue = [&](int s, uint32_t x) {
    if (x >= a.total) {
      st_p[s] = -1;
      return;
    }
    const int p = (int)(x % (uint32_t)a.BH), ts = (int)(x / (uint32_t)a.BH);
    st_p[s] = p;
    st_t[s] = ts;
    const int tr = kRev ? a.T - 1 - ts : ts;
    const int64_t lo = (int64_t)tr * tile_rows, hi = min(a.N, lo + tile_rows);
    const uint32_t bytes = (uint32_t)((hi - lo) * D * (int64_t)sizeof(T));
    uint8_t* st = lsm + (size_t)s * a.stage_bytes;
    const int64_t e0 = ((int64_t)p * a.N + lo) * D;
    ptx::mbar_arrive_expect_tx(&full[s], kIn * bytes);
    ptx::bulk_load(st, static_cast<const T*>(src) + e0, bytes, &full[s]);
    if (kIn == 2)
      ptx::bulk_load(st + a.in_bytes, static_cast<const T*>(other) + e0, bytes, &full[s]);
  };

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) ptx::mbar_init(&full[s], 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  uint32_t next = 0;  // thread 0: the ticket the next refill takes
  if (tid == 0) {
    for (int s = 0; s < S; ++s) issue(s, atomicAdd(a.ticket, 1u) + 1u);
    next = atomicAdd(a.ticket, 1u) + 1u;
  }
  __syncthreads();

  int pending_from = -1;  // on failure: first iteration whose copies may be in flight
  for (int it = 0;; ++it) {
    const int s = it % S;
    const int p = st_p[s];
    if (p < 0) break;
    const int ts = st_t[s];
    const int tr = kRev ? a.T - 1 - ts : ts;
    const int64_t lo = (int64_t)tr * tile_rows;
    const int nrows = (int)min((int64_t)tile_rows, a.N - lo);
    const int64_t base = (int64_t)p * a.N;
    const int64_t tix = (int64_t)p * a.T + ts;  // this tile in the look-back arrays

    const bool got = ptx::mbar_wait(&full[s], (uint32_t)((it / S) & 1), &abort_flag);
    if (!got) lb_record_timeout(a.status, &abort_flag);
    if (__syncthreads_or(!got)) {
      pending_from = it;
      break;
    }
    // ---- this thread's rows, from the stage (scan order); rl = row - lo
    const uint8_t* st = lsm + (size_t)s * a.stage_bytes;
    R xs[RPT][K];
    R qs[kTwo ? RPT : 1][K];
    float gz[RPT];
    int rl[RPT];
    bool valid[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      rl[i] = kRev ? nrows - 1 - (sp0 + i) : sp0 + i;
      valid[i] = kRev ? rl[i] >= 0 : rl[i] < nrows;
      const int e0 = rl[i] * D;
#pragma unroll
      for (int kk = 0; kk < K; ++kk) {
        const bool ok = valid[i] && colv[kk];
        xs[i][kk] = ok ? IO::lds(st, e0 + col[kk]) : IO::zero();
        if constexpr (kTwo) qs[i][kk] = ok ? IO::lds(st + a.in_bytes, e0 + col[kk]) : IO::zero();
      }
      gz[i] = (MODE != kZ && valid[i]) ? __ldg(a.grad_z + base + lo + rl[i]) : 0.f;
    }

    // ---- levels 1 and 2: this thread's rows, then across the warp's row
    // groups (pairs of columns in packed fp32x2 arithmetic)
    float2 sum[K][V2];
#pragma unroll
    for (int kk = 0; kk < K; ++kk)
#pragma unroll
      for (int j = 0; j < V2; ++j) sum[kk][j] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float2 g2 = make_float2(gz[i], gz[i]);
#pragma unroll
      for (int kk = 0; kk < K; ++kk) {
        float2 f[V2];
        IO::unpack2(xs[i][kk], f);
        if constexpr (FEAT) {
          // phi of the padding would be 1: map real elements only
          if (valid[i] && colv[kk]) {
#pragma unroll
            for (int j = 0; j < V2; ++j) {
              float2 d_;
              elu1_pair(f[j], f[j], d_);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < V2; ++j)
          sum[kk][j] = MODE == kDK ? __ffma2_rn(g2, f[j], sum[kk][j]) : __fadd2_rn(sum[kk][j], f[j]);
      }
    }
#pragma unroll
    for (int step = 0; step < 5; ++step) {
      const int o = TPR << step;
      if (o < 32) {
#pragma unroll
        for (int kk = 0; kk < K; ++kk)
#pragma unroll
          for (int j = 0; j < V2; ++j) {
            const float yx = __shfl_up_sync(0xffffffffu, sum[kk][j].x, o);
            const float yy = __shfl_up_sync(0xffffffffu, sum[kk][j].y, o);
            if (lane >= o) sum[kk][j] = __fadd2_rn(sum[kk][j], make_float2(yx, yy));
          }
      }
    }
    float2 ex[K][V2];
#pragma unroll
    for (int kk = 0; kk < K; ++kk)
#pragma unroll
      for (int j = 0; j < V2; ++j) {
        const float yx = __shfl_up_sync(0xffffffffu, sum[kk][j].x, TPR);
        const float yy = __shfl_up_sync(0xffffffffu, sum[kk][j].y, TPR);
        ex[kk][j] = gw == 0 ? make_float2(0.f, 0.f) : make_float2(yx, yy);
      }
    if (gw == gpw - 1) {
#pragma unroll
      for (int kk = 0; kk < K; ++kk)
        if (colv[kk])
#pragma unroll
          for (int j = 0; j < V2; ++j)
            *reinterpret_cast<float2*>(wt + warp * D + col[kk] + 2 * j) = sum[kk][j];
    }
    // every thread has its rows (read with ordinary loads): order those reads
    // before the bulk copy that refills the stage (async proxy)
    ptx::fence_proxy_async_smem();
    __syncthreads();  // wt complete; every thread has its rows: refill the stage
    if (tid == 0) {
      issue(s, next);
      if (next < a.total) next = atomicAdd(a.ticket, 1u) + 1u;
    }
    // ---- publish the tile's column sum (read by the next W - 1 tiles), and
    // look back: partial sums of agg(s_lo .. ts-1) over contiguous runs of
    // tiles, each value polled until it has been published
    const int s_lo = max(0, ts - a.W + 1);
    const int n_agg = ts - s_lo;
    const int run = (n_agg + nparts - 1) / nparts;
    bool wok = true;
    uint64_t t0 = 0;
    for (int d = lb_d; d < D && lb_pt < nparts; d += kLbThreads) {
      if (lb_pt == 0) {
        float c = 0.f;
        for (int w = 0; w < kLbWarps; ++w) c += wt[w * D + d];
        tsum[d] = c;
        if (ts + 1 < a.T) __stcg(a.agg + tix * D + d, c);
      }
      const int a0 = s_lo + lb_pt * run, a1 = min(ts, a0 + run);
      float c;
#pragma unroll 1
      for (int tries = 0;; ++tries) {
        bool ready = true;
        c = 0.f;
#pragma unroll 4
        for (int s2 = a0; s2 < a1; ++s2) {
          const float v = __ldcg(a.agg + (tix - ts + s2) * D + d);
          ready &= !unset(v);
          c += v;
        }
        if (ready) break;
        if (tries == 0) t0 = ptx::globaltimer();
        if (poll_expired(t0, a.status)) {
          wok = false;
          break;
        }
        __nanosleep(64);
      }
      part[lb_pt * D + d] = c;
    }
    __syncthreads();  // part and tsum complete
    // ---- exclusive prefix = incl(ts-W) + the runs in order; publish the
    // inclusive prefix; carry into each warp in warp order
    for (int d = tid; d < D && wok; d += kLbThreads) {
      float e = 0.f;
      if (ts >= a.W) {
#pragma unroll 1
        for (int tries = 0;; ++tries) {
          e = __ldcg(a.incl + (tix - a.W) * D + d);
          if (!unset(e)) break;
          if (tries == 0) t0 = ptx::globaltimer();
          if (poll_expired(t0, a.status)) {
            wok = false;
            break;
          }
          __nanosleep(64);
        }
      }
      for (int pt = 0; pt < nparts; ++pt) e += part[pt * D + d];
      if (ts + a.W < a.T) __stcg(a.incl + tix * D + d, e + tsum[d]);
#pragma unroll
      for (int w = 0; w < kLbWarps; ++w) {
        cw[w * D + d] = e;
        e += wt[w * D + d];
      }
    }
    if (!wok) lb_record_timeout(a.status, &abort_flag);
    if (__syncthreads_or(!wok)) {
      pending_from = it + 1;
      break;
    }
    // ---- outputs
    float2 c[K][V2];
#pragma unroll
    for (int kk = 0; kk < K; ++kk)
#pragma unroll
      for (int j = 0; j < V2; ++j) {
        const float2 w2 = colv[kk] ? *reinterpret_cast<const float2*>(cw + warp * D + col[kk] + 2 * j)
                                   : make_float2(0.f, 0.f);
        c[kk][j] = __fadd2_rn(w2, ex[kk][j]);
      }
    const int64_t gb = (base + lo) * D;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      float2 zp = make_float2(0.f, 0.f);
      const float2 g2 = make_float2(gz[i], gz[i]);
#pragma unroll
      for (int kk = 0; kk < K; ++kk) {
        float2 f[V2];
        IO::unpack2(xs[i][kk], f);
        if constexpr (FEAT) {
          if (valid[i] && colv[kk]) {
#pragma unroll
            for (int j = 0; j < V2; ++j) {
              float2 d_;
              elu1_pair(f[j], f[j], d_);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < V2; ++j)
          c[kk][j] = MODE == kDK ? __ffma2_rn(g2, f[j], c[kk][j]) : __fadd2_rn(c[kk][j], f[j]);
        if constexpr (MODE == kZ) {
          float2 qf[V2];
          IO::unpack2(qs[i][kk], qf);
          if constexpr (FEAT) {
            if (valid[i] && colv[kk]) {
#pragma unroll
              for (int j = 0; j < V2; ++j) {
                float2 d_;
                elu1_pair(qf[j], qf[j], d_);
              }
            }
          }
#pragma unroll
          for (int j = 0; j < V2; ++j) zp = __ffma2_rn(qf[j], c[kk][j], zp);
        } else {
          float2 o[V2];
#pragma unroll
          for (int j = 0; j < V2; ++j) o[j] = MODE == kDQ ? __fmul2_rn(g2, c[kk][j]) : c[kk][j];
          if constexpr (FEAT) {
            // chain rule through phi of the output's own raw input
            float2 xo[V2];
            IO::unpack2(qs[i][kk], xo);
#pragma unroll
            for (int j = 0; j < V2; ++j) {
              float2 p_, d_;
              elu1_pair(xo[j], p_, d_);
              o[j] = __fmul2_rn(o[j], d_);
            }
          }
          if (valid[i] && colv[kk]) IO::store2(a.out, gb + rl[i] * D + col[kk], o);
        }
      }
      if constexpr (MODE == kZ) {
        float zs = zp.x + zp.y;
        for (int o = TPR >> 1; o >= 1; o >>= 1) zs += __shfl_xor_sync(0xffffffffu, zs, o);
        if (valid[i] && (i & (TPR - 1)) == cc) a.z[base + lo + rl[i]] = zs;
      }
    }
  }
  // after a failure, let the copies still in flight land before the CTA
  // exits (their stages are never read)
  if (pending_from >= 0 && tid == 0) {
    for (int j = pending_from; j < pending_from + S; ++j) {
      const int s = j % S;
      if (st_p[s] >= 0) ptx::mbar_wait_timeout(&full[s], (uint32_t)((j / S) & 1), 1000000000ull);
    }
  }
}

// How a row of D elements is spread over lanes, and the rows of a tile of
// a CTA with `warps` warps.
struct NormShape {
  int V, K, TPR, RPT, rows;
};

NormShape norm_shape(int64_t D, cp_dtype_t dtype, int warps, int rows_per_thread) {
  NormShape sh{};
  sh.V = dtype != CP_DTYPE_F32 ? 8 : (D % 4 == 0 ? 4 : 1);
  const int64_t per_row = (D + sh.V - 1) / sh.V;  // accesses per row
  int K = 1;
  while ((per_row + K - 1) / K > 32) K <<= 1;
  sh.K = K;
  const int64_t need = (per_row + K - 1) / K;
  int tpr = 1;
  while (tpr < need) tpr <<= 1;
  sh.TPR = tpr;
  sh.RPT = rows_per_thread / K;
  sh.rows = sh.RPT * warps * (32 / tpr);
  return sh;
}

bool single_pass(int64_t D, cp_dtype_t dtype) {
  return norm_shape(D, dtype, kLbWarps, kLbRowsPerThread).V > 1;
}

// ---- two-pass plan (scalar fp32 rows)
struct NormPlan {
  NormShape sh;
  int G;
  int64_t seg_rows;
  size_t agg_bytes;
};

NormPlan norm_plan(int64_t BH, int64_t N, int64_t D, cp_dtype_t dtype) {
  NormPlan pl{};
  pl.sh = norm_shape(D, dtype, kNormWarps, 8);
  const int64_t n_tiles = std::max<int64_t>(1, (N + pl.sh.rows - 1) / pl.sh.rows);
  // two resident CTAs per SM; every segment holds at least one tile
  int64_t G = std::max<int64_t>(1, (2 * kPlanSMs) / std::max<int64_t>(BH, 1));
  G = std::min<int64_t>(G, n_tiles);
  const int64_t tiles_per_seg = (n_tiles + G - 1) / G;
  pl.seg_rows = tiles_per_seg * pl.sh.rows;
  pl.G = (int)std::max<int64_t>(1, (N + pl.seg_rows - 1) / pl.seg_rows);
  pl.agg_bytes = pl.G > 1 ? sizeof(float) * (size_t)BH * pl.G * D : 0;
  return pl;
}

// ---- single-pass plan: the workspace holds the ticket counter, then the
// tiles' sums and inclusive prefixes; all of it is filled with ones before
// every launch
struct LbPlan {
  NormShape sh;
  int T, W;
  size_t bytes;
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

LbPlan lb_plan(int64_t BH, int64_t N, int64_t D, cp_dtype_t dtype) {
  LbPlan pl{};
  pl.sh = norm_shape(D, dtype, kLbWarps, kLbRowsPerThread);
  pl.T = (int)std::max<int64_t>(1, (N + pl.sh.rows - 1) / pl.sh.rows);
  // the inclusive prefixes form chains of T / W hops; W - 1 sums are read
  // per tile
  pl.W = (int)std::min<int64_t>(64, std::max<int64_t>(8, (pl.T + 3) / 4));
  const size_t tiles = (size_t)BH * pl.T;
  pl.bytes = 256 + up256(2 * tiles * D * sizeof(float));
  return pl;
}

template <typename T, int V, int K, int MODE>
cudaError_t norm_run(NormArgs a, int64_t BH, const NormPlan& pl, float* agg, cudaStream_t st) {
  a.G = pl.G;
  a.seg_rows = pl.seg_rows;
  a.tpr = pl.sh.TPR;
  if (pl.G > 1) {
    // first pass: the column sums of every segment some later segment needs
    NormArgs b = a;
    b.agg_only = 1;
    b.agg_out = agg;
    b.GL = pl.G - 1;
    b.seg_base = MODE == kDK ? 1 : 0;
    norm_kernel<T, V, K, MODE><<<(unsigned)(BH * b.GL), kNormThreads, 0, st>>>(b);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    a.agg_in = agg;
  }
  a.GL = pl.G;
  a.seg_base = 0;
  norm_kernel<T, V, K, MODE><<<(unsigned)(BH * pl.G), kNormThreads, 0, st>>>(a);
  return cudaGetLastError();
}

template <typename T, int V, int K>
cudaError_t norm_modes(int mode, const NormArgs& a, int64_t BH, const NormPlan& pl, float* agg,
                       cudaStream_t st) {
  if (mode == kZ) return norm_run<T, V, K, kZ>(a, BH, pl, agg, st);
  if (mode == kDQ) return norm_run<T, V, K, kDQ>(a, BH, pl, agg, st);
  return norm_run<T, V, K, kDK>(a, BH, pl, agg, st);
}

template <typename T, int V, int K, int MODE, bool FEAT>
cudaError_t lb_run(LbArgs a, const LbPlan& pl, uint8_t* ws, cudaStream_t st) {
  constexpr int kIn = (MODE == kZ || FEAT) ? 2 : 1;
  const uint32_t in_bytes =
      (uint32_t)((pl.sh.rows * (size_t)a.D * sizeof(T) + 127) / 128 * 128);
  const uint32_t stage = kIn * in_bytes;
  int S = (int)(kLbRingBytes / stage);
  S = std::max(1, std::min(kLbMaxStages, S));
  const size_t aux = sizeof(float) * ((2 * kLbWarps + 1) * (size_t)a.D +
                                      std::max<size_t>(kLbThreads, a.D));
  const size_t smem = (size_t)S * stage + aux;
  auto kern = norm_lb_kernel<T, V, K, MODE, FEAT>;
  // the dynamic shared-memory opt-in of this kernel on each device: raised
  // when a launch needs more than any before it
  static std::mutex mu;
  static int opted[kMaxDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (opted[dev] < (int)smem) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      opted[dev] = (int)smem;
    }
  }
  int n_sm = 0, per_sm = 0;
  if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kLbThreads, smem)) !=
      cudaSuccess)
    return e;
  a.tpr = pl.sh.TPR;
  a.T = pl.T;
  a.W = pl.W;
  a.n_stages = S;
  a.stage_bytes = stage;
  a.in_bytes = in_bytes;
  if ((int64_t)a.BH * pl.T >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  a.total = (uint32_t)((int64_t)a.BH * pl.T);
  a.ticket = reinterpret_cast<unsigned int*>(ws);
  a.agg = reinterpret_cast<float*>(ws + 256);
  a.incl = a.agg + a.total * a.D;
  // counter = all ones (the first atomic increment hands out ticket 0) and
  // every sum and prefix unpublished
  const size_t fill = 256 + (size_t)a.total * a.D * 2 * sizeof(float);
  if ((e = cudaMemsetAsync(ws, 0xff, fill, st)) != cudaSuccess) return e;
  const long long grid = std::min<long long>((long long)a.total, (long long)n_sm * std::max(per_sm, 1));
  kern<<<(unsigned)grid, kLbThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <typename T, int V, int K>
cudaError_t lb_modes(int mode, bool feat, const LbArgs& a, const LbPlan& pl, uint8_t* ws,
                     cudaStream_t st) {
  if (feat) {
    if (mode == kZ) return lb_run<T, V, K, kZ, true>(a, pl, ws, st);
    if (mode == kDQ) return lb_run<T, V, K, kDQ, true>(a, pl, ws, st);
    return lb_run<T, V, K, kDK, true>(a, pl, ws, st);
  }
  if (mode == kZ) return lb_run<T, V, K, kZ, false>(a, pl, ws, st);
  if (mode == kDQ) return lb_run<T, V, K, kDQ, false>(a, pl, ws, st);
  return lb_run<T, V, K, kDK, false>(a, pl, ws, st);
}

}  // namespace

size_t norm_scratch_bytes(int64_t BH, int64_t N, int64_t D, cp_dtype_t dtype) {
  if (N == 0) return 0;
  if (single_pass(D, dtype)) return lb_plan(BH, N, D, dtype).bytes;
  return norm_plan(BH, N, D, dtype).agg_bytes;
}

bool norm_feature_supported(int64_t D, cp_dtype_t dtype) { return single_pass(D, dtype); }

int norm_launch_count(int64_t BH, int64_t N, int64_t D, cp_dtype_t dtype) {
  if (N == 0) return 0;
  if (single_pass(D, dtype)) return 1;
  return norm_plan(BH, N, D, dtype).G > 1 ? 2 : 1;
}

cudaError_t norm_launch(int mode, const void* q, const void* k, const float* grad_z, float* z,
                        void* out, int64_t BH, int64_t N, int64_t D, cp_dtype_t dtype,
                        void* scratch, int* status, cudaStream_t stream, int feature) {
  const bool feat = feature != 0;
  if (norm_pp_eligible(mode, feature, BH, N, D) && (!feat || single_pass(D, dtype)))
    return norm_pp_launch(mode, q, k, grad_z, z, out, BH, N, dtype, status, stream, feature);
  if (single_pass(D, dtype)) {
    const LbPlan pl = lb_plan(BH, N, D, dtype);
    LbArgs a{};
    a.q = q;
    a.k = k;
    a.grad_z = grad_z;
    a.z = z;
    a.out = out;
    a.N = N;
    a.D = (int)D;
    a.BH = (int)BH;
    a.status = status;
    uint8_t* ws = static_cast<uint8_t*>(scratch);
    if (dtype == CP_DTYPE_BF16)
      return lb_modes<__nv_bfloat16, 8, 1>(mode, feat, a, pl, ws, stream);
    if (dtype == CP_DTYPE_F16) return lb_modes<__half, 8, 1>(mode, feat, a, pl, ws, stream);
    if (pl.sh.K == 1) return lb_modes<float, 4, 1>(mode, feat, a, pl, ws, stream);
    return lb_modes<float, 4, 2>(mode, feat, a, pl, ws, stream);
  }
  if (feat) return cudaErrorInvalidValue;  // the feature map needs 16-byte rows
  const NormPlan pl = norm_plan(BH, N, D, dtype);
  NormArgs a{};
  a.q = q;
  a.k = k;
  a.grad_z = grad_z;
  a.z = z;
  a.out = out;
  a.N = N;
  a.D = (int)D;
  float* agg = static_cast<float*>(scratch);
  switch (pl.sh.K) {
    case 1: return norm_modes<float, 1, 1>(mode, a, BH, pl, agg, stream);
    case 2: return norm_modes<float, 1, 2>(mode, a, BH, pl, agg, stream);
    case 4: return norm_modes<float, 1, 4>(mode, a, BH, pl, agg, stream);
    default: return norm_modes<float, 1, 8>(mode, a, BH, pl, agg, stream);
  }
}

}  // namespace cp
