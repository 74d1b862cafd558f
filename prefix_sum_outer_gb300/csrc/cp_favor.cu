// Positive random features ("FAVOR+", the Performer feature map the pages of
// triton-lang/triton issue #217 name when they offer the causal product as a
// drop-in for the Performers code) on the 5th-generation tensor cores:
//
//     phi(x)_d = exp(w_d . x - |x|^2 / 2) / sqrt(D),      d = 0 .. D-1,
//
// for rows x of r <= 64 input features and one projection W [D][r] shared by
// every row.  Two kernels:
//
//   favor_map_kernel    Y = phi(X): F = X W^T on tcgen05 (one M = 128,
//                       N = D chain per 128-row tile, fp32 in TMEM), then
//                       exp2(F log2 e - |x|^2 log2 e / 2 - log2 sqrt(D)) per
//                       element, rounded to bf16 and stored by TMA.
//                       Optionally also lo = bf16(phi - hi) beside hi = bf16(phi).
//   favor_chain_kernel  the chain rule of the map: with A = dL/dphi,
//                       dL/dx = sum_d A_d phi_d (w_d - x)
//                             = (A o phi) W - x rowsum(A o phi),
//                       the first term a tcgen05 product (K = D) of the
//                       elementwise product A o phi (bf16, formed in shared
//                       memory) with W.  A arrives in two parts (the
//                       gradients against phi's hi and lo parts), summed in
//                       fp32.
//
// Rows are [BH][N][.] bf16 tensors walked in 128-row tiles per problem (TMA
// zero-fills rows past N on load and clips them on store).  Every wait is
// bounded and records CP_ERR_TIMEOUT in the status word.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <utility>

#include "cp_internal.h"
#include "cp_tc_common.cuh"

namespace cp {
namespace tc {
namespace favor {

using namespace cp::ptx;

constexpr int kEpiWarps = 4;                  // one TMEM lane quarter each (warps 0..3)
constexpr int kProdWarp = 4, kMmaWarp = 5;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr float kLog2e = 1.4426950408889634f;

// W [D][r] in shared memory: 128-row boxes of 128 bytes per row (r <= 64
// bf16, zero-padded), the same bytes serve as the K-major B operand of
// X W^T (rows = features) and as the MN-major B operand of (A o phi) W
// (rows = the contraction index).
__host__ __device__ constexpr int w_bytes(int D) { return ((D + 127) / 128) * kBoxBytes; }

__device__ __forceinline__ float ex2_approx(float y) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
  return r;
}

// sum of squares of one 64-column bf16 row of a swizzled [128 x 64] box (the
// swizzle only permutes the row's 16-byte chunks, which a sum ignores)
__device__ __forceinline__ float row_sumsq(const uint8_t* box, int row) {
  const uint4* p = reinterpret_cast<const uint4*>(box + row * 128);
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 w = p[c];
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float a = __uint_as_float(u[x] << 16), b = __uint_as_float(u[x] & 0xffff0000u);
      s = fmaf(a, a, s);
      s = fmaf(b, b, s);
    }
  }
  return s;
}

struct TileWalk {
  int tiles_per_problem;
  int n_tiles;  // BH * tiles_per_problem
};

// ------------------------------------------------------------------ map
// LO: also write lo = bf16(phi - hi) next to hi = bf16(phi): rows of the
// output are [hi (D) | lo (D)] (the precision the gradients need, see
// favor_bwd in cp_api.cu); otherwise rows of D.
template <int D, bool LO>
struct MapLayout {
  static constexpr int kXStages = 3;
  static constexpr int kStgBoxes = 6;  // staging ring of [128 x 64] boxes, one TMA store each
  static constexpr int kSmem =
      w_bytes(D) + kXStages * kBoxBytes + kStgBoxes * kBoxBytes + 1024 + 1024;
  static constexpr int kTmemCols = 2 * D <= 128 ? 128 : (2 * D <= 256 ? 256 : 512);
  static_assert(D % 64 == 0 && D <= 256, "D: 64 .. 256 in steps of 64");
  static_assert(kSmem <= kSmemLimit, "shared memory overflow");
};

template <int D, bool LO>
__global__ void __launch_bounds__(kThreads, 1)
    favor_map_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_y, const TileWalk tw, int* status) {
  using L = MapLayout<D, LO>;
  constexpr int NX = L::kXStages, NSTG = L::kStgBoxes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* w_s = smem;
  uint8_t* x_ring = w_s + w_bytes(D);
  uint8_t* stg = x_ring + NX * kBoxBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg + NSTG * kBoxBytes);
  uint64_t* x_full = bars;            // [NX]
  uint64_t* x_empty = x_full + NX;    // [NX] epilogue read |x|^2 after the MMA
  uint64_t* w_full = x_empty + NX;
  uint64_t* mma_done = w_full + 1;    // [2]
  uint64_t* tmem_free = mma_done + 2; // [2]
  uint64_t* fin = tmem_free + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(fin + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(fin + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_my = tw.n_tiles > (int)blockIdx.x
                       ? (tw.n_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                       : 0;
  auto tile_of = [&](int i) { return (int)blockIdx.x + i * (int)gridDim.x; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < NX; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], 32 * kEpiWarps);
    }
    mbar_init(w_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&mma_done[i], 1);
      mbar_init(&tmem_free[i], kEpiWarps);
    }
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_holder, L::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == kProdWarp) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      mbar_arrive_expect_tx(w_full, w_bytes(D));
      for (int b = 0; b < w_bytes(D) / kBoxBytes; ++b)
        tma_load_3d(w_s + b * kBoxBytes, &tm_w, w_full, 0, b * kTile, 0, policy_evict_last());
      for (int i = 0; i < n_my; ++i) {
        const int s = i % NX;
        if (i >= NX && !mbar_wait(&x_empty[s], ((i / NX) - 1) & 1, abort_flag)) {
          record_timeout(status, abort_flag);
          break;
        }
        const int t = tile_of(i);
        mbar_arrive_expect_tx(&x_full[s], kBoxBytes);
        tma_load_3d(x_ring + s * kBoxBytes, &tm_x, &x_full[s], 0,
                    (t % tw.tiles_per_problem) * kTile, t / tw.tiles_per_problem, pol);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 0);  // X . W^T, both K-major
      constexpr uint32_t kHi = desc_hi(1024);
      bool ok = mbar_wait(w_full, 0, abort_flag);
      const uint32_t w_lo = desc_lo(smem_u32(w_s), 16);
      for (int i = 0; ok && i < n_my; ++i) {
        const int s = i % NX, b = i & 1;
        if (!mbar_wait(&x_full[s], (i / NX) & 1, abort_flag) ||
            (i >= 2 && !mbar_wait(&tmem_free[b], ((i / 2) - 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t x_lo = desc_lo(smem_u32(x_ring + s * kBoxBytes), 16);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss_lo<kHi, kHi>(tmem + b * D, x_lo + kk * 2, w_lo + kk * 2, idesc, kk > 0 ? 1u : 0u);
        mma_commit(&mma_done[b]);
      }
      if (!ok) record_timeout(status, abort_flag);
      mma_commit(fin);
      mbar_wait_timeout(fin, 0, CP_WAIT_TIMEOUT_NS);
    }
  } else {
    // epilogue: one tile row per thread (TMEM lane = row); each 64-column
    // box of phi goes through a staging ring slot and out by its own TMA
    // store (and so does its lo box)
    const int row = warp * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float log2_sqrt_d = 0.5f * log2f((float)D);
    bool ok = true;
    int slot = 0;  // staging boxes used so far
    // a free staging slot: the store that last read it (NSTG boxes ago) is
    // done reading
    auto next_slot = [&]() -> uint8_t* {
      if (threadIdx.x == 0)
        asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(NSTG - 1) : "memory");
      named_barrier_sync(1, 32 * kEpiWarps);
      return stg + (slot++ % NSTG) * kBoxBytes;
    };
    auto store_box = [&](const uint8_t* box, int col0, int t) {
      fence_proxy_async_smem();
      named_barrier_sync(1, 32 * kEpiWarps);
      if (threadIdx.x == 0) {
        tma_store_3d(&tm_y, box, col0, (t % tw.tiles_per_problem) * kTile,
                     t / tw.tiles_per_problem);
        tma_store_commit();
      }
    };
    for (int i = 0; i < n_my; ++i) {
      const int s = i % NX, b = i & 1, t = tile_of(i);
      // the TMA barrier of the X stage, not only the MMA's completion, makes
      // the landed tile visible to these threads' loads (the stage held
      // tile i - NX before)
      if (!mbar_wait(&x_full[s], (i / NX) & 1, abort_flag) ||
          !mbar_wait(&mma_done[b], (i / 2) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float cst = -0.5f * kLog2e * row_sumsq(x_ring + s * kBoxBytes, row) - log2_sqrt_d;
      release_to_tma(&x_empty[s], cst);
#pragma unroll 1
      for (int bx = 0; bx < D / 64; ++bx) {
        uint32_t r[2][32];
        tmem_ld32(lane_base + b * D + bx * 64, r[0]);
        tmem_ld32(lane_base + b * D + bx * 64 + 32, r[1]);
        tmem_ld_wait();
        if (bx == D / 64 - 1) {
          // every column of this tile is read out: the MMA may reuse the buffer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tmem_free[b]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int x = 0; x < 32; ++x)
            r[h][x] = __float_as_uint(ex2_approx(fmaf(__uint_as_float(r[h][x]), kLog2e, cst)));
        uint8_t* hb = next_slot();
        store_chunk32(hb, row, 0, kBoxBytes, r[0]);
        store_chunk32(hb, row, 32, kBoxBytes, r[1]);
        store_box(hb, bx * 64, t);
        if (LO) {
          // lo = bf16(phi - bf16(phi)), in place of phi
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int x = 0; x < 32; x += 2) {
              const float a = __uint_as_float(r[h][x]), c = __uint_as_float(r[h][x + 1]);
              const uint32_t hw = pack_bf16x2(a, c);
              r[h][x] = __float_as_uint(a - __uint_as_float(hw << 16));
              r[h][x + 1] = __float_as_uint(c - __uint_as_float(hw & 0xffff0000u));
            }
          uint8_t* lb = next_slot();
          store_chunk32(lb, row, 0, kBoxBytes, r[0]);
          store_chunk32(lb, row, 32, kBoxBytes, r[1]);
          store_box(lb, D + bx * 64, t);
        }
      }
    }
    if (!ok) record_timeout(status, abort_flag);
    if (threadIdx.x == 0) tma_store_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// ------------------------------------------------------------------ chain rule
// A K-chunk ring: stage = (A hi-half box, A lo-half box, phi box) of one
// tile, 64 features each.  A = dL/dphi arrives as [hi-part | lo-part]
// halves of 2D columns (gradients taken against phi's hi and lo parts);
// a = hi-part + lo-part in fp32.
template <int D>
struct ChainLayout {
  static constexpr int kStages = 3;
  static constexpr int kStageBytes = 3 * kBoxBytes;
  static constexpr int kChunks = D / 64;
  static constexpr int kSmem = w_bytes(D) + kStages * kStageBytes + 2 * kBoxBytes /* x */ +
                               kBoxBytes /* dx staging */ + 1024 + 1024;
  static_assert(kSmem <= kSmemLimit, "shared memory overflow");
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    favor_chain_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_p,
                       const __grid_constant__ CUtensorMap tm_dx, const TileWalk tw, int* status) {
  using L = ChainLayout<D>;
  constexpr int NS = L::kStages, NC = L::kChunks;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* w_s = smem;
  uint8_t* ring = w_s + w_bytes(D);
  uint8_t* x_s = ring + NS * L::kStageBytes;  // [2] x tiles
  uint8_t* o_s = x_s + 2 * kBoxBytes;         // dx staging
  uint64_t* bars = reinterpret_cast<uint64_t*>(o_s + kBoxBytes);
  uint64_t* c_full = bars;              // [NS] TMA -> elementwise
  uint64_t* c_ready = c_full + NS;      // [NS] elementwise -> MMA: A o phi in place
  uint64_t* c_empty = c_ready + NS;     // [NS] MMA -> TMA
  uint64_t* x_full = c_empty + NS;      // [2]
  uint64_t* x_empty = x_full + 2;       // [2] epilogue -> TMA
  uint64_t* acc_done = x_empty + 2;     // [2] MMA -> epilogue
  uint64_t* acc_free = acc_done + 2;    // [2] epilogue -> MMA
  uint64_t* w_full = acc_free + 2;
  uint64_t* fin = w_full + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(fin + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(fin + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_my = tw.n_tiles > (int)blockIdx.x
                       ? (tw.n_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                       : 0;
  auto tile_of = [&](int i) { return (int)blockIdx.x + i * (int)gridDim.x; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&c_full[i], 1);
      mbar_init(&c_ready[i], kEpiWarps);
      mbar_init(&c_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], 32 * kEpiWarps);
      mbar_init(&acc_done[i], 1);
      mbar_init(&acc_free[i], kEpiWarps);
    }
    mbar_init(w_full, 1);
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_holder, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == kProdWarp) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      mbar_arrive_expect_tx(w_full, w_bytes(D));
      for (int b = 0; b < w_bytes(D) / kBoxBytes; ++b)
        tma_load_3d(w_s + b * kBoxBytes, &tm_w, w_full, 0, b * kTile, 0, policy_evict_last());
      int n = 0;  // chunks issued
      bool ok = true;
      for (int i = 0; ok && i < n_my; ++i) {
        const int t = tile_of(i);
        const int row0 = (t % tw.tiles_per_problem) * kTile, bh = t / tw.tiles_per_problem;
        const int xb = i & 1;
        if (i >= 2 && !mbar_wait(&x_empty[xb], ((i / 2) - 1) & 1, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(&x_full[xb], kBoxBytes);
        tma_load_3d(x_s + xb * kBoxBytes, &tm_x, &x_full[xb], 0, row0, bh, pol);
        for (int c = 0; c < NC; ++c, ++n) {
          const int s = n % NS;
          if (n >= NS && !mbar_wait(&c_empty[s], ((n / NS) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* st = ring + s * L::kStageBytes;
          mbar_arrive_expect_tx(&c_full[s], L::kStageBytes);
          tma_load_3d(st, &tm_a, &c_full[s], c * 64, row0, bh, pol);
          tma_load_3d(st + kBoxBytes, &tm_a, &c_full[s], D + c * 64, row0, bh, pol);
          tma_load_3d(st + 2 * kBoxBytes, &tm_p, &c_full[s], c * 64, row0, bh, pol);
        }
      }
      if (!ok) record_timeout(status, abort_flag);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // C += (A o phi)_chunk W_chunk: A K-major (features along K), W MN-major
      constexpr uint32_t idesc = idesc_bf16_f32(128, 64, 0, 1);
      constexpr uint32_t kHi = desc_hi(1024);
      bool ok = mbar_wait(w_full, 0, abort_flag);
      const uint32_t w_lo = desc_lo(smem_u32(w_s), kBoxBytes);
      int n = 0;
      for (int i = 0; ok && i < n_my; ++i) {
        const int b = i & 1;
        if (i >= 2 && !mbar_wait(&acc_free[b], ((i / 2) - 1) & 1, abort_flag)) { ok = false; break; }
        for (int c = 0; c < NC; ++c, ++n) {
          const int s = n % NS;
          if (!mbar_wait(&c_ready[s], (n / NS) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_lo = desc_lo(smem_u32(ring + s * L::kStageBytes), 16);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss_lo<kHi, kHi>(tmem + b * 64, a_lo + kk * 2,
                                w_lo + ((c * 64 * 128 + kk * 2048) >> 4), idesc,
                                (c > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&c_empty[s]);
        }
        if (!ok) break;
        mma_commit(&acc_done[b]);
      }
      if (!ok) record_timeout(status, abort_flag);
      mma_commit(fin);
      mbar_wait_timeout(fin, 0, CP_WAIT_TIMEOUT_NS);
    }
  } else {
    // elementwise (a_hi + a_lo) o phi (in place of a_hi, bf16) and its row
    // sum, then the epilogue dx = C - x rowsum; one tile row per thread
    const int row = warp * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    bool ok = true;
    int n = 0;
    for (int i = 0; ok && i < n_my; ++i) {
      const int b = i & 1;
      float rs = 0.f;
      for (int c = 0; c < NC; ++c, ++n) {
        const int s = n % NS;
        if (!mbar_wait(&c_full[s], (n / NS) & 1, abort_flag)) { ok = false; break; }
        uint8_t* st = ring + s * L::kStageBytes + row * 128;
        uint4* pa = reinterpret_cast<uint4*>(st);
        const uint4* pl = reinterpret_cast<const uint4*>(st + kBoxBytes);
        const uint4* pp = reinterpret_cast<const uint4*>(st + 2 * kBoxBytes);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 wa = pa[q], wl = pl[q], wp = pp[q];
          const uint32_t ua[4] = {wa.x, wa.y, wa.z, wa.w}, ul[4] = {wl.x, wl.y, wl.z, wl.w};
          const uint32_t up[4] = {wp.x, wp.y, wp.z, wp.w};
          uint32_t o[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const float a0 = __uint_as_float(ua[x] << 16) + __uint_as_float(ul[x] << 16);
            const float a1 =
                __uint_as_float(ua[x] & 0xffff0000u) + __uint_as_float(ul[x] & 0xffff0000u);
            const float t0 = a0 * __uint_as_float(up[x] << 16);
            const float t1 = a1 * __uint_as_float(up[x] & 0xffff0000u);
            rs += t0 + t1;
            o[x] = pack_bf16x2(t0, t1);
          }
          pa[q] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c_ready[s]);
      }
      if (!ok) break;
      const int xb = i & 1;
      if (!mbar_wait(&x_full[xb], (i / 2) & 1, abort_flag) ||
          !mbar_wait(&acc_done[b], (i / 2) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t r[2][32];
      tmem_ld32(lane_base + b * 64, r[0]);
      tmem_ld32(lane_base + b * 64 + 32, r[1]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_free[b]);
      // x row (swizzled: logical 16-byte chunk j sits at chunk j ^ (row % 8))
      const uint8_t* xr = x_s + xb * kBoxBytes + row * 128;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 w = *reinterpret_cast<const uint4*>(xr + ((j ^ (row & 7)) << 4));
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          uint32_t& c0 = r[j >> 2][(j & 3) * 8 + 2 * x];
          uint32_t& c1 = r[j >> 2][(j & 3) * 8 + 2 * x + 1];
          c0 = __float_as_uint(fmaf(-rs, __uint_as_float(u[x] << 16), __uint_as_float(c0)));
          c1 = __float_as_uint(fmaf(-rs, __uint_as_float(u[x] & 0xffff0000u), __uint_as_float(c1)));
        }
      }
      release_to_tma(&x_empty[xb], __uint_as_float(r[0][0]) + __uint_as_float(r[1][31]));
      // the previous tile's store has read the staging box
      if (threadIdx.x == 0) tma_store_wait_read_all();
      named_barrier_sync(1, 32 * kEpiWarps);
      store_chunk32(o_s, row, 0, kBoxBytes, r[0]);
      store_chunk32(o_s, row, 32, kBoxBytes, r[1]);
      fence_proxy_async_smem();
      named_barrier_sync(1, 32 * kEpiWarps);
      if (threadIdx.x == 0) {
        const int t = tile_of(i);
        tma_store_3d(&tm_dx, o_s, 0, (t % tw.tiles_per_problem) * kTile, t / tw.tiles_per_problem);
        tma_store_commit();
      }
    }
    if (!ok) record_timeout(status, abort_flag);
    if (threadIdx.x == 0) tma_store_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// ------------------------------------------------------------------ host
template <typename... KArgs, typename... Act>
cudaError_t launch(void (*kern)(KArgs...), int smem, unsigned grid, cudaStream_t stream,
                   std::atomic<uint64_t>& configured, Act&&... args) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if ((configured.load(std::memory_order_acquire) & bit) == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Act>(args)...);
}

unsigned grid_for(int n_tiles) {
  int dev = 0, n_sm = kPlanSMs;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    n_sm = kPlanSMs;
  return (unsigned)std::max(1, std::min(n_tiles, n_sm));
}

}  // namespace favor
}  // namespace tc

bool favor_supported(int64_t R, int64_t D) {
  return R >= 8 && R <= 64 && R % 8 == 0 && D >= 64 && D <= 256 && D % 64 == 0;
}

cp_status_t favor_map_launch(const void* x, const void* W, void* y, int64_t BH, int64_t N,
                             int64_t R, int64_t D, bool lo, int* status, cudaStream_t stream) {
  using namespace tc;
  if (!favor_supported(R, D)) return CP_ERR_UNSUPPORTED_SHAPE;
  if (N == 0) return CP_OK;
  CUtensorMap maps[3];
  if (!make_map(&maps[0], x, BH, N, R) || !make_map(&maps[1], W, 1, D, R) ||
      !make_map(&maps[2], y, BH, N, lo ? 2 * D : D))
    return CP_ERR_UNSUPPORTED_SHAPE;
  favor::TileWalk tw;
  tw.tiles_per_problem = (int)((N + kTile - 1) / kTile);
  tw.n_tiles = (int)(BH * tw.tiles_per_problem);
  const unsigned grid = favor::grid_for(tw.n_tiles);
  cudaError_t e;
#define CP_FAVOR_MAP(DV, LOV)                                                                   \
  if (D == DV && lo == LOV) {                                                                  \
    static std::atomic<uint64_t> configured{0};                                                \
    e = favor::launch(favor::favor_map_kernel<DV, LOV>, favor::MapLayout<DV, LOV>::kSmem,      \
                      grid, stream, configured, maps[0], maps[1], maps[2], tw, status);         \
  } else
  CP_FAVOR_MAP(64, false) CP_FAVOR_MAP(128, false) CP_FAVOR_MAP(192, false)
  CP_FAVOR_MAP(256, false) CP_FAVOR_MAP(64, true) CP_FAVOR_MAP(128, true)
  CP_FAVOR_MAP(192, true) CP_FAVOR_MAP(256, true) return CP_ERR_UNSUPPORTED_SHAPE;
#undef CP_FAVOR_MAP
  return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

cp_status_t favor_chain_launch(const void* x, const void* W, const void* a, const void* phi,
                               int64_t phi_pitch, void* dx, int64_t BH, int64_t N, int64_t R,
                               int64_t D, int* status, cudaStream_t stream) {
  using namespace tc;
  if (!favor_supported(R, D)) return CP_ERR_UNSUPPORTED_SHAPE;
  if (N == 0) return CP_OK;
  CUtensorMap maps[5];
  if (!make_map(&maps[0], x, BH, N, R) || !make_map(&maps[1], W, 1, D, R) ||
      !make_map(&maps[2], a, BH, N, 2 * D) || !make_map(&maps[3], phi, BH, N, D, phi_pitch) ||
      !make_map(&maps[4], dx, BH, N, R))
    return CP_ERR_UNSUPPORTED_SHAPE;
  favor::TileWalk tw;
  tw.tiles_per_problem = (int)((N + kTile - 1) / kTile);
  tw.n_tiles = (int)(BH * tw.tiles_per_problem);
  const unsigned grid = favor::grid_for(tw.n_tiles);
  cudaError_t e;
#define CP_FAVOR_CHAIN(DV)                                                                       \
  if (D == DV) {                                                                                \
    static std::atomic<uint64_t> configured{0};                                                 \
    e = favor::launch(favor::favor_chain_kernel<DV>, favor::ChainLayout<DV>::kSmem, grid,       \
                      stream, configured, maps[0], maps[1], maps[2], maps[3], maps[4], tw,      \
                      status);                                                                  \
  } else
  CP_FAVOR_CHAIN(64) CP_FAVOR_CHAIN(128) CP_FAVOR_CHAIN(192) CP_FAVOR_CHAIN(256) return CP_ERR_UNSUPPORTED_SHAPE;
#undef CP_FAVOR_CHAIN
  return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

}  // namespace cp
