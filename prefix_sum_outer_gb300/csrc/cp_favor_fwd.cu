// The causal product of positive random features with the feature map fused
// into the product kernel: out_i = sum_{j<=i} (phi(xq_i) . phi(xk_j)) v_j,
// phi(x)_d = exp(w_d . x - |x|^2 / 2) / sqrt(D), computed from the raw rows
// xq, xk (R <= 64 input features) inside the CTA, so that phi(xq) and
// phi(xk) never exist in global memory.  (The pages of triton-lang/triton
// issue #217 discuss the causal product as a drop-in for the Performers
// code, whose feature map this is.)
//
// One CTA walks one (segment, problem, 64-column value block) in 128-row
// tiles, as the plain product kernel does (the same tile algebra: with S the
// fp32 D x 64 state before tile t,
//     P = phi(Q) phi(K)^T masked to j <= i,  O = phi(Q) S + P V,  S += phi(K)^T V),
// but the features of a tile are produced and consumed 128 at a time (a
// "pair" of 64-column boxes): for pair p the CTA computes
//     F = X W_p^T on the tensor cores (fp32 in TMEM, 64 columns per chunk),
//     phi = exp2(F log2 e - |x|^2 log2 e / 2 - log2 sqrt(D)), rounded to bf16
// into a shared-memory pair stage, and the MMAs of the pair (P partial sum,
// the pair's rows of phi(Q) S, the pair's 128-row block of S) read it before
// the next pair overwrites it.  A whole [128 x 256] feature tile of q and k
// (128 KB) would not fit beside the state copy and the rings.
//
// CTA = 16 warps:
//   warp 0        TMA producer: W once, the X tile pair (xq | xk), V ring
//   warp 1        TMEM allocator; MMA issuer A: per pair, P, phi(Q) S and S
//   warps 2..5    state group: bf16 hi/lo copy of S per tile, read-out of O
//                 (TMA store), the segment aggregates of the first pass
//   warps 6..9    P group: mask P, split into bf16 hi + lo, pack in TMEM
//   warps 10..13  mapping group: |x|^2, F -> phi into the pair stage
//   warp 14       MMA issuer F: the F chunks, as far ahead as TMEM allows
//   warp 15       MMA issuer C: P V, once P is packed
// The aggregate pass (phi(K) and S only) double-buffers the pair stage.
// Every wait is bounded and records CP_ERR_TIMEOUT in the status word.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <utility>

#include "cp_internal.h"
#include "cp_tc_common.cuh"

namespace cp {
namespace tc {
namespace ffwd {

using namespace cp::ptx;

constexpr int kMB = 64;                       // value columns per CTA
constexpr int kSWarp0 = 2, kPWarp0 = 6, kMWarp0 = 10, kFWarp = 14, kCWarp = 15;
constexpr int kThreads = 32 * 16;
constexpr int kFSlots = 3;                    // F chunks in TMEM (64 columns each)
constexpr float kLog2e = 1.4426950408889634f;
// TMEM columns
constexpr int kColS = 0;    // state: D/128 blocks of 64 columns
constexpr int kColP = 128;  // P (128 columns; later packed bf16 hi|lo)
constexpr int kColO = 256;  // output accumulator (64 columns)
constexpr int kColF = 320;  // kFSlots F chunks
constexpr int kColsAlloc = 512;
static_assert(kColF + kFSlots * 64 <= kColsAlloc, "TMEM");

struct FArgs {
  int64_t N;
  int n_tiles, seg_tiles, G, BH, n_mb, M;
  const float* agg_in;  // [P][G][D][64] segment starting states (prefixed), or null
  float* agg_out;       // aggregate pass: [P][G][D][64]
  int* status;
};

template <int D, bool AGG>
struct FLayout {
  static constexpr int NPAIR = D / 128;
  static constexpr int kWBytes = D * 128;                    // W [D][64] bf16
  static constexpr int kXBytes = (AGG ? 1 : 2) * kBoxBytes;  // xk (| xq)
  static constexpr int kKOff = AGG ? 0 : 2 * kBoxBytes;      // phi(K) pair within the stage
  static constexpr int kPhiBytes = (AGG ? 2 : 4) * kBoxBytes;  // one pair stage
  static constexpr int NPHI = AGG ? 2 : 1;                      // pair stages
  static constexpr int kSOneBytes = D * 128;                 // D x 64 bf16
  static constexpr int kSBytes = AGG ? 0 : 2 * kSOneBytes;   // hi | lo
  static constexpr int kOBytes = AGG ? 0 : kBoxBytes;
  static constexpr int kFixed = kWBytes + kXBytes + NPHI * kPhiBytes + kSBytes + kOBytes;
  static constexpr int kAvail = kSmemLimit - 2048;
  static constexpr int NV = std::min(3, (kAvail - kFixed) / kBoxBytes);
  static constexpr int kSmemBytes = kFixed + NV * kBoxBytes + 2048;
  static_assert(D == 128 || D == 256, "pairs of 64-column boxes");
  static_assert(NV >= 1 && kSmemBytes <= kSmemLimit, "shared memory");
};

__device__ __forceinline__ float ex2_approx(float y) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
  return r;
}

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

template <int D, bool AGG>
__global__ void __launch_bounds__(kThreads, 1)
    favor_causal_kernel(const __grid_constant__ CUtensorMap tm_xq,
                        const __grid_constant__ CUtensorMap tm_xk,
                        const __grid_constant__ CUtensorMap tm_w,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_o, const FArgs a) {
  using L = FLayout<D, AGG>;
  constexpr int NPAIR = L::NPAIR, NV = L::NV, NPHI = L::NPHI;
  constexpr int kChunks = AGG ? 2 : 4;  // F chunks per pair: (q0, q1,) k0, k1
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* w_s = smem;
  uint8_t* x_s = w_s + L::kWBytes;        // [xq box |] xk box (xk last)
  uint8_t* phi_s = x_s + L::kXBytes;      // [phi(Q) pair (2 boxes) |] phi(K) pair
  uint8_t* s_tile = phi_s + NPHI * L::kPhiBytes; // hi | lo state copy
  uint8_t* o_tile = s_tile + L::kSBytes;
  uint8_t* v_ring = o_tile + L::kOBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(v_ring + NV * kBoxBytes);
  uint64_t* w_full = bars;
  uint64_t* x_full = w_full + 1;
  uint64_t* x_empty = x_full + 1;      // mapping threads (|x|^2 read) + issuer (F MMAs done)
  uint64_t* v_full = x_empty + 1;      // [NV]
  uint64_t* v_empty = v_full + NV;     // [NV]
  uint64_t* f_full = v_empty + NV;     // [kFSlots] issuer -> mapping
  uint64_t* f_free = f_full + kFSlots; // [kFSlots] mapping -> issuer
  uint64_t* pair_mapped = f_free + kFSlots;  // [NPHI] mapping -> issuer A
  uint64_t* pair_done = pair_mapped + NPHI;  // [NPHI] issuer A -> mapping: stage read
  uint64_t* p_done = pair_done + NPHI;       // issuer A -> P group
  uint64_t* p_ready = p_done + 1;            // P group -> issuer
  uint64_t* s_done = p_ready + 1;            // issuer -> state group: S updated
  uint64_t* s_ready = s_done + 1;            // state group -> issuer: copy written
  uint64_t* o_done = s_ready + 1;            // issuer -> state group: O final
  uint64_t* o_free = o_done + 1;             // state group -> issuer: O read out
  uint64_t* pv_done = o_free + 1;            // issuer -> issuer: P buffer free
  uint64_t* fin = pv_done + 1;               // [3] issuers A, F, C drain
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(fin + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(fin + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- block -> (segment, problem, value block)
  int idx = (int)blockIdx.x;
  const int mb = idx % a.n_mb;
  idx /= a.n_mb;
  const int bh = idx % a.BH;
  const int seg = idx / a.BH;  // the aggregate pass runs segments 0 .. G-2
  const int t_first = seg * a.seg_tiles;
  const int n_it = min(a.n_tiles, t_first + a.seg_tiles) - t_first;
  const int pidx = bh * a.n_mb + mb;
  const bool has_prefix = !AGG && a.agg_in != nullptr && seg > 0;

  if (threadIdx.x == 0) {
    mbar_init(w_full, 1);
    mbar_init(x_full, 1);
    mbar_init(x_empty, 32 * 4 + 1);
    for (int i = 0; i < NV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < kFSlots; ++i) {
      mbar_init(&f_full[i], 1);
      mbar_init(&f_free[i], 4);
    }
    for (int i = 0; i < NPHI; ++i) {
      mbar_init(&pair_mapped[i], 4);
      mbar_init(&pair_done[i], 1);
    }
    mbar_init(p_done, 1);
    mbar_init(p_ready, 4);
    mbar_init(s_done, 1);
    mbar_init(s_ready, 4);
    mbar_init(o_done, 1);
    mbar_init(o_free, 4);
    mbar_init(pv_done, 1);
    for (int i = 0; i < 3; ++i) mbar_init(&fin[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_xk);
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_v);
    if (!AGG) {
      tma_prefetch_desc(&tm_xq);
      tma_prefetch_desc(&tm_o);
    }
  }
  if (warp == 1) tmem_alloc(tmem_holder, kColsAlloc);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_wait();
  const uint32_t tmem = *tmem_holder;
  const int wq = warp & 3;
  const int row = wq * 32 + lane;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      mbar_arrive_expect_tx(w_full, L::kWBytes);
      for (int b = 0; b < D / 128; ++b)
        tma_load_3d(w_s + b * kBoxBytes, &tm_w, w_full, 0, b * kTile, 0, policy_evict_last());
      int nx = 0, nv = 0;
      uint64_t t0 = globaltimer();
      uint32_t idle = 0;
      while (nx < n_it || nv < n_it) {
        bool progressed = false;
        if (nx < n_it && (nx == 0 || mbar_test_wait(x_empty, (nx - 1) & 1))) {
          const int row0 = (t_first + nx) * kTile;
          mbar_arrive_expect_tx(x_full, L::kXBytes);
          if (!AGG) tma_load_3d(x_s, &tm_xq, x_full, 0, row0, bh, pol);
          tma_load_3d(x_s + L::kXBytes - kBoxBytes, &tm_xk, x_full, 0, row0, bh, pol);
          ++nx;
          progressed = true;
        }
        if (nv < nx && (nv < NV || mbar_test_wait(&v_empty[nv % NV], ((nv / NV) - 1) & 1))) {
          const int st = nv % NV;
          mbar_arrive_expect_tx(&v_full[st], kBoxBytes);
          tma_load_3d(v_ring + st * kBoxBytes, &tm_v, &v_full[st], mb * kMB,
                      (t_first + nv) * kTile, bh, pol);
          ++nv;
          progressed = true;
        }
        if (progressed) {
          idle = 0;
        } else if ((++idle & 63u) == 0) {
          if (idle == 64) t0 = globaltimer();
          if (*abort_flag || globaltimer() - t0 > CP_WAIT_TIMEOUT_NS) {
            record_timeout(a.status, abort_flag);
            break;
          }
        }
      }
      if (*abort_flag) {
        // let the copies already issued land before the CTA's memory goes away
        if (nx > 0) mbar_wait_timeout(x_full, (nx - 1) & 1, CP_WAIT_TIMEOUT_NS);
        for (int j = max(0, nv - NV); j < nv; ++j)
          mbar_wait_timeout(&v_full[j % NV], (j / NV) & 1, CP_WAIT_TIMEOUT_NS);
        mbar_wait_timeout(w_full, 0, CP_WAIT_TIMEOUT_NS);
      }
    }
  } else if (warp == kFWarp) {
    // ------------------------------------------------------------ MMA issuer F
    // F = X W_b^T per 64-column chunk b, into the next free F slot
    if (lane == 0) {
      constexpr uint32_t kHi = desc_hi(1024);
      constexpr uint32_t idesc_f = idesc_bf16_f32(128, 64, 0, 0);  // X . W_b^T
      const uint32_t w_lo = desc_lo(smem_u32(w_s), 16);
      bool ok = mbar_wait(w_full, 0, abort_flag);
      int gc = 0;  // F chunks issued
      for (int it = 0; ok && it < n_it; ++it) {
        if (!mbar_wait(x_full, it & 1, abort_flag)) { ok = false; break; }
        for (int pp = 0; ok && pp < NPAIR; ++pp) {
          for (int c = 0; c < kChunks; ++c, ++gc) {
            const int slot = gc % kFSlots;
            if (gc >= kFSlots &&
                !mbar_wait(&f_free[slot], ((gc / kFSlots) - 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const bool is_q = !AGG && c < 2;
            const uint32_t x_lo =
                desc_lo(smem_u32(is_q ? x_s : x_s + L::kXBytes - kBoxBytes), 16);
            const int wb = 2 * pp + (c & 1);  // W rows 64 wb .. 64 wb + 63
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss_lo<kHi, kHi>(tmem + kColF + slot * 64, x_lo + kk * 2,
                                  w_lo + ((wb * 64 * 128) >> 4) + kk * 2, idesc_f,
                                  kk > 0 ? 1u : 0u);
            mma_commit(&f_full[slot]);
          }
        }
        if (ok) mma_commit(x_empty);  // the tile's X is read by the MMAs
      }
      if (!ok) record_timeout(a.status, abort_flag);
      mma_commit(fin + 1);
      mbar_wait_timeout(fin + 1, 0, CP_WAIT_TIMEOUT_NS);
    }
  } else if (warp == kCWarp) {
    // ------------------------------------------------------------ MMA issuer C
    // O += P_hi V + P_lo V once P is packed (after phi(Q) S: p_done follows
    // every MMA of issuer A for the tile)
    if (lane == 0 && !AGG) {
      constexpr uint32_t kHi = desc_hi(1024);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, kMB, 0, 1);
      bool ok = true;
      for (int it = 0; it < n_it; ++it) {
        const int vs = it % NV;
        if (!mbar_wait(p_ready, it & 1, abort_flag) ||
            !mbar_wait(&v_full[vs], (it / NV) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t v_lo = desc_lo(smem_u32(v_ring + vs * kBoxBytes), kBoxBytes);
#pragma unroll
        for (int part = 0; part < kPParts; ++part) {
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t acol = (kk >> 1) * 32 + part * 16 + (kk & 1) * 8;
            mma_ts_lo<kHi>(tmem + kColO, tmem + kColP + acol, v_lo + ((kk * 2048) >> 4), idesc_o,
                           1u);
          }
        }
        mma_commit(o_done);
        mma_commit(pv_done);
        mma_commit(&v_empty[vs]);
      }
      if (!ok) record_timeout(a.status, abort_flag);
      mma_commit(fin + 2);
      mbar_wait_timeout(fin + 2, 0, CP_WAIT_TIMEOUT_NS);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer A
    if (lane == 0) {
      constexpr uint32_t kHi = desc_hi(1024);
      constexpr uint32_t idesc_p = idesc_bf16_f32(128, 128, 0, 0);   // phi(Q) phi(K)^T
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kMB, 1, 1);   // phi(K)^T V
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, kMB, 0, 1);   // phi(Q) S
      const uint32_t s_lo = desc_lo(smem_u32(s_tile), D * 128);
      bool ok = true;
      for (int it = 0; ok && it < n_it; ++it) {
        const bool fresh_state = it == 0 && !has_prefix;
        const int vs = it % NV;
        const uint32_t v_lo = desc_lo(smem_u32(v_ring + vs * kBoxBytes), kBoxBytes);
        for (int pp = 0; ok && pp < NPAIR; ++pp) {
          const int gp = it * NPAIR + pp;  // pairs so far
          const int st = gp % NPHI;
          uint8_t* stage = phi_s + st * L::kPhiBytes;
          const uint32_t phq_lo = desc_lo(smem_u32(stage), 16);                     // K-major
          const uint32_t phk_lo = desc_lo(smem_u32(stage + L::kKOff), 16);          // K-major
          const uint32_t phk_mn = desc_lo(smem_u32(stage + L::kKOff), kBoxBytes);   // MN-major
          if (!mbar_wait(&pair_mapped[st], (gp / NPHI) & 1, abort_flag)) { ok = false; break; }
          if (pp == 0) {
            if (!mbar_wait(&v_full[vs], (it / NV) & 1, abort_flag)) { ok = false; break; }
            if (!AGG) {
              // the P buffer (P V of the previous tile), the output buffer
              // (read out) and the state copy of this tile
              if ((it > 0 && !mbar_wait(pv_done, (it - 1) & 1, abort_flag)) ||
                  (it > 0 && !mbar_wait(o_free, (it - 1) & 1, abort_flag)) ||
                  !mbar_wait(s_ready, it & 1, abort_flag)) {
                ok = false;
                break;
              }
            }
          }
          tc_fence_after();
          if (!AGG) {
            // P += phi(Q)_pair phi(K)_pair^T (K = 128 features of the pair)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
              mma_ss_lo<kHi, kHi>(tmem + kColP, phq_lo + off, phk_lo + off, idesc_p,
                                  (pp > 0 || kk > 0) ? 1u : 0u);
            }
            // O (+)= phi(Q)_pair S[pair rows] (hi, then lo)
#pragma unroll
            for (int part = 0; part < 2; ++part) {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
                mma_ss_lo<kHi, kHi>(
                    tmem + kColO, phq_lo + off,
                    s_lo + ((part * L::kSOneBytes + (pp * 8 + kk) * 2048) >> 4), idesc_o,
                    (pp > 0 || part > 0 || kk > 0) ? 1u : 0u);
              }
            }
          }
          // S[pair rows] += phi(K)_pair^T V (A MN-major: 128 features, K = rows)
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ss_lo<kHi, kHi>(tmem + kColS + pp * kMB, phk_mn + ((kk * 2048) >> 4),
                                v_lo + ((kk * 2048) >> 4), idesc_s,
                                (fresh_state && kk == 0) ? 0u : 1u);
          mma_commit(&pair_done[st]);  // the pair stage may be overwritten
        }
        if (!ok) break;
        if (AGG) {
          mma_commit(&v_empty[vs]);
          continue;
        }
        mma_commit(s_done);
        mma_commit(p_done);
      }
      // the aggregate pass hands its state on once, after the last tile
      if (AGG && ok) mma_commit(s_done);
      if (!ok) record_timeout(a.status, abort_flag);
      mma_commit(fin);
      mbar_wait_timeout(fin, 0, CP_WAIT_TIMEOUT_NS);
    }
  } else if (warp >= kMWarp0) {
    // ------------------------------------------------------------ mapping group
    const float log2_sqrt_d = 0.5f * log2f((float)D);
    bool ok = true;
    int gc = 0;
    for (int it = 0; ok && it < n_it; ++it) {
      if (!mbar_wait(x_full, it & 1, abort_flag)) { ok = false; break; }
      const float ck = -0.5f * kLog2e * row_sumsq(x_s + L::kXBytes - kBoxBytes, row) - log2_sqrt_d;
      const float cq =
          AGG ? 0.f : -0.5f * kLog2e * row_sumsq(x_s, row) - log2_sqrt_d;
      // the X tile goes back to the TMA engine once the F MMAs are done too
      asm volatile("" ::"f"(ck), "f"(cq));
      fence_proxy_async_smem();
      mbar_arrive(x_empty);
      for (int pp = 0; ok && pp < NPAIR; ++pp) {
        const int gp = it * NPAIR + pp;
        const int st = gp % NPHI;
        uint8_t* stage = phi_s + st * L::kPhiBytes;
        // the MMAs of the pair that last used this stage have read it
        if (gp >= NPHI && !mbar_wait(&pair_done[st], ((gp / NPHI) - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        for (int c = 0; c < kChunks; ++c, ++gc) {
          const int slot = gc % kFSlots;
          if (!mbar_wait(&f_full[slot], (gc / kFSlots) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          uint32_t r[2][32];
          tmem_ld32(lane_base + kColF + slot * 64, r[0]);
          tmem_ld32(lane_base + kColF + slot * 64 + 32, r[1]);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&f_free[slot]);
          const bool is_q = !AGG && c < 2;
          const float cst = is_q ? cq : ck;
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int x = 0; x < 32; ++x)
              r[h][x] = __float_as_uint(ex2_approx(fmaf(__uint_as_float(r[h][x]), kLog2e, cst)));
          uint8_t* box = stage + (is_q ? 0 : L::kKOff) + (c & 1) * kBoxBytes;
          store_chunk32(box, row, 0, kBoxBytes, r[0]);
          store_chunk32(box, row, 32, kBoxBytes, r[1]);
        }
        if (!ok) break;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pair_mapped[st]);
      }
    }
    if (!ok) record_timeout(a.status, abort_flag);
  } else if (warp >= kPWarp0) {
    // ------------------------------------------------------------ P group
    bool ok = true;
    for (int it = 0; !AGG && it < n_it; ++it) {
      if (!mbar_wait(p_done, it & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t pc = lane_base + kColP;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const bool z = c > wq;  // chunk entirely above the diagonal
        uint32_t r[32];
        if (!z) {
          tmem_ld32(pc + 32 * c, r);
          tmem_ld_wait();
        }
        split_pack_p(r, z, c == wq, lane, 0);
        store_packed_p(pc + 32 * c, r);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_ready);
    }
    if (!ok) record_timeout(a.status, abort_flag);
  } else if (warp >= kSWarp0) {
    // ------------------------------------------------------------ state group
    bool ok = true;
    if (AGG) {
      if (n_it > 0 && mbar_wait(s_done, 0, abort_flag)) {
        tc_fence_after();
        float* dst = a.agg_out + ((size_t)pidx * a.G + seg) * (size_t)D * kMB;
#pragma unroll 1
        for (int sb = 0; sb < D / 128; ++sb) {
          const int d = sb * 128 + row;
#pragma unroll
          for (int c = 0; c < kMB / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(lane_base + kColS + sb * kMB + c * 32, r);
            tmem_ld_wait();
            float4* o4 = reinterpret_cast<float4*>(dst + (size_t)d * kMB + c * 32);
#pragma unroll
            for (int x = 0; x < 8; ++x)
              o4[x] = make_float4(__uint_as_float(r[4 * x]), __uint_as_float(r[4 * x + 1]),
                                  __uint_as_float(r[4 * x + 2]), __uint_as_float(r[4 * x + 3]));
          }
        }
      } else if (n_it > 0) {
        ok = false;
      }
    } else {
      const int s_tid = threadIdx.x - 32 * kSWarp0;
      // initial state: the prefix of the earlier segments
      if (has_prefix) {
#pragma unroll 1
        for (int sb = 0; sb < D / 128; ++sb) {
          const int d = sb * 128 + row;
#pragma unroll
          for (int c = 0; c < kMB / 32; ++c) {
            const float4* src = reinterpret_cast<const float4*>(
                a.agg_in + (((size_t)pidx * a.G + seg) * D + d) * kMB + c * 32);
            uint32_t r[32];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
              const float4 f = __ldg(src + x);
              r[4 * x] = __float_as_uint(f.x);
              r[4 * x + 1] = __float_as_uint(f.y);
              r[4 * x + 2] = __float_as_uint(f.z);
              r[4 * x + 3] = __float_as_uint(f.w);
            }
            tmem_st32(lane_base + kColS + sb * kMB + c * 32, r);
          }
        }
        tmem_st_wait();
      }
      // two sequences, whichever is ready: the state copy before tile ns, the
      // read-out of tile no
      int ns = 0, no = 0;
      uint64_t t0 = globaltimer();
      uint32_t idle = 0;
      while (ns < n_it || no < n_it) {
        bool progressed = false;
        bool ready = false;
        if (ns < n_it && lane == 0) ready = ns == 0 || mbar_test_wait(s_done, (ns - 1) & 1);
        if (__shfl_sync(0xffffffffu, ready, 0)) {
          tc_fence_after();
#pragma unroll 1
          for (int sb = 0; sb < D / 128; ++sb) {
            const int d = sb * 128 + row;
#pragma unroll 1
            for (int c = 0; c < kMB / 32; ++c) {
              if (ns == 0 && !has_prefix) {
                store_zero32(s_tile, d, c * 32, D * 128);
                store_zero32(s_tile + L::kSOneBytes, d, c * 32, D * 128);
              } else {
                uint32_t r[32];
                tmem_ld32(lane_base + kColS + sb * kMB + c * 32, r);
                tmem_ld_wait();
                store_chunk32_split(s_tile, s_tile + L::kSOneBytes, d, c * 32, D * 128, r);
              }
            }
          }
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_ready);
          ++ns;
          progressed = true;
        }
        ready = false;
        if (no < ns && lane == 0) ready = mbar_test_wait(o_done, no & 1);
        if (__shfl_sync(0xffffffffu, ready, 0)) {
          tc_fence_after();
          uint32_t r[2][32];
          tmem_ld32(lane_base + kColO, r[0]);
          tmem_ld32(lane_base + kColO + 32, r[1]);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_free);
          // the previous tile's store has finished reading the staging box
          if (s_tid == 0) tma_store_wait_read_all();
          named_barrier_sync(1, 128);
          store_chunk32(o_tile, row, 0, kBoxBytes, r[0]);
          store_chunk32(o_tile, row, 32, kBoxBytes, r[1]);
          fence_proxy_async_smem();
          named_barrier_sync(1, 128);
          if (s_tid == 0) {
            tma_store_3d(&tm_o, o_tile, mb * kMB, (t_first + no) * kTile, bh);
            tma_store_commit();
          }
          ++no;
          progressed = true;
        }
        if (progressed) {
          idle = 0;
        } else if ((++idle & 63u) == 0) {
          if (idle == 64) t0 = globaltimer();
          if (*abort_flag || globaltimer() - t0 > CP_WAIT_TIMEOUT_NS) {
            ok = false;
            break;
          }
        }
      }
      if (s_tid == 0) tma_store_wait_all();
    }
    if (!ok) record_timeout(a.status, abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  grid_dep_launch_dependents();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kColsAlloc);
  }
}

template <int D, bool AGG>
cudaError_t launch(const CUtensorMap* maps, const FArgs& fa, unsigned grid, cudaStream_t st) {
  using L = FLayout<D, AGG>;
  auto kern = favor_causal_kernel<D, AGG>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if ((configured.load(std::memory_order_acquire) & bit) == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], fa);
}

}  // namespace ffwd
}  // namespace tc

bool favor_fused_supported(int64_t R, int64_t D) {
  return favor_supported(R, D) && (D == 128 || D == 256);
}

FavorPlan favor_fused_plan(int64_t BH, int64_t N, int64_t D, int64_t M) {
  FavorPlan p{};
  p.n_mb = (int)((M + 63) / 64);
  p.n_tiles = (int)((N + tc::kTile - 1) / tc::kTile);
  const int64_t problems = BH * p.n_mb;
  int64_t G = 1;
  if (problems * 4 < (int64_t)kPlanSMs * 3) G = std::max<int64_t>(1, kPlanSMs / problems);
  G = std::min<int64_t>(G, std::max(1, p.n_tiles));
  p.seg_tiles = (int)((p.n_tiles + G - 1) / G);
  p.G = p.seg_tiles > 0 ? (p.n_tiles + p.seg_tiles - 1) / p.seg_tiles : 1;
  if (p.G < 1) p.G = 1;
  p.agg_bytes = p.G > 1 ? sizeof(float) * (size_t)problems * p.G * D * 64 : 0;
  return p;
}

cp_status_t favor_fused_fwd_launch(const void* xq, const void* xk, const void* v, const void* W,
                                   void* out, int64_t BH, int64_t N, int64_t R, int64_t D,
                                   int64_t M, float* agg, int* status, cudaStream_t stream) {
  using namespace tc;
  if (!favor_fused_supported(R, D)) return CP_ERR_UNSUPPORTED_SHAPE;
  if (N == 0) return CP_OK;
  CUtensorMap maps[5];
  if (!make_map(&maps[0], xq, BH, N, R) || !make_map(&maps[1], xk, BH, N, R) ||
      !make_map(&maps[2], W, 1, D, R) || !make_map(&maps[3], v, BH, N, M) ||
      !make_map(&maps[4], out, BH, N, M))
    return CP_ERR_UNSUPPORTED_SHAPE;
  const FavorPlan plan = favor_fused_plan(BH, N, D, M);
  ffwd::FArgs fa{};
  fa.N = N;
  fa.n_tiles = plan.n_tiles;
  fa.seg_tiles = plan.seg_tiles;
  fa.G = plan.G;
  fa.BH = (int)BH;
  fa.n_mb = plan.n_mb;
  fa.M = (int)M;
  fa.status = status;
  const int64_t problems = BH * plan.n_mb;
  cudaError_t e = cudaSuccess;
  if (plan.G > 1) {
    ffwd::FArgs fb = fa;
    fb.agg_out = agg;
    const unsigned g1 = (unsigned)(problems * (plan.G - 1));
    e = D == 128 ? ffwd::launch<128, true>(maps, fb, g1, stream)
                 : ffwd::launch<256, true>(maps, fb, g1, stream);
    if (e == cudaSuccess) e = seg_prefix_launch(agg, problems, plan.G, D * 64, false, stream);
    if (e != cudaSuccess) return CP_ERR_CUDA;
    fa.agg_in = agg;
  }
  const unsigned g2 = (unsigned)(problems * plan.G);
  e = D == 128 ? ffwd::launch<128, false>(maps, fa, g2, stream)
               : ffwd::launch<256, false>(maps, fa, g2, stream);
  return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

}  // namespace cp
