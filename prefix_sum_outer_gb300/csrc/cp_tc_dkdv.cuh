// Fused backward of the causal product for dk and dv (bf16, D and M <= 64).
//
// With g = dL/d out, the gradients of out_i = sum_{j<=i} (q_i . k_j) v_j
// ("Transformers are RNNs", the gradient of the causal product, written as
// cumulative sums in reverse order) are
//     dv_j = sum_{i>=j} (k_j . q_i) g_i,        dk_j = sum_{i>=j} (v_j . g_i) q_i.
// Both reverse-order sums read one running state, R = sum_{i>=j} q_i g_i^T
// (D x M): dv_j = R^T k_j and dk_j = R v_j plus the terms inside the tile.
// A CTA walks its segment of 128-row tiles from the last to the first; with
// R the fp32 state before tile t (the sum over the later tiles):
//     P1   = K_t Q_t^T    masked to i >= j inside the tile
//     P2   = V_t G_t^T    masked to i >= j
//     dV_t = K_t R   + P1 G_t
//     dK_t = V_t R^T + P2 Q_t
//     R   += Q_t^T G_t
// so one pass reads q, k, v and g once and writes dk and dv, where two
// separate reverse products would read six tiles per tile step.  R^T is the
// same bf16 copy of the state read as a K-major operand instead of an
// MN-major one.
//
// CTA = 16 warps:
//   warp 0        TMA producer: Q, K, V, G tiles into a 3-stage ring
//   warp 1        TMEM allocator; MMA issuer of R += Q^T G
//   warps 2..5    state copy (fp32 R -> bf16 hi/lo) and packing of P2
//   warps 6..9    packing of P1 (mask, split into bf16 hi/lo, in TMEM)
//   warps 10..13  dV and dK: fp32 -> bf16, staged in the stage's K and V
//                 boxes (no longer read once the output is final), TMA store
//   warp 14       MMA issuer of dV: P1, then K R and P1 G into one accumulator
//   warp 15       MMA issuer of dK: P2, then V R^T and P2 Q
// Each output's inter- and intra-tile terms come from one thread, so they
// accumulate in issue order.
#pragma once
#include "cp_tc_common.cuh"

namespace cp {
namespace tc {
namespace dkdv {

using namespace cp::ptx;

constexpr int kW = 64;                      // D and M padded to one 64-column box
constexpr int kNS = 3;                      // ring stages
constexpr int kStageBytes = 4 * kBoxBytes;  // Q | K | V | G
constexpr int kSOneBytes = kW * 128;        // 64 x 64 bf16 state copy
constexpr int kSBufBytes = 2 * kSOneBytes;  // hi | lo
constexpr int kNSB = 2;                     // state copies in flight
constexpr int kSmemBytes = kNS * kStageBytes + kNSB * kSBufBytes + 1024 + 1024;
static_assert(kSmemBytes <= kSmemLimit, "shared memory overflow");

// TMEM columns
constexpr int kColP1 = 0;
constexpr int kColP2 = 128;
constexpr int kColO1 = 256;  // dV accumulator, 2 x 64: [K R_hi + P1 G | K R_lo]
constexpr int kColO2 = 384;  // dK accumulator (D columns)
constexpr int kColS = 448;   // state R (D lanes x M columns)
constexpr int kColsAlloc = 512;

constexpr int kSWarp0 = 2, kPWarp0 = 6, kOWarp0 = 10;
constexpr int kI1Warp = 14, kI2Warp = 15;
constexpr int kThreads = 512;
static_assert(kPWarp0 == kSWarp0 + 4 && kOWarp0 == kPWarp0 + 4 && kI1Warp == kOWarp0 + 4,
              "four consecutive warps (one per TMEM lane quarter) per converter group");

struct DkdvArgs {
  int64_t N;
  int n_tiles;
  int seg_tiles;
  int G;
  int BH;
  int D, M;
  const float* agg_in;  // [BH][G][64][64] per-segment sums of q g^T; null when G == 1
  const float* state_in;  // [BH][D][M] dL/dS_N seeding R (null: zero)
  float* state_out;       // [BH][D][M] receives dL/dS_0 = R after row 0 (null: not written)
  int* status;
};

// P of one tile, in place in TMEM: mask to i >= j, split into bf16 hi + lo,
// pack (chunk c of 32 columns: hi at +[0,16), lo at +[16,32)).
__device__ __forceinline__ void pack_p_reverse(uint32_t pc, int wq, int lane) {
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    const bool z = c < wq;  // every column of the chunk is left of the diagonal
    uint32_t r[32];
    if (!z) {
      tmem_ld32(pc + 32 * c, r);
      tmem_ld_wait();
    }
    split_pack_p(r, z, c == wq, lane, 1);
    store_packed_p(pc + 32 * c, r);
  }
  tmem_st_wait();
}

// One CTA's work: the fused reverse scan of one (segment, problem).  The
// tensor maps are the kernel's __grid_constant__ parameters.  STATE_OUT: the
// launch writes dL/dS_0 (a separate instantiation, as for the product).
// FEAT: q and k are raw rows of the feature map phi = elu + 1: the output
// group maps the Q and K boxes of each stage in place one tile ahead (the
// MMAs wait for the map), and dK, read out before dV overwrites the K box,
// is multiplied by phi'(k) = min(1, phi(k)) from that box, so that dK and
// dV are the gradients with respect to the raw k and v.
// Returns false when a wait gave up.
template <bool STATE_OUT, bool FEAT = false>
__device__ __forceinline__ bool dkdv_body(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                          const CUtensorMap& tm_v, const CUtensorMap& tm_g,
                                          const CUtensorMap& tm_dk, const CUtensorMap& tm_dv,
                                          const DkdvArgs& a, const Phase ph) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;                              // [kNS] x (Q | K | V | G)
  uint8_t* s_tile = ring + kNS * kStageBytes;        // [kNSB] x (hi | lo) bf16 copies of R
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_tile + kNSB * kSBufBytes);
  uint64_t* full = bars;                    // [kNS] TMA -> issuers
  uint64_t* empty = full + kNS;             // [kNS] state issuer + output group -> TMA
  uint64_t* p_done = empty + kNS;           // [2] issuer x -> packers: P in TMEM
  uint64_t* p_ready = p_done + 2;           // [2] packers -> issuer x: P packed
  uint64_t* o_done = p_ready + 2;           // [2] issuer x -> output group, issuer x: output final
  uint64_t* o_free = o_done + 2;            // [2] output group -> issuer x: read out
  uint64_t* copy_ready = o_free + 2;        // [kNSB] state group -> issuers: copy of R written
  uint64_t* qs_done = copy_ready + kNSB;    // [kNSB] issuers 1, 2 -> state group: copy read
  uint64_t* s_done = qs_done + kNSB;        // state issuer -> state group: R updated
  uint64_t* fin = s_done + 1;               // [3]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(fin + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(fin + 4);
  uint64_t* qk_mapped = fin + 5;            // [kNS] FEAT: output group -> issuers: Q, K mapped
  // what an MMA that reads Q or K waits for
  uint64_t* const qk_bar = FEAT ? qk_mapped : full;
  static_assert(!(FEAT && STATE_OUT), "the feature backward carries no state");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int bh = ph.work % a.BH;
  const int seg = ph.work / a.BH;
  const int t_first = seg * a.seg_tiles;
  const int t_end = min(a.n_tiles, t_first + a.seg_tiles);
  const int n_it = t_end - t_first;
  const bool has_prefix = a.agg_in != nullptr && seg < a.G - 1;
  // R does not start at zero: later segments or a carried final-state gradient
  const bool has_init = has_prefix || a.state_in != nullptr;
  auto tile_of = [&](int it) { return t_end - 1 - it; };  // reverse order

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&p_done[x], 1);
      mbar_init(&p_ready[x], 4);
      mbar_init(&o_done[x], 1);
      mbar_init(&o_free[x], 4);
    }
    for (int i = 0; i < kNSB; ++i) {
      mbar_init(&copy_ready[i], 4);
      mbar_init(&qs_done[i], 2);
    }
    mbar_init(s_done, 1);
    for (int i = 0; i < 3; ++i) mbar_init(&fin[i], 1);
    for (int i = 0; FEAT && i < kNS; ++i) mbar_init(&qk_mapped[i], 4);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_g);
    tma_prefetch_desc(&tm_dk);
    tma_prefetch_desc(&tm_dv);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kColsAlloc);
    if (ph.last) tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (ph.first) grid_dep_wait();  // inputs written by the previous kernel are visible from here
  const uint32_t tmem = *tmem_holder;
  const int wq = warp & 3;                 // TMEM lane quarter of this warp
  const int row = wq * 32 + lane;          // tile row = TMEM lane
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);

  constexpr uint32_t kHi = desc_hi(1024);  // SBO = 1024, 128-byte swizzle
  auto stage_addr = [&](int it) { return smem_u32(ring + (it % kNS) * kStageBytes); };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int n = 0;
      for (; n < n_it; ++n) {
        const int st = n % kNS;
        if (n >= kNS && !mbar_wait_t<FEAT>(&empty[st], ((n / kNS) - 1) & 1, abort_flag)) {
          record_timeout(a.status, abort_flag);
          break;
        }
        const int row0 = tile_of(n) * kTile;
        uint8_t* base = ring + st * kStageBytes;
        mbar_arrive_expect_tx(&full[st], kStageBytes);
        tma_load_3d(base, &tm_q, &full[st], 0, row0, bh, pol);
        tma_load_3d(base + kBoxBytes, &tm_k, &full[st], 0, row0, bh, pol);
        tma_load_3d(base + 2 * kBoxBytes, &tm_v, &full[st], 0, row0, bh, pol);
        tma_load_3d(base + 3 * kBoxBytes, &tm_g, &full[st], 0, row0, bh, pol);
      }
      if (*abort_flag) {
        // let the copies already issued land before the CTA's memory goes away
        for (int j = max(0, n - kNS); j < n; ++j)
          mbar_wait_timeout(&full[j % kNS], (j / kNS) & 1, CP_WAIT_TIMEOUT_NS);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ state issuer
    // R(t) update needs tile t landed and R copied out for tile t.
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kW, 1, 1);  // Q^T . G
      const uint32_t t_s = tmem + kColS;
      bool ok = true;
      for (int it = 0; it < n_it; ++it) {
        if (!mbar_wait_t<FEAT>(&qk_bar[it % kNS], (it / kNS) & 1, abort_flag) ||
            !mbar_wait_t<FEAT>(&copy_ready[it % kNSB], (it / kNSB) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // R += Q^T G (A = Q^T, B = G, both MN-major)
        const uint32_t base = stage_addr(it);
        const uint32_t qt_lo = desc_lo(base, kBoxBytes);
        const uint32_t g_lo = desc_lo(base + 3 * kBoxBytes, kBoxBytes);
        const bool fresh = (it == 0) && !has_init;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ss_lo<kHi, kHi>(t_s, qt_lo + ((kk * 2048) >> 4), g_lo + ((kk * 2048) >> 4), idesc_s,
                              (fresh && kk == 0) ? 0u : 1u);
        mma_commit(s_done);
        mma_commit(&empty[it % kNS]);
      }
      if (!ok) record_timeout(a.status, abort_flag);
      mma_commit(&fin[0]);
      mbar_wait_timeout(&fin[0], 0, CP_WAIT_TIMEOUT_NS);
    }
  } else if (warp == kI1Warp || warp == kI2Warp) {
    // ------------------------------------------------------------ product issuers
    // x = 0: P1 = K Q^T, dV = K R + P1 G;  x = 1: P2 = V G^T, dK = V R^T + P2 Q.
    // P(t) overwrites the buffer P(t - 1) was read from, so it waits for the
    // output MMAs of t - 1; the inter-tile term waits for the copy of R and
    // for the output group to have read the accumulator for t - 1.
    if (lane == 0) {
      const int x = warp == kI1Warp ? 0 : 1;
      constexpr uint32_t idesc_p = idesc_bf16_f32(128, 128, 0, 0);  // [K|V] . [Q|G]^T
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, kW, 0, 1);   // P . [G|Q], K . R
      constexpr uint32_t idesc_ot = idesc_bf16_f32(128, kW, 0, 0);  // V . R^T (R K-major)
      constexpr uint32_t idesc_ow = idesc_bf16_f32(128, 2 * kW, 0, 1);  // K . [R_hi | R_lo]
      const uint32_t t_p = tmem + (x == 0 ? kColP1 : kColP2);
      const uint32_t t_o = tmem + (x == 0 ? kColO1 : kColO2);
      const uint32_t s_addr = smem_u32(s_tile);
      // operand boxes within a stage: A of P (and of the inter-tile term),
      // B of P, B of P . X
      const uint32_t off_a = (x == 0 ? 1 : 2) * kBoxBytes;  // K or V
      const uint32_t off_b = (x == 0 ? 0 : 3) * kBoxBytes;  // Q or G
      const uint32_t off_x = (x == 0 ? 3 : 0) * kBoxBytes;  // G or Q
      bool ok = true;
      for (int it = 0; it < n_it; ++it) {
        // P1 = K Q^T reads mapped boxes; P2 = V G^T does not
        if (!mbar_wait_t<FEAT>(x == 0 ? &qk_bar[it % kNS] : &full[it % kNS], (it / kNS) & 1, abort_flag) ||
            (it > 0 && !mbar_wait_t<FEAT>(&o_done[x], (it - 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = stage_addr(it);
        const uint32_t a_lo = desc_lo(base + off_a, 16);
        const uint32_t b_lo = desc_lo(base + off_b, 16);
#pragma unroll
        for (int kk = 0; kk < kW / 16; ++kk)
          mma_ss_lo<kHi, kHi>(t_p, a_lo + kk * 2, b_lo + kk * 2, idesc_p, kk > 0 ? 1u : 0u);
        mma_commit(&p_done[x]);
        if (!mbar_wait_t<FEAT>(&copy_ready[it % kNSB], (it / kNSB) & 1, abort_flag) ||
            (it > 0 && !mbar_wait_t<FEAT>(&o_free[x], (it - 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // inter-tile term from the hi and lo copies of R.  dV: K [R_hi | R_lo]
        // in one N = 128 chain (the copies sit side by side as one MN-major
        // operand; the two halves are summed on read-out).  dK: V R_hi^T +
        // V R_lo^T, R read K-major (row d of R is column d of R^T).
        const uint32_t s_buf = s_addr + (it % kNSB) * kSBufBytes;
        if (x == 0) {
          const uint32_t r_lo = desc_lo(s_buf, kSOneBytes);
#pragma unroll
          for (int kk = 0; kk < kW / 16; ++kk)
            mma_ss_lo<kHi, kHi>(t_o, a_lo + kk * 2, r_lo + ((kk * 2048) >> 4), idesc_ow,
                                kk > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int part = 0; part < 2; ++part) {
#pragma unroll
            for (int kk = 0; kk < kW / 16; ++kk)
              mma_ss_lo<kHi, kHi>(t_o, a_lo + kk * 2,
                                  desc_lo(s_buf + part * kSOneBytes, 16) + kk * 2, idesc_ot,
                                  (part == 0 && kk == 0) ? 0u : 1u);
          }
        }
        mma_commit(&qs_done[it % kNSB]);
        if (!mbar_wait_t<FEAT>(&p_ready[x], it & 1, abort_flag) ||
            (FEAT && x == 1 && !mbar_wait_t<FEAT>(&qk_mapped[it % kNS], (it / kNS) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // out += P_hi X (+ P_lo X) (A = packed P in TMEM, B = X MN-major)
        const uint32_t x_lo = desc_lo(base + off_x, kBoxBytes);
#pragma unroll
        for (int part = 0; part < kPParts; ++part) {
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t acol = (kk >> 1) * 32 + part * 16 + (kk & 1) * 8;
            mma_ts_lo<kHi>(t_o, t_p + acol, x_lo + ((kk * 2048) >> 4), idesc_o, 1u);
          }
        }
        mma_commit(&o_done[x]);
      }
      if (!ok) record_timeout(a.status, abort_flag);
      mma_commit(&fin[1 + x]);
      mbar_wait_timeout(&fin[1 + x], 0, CP_WAIT_TIMEOUT_NS);
    }
  } else if (warp < kPWarp0) {
    // ------------------------------------------------------------ state group
    // Two independent sequences, taken whichever is ready: the bf16 copy of
    // R before each tile, and the packing of P2.
    if (has_init) {
      // initial state: the carried dL/dS_N plus the fixed-order sum of the
      // later segments' aggregates
      if (wq < 2) {
        const float* st = a.state_in != nullptr ? a.state_in + (int64_t)bh * a.D * a.M : nullptr;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float acc[32];
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int m = c * 32 + x;
            acc[x] = (st != nullptr && row < a.D && m < a.M) ? st[row * a.M + m] : 0.f;
          }
          // slot seg holds the sum of the later segments' aggregates
          if (has_prefix) {
            const float4* src = reinterpret_cast<const float4*>(
                a.agg_in + (((size_t)bh * a.G + seg) * kW + row) * kW + c * 32);
#pragma unroll
            for (int x = 0; x < 8; ++x) {
              const float4 f = __ldg(src + x);
              acc[4 * x] += f.x;
              acc[4 * x + 1] += f.y;
              acc[4 * x + 2] += f.z;
              acc[4 * x + 3] += f.w;
            }
          }
          uint32_t r[32];
#pragma unroll
          for (int x = 0; x < 32; ++x) r[x] = __float_as_uint(acc[x]);
          tmem_st32(lane_base + kColS + c * 32, r);
        }
        tmem_st_wait();
      }
    }
    bool ok = true;
    int ns = 0, np = 0;
    uint64_t t0 = globaltimer();
    uint32_t idle = 0;
    while (ns < n_it || np < n_it) {
      bool progressed = false;
      bool ready = false;
      if (ns < n_it && lane == 0) {
        const int b = ns % kNSB;
        ready = (ns < kNSB || mbar_test_wait(&qs_done[b], ((ns - kNSB) / kNSB) & 1)) &&
                (ns == 0 || mbar_test_wait(s_done, (ns - 1) & 1));
      }
      if (__shfl_sync(0xffffffffu, ready, 0)) {
        tc_fence_after();
        uint8_t* sbuf = s_tile + (ns % kNSB) * kSBufBytes;
        if (wq < 2) {  // rows d of R (D <= 64 lanes)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            if (ns == 0 && !has_init) {
              store_zero32(sbuf, row, c * 32, kW * 128);
              store_zero32(sbuf + kSOneBytes, row, c * 32, kW * 128);
            } else {
              uint32_t r[32];
              tmem_ld32(lane_base + kColS + c * 32, r);
              tmem_ld_wait();
              store_chunk32_split(sbuf, sbuf + kSOneBytes, row, c * 32, kW * 128, r);
            }
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&copy_ready[ns % kNSB]);
        ++ns;
        progressed = true;
      }
      ready = false;
      if (np < n_it && lane == 0) ready = mbar_test_wait(&p_done[1], np & 1);
      if (__shfl_sync(0xffffffffu, ready, 0)) {
        tc_fence_after();
        pack_p_reverse(lane_base + kColP2, wq, lane);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_ready[1]);
        ++np;
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
    // the first segment (last in scan order) hands on R after row 0: dL/dS_0
    if (STATE_OUT && ok && seg == 0 && n_it > 0) {
      if (!mbar_wait_t<FEAT>(s_done, (n_it - 1) & 1, abort_flag)) {
        ok = false;
      } else if (wq < 2) {
        tc_fence_after();
        float* st = a.state_out + (int64_t)bh * a.D * a.M;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[32];
          tmem_ld32(lane_base + kColS + c * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int m = c * 32 + x;
            if (row < a.D && m < a.M) st[row * a.M + m] = __uint_as_float(r[x]);
          }
        }
      }
    }
    if (!ok) record_timeout(a.status, abort_flag);
  } else if (warp < kOWarp0) {
    // ------------------------------------------------------------ P1 group
    bool ok = true;
    for (int it = 0; it < n_it && ok; ++it) {
      if (!mbar_wait_t<FEAT>(&p_done[0], it & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      pack_p_reverse(lane_base + kColP1, wq, lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_ready[0]);
    }
    if (!ok) record_timeout(a.status, abort_flag);
  } else if (warp < kI1Warp) {
    // ------------------------------------------------------------ output group
    // dV(t) is staged in the K box of tile t's stage and dK(t) in its V box:
    // once an output is final, every MMA that read that box has completed.
    // The stage is released after both stores have read it.
    const int o_tid = threadIdx.x - 32 * kOWarp0;
    bool ok = true;
    // FEAT: phi applied in place to the Q and K boxes of tile it (columns
    // D.. of a box are zero padding and stay zero; a box row is 8 chunks of
    // 16 bytes under the 128-byte swizzle: chunk c of row r holds logical
    // chunk c ^ (r % 8)).  Tile it + 1 is mapped before the read-out of tile
    // it: its stage was released at the end of iteration it - 2.
    [[maybe_unused]] auto map_stage = [&](int it) -> bool {
      if (!mbar_wait_t<FEAT>(&full[it % kNS], (it / kNS) & 1, abort_flag)) return false;
      uint4* p = reinterpret_cast<uint4*>(ring + (it % kNS) * kStageBytes);  // Q box, K box
      constexpr int kChunks = 2 * kBoxBytes / 16, kBoxChunks = kBoxBytes / 16;
      auto map_chunk = [&](int i) {
        uint4 w = p[i];
        w.x = elu1_bf16x2(w.x);
        w.y = elu1_bf16x2(w.y);
        w.z = elu1_bf16x2(w.z);
        w.w = elu1_bf16x2(w.w);
        p[i] = w;
      };
      if (a.D == kW) {
#pragma unroll 2
        for (int i = o_tid; i < kChunks; i += 128) map_chunk(i);
      } else {
        for (int i = o_tid; i < kChunks; i += 128) {
          const int rc = i % kBoxChunks;
          if ((((rc & 7) ^ ((rc >> 3) & 7)) << 3) < a.D) map_chunk(i);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&qk_mapped[it % kNS]);
      return true;
    };
    if (FEAT && n_it > 0) ok = map_stage(0);
    for (int it = 0; it < n_it && ok; ++it) {
      const int st = it % kNS;
      const int row0 = tile_of(it) * kTile;
      if (FEAT && it + 1 < n_it && !map_stage(it + 1)) {
        ok = false;
        break;
      }
      for (int xi = 0; xi < 2; ++xi) {
        // FEAT: dK first, while the K box still holds phi(k)
        const int x = FEAT ? 1 - xi : xi;
        if (!mbar_wait_t<FEAT>(&o_done[x], it & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (!FEAT) {
          // a chunk of 32 columns at a time (one copy of the conversion in
          // the instruction stream: the one-launch backward measured 122.6
          // against 124.4 us)
          uint8_t* ob = ring + st * kStageBytes + (x == 0 ? 1 : 2) * kBoxBytes;
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t r1[32];
            tmem_ld32(lane_base + (x == 0 ? kColO1 : kColO2) + c * 32, r1);
            tmem_ld_wait();
            if (x == 0) {
              uint32_t u[32];
              tmem_ld32(lane_base + kColO1 + kW + c * 32, u);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e)
                r1[e] = __float_as_uint(__uint_as_float(r1[e]) + __uint_as_float(u[e]));
            }
            store_chunk32(ob, row, c * 32, kBoxBytes, r1);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&o_free[x]);
          fence_proxy_async_smem();
          named_barrier_sync(1, 128);
          if (o_tid == 0) {
            tma_store_3d(x == 0 ? &tm_dv : &tm_dk, ob, 0, row0, bh);
            tma_store_commit();
          }
          continue;
        }
        uint32_t r[2][32];
        tmem_ld32(lane_base + (x == 0 ? kColO1 : kColO2), r[0]);
        tmem_ld32(lane_base + (x == 0 ? kColO1 : kColO2) + 32, r[1]);
        tmem_ld_wait();
        if (x == 0) {
          // add the K R_lo half
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t u[32];
            tmem_ld32(lane_base + kColO1 + kW + c * 32, u);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e)
              r[c][e] = __float_as_uint(__uint_as_float(r[c][e]) + __uint_as_float(u[e]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&o_free[x]);
        uint8_t* ob = ring + st * kStageBytes + (x == 0 ? 1 : 2) * kBoxBytes;
        if (FEAT && x == 1) {
          const uint8_t* kb = ring + st * kStageBytes + kBoxBytes;
          scale_store_chunk32_phi(ob, kb, row, 0, kBoxBytes, r[0]);
          scale_store_chunk32_phi(ob, kb, row, 32, kBoxBytes, r[1]);
        } else {
          store_chunk32(ob, row, 0, kBoxBytes, r[0]);
          store_chunk32(ob, row, 32, kBoxBytes, r[1]);
        }
        fence_proxy_async_smem();
        named_barrier_sync(1, 128);
        if (o_tid == 0) {
          tma_store_3d(x == 0 ? &tm_dv : &tm_dk, ob, 0, row0, bh);
          tma_store_commit();
        }
      }
      if (o_tid == 0 && ok) {
        tma_store_wait_read_all();
        mbar_arrive(&empty[st]);
      }
    }
    if (!ok) record_timeout(a.status, abort_flag);
    if (o_tid == 0) tma_store_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  // this CTA's work is done: the next kernel in the stream may be scheduled
  // once every CTA has got here (its blocks still wait in grid_dep_wait for
  // this whole grid).  Triggering at the start instead let the next kernel's
  // CTAs take the SMs this grid's blocks freed, which cost up to 80 us when
  // the forward and backward kernels alternate.
  if (ph.last) grid_dep_launch_dependents();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kColsAlloc);
  }
  const bool completed = *abort_flag == 0;
  if (!ph.last) {
    // a later scan of this CTA reuses the barriers' memory
    __syncthreads();
    if (threadIdx.x == 0) {
      for (uint64_t* b = bars; b < fin + 3; ++b) mbar_inval(b);
      for (int i = 0; FEAT && i < kNS; ++i) mbar_inval(&qk_mapped[i]);
    }
    __syncthreads();
  }
  return completed;
}

}  // namespace dkdv
}  // namespace tc
}  // namespace cp
