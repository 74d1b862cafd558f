// The causal-product scan of one CTA on the 5th-generation tensor cores
// (sm_103a), as a device function (the body of the product kernel).
//
// The recurrence "state += k v^T; out = state^T q" (triton-lang/triton issue
// #217, the loop listing; the issue's opening comment calls it the prefix
// sum of Algorithm 1 of "Transformers are RNNs") is regrouped into tiles of
// 128 rows.  With S the fp32 D x M state before tile t:
//     P   = Q_t K_t^T            masked to j <= i inside the tile (128x128)
//     O_t = Q_t S + P V_t        (inter-tile readout, then the intra-tile part
//                                 accumulated onto it)
//     S  += K_t^T V_t
// All four are dense contractions and run as tcgen05.mma with bf16 operands
// in shared memory and fp32 accumulators in tensor memory (TMEM).  The state
// never leaves TMEM while a CTA walks its segment; a bf16 copy of it is
// written to shared memory once per tile to serve as the MMA operand of
// Q_t S.  P is masked and rounded to bf16 on its way from TMEM to shared
// memory.
//
// CTA = 16 warps:
//   warp 0        TMA producer: Q/K tiles and V tiles into two rings
//   warp 1        TMEM allocator; MMA issuer of the state chain S and of Q S
//   warps 2..5    state group: fp32 S -> bf16 hi/lo operand copy
//   warps 6..9    P group: mask P, split into bf16 hi/lo, pack in TMEM
//   warps 10..13  O group: fp32 O -> bf16, TMA store
//   warps 14, 15  MMA issuers of P and of P V
// (the converter groups run one thread per TMEM lane = tile row)
//
// Product kernels are launched as programmatic dependents: the set-up
// (barriers, TMEM allocation, descriptor prefetch) overlaps the previous
// kernel in the stream, and no global memory is touched before it has
// completed.  A CTA lets the next kernel be scheduled only when its own
// work is done.
//
// With a feature map (the FEAT instantiation), the loaded Q and K tiles are
// raw inputs x: the O group (the state group in the aggregate-only mode)
// maps them in shared memory, phi(x) = elu(x) + 1 (x + 1 for x > 0, e^x
// otherwise, rounded to bf16), before any MMA reads them, so phi(q) and
// phi(k) never exist in global memory.
//
// With the normaliser (the NORM instantiation, forward, D <= 64, one
// segment per problem) the CTA also writes z_i = q_i . sum_{j<=i} k_j.  The
// state group, whose warps of lane quarters 2 and 3 hold no state rows at
// D <= 64 and whose chain has slack, computes q_i . s_k for the tile (s_k =
// the sum of k over the earlier tiles, in shared memory) and the tile's
// column sums of k, off the P chain; the P group sums each masked fp32 row
// of P while packing it (the terms j of the tile) and writes z.
//
// FEAT_V maps the value tiles the same way (the value operand is a raw
// input), and EPI multiplies every output element by phi'(x) = min(1,
// phi(x)) of a raw row given apart (a.epi_x): the chain rule of the feature
// map, for the products of a backward whose inputs are raw rows.
//
// Long sequences with few problems are split into G segments per problem;
// a first launch of the same kernel in aggregate-only mode writes each
// segment's sum of k v^T, and every segment of the second launch starts
// from the fixed-order sum of its predecessors' aggregates (a two-pass scan
// across segments, deterministic).
#pragma once
#include <type_traits>
#include "cp_tc_common.cuh"

namespace cp {
namespace tc {

using namespace cp::ptx;

// Warp roles: 0 TMA producer; 1, 14 and 15 MMA issuers (the issuing
// thread's instruction rate, not the tensor pipe, bounds a single issuer);
// three converter groups that each own one lane quarter of TMEM per warp.
// Sixteen warps keep every sub-partition at four warps, which leaves 128
// registers per thread.
constexpr int kSWarp0 = 2, kSWarps = 4;    // state: fp32 S -> bf16 hi/lo operand copy
constexpr int kPWarp0 = 6, kPWarps = 4;    // P: mask, split hi/lo, pack in TMEM
constexpr int kOWarp0 = 10, kOWarps = 4;   // O: fp32 -> bf16 -> TMA store
constexpr int kBWarp = 14;                 // MMA issuer of P
constexpr int kCWarp = 15;                 // MMA issuer of P V
constexpr int kThreads = 32 * (kCWarp + 1);
static_assert(kPWarp0 == kSWarp0 + kSWarps && kOWarp0 == kPWarp0 + kPWarps &&
                  kBWarp == kOWarp0 + kOWarps,
              "converter groups of consecutive warps, one per TMEM lane quarter");
constexpr int kOThreads = 32 * kOWarps;

struct Args {
  int64_t N;
  int n_tiles;
  int seg_tiles;
  int G;
  int BH;
  int n_mb;
  int reverse;
  const float* agg_in;   // [P][G][DP][MB]; null when G == 1
  float* agg_out;        // aggregate-only launch writes here
  int* status;
  // carried state (see Product): read by every segment, written by the last
  // one in scan order; Dr x Mc per problem
  const float* state_in;
  float* state_out;
  int64_t st_ld_r, st_ld_c;
  int Dr, Mc;
  int feature;  // 0: q, k used as given; 1: phi = elu + 1 (FEAT instantiation)
};

// The arguments of the checkpoint-writing (CKPT) and seeded (SEED)
// instantiations.  The plain kernels take Args alone: measured on
// B=8 H=16 N=4096 D=M=64, these fields in every kernel's parameters made the
// plain forward launch 3.5 us slower (44.4 -> 48.0 us) through code
// generation, with the same code path at run time.
struct ArgsX : Args {
  // Checkpoints of the state every ck_tiles tiles, in the caller's state
  // layout: ckpt[((bh * (ck_G - 1) + s - 1) * Dr + d) * Mc + m] is element
  // (d, m) of the state before tile s * ck_tiles, s = 1 .. ck_G - 1.  A
  // forward product with ckpt set (CKPT instantiation) writes them.
  float* ckpt;
  int ck_tiles, ck_G;
  // Seeded segments (SEED instantiation): every segment but the first in
  // scan order starts from a precomputed state instead of a segment-sum
  // pass: element (r, c) of the start of segment seg of problem bh is
  // seed[bh * seed_bh + (seg + seed_seg_off) * seed_seg + r * st_ld_r + c * st_ld_c]
  // (the carried-state strides; no carried state besides).
  const float* seed;
  int64_t seed_bh, seed_seg;
  int seed_seg_off;
  // NORM instantiation: z [BH][N] fp32, z_i = q_i . sum_{j<=i} k_j
  float* z;
  // EPI instantiation: raw rows x [BH][N][Mc] bf16; each output element is
  // multiplied by phi'(x) of its position (phi = elu + 1)
  const void* epi_x;
  // the one-launch split scan (tc_lookback_kernel): agg_out holds each
  // segment's own sum, slot s written once lb_flags[pidx * G + s] is nonzero;
  // agg_in (the prefix slots) is filled by the launch itself
  unsigned int* lb_flags;
};

// Kernel arguments: the extended set only where an instantiation reads it
// (the plain kernels keep the smaller parameter block).
template <bool EXT>
using KArgs = std::conditional_t<EXT, ArgsX, Args>;

// Shared memory of the NORM instantiation beyond the layout: q_i . s_k for
// the tile's 128 rows, s_k and one half of a tile's column sums of k (DP
// fp32 each).
template <int DP>
constexpr int kNormBytes = 128 * 4 + 2 * DP * 4;

// AGG: the aggregate-only pass.  It loads no Q and keeps neither state
// copies nor output staging, so its Q/K stages hold K alone and the whole
// budget goes to the rings (at DP = MB = 128: 3 K and 4 V stages instead of
// one of each).
template <int DP, int MB, bool AGG = false>
struct Layout {
  static constexpr int kQBoxes = DP / kBoxCols;
  static constexpr int kVBoxes = MB / kBoxCols;
  static constexpr int kSBlocks = (DP + 127) / 128;
  static constexpr int kQBytes = kQBoxes * kBoxBytes;
  static constexpr int kQKBytes = 2 * kQBytes;               // one Q tile + one K tile
  static constexpr int kQKStage = AGG ? kQBytes : kQKBytes;  // a Q/K ring stage
  static constexpr int kKOff = AGG ? 0 : kQBytes;            // K within a stage
  static constexpr int kVBytes = kVBoxes * kBoxBytes;
  static constexpr int kSOneBytes = kVBoxes * DP * 128;      // DP x MB bf16
  static constexpr int kOBytes = kVBoxes * kBoxBytes;        // 128 x MB bf16
  static constexpr int kBarBytes = 1024;
  static constexpr int kAlignSlack = 1024;
  static constexpr int kAvail = kSmemLimit - kBarBytes - kAlignSlack;
  // Q/K and V tiles live in two rings: Q and K are released once P, the
  // state update and Q S have been issued, V only after P V, so the V ring
  // gets one stage more when it fits.  Returns NQK * 8 + NV.
  static constexpr int rings(int budget) {
    for (int n = 4; n >= 1; --n) {
      if (n * kQKStage + (n + 1) * kVBytes <= budget) return n * 8 + n + 1;
      if (n * kQKStage + n * kVBytes <= budget) return n * 8 + n;
    }
    return 0;
  }
  // TMEM holds NP buffers of P (128 columns, fp32; later packed bf16 hi|lo),
  // NO output accumulators of MB columns (Q S, then P V accumulated on top)
  // and the state (kSBlocks x MB).  A P buffer is reused only after the P V
  // that read it has completed, an output buffer only after the output
  // group has read it out.
  static constexpr int cols(int np, int no) { return np * 128 + no * MB + kSBlocks * MB; }
  static constexpr int NP = cols(2, 1) <= 512 ? 2 : 1;
  static constexpr int NO = cols(NP, 3) <= 512 ? 3 : (cols(NP, 2) <= 512 ? 2 : 1);
  // bf16 copies of the state in shared memory (one per tile in flight, at
  // most two); the state operand of Q S is split into hi + lo parts when it
  // fits next to a one-stage ring.
  static constexpr int NSB =
      (NP >= 2 && rings(kAvail - 4 * kSOneBytes - 2 * kOBytes) / 8 >= 2) ? 2 : 1;
  static constexpr bool kSplit = rings(kAvail - NSB * 2 * kSOneBytes - kOBytes) / 8 >= 1;
  static constexpr int kSBufBytes = (kSplit ? 2 : 1) * kSOneBytes;
  // output staging: two buffers (one store in flight) when they fit next to
  // the state copies and rings of at least one Q/K and two V stages (a
  // single V stage would serialise each tile's V load behind the previous
  // tile's P V)
  static constexpr int kOBufs =
      (rings(kAvail - NSB * kSBufBytes - 2 * kOBytes) / 8 >= (NSB == 2 ? 2 : 1) &&
       rings(kAvail - NSB * kSBufBytes - 2 * kOBytes) >= 8 + 2)
          ? 2
          : 1;
  static constexpr int kSRegion = AGG ? 0 : NSB * kSBufBytes;
  static constexpr int kORegion = AGG ? 0 : kOBufs * kOBytes;
  static constexpr int kFixed = kSRegion + kORegion;
  static constexpr int NQK = rings(kAvail - kFixed) / 8;
  static constexpr int NV = rings(kAvail - kFixed) % 8;
  static constexpr int kSmemBytes =
      NQK * kQKStage + NV * kVBytes + kFixed + kBarBytes + kAlignSlack;
  static constexpr int kColP = 0;                        // + b * 128
  static constexpr int kColO = NP * 128;                 // + o * MB
  static constexpr int kColS = kColO + NO * MB;          // + sb * MB
  static constexpr int kColsUsed = kColS + kSBlocks * MB;
  static constexpr int kColsAlloc = kColsUsed <= 256 ? 256 : 512;
  static_assert(NQK >= 1 && NV >= 1, "tile does not fit in shared memory");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory overflow");
  static_assert(kColsUsed <= 512, "accumulators do not fit in TMEM");
  static_assert(DP % 64 == 0 && MB % 64 == 0, "64-column boxes");
};

// One CTA's work: the scan of one (segment, problem, value block).  The
// tensor maps are the kernel's __grid_constant__ parameters.  STATE_OUT:
// the launch writes the final state (a separate instantiation: the write,
// though it runs once, costs the whole kernel registers).
// FEAT: q and k are raw inputs mapped by phi = elu + 1 in shared memory.
// CKPT: a forward product writes its state at every checkpoint boundary.
// SEED: segments start from precomputed states (a.seed) instead of the
// prefix of a segment-sum pass (separate instantiations: both cost the
// plain scan registers and time when compiled in).
// NORM: the forward scan of an unsplit problem also writes z (a.z).
// FEAT_V: v is a raw input mapped by phi = elu + 1 in shared memory.
// EPI: every output element times phi'(x) of the raw row a.epi_x (tm_x: its
// tensor map, the output's shape).
// Returns false when a wait gave up.
template <int DP, int MB, bool AGG_ONLY, bool STATE_OUT, bool FEAT = false, bool CKPT = false,
          bool SEED = false, bool NORM = false, bool FEAT_V = false, bool EPI = false,
          typename A = Args>
__device__ __forceinline__ bool causal_body(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                            const CUtensorMap& tm_v, const CUtensorMap& tm_o,
                                            const A& a, const Phase ph,
                                            const CUtensorMap* tm_x = nullptr) {
  static_assert(!(CKPT || SEED || NORM || EPI) || sizeof(A) == sizeof(ArgsX),
                "CKPT, SEED, NORM and EPI take ArgsX");
  static_assert(!(FEAT_V || EPI) || !(FEAT || STATE_OUT || CKPT || SEED || NORM),
                "the value map and the derivative epilogue serve plain backward products");
  static_assert(!EPI || !AGG_ONLY, "the aggregate pass writes no output");
  static_assert(!NORM || !(AGG_ONLY || STATE_OUT || FEAT || CKPT || SEED),
                "the normaliser is written by the plain forward scan alone");
  static_assert(!NORM || DP == 64, "the normaliser uses the state group's two idle warps");
  // the feature-map and normaliser instantiations wait with the polling
  // loop out of line (their instruction stream is a leading stall reason:
  // the one-launch feature backward measured 172 against 183 us, the
  // forward with the normaliser 79 against 82.5 us; the plain kernels are
  // faster with it inline)
  constexpr bool kOutlineWaits = FEAT || FEAT_V || EPI || NORM;
  using L = Layout<DP, MB, AGG_ONLY>;
  constexpr int NQK = L::NQK;
  constexpr int NV = L::NV;
  constexpr int NP = L::NP;
  constexpr int NSB = L::NSB;
  constexpr int NO = L::NO;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* qk_ring = smem;                           // [NQK] x (Q tile | K tile), K alone (AGG)
  uint8_t* v_ring = qk_ring + NQK * L::kQKStage;     // [NV] x V tile
  uint8_t* s_tile = v_ring + NV * L::kVBytes;        // [NSB] x (hi | lo) bf16 state copies
  uint8_t* o_tile = s_tile + L::kSRegion;            // [kOBufs] output staging
  uint64_t* bars = reinterpret_cast<uint64_t*>(o_tile + L::kORegion);
  uint64_t* full_qk = bars;                 // [NQK] TMA -> MMA
  uint64_t* empty_qk = full_qk + NQK;       // [NQK] MMA -> TMA
  uint64_t* full_v = empty_qk + NQK;        // [NV]
  uint64_t* empty_v = full_v + NV;          // [NV]
  uint64_t* p_done = empty_v + NV;          // [NP] issuer B -> P group: P(t) in TMEM
  uint64_t* p_ready = p_done + NP;          // [NP] P group -> C: masked bf16 P (hi|lo) packed
  uint64_t* pv_done = p_ready + NP;         // [NP] C -> B: P V(t) done, P buffer free
  uint64_t* qs_done = pv_done + NP;         // [NSB] A -> S group: Q S(t) done, state copy free
  uint64_t* o_qs = qs_done + NSB;           // [NO] A -> C: Q S(t) in output buffer t % NO
  uint64_t* o_done = o_qs + NO;             // [NO] C -> O group: O(t) final
  uint64_t* o_free = o_done + NO;           // [NO] O group -> A: output buffer read out
  uint64_t* s_done = o_free + NO;           // A -> S group: state updated with tile t
  uint64_t* s_ready = s_done + 1;           // S group -> A: bf16 state copy written, S read
  uint64_t* fin = s_done + 2;               // [3] issuer drains before TMEM release
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(s_done + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(s_done + 6);
  uint64_t* qk_ready = s_done + 7;          // [NQK] S, O groups -> MMA: Q/K(t) mapped (FEAT)
  // NORM, after the barriers: q_i . s_k of the tile's rows, s_k, half a
  // tile's column sums
  float* z_q = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + L::kBarBytes);
  float* z_sk = z_q + 128;
  float* z_part = z_sk + DP;
  uint64_t* zq_ready = qk_ready + NQK;      // NORM: state group -> P group: z_q of tile t written
  uint64_t* zq_free = zq_ready + 1;         // NORM: P group -> state group: z_q read
  // the barrier the MMA issuers wait on before reading a Q/K stage
  uint64_t* const qk_bar = FEAT ? qk_ready : full_qk;
  // FEAT_V: V(t) mapped, by the same warps (after qk_ready; the normaliser's
  // barriers, which never meet FEAT_V, sit there too)
  uint64_t* v_ready = qk_ready + NQK;
  uint64_t* const v_bar = FEAT_V ? v_ready : full_v;
  // EPI: raw rows of tile t landed in output staging buffer t % kOBufs
  uint64_t* x_full = v_ready + NV;
  // FEAT: warps that map a tile: the O group, whose read-out has slack (NO
  // accumulators), not the state group, which sits on the state chain; the
  // state group only in the aggregate-only mode, which has no read-out
  constexpr int kMapWarps = AGG_ONLY ? kSWarps : kOWarps;
  // FEAT_V: with a state of at most 64 rows (TMEM lane quarters 0 and 1)
  // the state group's warps of quarters 2 and 3 have no rows: they map every
  // V tile as soon as it lands, apart from the state chain, and the O group
  // only reads out; wider states leave the map to the O group.  (Q and K
  // tiles, twice the elements, took longer on those two warps than on the
  // O group: measured 75 against 67 us for the feature forward at B=8 H=16
  // N=4096 D=M=64.)
  constexpr bool kVMapS = FEAT_V && !AGG_ONLY && DP <= 64;
  constexpr int kVMapWarps = kVMapS ? 2 : kMapWarps;
  // the state group's warps that arrive on s_ready
  constexpr int kSChainWarps = kVMapS ? 2 : kSWarps;
  // a group maps tile it + kAhead during its iteration it: as far ahead as
  // the Q/K ring allows, off the MMA chain (mapping tile it + kAhead needs
  // only the stage tile it - 1 releases)
  constexpr int kAhead = NQK - 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- block -> (segment, problem, value-column block)
  int idx = ph.work;
  const int mb = idx % a.n_mb;
  idx /= a.n_mb;
  const int bh = idx % a.BH;
  int seg = idx / a.BH;
  if (AGG_ONLY && a.reverse) seg += 1;  // the first segment in scan order is never needed
  const int t_first = seg * a.seg_tiles;
  const int t_end = min(a.n_tiles, t_first + a.seg_tiles);
  const int n_it = t_end - t_first;
  const int pidx = bh * a.n_mb + mb;
  const bool has_prefix =
      !AGG_ONLY && a.agg_in != nullptr && (a.reverse ? (seg < a.G - 1) : (seg > 0));
  // a segment seeded from a precomputed state
  const bool seeded = SEED && !AGG_ONLY && (a.reverse ? (seg < a.G - 1) : (seg > 0));
  // the state does not start at zero: earlier segments, a checkpoint or a
  // carried state
  const bool has_init = has_prefix || seeded || (!AGG_ONLY && a.state_in != nullptr);
  const bool last_seg = a.reverse ? (seg == 0) : (seg == a.G - 1);
  // The aggregate-only pass walks each segment against the order of the
  // scan pass that follows it, and keeps what it loads in L2: the scan pass
  // then starts on the tiles the aggregate pass read last (a segment's sum
  // is the same in either order; the order is fixed, so it is
  // deterministic).
  auto tile_of = [&](int it) {
    return (a.reverse != 0) != AGG_ONLY ? (t_end - 1 - it) : (t_first + it);
  };

  if (threadIdx.x == 0) {
    // a stage is released by both issuers (A: S / Q S, B: P / P V); in the
    // aggregate-only mode issuer A alone consumes the rings
    const uint32_t kRel = AGG_ONLY ? 1 : 2;  // A + B for Q/K, A + C for V
    for (int i = 0; i < NQK; ++i) {
      mbar_init(&full_qk[i], 1);
      // NORM: every state-group warp also reads Q (and two of them K)
      mbar_init(&empty_qk[i], kRel + (NORM ? kSWarps : 0));
      if (FEAT) mbar_init(&qk_ready[i], kMapWarps);
    }
    if (NORM) {
      mbar_init(zq_ready, kSWarps);
      mbar_init(zq_free, kPWarps);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&full_v[i], 1);
      mbar_init(&empty_v[i], kRel);
      if (FEAT_V) mbar_init(&v_ready[i], kVMapWarps);
    }
    for (int i = 0; EPI && i < L::kOBufs; ++i) mbar_init(&x_full[i], 1);
    for (int i = 0; i < NP; ++i) {
      mbar_init(&p_done[i], 1);
      mbar_init(&p_ready[i], kPWarps);
      mbar_init(&pv_done[i], 1);
    }
    for (int i = 0; i < NSB; ++i) mbar_init(&qs_done[i], 1);
    for (int i = 0; i < NO; ++i) {
      mbar_init(&o_qs[i], 1);
      mbar_init(&o_done[i], 1);
      mbar_init(&o_free[i], kOWarps);
    }
    mbar_init(s_done, 1);
    mbar_init(s_ready, kSChainWarps);
    mbar_init(&fin[0], 1);
    mbar_init(&fin[1], 1);
    mbar_init(&fin[2], 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    if (!AGG_ONLY) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_o);
      if (EPI) tma_prefetch_desc(tm_x);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, L::kColsAlloc);
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

  // CKPT: checkpoint s (>= 1) is the state before tile s * ck_tiles; 0
  // when the boundary before `tile` holds none (the start of the sequence)
  auto ckpt_slot = [&](int tile) -> int {
    if constexpr (CKPT) {
      if (a.reverse || tile <= 0 || tile >= a.n_tiles) return 0;
      return tile % a.ck_tiles == 0 ? tile / a.ck_tiles : 0;
    } else {
      return 0;
    }
  };
  // CKPT: row d of checkpoint s, columns m0 .. m0 + 31 of this value block
  auto ckpt_row = [&](int s_slot, int d, int m0) -> float* {
    if constexpr (CKPT)
      return a.ckpt + (((size_t)bh * (a.ck_G - 1) + s_slot - 1) * a.Dr + d) * a.Mc + m0;
    else
      return nullptr;
  };

  // FEAT: phi applied in place to the landed Q/K tiles of tile it (K only in
  // the aggregate-only mode, which loads no Q) by the kMapWarps mapping
  // warps, each thread taking every (32 kMapWarps)-th 16-byte chunk from
  // mtid on; the issuers wait on qk_ready for all of them
  auto map_qk = [&](int it, int mtid) -> bool {
    if (!mbar_wait_t<kOutlineWaits>(&full_qk[it % NQK], (it / NQK) & 1, abort_flag)) return false;
    uint8_t* q_s = qk_ring + (it % NQK) * L::kQKStage;
    uint4* p = reinterpret_cast<uint4*>(AGG_ONLY ? q_s + L::kKOff : q_s);
    constexpr int kChunks = (AGG_ONLY ? 1 : 2) * L::kQBytes / 16;
    constexpr int kTileChunks = L::kQBytes / 16, kBoxChunks = kBoxBytes / 16;
    auto map_chunk = [&](int i) {
      uint4 w = p[i];
      w.x = elu1_bf16x2(w.x);
      w.y = elu1_bf16x2(w.y);
      w.z = elu1_bf16x2(w.z);
      w.w = elu1_bf16x2(w.w);
      p[i] = w;
    };
    if (a.Dr == DP) {
      // four chunks in flight per thread (two: the feature forward at B=8
      // H=16 N=4096 D=M=64 took 67 us, four 59 us, eight 60 us)
#pragma unroll 4
      for (int i = mtid; i < kChunks; i += 32 * kMapWarps) map_chunk(i);
    } else {
      // columns D..DP-1 of the boxes are zero padding, and phi(0) would be
      // 1: leave them.  A box row is 128 bytes (8 chunks of 8 columns)
      // stored with the 128-byte swizzle, so chunk c of row r holds
      // logical chunk c ^ (r % 8).
      for (int i = mtid; i < kChunks; i += 32 * kMapWarps) {
        const int local = i % kTileChunks, b = local / kBoxChunks, rc = local % kBoxChunks;
        const int col0 = b * kBoxCols + (((rc & 7) ^ ((rc >> 3) & 7)) << 3);
        if (col0 < a.Dr) map_chunk(i);
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&qk_ready[it % NQK]);
    return true;
  };

  // FEAT_V: phi applied in place to the landed V tile of tile it (columns
  // mb * MB .. of the value), the same way; the issuers wait on v_ready
  auto map_v = [&](int it, int mtid) -> bool {
    if (!mbar_wait_t<kOutlineWaits>(&full_v[it % NV], (it / NV) & 1, abort_flag)) return false;
    uint4* p = reinterpret_cast<uint4*>(v_ring + (it % NV) * L::kVBytes);
    constexpr int kChunks = L::kVBytes / 16, kBoxChunks = kBoxBytes / 16;
    auto map_chunk = [&](int i) {
      uint4 w = p[i];
      w.x = elu1_bf16x2(w.x);
      w.y = elu1_bf16x2(w.y);
      w.z = elu1_bf16x2(w.z);
      w.w = elu1_bf16x2(w.w);
      p[i] = w;
    };
    if ((mb + 1) * MB <= a.Mc) {
#pragma unroll 2
      for (int i = mtid; i < kChunks; i += 32 * kVMapWarps) map_chunk(i);
    } else {
      // zero padding beyond column Mc stays zero (phi(0) would be 1)
      for (int i = mtid; i < kChunks; i += 32 * kVMapWarps) {
        const int b = i / kBoxChunks, rc = i % kBoxChunks;
        const int col0 = mb * MB + b * kBoxCols + (((rc & 7) ^ ((rc >> 3) & 7)) << 3);
        if (col0 < a.Mc) map_chunk(i);
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&v_ready[it % NV]);
    return true;
  };
  // a group maps V tile it + kAheadV during its iteration it (mapping it
  // needs only the stage tile it - 1 releases)
  constexpr int kAheadV = NV - 1;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Polls both rings and refills whichever has a free stage (V never runs
    // ahead of Q/K).
    if (lane == 0) {
      const uint64_t pol = AGG_ONLY ? policy_evict_last() : policy_evict_first();
      constexpr uint32_t kQKTx = AGG_ONLY ? L::kQBytes : L::kQKBytes;
      int nq = 0, nv = 0;
      uint64_t t0 = globaltimer();
      uint32_t idle = 0;
      while (nq < n_it || nv < n_it) {
        bool progressed = false;
        if (nq < n_it &&
            (nq < NQK || mbar_test_wait(&empty_qk[nq % NQK], ((nq / NQK) - 1) & 1))) {
          const int st = nq % NQK;
          const int row0 = tile_of(nq) * kTile;
          uint8_t* q_s = qk_ring + st * L::kQKStage;
          uint8_t* k_s = q_s + L::kKOff;
          mbar_arrive_expect_tx(&full_qk[st], kQKTx);
#pragma unroll
          for (int b = 0; b < L::kQBoxes; ++b) {
            if (!AGG_ONLY)
              tma_load_3d(q_s + b * kBoxBytes, &tm_q, &full_qk[st], b * kBoxCols, row0, bh, pol);
            tma_load_3d(k_s + b * kBoxBytes, &tm_k, &full_qk[st], b * kBoxCols, row0, bh, pol);
          }
          ++nq;
          progressed = true;
        }
        if (nv < nq && (nv < NV || mbar_test_wait(&empty_v[nv % NV], ((nv / NV) - 1) & 1))) {
          const int st = nv % NV;
          const int row0 = tile_of(nv) * kTile;
          uint8_t* v_s = v_ring + st * L::kVBytes;
          mbar_arrive_expect_tx(&full_v[st], L::kVBytes);
#pragma unroll
          for (int b = 0; b < L::kVBoxes; ++b)
            tma_load_3d(v_s + b * kBoxBytes, &tm_v, &full_v[st], mb * MB + b * kBoxCols, row0,
                        bh, pol);
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
        for (int j = max(0, nq - NQK); j < nq; ++j)
          mbar_wait_timeout(&full_qk[j % NQK], (j / NQK) & 1, CP_WAIT_TIMEOUT_NS);
        for (int j = max(0, nv - NV); j < nv; ++j)
          mbar_wait_timeout(&full_v[j % NV], (j / NV) & 1, CP_WAIT_TIMEOUT_NS);
      }
    }
  } else if (warp == 1 || warp == kBWarp || warp == kCWarp) {
    // ------------------------------------------------------------ MMA issuers
    // Issuer A (warp 1): the state chain S(t) and the inter-tile read-out
    // Q S(t) into output buffer t % NO.  Issuer B (warp kBWarp): P(t) =
    // Q K^T.  Issuer C (warp kCWarp): the intra-tile P V(t), accumulated onto
    // Q S(t) once that has completed, so the order of the sums is fixed.
    // With NO buffers the read-out of a tile never holds up the next one.  A
    // ring stage is released by a commit from each of its two users.
    if (lane == 0 && (warp == 1 || !AGG_ONLY)) {
      constexpr uint32_t idesc_p = idesc_bf16_f32(128, 128, 0, 0);   // Q . K^T
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, MB, 1, 1);    // K^T . V
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, MB, 0, 1);    // P . V, Q . S
      constexpr uint32_t kHi = desc_hi(1024);  // SBO = 1024, 128-byte swizzle
      const uint32_t t_s = tmem + L::kColS;
      auto t_out = [&](int it) { return tmem + L::kColO + (it % NO) * MB; };
      const uint32_t s_addr = smem_u32(s_tile);
      auto qk_addr = [&](int it) { return smem_u32(qk_ring + (it % NQK) * L::kQKStage); };
      auto v_addr = [&](int it) { return smem_u32(v_ring + (it % NV) * L::kVBytes); };
      // Descriptor low words advance by (byte offset >> 4) per K step.
      auto issue_s = [&](int it) {
        // S += K^T V (A = K^T and B = V, both MN-major), one 128-row block of
        // the state per 128 columns of K
        const uint32_t kt_lo = desc_lo(qk_addr(it) + L::kKOff, kBoxBytes);
        const uint32_t v_lo = desc_lo(v_addr(it), kBoxBytes);
        const bool fresh = (it == 0) && !has_init;
#pragma unroll
        for (int sb = 0; sb < L::kSBlocks; ++sb) {
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            mma_ss_lo<kHi, kHi>(t_s + sb * MB, kt_lo + ((2 * sb * kBoxBytes + kk * 2048) >> 4),
                                v_lo + ((kk * 2048) >> 4), idesc_s, (fresh && kk == 0) ? 0u : 1u);
          }
        }
      };
      bool ok = true;
      uint64_t t0 = globaltimer();
      uint32_t idle = 0;
      auto idle_tick = [&](bool progressed) -> bool {  // false: give up
        if (progressed) {
          idle = 0;
        } else if ((++idle & 63u) == 0) {
          if (idle == 64) t0 = globaltimer();
          if (*abort_flag || globaltimer() - t0 > CP_WAIT_TIMEOUT_NS) return false;
        }
        return true;
      };
      if (AGG_ONLY) {
        for (int it = 0; it < n_it; ++it) {
          if (!mbar_wait_t<kOutlineWaits>(&qk_bar[it % NQK], (it / NQK) & 1, abort_flag) ||
              !mbar_wait_t<kOutlineWaits>(&v_bar[it % NV], (it / NV) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(it);
          mma_commit(&empty_qk[it % NQK]);
          mma_commit(&empty_v[it % NV]);
        }
        if (ok) mma_commit(s_done);
      } else if (warp == 1) {
        // issuer A: S(t) needs Q/K(t), V(t) landed and the state copied out
        // (s_ready); Q S(t) needs S(t) issued and output buffer t % NO read
        // out for t - NO.
        int nS = 0, nQ = 0;
        while (nQ < n_it) {
          bool progressed = false;
          if (nS < n_it && mbar_test_wait(&qk_bar[nS % NQK], (nS / NQK) & 1) &&
              mbar_test_wait(&v_bar[nS % NV], (nS / NV) & 1) &&
              mbar_test_wait(s_ready, nS & 1)) {
            tc_fence_after();
            issue_s(nS);
            mma_commit(s_done);
            mma_commit(&empty_v[nS % NV]);
            ++nS;
            progressed = true;
          }
          if (nQ < nS &&
              (nQ < NO || mbar_test_wait(&o_free[nQ % NO], ((nQ - NO) / NO) & 1))) {
            tc_fence_after();
            const uint32_t q_lo = desc_lo(qk_addr(nQ), 16);
            const uint32_t s_lo = desc_lo(s_addr + (nQ % NSB) * L::kSBufBytes, DP * 128);
            // O(t) = Q S_hi (+ Q S_lo) into a free output buffer; P V(t)
            // accumulates on top once this has completed
#pragma unroll
            for (int part = 0; part < (L::kSplit ? 2 : 1); ++part) {
#pragma unroll
              for (int kk = 0; kk < DP / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
                mma_ss_lo<kHi, kHi>(t_out(nQ), q_lo + off,
                                    s_lo + ((part * L::kSOneBytes + kk * 2048) >> 4), idesc_o,
                                    (part == 0 && kk == 0) ? 0u : 1u);
              }
            }
            mma_commit(&qs_done[nQ % NSB]);
            mma_commit(&o_qs[nQ % NO]);
            mma_commit(&empty_qk[nQ % NQK]);
            ++nQ;
            progressed = true;
          }
          if (!idle_tick(progressed)) { ok = false; break; }
        }
      } else if (warp == kBWarp) {
        // issuer B: P(t) needs Q/K(t) landed and P buffer t%NP free (P V of
        // tile t - NP completed)
        for (int it = 0; it < n_it; ++it) {
          if (!mbar_wait_t<kOutlineWaits>(&qk_bar[it % NQK], (it / NQK) & 1, abort_flag) ||
              (it >= NP && !mbar_wait_t<kOutlineWaits>(&pv_done[it % NP], ((it - NP) / NP) & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t q_lo = desc_lo(qk_addr(it), 16);
          const uint32_t k_lo = desc_lo(qk_addr(it) + L::kKOff, 16);
          const uint32_t t_p = tmem + L::kColP + (it % NP) * 128;
#pragma unroll
          for (int kk = 0; kk < DP / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
            mma_ss_lo<kHi, kHi>(t_p, q_lo + off, k_lo + off, idesc_p, kk > 0);
          }
          mma_commit(&p_done[it % NP]);
          mma_commit(&empty_qk[it % NQK]);
        }
      } else {
        // issuer C: P V(t) needs P(t) packed, V(t) landed and Q S(t)
        // completed in the output buffer it accumulates onto
        for (int it = 0; it < n_it; ++it) {
          const int b = it % NP;
          if (!mbar_wait_t<kOutlineWaits>(&p_ready[b], (it / NP) & 1, abort_flag) ||
              !mbar_wait_t<kOutlineWaits>(&v_bar[it % NV], (it / NV) & 1, abort_flag) ||
              !mbar_wait_t<kOutlineWaits>(&o_qs[it % NO], (it / NO) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t t_p = tmem + L::kColP + b * 128;
          const uint32_t v_lo = desc_lo(v_addr(it), kBoxBytes);
          // O(t) += P_hi V (+ P_lo V) (A = packed bf16 P in TMEM, B = V
          // MN-major).  Chunk c of P (columns 32c..32c+31) holds hi in its
          // first 16 TMEM columns and lo in the next 16, two j per column.
#pragma unroll
          for (int part = 0; part < kPParts; ++part) {
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
              const uint32_t acol = (kk >> 1) * 32 + part * 16 + (kk & 1) * 8;
              mma_ts_lo<kHi>(t_out(it), t_p + acol, v_lo + ((kk * 2048) >> 4), idesc_o, 1u);
            }
          }
          mma_commit(&pv_done[b]);
          mma_commit(&o_done[it % NO]);
          mma_commit(&empty_v[it % NV]);
        }
      }
      if (!ok) record_timeout(a.status, abort_flag);
      // every MMA this thread issued completes before TMEM is released
      uint64_t* my_fin = &fin[warp == 1 ? 0 : (warp == kBWarp ? 1 : 2)];
      mma_commit(my_fin);
      mbar_wait_timeout(my_fin, 0, CP_WAIT_TIMEOUT_NS);
    }
  } else if (warp < kPWarp0) {
    // ------------------------------------------------------------ state group
    bool ok = true;
    if (AGG_ONLY) {
      for (int it = 0; FEAT && it < n_it && ok; ++it) ok = map_qk(it, threadIdx.x - 32 * kSWarp0);
      for (int it = 0; FEAT_V && it < n_it && ok; ++it) ok = map_v(it, threadIdx.x - 32 * kSWarp0);
      if (!ok) {
        record_timeout(a.status, abort_flag);
      } else if (!mbar_wait_t<kOutlineWaits>(s_done, 0, abort_flag)) {
        record_timeout(a.status, abort_flag);
      } else if (n_it > 0) {
        tc_fence_after();
        float* dst = a.agg_out + ((size_t)pidx * a.G + seg) * (size_t)DP * MB;
#pragma unroll
        for (int sb = 0; sb < L::kSBlocks; ++sb) {
          if (sb * 128 + wq * 32 >= DP) continue;  // warp-uniform
          const int d = sb * 128 + row;
#pragma unroll
          for (int c = 0; c < MB / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(lane_base + L::kColS + sb * MB + c * 32, r);
            tmem_ld_wait();
            float4* o4 = reinterpret_cast<float4*>(dst + (size_t)d * MB + c * 32);
#pragma unroll
            for (int x = 0; x < 8; ++x)
              o4[x] = make_float4(__uint_as_float(r[4 * x]), __uint_as_float(r[4 * x + 1]),
                                  __uint_as_float(r[4 * x + 2]), __uint_as_float(r[4 * x + 3]));
          }
        }
      }
    } else if (kVMapS && wq >= 2) {
      // the value map (no state rows in these lane quarters)
      for (int it = 0; it < n_it && ok; ++it) ok = map_v(it, row - 64);
      if (!ok) record_timeout(a.status, abort_flag);
    } else {
      // initial state: the carried state plus the sum of the preceding
      // segments' aggregates (slot seg of agg_in, prefixed between passes)
      if (has_init) {
        const int lo = has_prefix ? seg : 0;
        const int hi = has_prefix ? seg + 1 : 0;
        const float* st = a.state_in != nullptr ? a.state_in + (int64_t)bh * a.Dr * a.Mc : nullptr;
        if constexpr (SEED) {
          if (seeded)
            st = a.seed + (int64_t)bh * a.seed_bh + (int64_t)(seg + a.seed_seg_off) * a.seed_seg;
        }
#pragma unroll
        for (int sb = 0; sb < L::kSBlocks; ++sb) {
          if (sb * 128 + wq * 32 >= DP) continue;
          const int d = sb * 128 + row;
#pragma unroll
          for (int c = 0; c < MB / 32; ++c) {
            float acc[32];
            // columns m0 + x of row d of the carried state
            const int m0 = mb * MB + c * 32;
            const int nm = (st != nullptr && d < a.Dr) ? min(32, a.Mc - m0) : 0;
            const float* src = st + d * a.st_ld_r + m0 * a.st_ld_c;
#pragma unroll
            for (int x = 0; x < 32; ++x) acc[x] = x < nm ? src[x * a.st_ld_c] : 0.f;
            for (int s2 = lo; s2 < hi; ++s2) {
              const float4* src = reinterpret_cast<const float4*>(
                  a.agg_in + (((size_t)pidx * a.G + s2) * DP + d) * MB + c * 32);
#pragma unroll
              for (int x = 0; x < 8; ++x) {
                // (coherent loads: the one-launch split scan writes the
                // slot within the same launch)
                const float4 f = __ldcg(src + x);
                acc[4 * x] += f.x;
                acc[4 * x + 1] += f.y;
                acc[4 * x + 2] += f.z;
                acc[4 * x + 3] += f.w;
              }
            }
            uint32_t r[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) r[x] = __float_as_uint(acc[x]);
            tmem_st32(lane_base + L::kColS + sb * MB + c * 32, r);
          }
        }
        tmem_st_wait();
      }
      if (NORM) {
        for (int d = threadIdx.x - 32 * kSWarp0; d < DP; d += 32 * kSWarps) z_sk[d] = 0.f;
        named_barrier_sync(2, 32 * kSWarps);
      }
      for (int it = 0; it < n_it && ok; ++it) {
        const int b = it % NSB;
        uint8_t* sbuf = s_tile + b * L::kSBufBytes;
        // the Q S that last read this copy (tile it - NSB) has completed
        if (it >= NSB && !mbar_wait_t<kOutlineWaits>(&qs_done[b], ((it - NSB) / NSB) & 1, abort_flag)) {
          ok = false;
          break;
        }
        if (it == 0 && !has_init) {
#pragma unroll
          for (int sb = 0; sb < L::kSBlocks; ++sb) {
            if (sb * 128 + wq * 32 >= DP) continue;
#pragma unroll
            for (int c = 0; c < MB / 32; ++c) {
              store_zero32(sbuf, sb * 128 + row, c * 32, DP * 128);
              if (L::kSplit) store_zero32(sbuf + L::kSOneBytes, sb * 128 + row, c * 32, DP * 128);
            }
          }
        } else {
          if (it > 0) {
            if (!mbar_wait_t<kOutlineWaits>(s_done, (it - 1) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
          }
#pragma unroll
          for (int sb = 0; sb < L::kSBlocks; ++sb) {
            if (sb * 128 + wq * 32 >= DP) continue;
#pragma unroll
            for (int c = 0; c < MB / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(lane_base + L::kColS + sb * MB + c * 32, r);
              tmem_ld_wait();
              if (L::kSplit)
                store_chunk32_split(sbuf, sbuf + L::kSOneBytes, sb * 128 + row, c * 32, DP * 128,
                                    r);
              else
                store_chunk32(sbuf, sb * 128 + row, c * 32, DP * 128, r);
            }
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_ready);
        if constexpr (NORM) {
          // q_i . s_k for the tile's rows (thread = row), then s_k takes the
          // tile's k: column sums over 64 rows each by the warps of lane
          // quarters 2 and 3 (no state rows at D <= 64), lane l owning
          // columns 2l, 2l + 1, four interleaved partial sums; fixed order
          const int st = it % NQK;
          if (!mbar_wait_t<kOutlineWaits>(&full_qk[st], (it / NQK) & 1, abort_flag) ||
              (it > 0 && !mbar_wait_t<kOutlineWaits>(zq_free, (it - 1) & 1, abort_flag))) {
            ok = false;
            break;
          }
          const uint8_t* q_s = qk_ring + st * L::kQKStage;
          const uint8_t* k_s = q_s + L::kKOff;
          float qd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            const uint4 w =
                *reinterpret_cast<const uint4*>(q_s + sw128_offset(row, 8 * c8, kBoxBytes));
            const float4* skc = reinterpret_cast<const float4*>(z_sk + 8 * c8);
            const float4 s0 = skc[0], s1 = skc[1];
            qd[0] = fmaf(__uint_as_float(w.x << 16), s0.x, qd[0]);
            qd[1] = fmaf(__uint_as_float(w.x & 0xffff0000u), s0.y, qd[1]);
            qd[2] = fmaf(__uint_as_float(w.y << 16), s0.z, qd[2]);
            qd[3] = fmaf(__uint_as_float(w.y & 0xffff0000u), s0.w, qd[3]);
            qd[0] = fmaf(__uint_as_float(w.z << 16), s1.x, qd[0]);
            qd[1] = fmaf(__uint_as_float(w.z & 0xffff0000u), s1.y, qd[1]);
            qd[2] = fmaf(__uint_as_float(w.w << 16), s1.z, qd[2]);
            qd[3] = fmaf(__uint_as_float(w.w & 0xffff0000u), s1.w, qd[3]);
          }
          const float qdot = (qd[0] + qd[1]) + (qd[2] + qd[3]);
          z_q[row] = qdot;
          float cs0 = 0.f, cs1 = 0.f;
          if (wq >= 2) {  // warp-uniform
            float acc[4][2] = {};
#pragma unroll 4
            for (int r = 64 * (wq - 2); r < 64 * (wq - 2) + 64; r += 4) {
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(
                    k_s + sw128_offset(r + u, 2 * lane, kBoxBytes));
                acc[u][0] += __uint_as_float(w << 16);
                acc[u][1] += __uint_as_float(w & 0xffff0000u);
              }
            }
            cs0 = (acc[0][0] + acc[1][0]) + (acc[2][0] + acc[3][0]);
            cs1 = (acc[0][1] + acc[1][1]) + (acc[2][1] + acc[3][1]);
            if (wq == 3) {  // rows 64..127, for quarter 2 to add
              z_part[2 * lane] = cs0;
              z_part[2 * lane + 1] = cs1;
            }
          }
          // this warp's reads of the stage are done: hand it back
          asm volatile("" ::"f"(qdot + cs0 + cs1));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&empty_qk[st]);
            mbar_arrive(zq_ready);
          }
          named_barrier_sync(2, 32 * kSWarps);  // every read of s_k done; rows 64..127 summed
          if (wq == 2) {
            z_sk[2 * lane] += cs0 + z_part[2 * lane];
            z_sk[2 * lane + 1] += cs1 + z_part[2 * lane + 1];
          }
          named_barrier_sync(2, 32 * kSWarps);  // s_k advanced before the next tile reads it
        }
        // CKPT: the state before this tile is a checkpoint.  It is written
        // off the state chain, after the copy is handed on, from the hi + lo
        // copy this thread wrote (hi + lo carries 16 significant bits: the
        // precision the Q S operands use), which stays put until the copy
        // after the next NSB - 1 tiles.
        if (CKPT && L::kSplit && it > 0) {
          const int slot = ckpt_slot(tile_of(it));
          if (slot > 0) {
#pragma unroll 1
            for (int sb = 0; sb < L::kSBlocks; ++sb) {
              const int d = sb * 128 + row;
              if (sb * 128 + wq * 32 >= DP || d >= a.Dr) continue;
#pragma unroll 1
              for (int c8 = 0; c8 < MB / 8; ++c8) {
                const int m0 = mb * MB + c8 * 8;
                if (m0 + 8 > a.Mc) break;
                const uint32_t off = sw128_offset(d, c8 * 8, DP * 128);
                const uint4 h = *reinterpret_cast<const uint4*>(sbuf + off);
                const uint4 l = *reinterpret_cast<const uint4*>(sbuf + L::kSOneBytes + off);
                const uint32_t hw[4] = {h.x, h.y, h.z, h.w}, lw[4] = {l.x, l.y, l.z, l.w};
                float f[8];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  f[2 * u] = __uint_as_float(hw[u] << 16) + __uint_as_float(lw[u] << 16);
                  f[2 * u + 1] = __uint_as_float(hw[u] & 0xffff0000u) +
                                 __uint_as_float(lw[u] & 0xffff0000u);
                }
                float4* dst = reinterpret_cast<float4*>(ckpt_row(slot, d, m0));
                dst[0] = make_float4(f[0], f[1], f[2], f[3]);
                dst[1] = make_float4(f[4], f[5], f[6], f[7]);
              }
            }
          }
        }

      }
      // CKPT: a checkpoint boundary right after this segment's last tile
      // (the state is exact here: no copy follows it)
      if (CKPT && ok && n_it > 0 && ckpt_slot(tile_of(n_it - 1) + 1) > 0) {
        if (!mbar_wait_t<kOutlineWaits>(s_done, (n_it - 1) & 1, abort_flag)) {
          ok = false;
        } else {
          tc_fence_after();
          const int slot = ckpt_slot(tile_of(n_it - 1) + 1);
#pragma unroll 1
          for (int sb = 0; sb < L::kSBlocks; ++sb) {
            const int d = sb * 128 + row;
            if (sb * 128 + wq * 32 >= DP) continue;  // warp-uniform
#pragma unroll 1
            for (int c = 0; c < MB / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(lane_base + L::kColS + sb * MB + c * 32, r);
              tmem_ld_wait();
              const int m0 = mb * MB + c * 32;
              if (d >= a.Dr) continue;
#pragma unroll
              for (int x8 = 0; x8 < 4; ++x8) {
                if (m0 + 8 * x8 + 8 > a.Mc) break;
                float4* dst = reinterpret_cast<float4*>(ckpt_row(slot, d, m0 + 8 * x8));
                dst[0] = make_float4(__uint_as_float(r[8 * x8]), __uint_as_float(r[8 * x8 + 1]),
                                     __uint_as_float(r[8 * x8 + 2]), __uint_as_float(r[8 * x8 + 3]));
                dst[1] = make_float4(__uint_as_float(r[8 * x8 + 4]), __uint_as_float(r[8 * x8 + 5]),
                                     __uint_as_float(r[8 * x8 + 6]), __uint_as_float(r[8 * x8 + 7]));
              }
            }
          }
        }
      }
      // the last segment in scan order hands on the state after its last tile
      if (STATE_OUT && ok && last_seg && n_it > 0) {
        if (!mbar_wait_t<kOutlineWaits>(s_done, (n_it - 1) & 1, abort_flag)) {
          ok = false;
        } else {
          tc_fence_after();
          float* st = a.state_out + (int64_t)bh * a.Dr * a.Mc;
#pragma unroll
          for (int sb = 0; sb < L::kSBlocks; ++sb) {
            if (sb * 128 + wq * 32 >= DP) continue;  // warp-uniform
            const int d = sb * 128 + row;
#pragma unroll 1
            for (int c = 0; c < MB / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(lane_base + L::kColS + sb * MB + c * 32, r);
              tmem_ld_wait();
              const int m0 = mb * MB + c * 32;
              const int nm = d < a.Dr ? min(32, a.Mc - m0) : 0;
              float* dst = st + d * a.st_ld_r + m0 * a.st_ld_c;
#pragma unroll
              for (int x = 0; x < 32; ++x)
                if (x < nm) dst[x * a.st_ld_c] = __uint_as_float(r[x]);
            }
          }
        }
      }
      if (!ok) record_timeout(a.status, abort_flag);
    }
  } else if (warp < kOWarp0) {
    // ------------------------------------------------------------ P group
    // P of tile it: mask to the causal triangle of the tile, split into bf16
    // hi + lo and pack back into the chunk's own TMEM columns: chunk c
    // (j in [32c, 32c+32)) -> hi at 32c + [0,16), lo at 32c + [16,32), two j
    // per 32-bit column.
    bool ok = true;
    for (int it = 0; !AGG_ONLY && it < n_it && ok; ++it) {
      const int b = it % NP;
      if (!mbar_wait_t<kOutlineWaits>(&p_done[b], (it / NP) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t pc = lane_base + L::kColP + b * 128;
      float zrow = 0.f;  // NORM: sum over the row's unmasked fp32 entries, in column order
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const bool z = a.reverse ? (c < wq) : (c > wq);  // chunk entirely masked
        uint32_t r[32];
        if (!z) {
          tmem_ld32(pc + 32 * c, r);
          tmem_ld_wait();
          if (NORM) {
            // the chunk's kept entries summed as a pairwise tree (forward
            // mask: all of a chunk left of the diagonal, columns x <= lane of
            // the diagonal chunk)
            float t[16];
            if (c == wq) {  // warp-uniform
#pragma unroll
              for (int x = 0; x < 16; ++x)
                t[x] = (2 * x <= lane ? __uint_as_float(r[2 * x]) : 0.f) +
                       (2 * x + 1 <= lane ? __uint_as_float(r[2 * x + 1]) : 0.f);
            } else {
#pragma unroll
              for (int x = 0; x < 16; ++x) t[x] = __uint_as_float(r[2 * x]) + __uint_as_float(r[2 * x + 1]);
            }
#pragma unroll
            for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
              for (int x = 0; x < w; ++x) t[x] += t[x + w];
            zrow += t[0];
          }
        }
        split_pack_p(r, z, c == wq, lane, a.reverse);
        store_packed_p(pc + 32 * c, r);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_ready[b]);
      if constexpr (NORM) {
        // z_i = (row sum of P: the terms j of this tile) + q_i . s_k
        if (!mbar_wait_t<kOutlineWaits>(zq_ready, it & 1, abort_flag)) {
          ok = false;
          break;
        }
        const float zval = zrow + z_q[row];
        __syncwarp();
        if (lane == 0) mbar_arrive(zq_free);
        const int64_t grow = (int64_t)tile_of(it) * kTile + row;
        if (grow < a.N) a.z[(int64_t)bh * a.N + grow] = zval;
      }
    }
    if (!ok) record_timeout(a.status, abort_flag);
  } else {
    // ------------------------------------------------------------ O group
    const int o_tid = threadIdx.x - 32 * kOWarp0;   // 0..kOThreads-1
    bool ok = true;
    // EPI: the raw rows of tile j go by TMA into staging buffer j % kOBufs
    // (the output's box layout) once the store of tile j - kOBufs has read
    // it; the read-out multiplies each value by phi'(x) of the element at
    // its own staging position and stores the product there
    [[maybe_unused]] int x_next = 0;
    [[maybe_unused]] auto epi_load = [&]() {
      if constexpr (EPI) {
        const int b = x_next % L::kOBufs;
        uint8_t* xb = o_tile + b * L::kOBytes;
        mbar_arrive_expect_tx(&x_full[b], L::kOBytes);
#pragma unroll
        for (int bx = 0; bx < L::kVBoxes; ++bx)
          tma_load_3d(xb + bx * kBoxBytes, tm_x, &x_full[b], mb * MB + bx * kBoxCols,
                      tile_of(x_next) * kTile, bh, policy_evict_first());
        ++x_next;
      }
    };
    if (EPI && o_tid == 0 && n_it > 0 && !AGG_ONLY) epi_load();
    // FEAT: the O group maps every tile, tile it + kAhead before the
    // read-out of tile it
    for (int j = 0; FEAT && !AGG_ONLY && j < kAhead && j < n_it && ok; ++j)
      ok = map_qk(j, o_tid);
    for (int j = 0; FEAT_V && !kVMapS && !AGG_ONLY && j < kAheadV && j < n_it && ok; ++j)
      ok = map_v(j, o_tid);
    for (int it = 0; !AGG_ONLY && it < n_it && ok; ++it) {
      if (FEAT && it + kAhead < n_it && !map_qk(it + kAhead, o_tid)) {
        ok = false;
        break;
      }
      if (FEAT_V && !kVMapS && it + kAheadV < n_it && !map_v(it + kAheadV, o_tid)) {
        ok = false;
        break;
      }
      if (EPI && L::kOBufs == 2 && o_tid == 0 && it + 1 < n_it) {
        // the other buffer's last store (tile it - 1) has been read
        tma_store_wait_read_all();
        epi_load();
      }
      uint8_t* ob = o_tile + (it % L::kOBufs) * L::kOBytes;
      if (!mbar_wait_t<kOutlineWaits>(&o_done[it % NO], (it / NO) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t t_o = lane_base + L::kColO + (it % NO) * MB;
      auto wait_staging = [&]() {
        // the store that last read this staging buffer has finished reading it
        if (o_tid == 0) {
          if (L::kOBufs == 2)
            asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          else
            tma_store_wait_read_all();
        }
        named_barrier_sync(1, kOThreads);
      };
      // a chunk of 32 columns at a time, one copy of the conversion in the
      // instruction stream (reading the whole row first, then releasing the
      // buffer, measured slower in the one-launch backward, whose two scan
      // bodies share the instruction cache: 127.1 against 124.6 us; the
      // feature backward 192 against 181 us)
      if constexpr (EPI) {
        if (!mbar_wait_t<kOutlineWaits>(&x_full[it % L::kOBufs], (it / L::kOBufs) & 1, abort_flag)) {
          ok = false;
          break;
        }
      } else {
        wait_staging();
      }
#pragma unroll 1
      for (int c = 0; c < MB / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(t_o + c * 32, r);
        tmem_ld_wait();
        if constexpr (EPI)
          scale_store_chunk32(ob, row, c * 32, kBoxBytes, r);
        else
          store_chunk32(ob, row, c * 32, kBoxBytes, r);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[it % NO]);
      fence_proxy_async_smem();
      named_barrier_sync(1, kOThreads);
      if (o_tid == 0) {
        const int tile = tile_of(it);
#pragma unroll
        for (int bx = 0; bx < L::kVBoxes; ++bx)
          tma_store_3d(&tm_o, ob + bx * kBoxBytes, mb * MB + bx * kBoxCols, tile * kTile, bh);
        tma_store_commit();
        if (EPI && L::kOBufs == 1 && it + 1 < n_it) {
          tma_store_wait_read_all();
          epi_load();
        }
      }
    }
    if (!ok) record_timeout(a.status, abort_flag);
    if (EPI && o_tid == 0) {
      // raw-row loads still in flight land before the CTA's memory goes away
      for (int j = x_next - L::kOBufs; j < x_next; ++j)
        if (j >= 0) mbar_wait_timeout(&x_full[j % L::kOBufs], (j / L::kOBufs) & 1,
                                      CP_WAIT_TIMEOUT_NS);
    }
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
    tmem_dealloc(tmem, L::kColsAlloc);
  }
  const bool completed = *abort_flag == 0;
  if (!ph.last) {
    // a later scan of this CTA reuses the barriers' memory
    __syncthreads();
    if (threadIdx.x == 0) {
      for (uint64_t* b = bars; b < fin + 3; ++b) mbar_inval(b);
      if (FEAT)
        for (int i = 0; i < NQK; ++i) mbar_inval(&qk_ready[i]);
      if (FEAT_V)
        for (int i = 0; i < NV; ++i) mbar_inval(&v_ready[i]);
      if (EPI)
        for (int i = 0; i < L::kOBufs; ++i) mbar_inval(&x_full[i]);

    }
    __syncthreads();
  }
  return completed;
}

// The split forward scan in one launch (csrc/cp_tc_lookback.cu): a.agg_out
// the segments' sums and a.agg_in their prefixes, each [P][G][DP][MB];
// a.lb_flags [P][G] cleared; grid P * G CTAs, all resident at once.  Plain
// and checkpoint scans.
cudaError_t lookback_launch(int DP, int MB, const CUtensorMap& q, const CUtensorMap& k,
                            const CUtensorMap& v, const CUtensorMap& o, const ArgsX& a,
                            unsigned grid, cudaStream_t st);

}  // namespace tc
}  // namespace cp
