// Pieces shared by the tensor-core kernels: tile geometry, the 128-byte
// swizzled tile layout, bf16 conversion and hi/lo splitting, the in-TMEM
// packing of the intra-tile matrix P, timeout reporting and TMA maps.
#pragma once
#include <cstdint>
#include <mutex>

#include <cudaTypedefs.h>

#include "cp_internal.h"
#include "sm103_ptx.cuh"

namespace cp {
namespace tc {

constexpr int kTile = 128;             // rows per tile = MMA M
constexpr int kBoxCols = 64;           // bf16 columns per TMA box (128 bytes)
constexpr int kBoxBytes = kTile * 128; // one [128 x 64] bf16 box
constexpr int kSmemLimit = 232448;     // 227 KB opt-in dynamic shared memory

// One scan a CTA runs.  A CTA may run several scans one after another (the
// backward kernel does); `work` replaces the block index, `first` makes the
// scan wait for the previous kernel in the stream (and then let dependents
// start), `last` gives up the CTA's permit to allocate tensor memory and
// skips the barrier clean-up that lets a later scan reuse the memory.
struct Phase {
  int work;
  bool first;
  bool last;
};

// Byte offset of element (row, col) inside a [rows x 64k] bf16 tile stored
// as 64-column boxes of `box_stride` bytes with the 128-byte swizzle (the
// layout TMA writes and tcgen05 descriptors read): 16-byte chunk index
// XOR row % 8.
__device__ __forceinline__ uint32_t sw128_offset(int row, int col, int box_stride) {
  const int box = col >> 6;
  const int chunk = (col & 63) >> 3;
  return box * box_stride + row * 128 + ((chunk ^ (row & 7)) << 4) + ((col & 7) << 1);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Convert 32 fp32 values (columns col0..col0+31 of `row`) to bf16 and store
// them into a swizzled tile; col0 must be a multiple of 32.
__device__ __forceinline__ void store_chunk32(uint8_t* tile, int row, int col0, int box_stride,
                                              const uint32_t (&r)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 w;
    w.x = pack_bf16x2(__uint_as_float(r[8 * c + 0]), __uint_as_float(r[8 * c + 1]));
    w.y = pack_bf16x2(__uint_as_float(r[8 * c + 2]), __uint_as_float(r[8 * c + 3]));
    w.z = pack_bf16x2(__uint_as_float(r[8 * c + 4]), __uint_as_float(r[8 * c + 5]));
    w.w = pack_bf16x2(__uint_as_float(r[8 * c + 6]), __uint_as_float(r[8 * c + 7]));
    *reinterpret_cast<uint4*>(tile + sw128_offset(row, col0 + 8 * c, box_stride)) = w;
  }
}

// Split 32 fp32 values into hi = bf16(x) and lo = bf16(x - hi) and store
// both (hi into `hi_tile`, lo into `lo_tile`, same swizzled layout).
__device__ __forceinline__ void store_chunk32_split(uint8_t* hi_tile, uint8_t* lo_tile, int row,
                                                    int col0, int box_stride,
                                                    const uint32_t (&r)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float a = __uint_as_float(r[8 * c + 2 * x]);
      const float b = __uint_as_float(r[8 * c + 2 * x + 1]);
      h[x] = pack_bf16x2(a, b);
      const float ah = __uint_as_float(h[x] << 16);
      const float bh = __uint_as_float(h[x] & 0xffff0000u);
      l[x] = pack_bf16x2(a - ah, b - bh);
    }
    const uint32_t off = sw128_offset(row, col0 + 8 * c, box_stride);
    *reinterpret_cast<uint4*>(hi_tile + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo_tile + off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

__device__ __forceinline__ void store_zero32(uint8_t* tile, int row, int col0, int box_stride) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(tile + sw128_offset(row, col0 + 8 * c, box_stride)) =
        make_uint4(0, 0, 0, 0);
}

// P = Q K^T is rounded to bf16 for the P V product either once (hi) or as
// hi + lo (lo = bf16(P - hi)), which doubles the P V MMAs.
constexpr bool kSplitP = true;
constexpr int kPParts = kSplitP ? 2 : 1;

// In place: mask a 32-column chunk of P to the causal triangle of the tile
// (only the diagonal chunk needs it; an entirely masked chunk becomes zero)
// and round to bf16 pairs: columns 0..15 <- hi pairs, and with the split
// columns 16..31 <- lo pairs.
__device__ __forceinline__ void split_pack_p(uint32_t (&r)[32], bool zero, bool diag, int lane,
                                             int reverse) {
  if (zero) {
#pragma unroll
    for (int x = 0; x < 32; ++x) r[x] = 0u;
    return;
  }
  if (diag) {
#pragma unroll
    for (int x = 0; x < 32; ++x) {
      const bool keep = reverse ? (x >= lane) : (x <= lane);
      if (!keep) r[x] = 0u;
    }
  }
  // hi of pair x goes to r[x] (already consumed), lo waits in a 16-entry
  // temporary until the pairs it would overwrite are consumed
  uint32_t lo[16];
#pragma unroll
  for (int x = 0; x < 16; ++x) {
    const float a0 = __uint_as_float(r[2 * x]), a1 = __uint_as_float(r[2 * x + 1]);
    const uint32_t h = pack_bf16x2(a0, a1);
    if (kSplitP)
      lo[x] = pack_bf16x2(a0 - __uint_as_float(h << 16), a1 - __uint_as_float(h & 0xffff0000u));
    r[x] = h;
  }
  if (kSplitP) {
#pragma unroll
    for (int x = 0; x < 16; ++x) r[16 + x] = lo[x];
  }
}

// Store a packed chunk back to its TMEM columns (16 or 32 of them).
__device__ __forceinline__ void store_packed_p(uint32_t taddr, const uint32_t (&r)[32]) {
  if (kSplitP)
    cp::ptx::tmem_st32(taddr, r);
  else
    cp::ptx::tmem_st16(taddr, r);
}

// Hand a shared-memory stage this thread has read with ordinary loads back
// to the TMA engine, which will overwrite it: every reading thread orders
// its loads before the async proxy's later writes (fence.proxy.async) and
// arrives itself (the barrier counts every reader).  `v` is a value computed
// from the loads, so they have returned before the fence.  (A single lane
// arriving after __syncwarp let the next tile's TMA load overwrite rows some
// lanes were still reading.)
__device__ __forceinline__ void release_to_tma(uint64_t* bar, float v) {
  asm volatile("" ::"f"(v));
  cp::ptx::fence_proxy_async_smem();
  cp::ptx::mbar_arrive(bar);
}

__device__ __forceinline__ void record_timeout(int* status, volatile int* abort_flag) {
  *abort_flag = 1;
  if (status != nullptr) atomicCAS(status, 0, (int)CP_ERR_TIMEOUT);
}

// ------------------------------------------------------------------ host
inline PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [BH][N][cols] bf16, boxes of 64 columns x 128 rows x 1 problem, 128-byte
// swizzle.  `pitch` (elements between rows, 0: cols) lets the map cover the
// first `cols` columns of wider rows.
inline bool make_map(CUtensorMap* m, const void* ptr, int64_t BH, int64_t N, int64_t cols,
                     int64_t pitch = 0) {
  auto enc = get_encode();
  if (enc == nullptr) return false;
  if (pitch == 0) pitch = cols;
  if (pitch < cols) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)pitch * 2, (cuuint64_t)(N * pitch * 2)};
  cuuint32_t box[3] = {(cuuint32_t)kBoxCols, (cuuint32_t)kTile, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// phi(x) = elu(x) + 1 on a pair of bf16 values, in packed bf16x2
// arithmetic: phi(x) = e^min(x, 0) + max(x, 0), with min and max exact
// (NaN-propagating) and e^n = 2^(n log2 e) by the change of base.  log2 e
// is split into two bf16 parts (0x3fb9 = 1.4453125 and 0xbb2c =
// -0.00262451171875, together within 5e-6 of it) so the product n log2 e
// is rounded once, by the FMA; 2^y is the hardware base-2 exponential on
// bf16 pairs, and the sum is rounded to bf16 once.
__device__ __forceinline__ uint32_t elu1_bf16x2(uint32_t w) {
  constexpr uint32_t kLog2eHi = 0x3fb93fb9u, kLog2eLo = 0xbb2cbb2cu;
  uint32_t mn, mx, t, y, e, r;
  asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(mn) : "r"(w), "r"(0u));
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(mx) : "r"(w), "r"(0u));
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(t) : "r"(mn), "r"(kLog2eLo));
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(y) : "r"(mn), "r"(kLog2eHi), "r"(t));
  asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(e) : "r"(y));
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(e), "r"(mx));
  return r;
}

// e^min(x, 0) on a bf16 pair: phi'(x) for phi = elu + 1 (1 for x > 0, e^x
// otherwise), with the exponent formed as in elu1_bf16x2.
__device__ __forceinline__ uint32_t exp_min0_bf16x2(uint32_t w) {
  constexpr uint32_t kLog2eHi = 0x3fb93fb9u, kLog2eLo = 0xbb2cbb2cu;
  uint32_t mn, t, y, e;
  asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(mn) : "r"(w), "r"(0u));
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(t) : "r"(mn), "r"(kLog2eLo));
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(y) : "r"(mn), "r"(kLog2eHi), "r"(t));
  asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(e) : "r"(y));
  return e;
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// The chain rule of phi = elu + 1 on 32 fp32 values of a row: each value,
// rounded to bf16, times phi'(x) = e^min(x, 0) in bf16, x the bf16 element at
// the same position of a staged tile (the raw row), and the product stored
// over it (two bf16 roundings and the bf16 exponential: within the bf16
// output's own error).
__device__ __forceinline__ void scale_store_chunk32(uint8_t* tile, int row, int col0,
                                                    int box_stride, const uint32_t (&r)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4* p = reinterpret_cast<uint4*>(tile + sw128_offset(row, col0 + 8 * c, box_stride));
    const uint4 xw = *p;
    const uint32_t u[4] = {xw.x, xw.y, xw.z, xw.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      o[e] = mul_bf16x2(pack_bf16x2(__uint_as_float(r[8 * c + 2 * e]),
                                    __uint_as_float(r[8 * c + 2 * e + 1])),
                        exp_min0_bf16x2(u[e]));
    }
    *p = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// The same chain rule with phi'(x) = min(1, phi(x)) read from a staged
// tile of phi(x) (the mapped operand; 1 for x > 0, where phi(x) = x + 1 >=
// 1, and e^x otherwise), the product stored at the same position of `dst`.
__device__ __forceinline__ void scale_store_chunk32_phi(uint8_t* dst, const uint8_t* phi_tile,
                                                        int row, int col0, int box_stride,
                                                        const uint32_t (&r)[32]) {
  constexpr uint32_t kOnes = 0x3f803f80u;  // bf16 pair (1, 1)
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t off = sw128_offset(row, col0 + 8 * c, box_stride);
    const uint4 fw = *reinterpret_cast<const uint4*>(phi_tile + off);
    const uint32_t f[4] = {fw.x, fw.y, fw.z, fw.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t d;
      asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(f[e]), "r"(kOnes));
      o[e] = mul_bf16x2(pack_bf16x2(__uint_as_float(r[8 * c + 2 * e]),
                                    __uint_as_float(r[8 * c + 2 * e + 1])),
                        d);
    }
    *reinterpret_cast<uint4*>(dst + off) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace tc
}  // namespace cp
