// tc_tile.cuh -- 128 x 128 tile building blocks on tcgen05 shared by the
// threshold-attention forward and backward kernels.
//
// Tiles of 128 rows x D bf16 live in shared memory as D/64 panels of 128 rows
// x 128 bytes, written by TMA with 128-byte swizzle (1024-byte aligned).  One
// such tile serves both as a K-major operand (rows = M or N, D along K) and
// as an MN-major operand (rows along K, D along N).
#pragma once

#include "kernels.h"
#include "ptx.cuh"

namespace bsa {
namespace tile {

constexpr int ROWS = 128;               // rows of a tile (and keys/queries per MMA tile)
constexpr int PANEL_BYTES = 128 * 128;  // 128 rows x 128 B (64 bf16) swizzle panel

// C_tmem[128 x 128] = A[128 x D] * B[128 x D]^T, both K-major tiles in smem:
// D/16 MMAs of K = 16 (32 bytes of each 128-byte row).  `leader`: the one
// thread that issues; a converged warp computes the descriptors together
// (warp-uniform values) and only the leader issues -- measured to issue a
// tcgen05.mma every ~32 cycles, against ~48 for a lone thread that builds
// its own descriptors.
template <int D>
__device__ __forceinline__ void mma_abt(uint32_t tC, uint32_t sA, uint32_t sB, bool leader = true) {
  constexpr uint32_t IDESC = idesc_bf16_f32(ROWS, ROWS, 0, 0);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * PANEL_BYTES + (kk & 3) * 32;
    const uint64_t a = smem_desc_sw128(sA + off, 16, 1024), b = smem_desc_sw128(sB + off, 16, 1024);
    if (leader) mma_ss(tC, a, b, IDESC, kk > 0 ? 1u : 0u);
  }
}

// C_tmem[128 x D] (+)= P_tmem[128 x 128] * B[128 x D] for the K range
// [16*kk0, 16*kk1): P is bf16 packed two per TMEM column, B an MN-major tile
// in smem (its rows run along K).  `first` starts a new accumulation.
template <int D>
__device__ __forceinline__ void mma_tmem_a(uint32_t tC, uint32_t tP, uint32_t sB, int kk0, int kk1, bool first,
                                           bool leader = true) {
  constexpr uint32_t IDESC = idesc_bf16_f32(ROWS, D, 0, 1);
  constexpr int NP = D / 64;
#pragma unroll
  for (int kk = kk0; kk < kk1; ++kk) {
    const uint64_t bdesc = smem_desc_sw128(sB + kk * 16 * 128, NP > 1 ? PANEL_BYTES : 1024, 1024);
    if (leader) mma_ts(tC, tP + kk * 8, bdesc, IDESC, (!first || kk > 0) ? 1u : 0u);
  }
}

// Columns [c*32, c*32+32) of this thread's TMEM lane (fp32) -> bf16 -> 64
// bytes of global memory at dst (skipped when !in_range).
__device__ __forceinline__ void store_row_chunk(uint32_t tC, int c, __nv_bfloat16* row, bool in_range) {
  uint32_t v[32];
  tmem_ld32(tC + c * 32, v);
  tmem_wait_ld();
  if (in_range) {
    uint4* dst = reinterpret_cast<uint4*>(row + c * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 u;
      u.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
      u.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
      u.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
      u.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
      dst[q] = u;
    }
  }
}

// The first `ncols` (16 or 32) of the 32 columns [c*32, c*32+32) of this
// thread's TMEM lane -> bf16 -> global memory at row + c*32 (skipped when
// !in_range): the last, partial chunk of a row whose head dim is not a
// multiple of 32.
__device__ __forceinline__ void store_row_part(uint32_t tC, int c, __nv_bfloat16* row, bool in_range, int ncols) {
  uint32_t v[32];
  tmem_ld32(tC + c * 32, v);
  tmem_wait_ld();
  if (in_range) {
    uint4* dst = reinterpret_cast<uint4*>(row + c * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // (static register indices; ncols / 8 of the four are stored)
      if (q >= ncols / 8) break;
      uint4 u;
      u.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
      u.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
      u.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
      u.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
      dst[q] = u;
    }
  }
}

// tau(i) = beta * sqrt(2 ln(i+1) / D), in fp32 as the page computes it.
__device__ __forceinline__ float tau_of_row(int row, float beta, int D) {
  return beta * sqrtf(2.0f * logf(static_cast<float>(row + 1)) / static_cast<float>(D));
}

// Block order of the non-persistent kernels: the BH (b, h) heads split into
// G groups whose sizes differ by at most one (the first BH % G groups hold one
// head more); inside a group the tile rank goes first (rank 0 = the longest
// item) and the group's heads round-robin, so the CTAs resident at one time
// stream the tiles of a few heads, which stay in L2, instead of touching every
// head at once.  Block idx in [0, BH * nT) maps onto every (rank, bh) once.
struct HeadItem {
  int rank, bh;
};
__device__ __forceinline__ HeadItem head_group_item(int idx, int BH, int nT, int G) {
  const int b = BH / G, r = BH % G;
  const int big = (b + 1) * nT;  // items of each of the first r groups
  int h0, hg, i;
  if (idx < r * big) {
    const int g = idx / big;
    h0 = g * (b + 1);
    hg = b + 1;
    i = idx - g * big;
  } else {
    const int i2 = idx - r * big;
    const int g = i2 / (b * nT);
    h0 = r * (b + 1) + g * b;
    hg = b;
    i = i2 - g * b * nT;
  }
  return {i / hg, h0 + i % hg};
}

#ifndef BSA_HEAD_GROUP_MB
#define BSA_HEAD_GROUP_MB 32  // L2 bytes (MB) a group of heads streams; 0 = one group
#endif

// Number of head groups G for head_group_item.  A group holds the heads whose
// streamed tiles (stream_bytes per head) fill about BSA_HEAD_GROUP_MB of L2,
// but at least enough heads that the group's work, spread over `slots`
// resident CTAs, is twice its longest item: heads * nT (nT + 1) / 2 tile
// steps >= 2 * slots * nT.  The longest items start when their group does, so
// a smaller last group would leave the GPU idle behind them.
inline int head_groups(int BH, int nT, long long stream_bytes, int slots) {
  if (BSA_HEAD_GROUP_MB <= 0 || stream_bytes <= 0 || BH < 2) return 1;
  long long hg = (static_cast<long long>(BSA_HEAD_GROUP_MB) << 20) / stream_bytes;
  const long long hmin = (4LL * slots + nT) / (nT + 1);  // ceil(4 slots / (nT + 1))
  if (hg < hmin) hg = hmin;
  if (hg < 1) hg = 1;
  const long long g = BH / hg;
  return static_cast<int>(g < 1 ? 1 : g);
}

// Load the D/64 panels of tile row block `row0` of head `bh` into smem.
template <int D>
__device__ __forceinline__ void tma_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int row0, int bh) {
#pragma unroll
  for (int pnl = 0; pnl < D / 64; ++pnl) tma_load_3d(dst + pnl * PANEL_BYTES, map, bar, 64 * pnl, row0, bh);
}

}  // namespace tile
}  // namespace bsa
