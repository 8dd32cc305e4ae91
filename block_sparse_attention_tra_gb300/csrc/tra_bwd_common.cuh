// tra_bwd_common.cuh -- pieces shared by the two threshold-attention
// backward kernels (the recompute pair in tra_bwd.cu and the fused kernel in
// tra_bwd_fused.cu).
//
// Method: page "triton_threshold_attention.py", ThresholdRelaFunction.backward:
// with x_ij = q_i.k_j - tau(i) over the causal pairs j <= i,
//     W_ij = ReLU(x_ij)^p,   dA_ij = (dO_i . v_j) p ReLU(x_ij)^(p-1)
// (derivative 0 where x <= 0, as on the page).
#pragma once

#include "kernels.h"
#include "ptx.cuh"
#include "tc_tile.cuh"

namespace bsa {
namespace bwd {

__device__ __forceinline__ float ex2a(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2a(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ReLU(x)^p and its derivative p ReLU(x)^(p-1) (0 for x <= 0).  For p > 1
// (POW_GENERAL_MIX) the factor p goes into the exponent, g = exp2((p - 1)
// log2 r + log2 p) with lp = log2 p, and r = 0 needs no test: (p - 1) (-inf)
// is -inf and exp2 of it 0.  Other general powers (p < 1, where (p - 1)
// (-inf) is +inf) test x.
template <int PC>
__device__ __forceinline__ void weight_and_grad(float x, float p, float lp, float& w, float& g) {
  const float r = fmaxf(x, 0.0f);
  if constexpr (PC == POW_ONE) {
    w = r;
    g = x > 0.0f ? 1.0f : 0.0f;
  } else if constexpr (PC == POW_TWO) {
    w = r * r;
    g = 2.0f * r;
  } else if constexpr (PC == POW_GENERAL_MIX) {
    const float l = lg2a(r);  // -inf for r = 0
    w = ex2a(p * l);
    g = ex2a(fmaf(p - 1.0f, l, lp));
  } else {
    const float l = lg2a(r);
    w = ex2a(p * l);
    g = x > 0.0f ? p * ex2a((p - 1.0f) * l) : 0.0f;
  }
}

// Backward power class: p = 1, p = 2, p > 1 (POW_GENERAL_MIX) or any other.
__host__ __device__ inline int bwd_power_class(float p) {
  if (p == 1.0f) return POW_ONE;
  if (p == 2.0f) return POW_TWO;
  return p > 1.0f ? POW_GENERAL_MIX : POW_GENERAL;
}

// TMA producer of a backward block: two resident 128-row tiles (row res_row
// of maps r0 and r1) into res0 / res1, completing on res_full; then, for
// j = 0 .. count-1, tile (first + j) of map g0 into slot j % NS0 of ring0 and
// of map g1 into slot j % NS1 of ring1, each slot waiting for its release on
// empty0 / empty1 and completing on full0 / full1.  Every wait is bounded; on
// a failed wait it stops issuing and waits (bounded) for what is in flight.
template <int D, int NS0, int NS1>
__device__ __forceinline__ void produce(uint8_t* res0, uint8_t* res1, uint64_t* res_full, uint8_t* ring0,
                                        uint64_t* full0, uint64_t* empty0, uint8_t* ring1, uint64_t* full1,
                                        uint64_t* empty1, const CUtensorMap* r0, const CUtensorMap* r1, int res_row,
                                        const CUtensorMap* g0, const CUtensorMap* g1, int first, int count, int bh) {
  constexpr int TILE = D / 64 * tile::PANEL_BYTES;
  tma_prefetch_desc(r0);
  tma_prefetch_desc(r1);
  tma_prefetch_desc(g0);
  tma_prefetch_desc(g1);
  debug_check(res_row >= 0 && first >= 0 && bh >= 0);
  mbar_arrive_expect_tx(res_full, 2 * TILE);
  tile::tma_tile<D>(res0, r0, res_full, res_row, bh);
  tile::tma_tile<D>(res1, r1, res_full, res_row, bh);
  int issued0 = 0, issued1 = 0;
  bool ok = true;
  for (int j = 0; j < count && ok; ++j) {
    const int row = (first + j) * tile::ROWS;
    const int s0 = j % NS0, s1 = j % NS1;
    if (!(ok = mbar_wait(&empty0[s0], ((j / NS0) & 1) ^ 1))) break;
    mbar_arrive_expect_tx(&full0[s0], TILE);
    tile::tma_tile<D>(ring0 + s0 * TILE, g0, &full0[s0], row, bh);
    issued0 = j + 1;
    if (!(ok = mbar_wait(&empty1[s1], ((j / NS1) & 1) ^ 1))) break;
    mbar_arrive_expect_tx(&full1[s1], TILE);
    tile::tma_tile<D>(ring1 + s1 * TILE, g1, &full1[s1], row, bh);
    issued1 = j + 1;
  }
  if (!ok) {  // drain what is still landing before the CTA may exit
    mbar_wait(res_full, 0);
    for (int j = (issued0 > NS0 ? issued0 - NS0 : 0); j < issued0; ++j) mbar_wait(&full0[j % NS0], (j / NS0) & 1);
    for (int j = (issued1 > NS1 ? issued1 - NS1 : 0); j < issued1; ++j) mbar_wait(&full1[j % NS1], (j / NS1) & 1);
  }
}

}  // namespace bwd
}  // namespace bsa
