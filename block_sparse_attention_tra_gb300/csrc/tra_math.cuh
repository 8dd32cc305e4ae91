// tra_math.cuh -- the threshold-attention weight ReLU(s - tau)^p in the
// epilogue registers: power classes p = 1, p = 2 and general p through
// exp2(p log2 x), with an optional FMA-pipe log2 for part of the elements.
// Shared by the forward kernels (plain and differential).
#pragma once

#include "kernels.h"
#include "ptx.cuh"

namespace bsa {
namespace {

// General power: pairs (of 16 per 32 columns) whose log2 is evaluated on the
// FMA pipe by a polynomial instead of the MUFU lg2 (the MUFU unit, shared by
// lg2 and ex2, bounds the general path).
#ifndef BSA_EMU_LOG2_PAIRS
#define BSA_EMU_LOG2_PAIRS 0
#endif
constexpr int EMU_LOG2_PAIRS = BSA_EMU_LOG2_PAIRS;
static_assert(EMU_LOG2_PAIRS >= 0 && EMU_LOG2_PAIRS <= 16, "pairs per 16");

// log2(m) ~= sum_k LOG2_Ck m^k for m in [1, 2): degree-4 least-squares fit
// on Chebyshev nodes (fit_log2.py); max |error| 1.0e-4, i.e. a relative error
// <= p * ln2 * 1e-4 in the weight, well below its bf16 rounding (2^-9).
constexpr float LOG2_C0 = -2.505614662e+00f, LOG2_C1 = 4.049616893e+00f, LOG2_C2 = -2.099402281e+00f,
                LOG2_C3 = 6.355111165e-01f, LOG2_C4 = -8.001087691e-02f;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// ReLU then round both to bf16: {lo, hi} packed, lo in the low half.
__device__ __forceinline__ uint32_t relu_pack(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.relu.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Round two non-negative fp32 weights to bf16 (nearest, ties away from zero)
// and pack them, with integer adds and a byte permute on the ALU pipe instead
// of the conversion unit, which the general path keeps busy with lg2/ex2.
#ifndef BSA_INT_PACK
#define BSA_INT_PACK 0
#endif
__device__ __forceinline__ uint32_t pack_bf16x2_alu(float lo, float hi) {
#if BSA_INT_PACK
  const uint32_t a = __float_as_uint(lo) + 0x8000u, b = __float_as_uint(hi) + 0x8000u;
  return __byte_perm(a, b, 0x7632);
#else
  return pack_bf16x2(lo, hi);
#endif
}

// p * log2(x) on the FMA/ALU pipes: x = 2^e m with m in [1, 2) taken from
// the bits, log2(m) from the LOG2_Ck polynomial with p folded into pc[].
// Any x <= 0 (the ReLU's zeros) returns -inf, so that exp2 of it is 0.
__device__ __forceinline__ float p_log2_poly(float x, float p, const float (&pc)[5]) {
  const uint32_t b = __float_as_uint(x);
  const float m = __uint_as_float((b & 0x007fffffu) | 0x3f800000u);
  const float e = __uint_as_float((b >> 23) | 0x4b000000u) - (8388608.0f + 127.0f);
  float acc = fmaf(pc[4], m, pc[3]);
  acc = fmaf(acc, m, pc[2]);
  acc = fmaf(acc, m, pc[1]);
  acc = fmaf(acc, m, pc[0]);
  return x > 0.0f ? fmaf(p, e, acc) : -INFINITY;
}

// Weights of two adjacent keys from their scores: ReLU(s - tau)^p, bf16x2.
template <int PC, bool EMU>
__device__ __forceinline__ uint32_t weights2(float s0, float s1, float tau, float p, const float (&pc)[5]) {
  const float x0 = s0 - tau, x1 = s1 - tau;
  if constexpr (PC == POW_ONE) {
    return relu_pack(x0, x1);
  } else if constexpr (PC == POW_TWO) {
    const uint32_t h = relu_pack(x0, x1);
    return mul_bf16x2(h, h);
  } else {
    // x^p = exp2(p log2 x); log2 of the ReLU's zeros is -inf and ex2 of it 0.
    float y0, y1;
    if constexpr (EMU) {
      y0 = p_log2_poly(x0, p, pc);
      y1 = p_log2_poly(x1, p, pc);
    } else {
      y0 = p * lg2_approx(fmaxf(x0, 0.0f));
      y1 = p * lg2_approx(fmaxf(x1, 0.0f));
    }
    return pack_bf16x2_alu(ex2_approx(y0), ex2_approx(y1));
  }
}

}  // namespace
}  // namespace bsa
