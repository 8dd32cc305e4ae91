// tra_math.cuh -- the threshold-attention weight ReLU(s - tau)^p in the
// epilogue registers: power classes p = 1, p = 2, general p through
// exp2(p log2 x) (with an FMA-pipe log2 for part of the elements when
// p >= 1), and, on request, p = k + 1/2 as x^k sqrt(x).
// Shared by the forward kernels (plain and differential).
#pragma once

#include "kernels.h"
#include "ptx.cuh"

namespace bsa {
namespace {

// General power with p >= 1: pairs (of 16 per 32 columns) whose log2 is
// evaluated on the FMA pipe by a polynomial instead of the MUFU lg2.
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
__device__ __forceinline__ float sqrt_approx(float x) {
  float y;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
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

// Two fp32 values in one 64-bit register (lo = first) and the packed
// f32x2 arithmetic of the sm_100 family: one instruction for both keys of a
// pair on the FMA pipe.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Per-row constants of the weight: tau and p (and p * LOG2_Ck) duplicated
// into both halves of a packed pair.
struct PowParams {
  uint64_t tau2, p2, pc2[5];
};
__device__ __forceinline__ PowParams pow_params(float tau, float p) {
  PowParams w;
  w.tau2 = f2_pack(tau, tau);
  w.p2 = f2_pack(p, p);
  const float c[5] = {LOG2_C0, LOG2_C1, LOG2_C2, LOG2_C3, LOG2_C4};
#pragma unroll
  for (int k = 0; k < 5; ++k) w.pc2[k] = f2_pack(p * c[k], p * c[k]);
  return w;
}

// p * log2(x) of two non-negative x on the FMA/ALU pipes: x = 2^e m with
// m in [1, 2) taken from the bits, log2(m) from the LOG2_Ck polynomial with p
// folded into pc2.  x = 0 reads as e = -127, m = 1, i.e. about -127 p, whose
// exp2 flushes to 0 for p >= 1: callers use this path only when p >= 1.
__device__ __forceinline__ uint64_t p_log2_poly2(float x0, float x1, const PowParams& w) {
  const uint32_t b0 = __float_as_uint(x0), b1 = __float_as_uint(x1);
  const uint64_t m = f2_pack(__uint_as_float((b0 & 0x007fffffu) | 0x3f800000u),
                             __uint_as_float((b1 & 0x007fffffu) | 0x3f800000u));
  const float bias = 8388608.0f + 127.0f;
  const uint64_t e = f2_sub(f2_pack(__uint_as_float((b0 >> 23) | 0x4b000000u), __uint_as_float((b1 >> 23) | 0x4b000000u)),
                            f2_pack(bias, bias));
  uint64_t acc = f2_fma(w.pc2[4], m, w.pc2[3]);
  acc = f2_fma(acc, m, w.pc2[2]);
  acc = f2_fma(acc, m, w.pc2[1]);
  acc = f2_fma(acc, m, w.pc2[0]);
  return f2_fma(w.p2, e, acc);
}

// Weights of two adjacent keys from their scores: ReLU(s - tau)^p, bf16x2.
// EMU: p * log2 on the FMA pipe (requires p >= 1), else on the MUFU unit.
template <int PC, bool EMU>
__device__ __forceinline__ uint32_t weights2(float s0, float s1, const PowParams& w) {
  float x0, x1;
  f2_unpack(f2_sub(f2_pack(s0, s1), w.tau2), x0, x1);
  if constexpr (PC == POW_ONE) {
    return relu_pack(x0, x1);
  } else if constexpr (PC == POW_TWO) {
    const uint32_t h = relu_pack(x0, x1);
    return mul_bf16x2(h, h);
  } else if constexpr (PC >= POW_HALF0) {
    // p = k + 1/2: x^p = x^k sqrt(x), one MUFU operation per score; the
    // ReLU's zeros give sqrt(0) = 0 exactly.
    x0 = fmaxf(x0, 0.0f);
    x1 = fmaxf(x1, 0.0f);
    uint64_t r = f2_pack(sqrt_approx(x0), sqrt_approx(x1));
    const uint64_t x = f2_pack(x0, x1);
#pragma unroll
    for (int j = 0; j < PC - POW_HALF0; ++j) r = f2_mul(r, x);
    float r0, r1;
    f2_unpack(r, r0, r1);
    return pack_bf16x2_alu(r0, r1);
  } else {
    // x^p = exp2(p log2 x); the ReLU's zeros give log2 = -inf (MUFU) or about
    // -127 p (polynomial, p >= 1), and exp2 of either is 0.
    x0 = fmaxf(x0, 0.0f);
    x1 = fmaxf(x1, 0.0f);
    const uint64_t y = EMU ? p_log2_poly2(x0, x1, w) : f2_mul(f2_pack(lg2_approx(x0), lg2_approx(x1)), w.p2);
    float y0, y1;
    f2_unpack(y, y0, y1);
    return pack_bf16x2_alu(ex2_approx(y0), ex2_approx(y1));
  }
}

}  // namespace
}  // namespace bsa
