// tra_math.cuh -- the threshold-attention weight ReLU(s - tau)^p in the
// epilogue registers: power classes p = 1, p = 2, general p through
// exp2(p log2 x), and, on request, p = k + 1/2 as x^k sqrt(x).
// Shared by the forward kernels (plain and differential).
#pragma once

#include "kernels.h"
#include "ptx.cuh"

namespace bsa {
namespace {

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
// Per-row constants of the weight: tau and p duplicated into both halves of
// a packed pair.
struct PowParams {
  uint64_t tau2, p2;
};
__device__ __forceinline__ PowParams pow_params(float tau, float p) {
  PowParams w;
  w.tau2 = f2_pack(tau, tau);
  w.p2 = f2_pack(p, p);
  return w;
}

// Weights of two adjacent keys from their scores: ReLU(s - tau)^p, bf16x2.
template <int PC>
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
    return pack_bf16x2(r0, r1);
  } else {
    // x^p = exp2(p log2 x); the ReLU's zeros give log2 = -inf and exp2 of it 0.
    x0 = fmaxf(x0, 0.0f);
    x1 = fmaxf(x1, 0.0f);
    const uint64_t y = f2_mul(f2_pack(lg2_approx(x0), lg2_approx(x1)), w.p2);
    float y0, y1;
    f2_unpack(y, y0, y1);
    return pack_bf16x2(ex2_approx(y0), ex2_approx(y1));
  }
}

}  // namespace
}  // namespace bsa
