// tra_math.cuh -- the threshold-attention weight ReLU(s - tau)^p in the
// epilogue registers: power classes p = 1, p = 2, general p through
// exp2(p log2 x), and, on request, p = k + 1/2 as x^k sqrt(x).
// Shared by the forward kernels (plain and differential).
//
// The general path's log2 runs on two units.  MUFU lg2 issues at half the
// ex2 rate (16 against 32 results per clock and SM), so with one lg2 and one
// ex2 per score it bounds the epilogue.  POW_GENERAL_MIX evaluates log2 of
// a share of the scores on the FMA pipe instead: x = 2^e m with m in [1, 2)
// taken from the float's exponent and mantissa fields (one funnel shift and
// one LOP3), log2 m from a degree-5 minimax polynomial (Remez exchange fit,
// block_sparse_attention_tra_gb300/log2_poly.py; max error 1.6e-5 evaluated
// in float32) by Horner's rule on packed f32x2 FMAs, with p folded into the
// coefficients.  exp2 can leave MUFU for a share of the pairs too
// (exp2_fma: n = round(y), f = y - n, 2^f from a degree-4 minimax
// polynomial, the exponent raised by n with one integer add), but every
// share of it measured slower, so none is taken by default.
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
// max(w, 0) per bf16 half; a NaN half gives 0 (max returns the operand that
// is not NaN).
__device__ __forceinline__ uint32_t relu_nan_bf16x2(uint32_t w) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(w), "r"(0u));
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
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
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

// log2(m) ~= sum_k LOG2_M[k] m^k on m in [1, 2): the Remez minimax fit of
// log2(1 + t) on t in [0, 1) (through 0 at t = 0), written in m = 1 + t.
constexpr int LOG2_DEG = 5;
__device__ constexpr float LOG2_M[LOG2_DEG + 1] = {-2.811879280e+00f, 5.131084173e+00f, -3.603921890e+00f,
                                                  1.666528133e+00f, -4.281965043e-01f, 4.638536892e-02f};
constexpr float EXP_FIELD_BIAS = 8388735.0f;  // 2^23 + 127: float of (0x4B000000 | e_field) minus this = e

// Per-row constants of the weight: tau and p duplicated into both halves of
// a packed pair; for POW_GENERAL_MIX also p times the log2 coefficients and
// the exponent-field bias.
struct PowParams {
  uint64_t tau2, p2;
  uint64_t lc[LOG2_DEG + 1];
  uint64_t ebias2;
};
__device__ __forceinline__ PowParams pow_params(float tau, float p) {
  PowParams w;
  w.tau2 = f2_pack(tau, tau);
  w.p2 = f2_pack(p, p);
#pragma unroll
  for (int k = 0; k <= LOG2_DEG; ++k) w.lc[k] = f2_pack(p * LOG2_M[k], p * LOG2_M[k]);
  w.ebias2 = f2_pack(EXP_FIELD_BIAS, EXP_FIELD_BIAS);
  return w;
}

// p log2(x0), p log2(x1) for x >= 0 on the FMA pipe (x = 0 gives -127 p, and
// exp2 of it flushes to 0 for p >= 1).
__device__ __forceinline__ uint64_t p_log2_fma(float x0, float x1, const PowParams& w) {
  const uint32_t i0 = __float_as_uint(x0), i1 = __float_as_uint(x1);
  // mantissa with a zero exponent field: m in [1, 2)
  const uint64_t m = f2_pack(__uint_as_float((i0 & 0x007fffffu) | 0x3f800000u),
                             __uint_as_float((i1 & 0x007fffffu) | 0x3f800000u));
  // 0x4B000000 | exponent field (x >= 0: the sign bit is 0), as a float 2^23 + field
  const uint64_t ef = f2_sub(f2_pack(__uint_as_float(__funnelshift_r(i0, 0x00258000u, 23)),
                                     __uint_as_float(__funnelshift_r(i1, 0x00258000u, 23))),
                             w.ebias2);
  uint64_t r = w.lc[LOG2_DEG];
#pragma unroll
  for (int k = LOG2_DEG - 1; k >= 0; --k) r = f2_fma(r, m, w.lc[k]);
  return f2_fma(ef, w.p2, r);
}

// exp2(y0), exp2(y1) on the FMA pipe (then rounded to bf16x2).  y is clamped to
// [-127, 128]; t = y + 1.5 * 2^23 holds n = round(y) in its low mantissa bits
// (round to nearest), f = y - (t - 1.5 * 2^23) lies in [-1/2, 1/2], and
// 2^f ~= 1 + f (c1 + c2 f + c3 f^2 + c4 f^3): the Remez fit with p(0) = 1 of
// block_sparse_attention_tra_gb300/exp2_poly.py (relative error 2.9e-6
// evaluated in float32, against 2^-9 for the bf16 rounding that follows).
// Adding t's bits shifted left by 23 adds n to the exponent field (the
// constant part of t shifts out).  y = -127 (the ReLU's zeros, p >= 1) gives
// the bits of +0.0 exactly and y = 128 those of +inf; between -127 and -126
// the pattern is a small subnormal (the MUFU form flushes those to 0).
#ifndef BSA_EXP2_DEG
#define BSA_EXP2_DEG 4
#endif
#if BSA_EXP2_DEG == 4
__device__ constexpr float EXP2_C[4] = {6.931241934e-01f, 2.402409861e-01f, 5.590642460e-02f, 9.582853096e-03f};
#elif BSA_EXP2_DEG == 3
__device__ constexpr float EXP2_C[3] = {6.932829271e-01f, 2.422109593e-01f, 5.500893113e-02f};  // 1.0e-4
#else
#error "BSA_EXP2_DEG must be 3 or 4"
#endif
constexpr float ROUND_MAGIC = 12582912.0f;  // 1.5 * 2^23
__device__ __forceinline__ uint64_t exp2_fma2(uint64_t y2) {
  float y0, y1;
  f2_unpack(y2, y0, y1);
  const uint64_t y = f2_pack(fminf(fmaxf(y0, -127.0f), 128.0f), fminf(fmaxf(y1, -127.0f), 128.0f));
  const uint64_t magic = f2_pack(ROUND_MAGIC, ROUND_MAGIC);
  const uint64_t t = f2_add(y, magic);
  const uint64_t f = f2_sub(y, f2_sub(t, magic));
  uint64_t r = f2_pack(EXP2_C[BSA_EXP2_DEG - 1], EXP2_C[BSA_EXP2_DEG - 1]);
#pragma unroll
  for (int k = BSA_EXP2_DEG - 2; k >= 0; --k) r = f2_fma(r, f, f2_pack(EXP2_C[k], EXP2_C[k]));
  r = f2_fma(r, f, f2_pack(1.0f, 1.0f));
  float r0, r1, t0, t1;
  f2_unpack(r, r0, r1);
  f2_unpack(t, t0, t1);
  return f2_pack(__uint_as_float(__float_as_uint(r0) + (__float_as_uint(t0) << 23)),
                 __uint_as_float(__float_as_uint(r1) + (__float_as_uint(t1) << 23)));
}
__device__ __forceinline__ uint32_t exp2_fma_bf16x2(uint64_t y2) {
  float w0, w1;
  f2_unpack(exp2_fma2(y2), w0, w1);
  return pack_bf16x2(w0, w1);
}

// Which units each pair of a 16-pair quarter uses under POW_GENERAL_MIX, as a
// plan MUFU_LOG + 32 EXP_FMA: MUFU_LOG of every 16 pairs take MUFU lg2 (the
// rest the FMA-pipe log2), and EXP_FMA of those MUFU_LOG pairs take the
// FMA-pipe exp2 (the rest MUFU ex2), each share spread evenly.  The shares
// are chosen per head dim (measured on the T=8192 D=64 and the T=4096 D=128
// p = 1.5 workloads with two epilogue warpgroups per query tile); more
// FMA-pipe pairs than that are slower, since the packed f32x2 FMAs, LOP3 and
// funnel shifts of the polynomial paths all run at half rate.
#ifndef BSA_MIX_MUFU_PAIRS_D64
#define BSA_MIX_MUFU_PAIRS_D64 10
#endif
#ifndef BSA_MIX_MUFU_PAIRS_D128
#define BSA_MIX_MUFU_PAIRS_D128 10
#endif
#ifndef BSA_MIX_EXP_FMA_PAIRS_D64
#define BSA_MIX_EXP_FMA_PAIRS_D64 0
#endif
#ifndef BSA_MIX_EXP_FMA_PAIRS_D128
#define BSA_MIX_EXP_FMA_PAIRS_D128 0
#endif
template <int D>
__host__ __device__ constexpr int mix_mufu_pairs() {
  return D == 64 ? BSA_MIX_MUFU_PAIRS_D64 + 32 * BSA_MIX_EXP_FMA_PAIRS_D64
                 : BSA_MIX_MUFU_PAIRS_D128 + 32 * BSA_MIX_EXP_FMA_PAIRS_D128;
}
template <int PLAN>
__host__ __device__ constexpr bool mix_pair_on_fma(int e) {
  constexpr int M = PLAN % 32;
  return ((e % 16) * M) % 16 >= M;
}
template <int PLAN>
__host__ __device__ constexpr bool mix_exp_on_fma(int e) {
  constexpr int M = PLAN % 32, E = PLAN / 32;
  if (E == 0 || mix_pair_on_fma<PLAN>(e)) return false;
  int k = 0;  // rank of pair e among the MUFU-log2 pairs
  for (int j = 0; j < e % 16; ++j) k += mix_pair_on_fma<PLAN>(j) ? 0 : 1;
  return (k * E) % M < E;
}

// p = 2: round x to bf16 and square in bf16 (0: two roundings, at most ~1.5
// bf16 ulp per weight), or square in fp32 and round once (1: half an ulp, one
// instruction more per key pair; measured 8.6% slower at B4 H16 T4096 D128
// and 4% at B2 H32 T8192 D64, whose epilogues share the SMSPs with the MMA
// issue).
#ifndef BSA_POW2_SINGLE_ROUNDING
#define BSA_POW2_SINGLE_ROUNDING 0
#endif

// Weights of two adjacent keys from x = s - tau (packed): ReLU(x)^p, bf16x2.
// FMA_LOG2, FMA_EXP2 (POW_GENERAL_MIX only): this pair's log2, exp2 runs on
// the FMA pipe.
template <int PC, bool FMA_LOG2 = false, bool FMA_EXP2 = false>
__device__ __forceinline__ uint32_t weights2_x(uint64_t x2, const PowParams& w) {
  float x0, x1;
  f2_unpack(x2, x0, x1);
  if constexpr (PC == POW_ONE) {
    return relu_pack(x0, x1);
  } else if constexpr (PC == POW_TWO) {
#if BSA_POW2_SINGLE_ROUNDING
    // x |x| is x^2 where x > 0 and negative elsewhere, so the ReLU of the
    // conversion keeps exactly the positive part: one rounding, from fp32.
    return relu_pack(x0 * fabsf(x0), x1 * fabsf(x1));
#else
    const uint32_t h = relu_pack(x0, x1);  // x rounded to bf16, then squared in bf16
    return mul_bf16x2(h, h);
#endif
  } else if constexpr (PC == POW_GENERAL_MIX) {
    if constexpr (FMA_LOG2) {
      // the exponent and mantissa fields need x >= 0
      const uint64_t y = p_log2_fma(fmaxf(x0, 0.0f), fmaxf(x1, 0.0f), w);
      if constexpr (FMA_EXP2) return exp2_fma_bf16x2(y);
      float y0, y1;
      f2_unpack(y, y0, y1);
      return pack_bf16x2(ex2_approx(y0), ex2_approx(y1));
    } else {
      // MUFU lg2 of x <= 0 is -inf (x = 0) or NaN (x < 0): exp2 gives 0 or
      // NaN, and the ReLU is applied after the rounding to bf16 (max with 0,
      // which maps NaN to 0) -- one instruction per pair instead of two.
      // The FMA-pipe exp2 clamps its input, which also maps NaN to 0.
      const uint64_t y = f2_mul(f2_pack(lg2_approx(x0), lg2_approx(x1)), w.p2);
      if constexpr (FMA_EXP2) return exp2_fma_bf16x2(y);
      float y0, y1;
      f2_unpack(y, y0, y1);
      return relu_nan_bf16x2(pack_bf16x2(ex2_approx(y0), ex2_approx(y1)));
    }
  } else if constexpr (PC >= POW_HALF0 && PC <= POW_HALF3) {
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
    // x^p = exp2(p log2 x); lg2 of x = 0 is -inf (exp2 of it 0) and of x < 0
    // NaN, which the ReLU after the bf16 rounding maps to 0.
    const uint64_t y = f2_mul(f2_pack(lg2_approx(x0), lg2_approx(x1)), w.p2);
    float y0, y1;
    f2_unpack(y, y0, y1);
    return relu_nan_bf16x2(pack_bf16x2(ex2_approx(y0), ex2_approx(y1)));
  }
}

// Weights of two adjacent keys from their scores: ReLU(s - tau)^p, bf16x2.
template <int PC, bool FMA_LOG2 = false, bool FMA_EXP2 = false>
__device__ __forceinline__ uint32_t weights2(float s0, float s1, const PowParams& w) {
  return weights2_x<PC, FMA_LOG2, FMA_EXP2>(f2_sub(f2_pack(s0, s1), w.tau2), w);
}

}  // namespace
}  // namespace bsa
