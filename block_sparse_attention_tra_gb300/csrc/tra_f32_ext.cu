// tra_f32_ext.cu -- the fp32 forms of the threshold-attention backward and of
// the differential forward, on the CUDA cores (FFMA throughout, like the fp32
// forward in tra_f32.cu: TF32 tensor cores would miss a 1e-4 relative bar).
//
// Backward -- page "triton_threshold_attention.py", ThresholdRelaFunction.
// backward with _threshold_rela_bwd_kernel_dq / _dkv, which compute in fp32:
// over the causal pairs j <= i, with x_ij = q_i.k_j - tau(i),
//     W_ij = ReLU(x_ij)^p,            dV_j = sum_i W_ij dO_i,
//     dA_ij = (dO_i . v_j) p ReLU(x_ij)^(p-1)   (0 where x_ij <= 0),
//     dQ_i = sum_j dA_ij k_j,          dK_j = sum_i dA_ij q_i.
// Two kernels: one CTA per 64-row query tile walks key tiles 0..m and
// accumulates dQ; one CTA per 64-key tile walks query tiles n..last and
// accumulates dK and dV.  Scores and dO.v are recomputed in each.
//
// Differential forward -- same page, differential_threshold_rela_triton:
//     out = TRA(n(q1), n(k1), v) - clamp(lambda, 0, 1) TRA(n(q2), n(k2), v),
// n = row-wise L2 normalisation x / max(||x||, 1e-12) when requested.  One CTA
// per 64-row query tile runs both score streams on the same key tiles and
// accumulates the combined weights times V; the normalisation is folded into
// the scores (s * r(q) * r(k), r = 1 / max(||row||, 1e-12)), computed from
// the rows already in shared memory, so no scratch memory is needed.
#include "kernels.h"
#include "ptx.cuh"

namespace bsa {
namespace {

constexpr int XB = 64;         // rows per tile (queries or keys)
constexpr int XTHREADS = 256;  // 16 x 16 threads, 4 x 4 outputs each

__device__ __forceinline__ float tau_f32(int row, float beta, int D) {
  return beta * sqrtf(2.0f * logf(static_cast<float>(row + 1)) / static_cast<float>(D));
}

// ReLU(x)^p and its derivative (0 for x <= 0), in fp32.
template <int PC>
__device__ __forceinline__ void wgrad_f32(float x, float p, float& w, float& g) {
  const float r = fmaxf(x, 0.0f);
  if constexpr (PC == POW_ONE) {
    w = r;
    g = x > 0.0f ? 1.0f : 0.0f;
  } else if constexpr (PC == POW_TWO) {
    w = r * r;
    g = 2.0f * r;
  } else {
    if (x > 0.0f) {
      const float l = log2f(r);
      w = exp2f(p * l);
      g = p * exp2f((p - 1.0f) * l);
    } else {
      w = 0.0f;
      g = 0.0f;
    }
  }
}

template <int PC>
__device__ __forceinline__ float relu_pow(float x, float p) {
  float w, g;
  if constexpr (PC == POW_ONE) return fmaxf(x, 0.0f);
  if constexpr (PC == POW_TWO) {
    const float r = fmaxf(x, 0.0f);
    return r * r;
  }
  wgrad_f32<PC>(x, p, w, g);
  return w;
}

// Rows [row0, row0 + 64) of a [T, D] head into smem rows of stride QS (zero
// beyond T).
template <int D>
__device__ __forceinline__ void load_rows(float* dst, const float* __restrict__ src, int row0, int T) {
  constexpr int QS = D + 1;
  for (int e = threadIdx.x; e < XB * D; e += XTHREADS) {
    const int r = e / D, d = e % D;
    const int row = row0 + r;
    dst[r * QS + d] = row < T ? src[static_cast<size_t>(row) * D + d] : 0.0f;
  }
}

// a[r][c] = sum_d A[ty + 16 r][d] B[tx + 16 c][d] for the thread's 4 x 4 block.
template <int D>
__device__ __forceinline__ void dot4x4(const float* A, const float* B, int ty, int tx, float (&a)[4][4]) {
  constexpr int QS = D + 1;
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) a[r][c] = 0.0f;
#pragma unroll 8
  for (int d = 0; d < D; ++d) {
    float x[4], y[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) x[r] = A[(ty + 16 * r) * QS + d];
#pragma unroll
    for (int c = 0; c < 4; ++c) y[c] = B[(tx + 16 * c) * QS + d];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) a[r][c] = fmaf(x[r], y[c], a[r][c]);
  }
}

// acc[r][c] += sum_j W[ty + 16 r][j] X[j][tx + 16 c] (W stride XB + 1, X stride D + 1).
template <int D>
__device__ __forceinline__ void accum_wx(const float* W, const float* X, int ty, int tx, float (&acc)[4][D / 16]) {
  constexpr int QS = D + 1;
#pragma unroll 4
  for (int j = 0; j < XB; ++j) {
    float wa[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) wa[r] = W[(ty + 16 * r) * (XB + 1) + j];
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      const float xv = X[j * QS + tx + 16 * c];
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[r][c] = fmaf(wa[r], xv, acc[r][c]);
    }
  }
}

template <int D>
__device__ __forceinline__ void store_rows(float* __restrict__ dst, int row0, int T, int ty, int tx,
                                           const float (&acc)[4][D / 16]) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = row0 + ty + 16 * r;
    if (row < T) {
#pragma unroll
      for (int c = 0; c < D / 16; ++c) dst[static_cast<size_t>(row) * D + tx + 16 * c] = acc[r][c];
    }
  }
}

// ------------------------------------------------------------------ backward

// dQ: one CTA per (query tile m, head), m = nM-1 .. 0 (longest first).
template <int D, int PC>
__global__ void __launch_bounds__(XTHREADS) tra_f32_bwd_dq_kernel(const float* __restrict__ q,
                                                                  const float* __restrict__ k,
                                                                  const float* __restrict__ v,
                                                                  const float* __restrict__ dout,
                                                                  float* __restrict__ dq, int BH, int T, int nM,
                                                                  float beta, float p) {
  constexpr int QS = D + 1;
  extern __shared__ float xsm[];
  float* Qs = xsm;              // [64][QS]
  float* Os = Qs + XB * QS;     // dO rows
  float* Ks = Os + XB * QS;
  float* Vs = Ks + XB * QS;
  float* As = Vs + XB * QS;     // dA [64][65]
  const int m = nM - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const size_t base = static_cast<size_t>(bh) * T * D;
  load_rows<D>(Qs, q + base, m * XB, T);
  load_rows<D>(Os, dout + base, m * XB, T);
  float tau[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) tau[r] = tau_f32(m * XB + ty + 16 * r, beta, D);
  float acc[4][D / 16];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < D / 16; ++c) acc[r][c] = 0.0f;

  for (int n = 0; n <= m; ++n) {
    __syncthreads();
    load_rows<D>(Ks, k + base, n * XB, T);
    load_rows<D>(Vs, v + base, n * XB, T);
    __syncthreads();
    float s[4][4], dp[4][4];
    dot4x4<D>(Qs, Ks, ty, tx, s);
    dot4x4<D>(Os, Vs, ty, tx, dp);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int row = m * XB + ty + 16 * r;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int key = n * XB + tx + 16 * c;
        float w, g;
        wgrad_f32<PC>(s[r][c] - tau[r], p, w, g);
        As[(ty + 16 * r) * (XB + 1) + tx + 16 * c] = key <= row ? dp[r][c] * g : 0.0f;
      }
    }
    __syncthreads();
    accum_wx<D>(As, Ks, ty, tx, acc);
  }
  store_rows<D>(dq + base, m * XB, T, ty, tx, acc);
}

// dK, dV: one CTA per (key tile n, head), n = 0 .. nM-1 (longest first).
template <int D, int PC>
__global__ void __launch_bounds__(XTHREADS) tra_f32_bwd_dkdv_kernel(const float* __restrict__ q,
                                                                    const float* __restrict__ k,
                                                                    const float* __restrict__ v,
                                                                    const float* __restrict__ dout,
                                                                    float* __restrict__ dk, float* __restrict__ dv,
                                                                    int BH, int T, int nM, float beta, float p) {
  constexpr int QS = D + 1;
  extern __shared__ float xsm[];
  float* Ks = xsm;              // [64][QS]
  float* Vs = Ks + XB * QS;
  float* Qs = Vs + XB * QS;
  float* Os = Qs + XB * QS;     // dO rows
  float* Wt = Os + XB * QS;     // W^T [64 keys][65]
  float* At = Wt + XB * (XB + 1);  // dA^T
  const int n = static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const size_t base = static_cast<size_t>(bh) * T * D;
  load_rows<D>(Ks, k + base, n * XB, T);
  load_rows<D>(Vs, v + base, n * XB, T);
  float adk[4][D / 16], adv[4][D / 16];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < D / 16; ++c) adk[r][c] = adv[r][c] = 0.0f;

  for (int m = n; m < nM; ++m) {
    __syncthreads();
    load_rows<D>(Qs, q + base, m * XB, T);
    load_rows<D>(Os, dout + base, m * XB, T);
    __syncthreads();
    float s[4][4], dp[4][4];  // rows = keys ty + 16 r, columns = queries tx + 16 c
    dot4x4<D>(Ks, Qs, ty, tx, s);
    dot4x4<D>(Vs, Os, ty, tx, dp);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int row = m * XB + tx + 16 * c;  // query
      const float t = tau_f32(row, beta, D);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int key = n * XB + ty + 16 * r;
        float w, g;
        wgrad_f32<PC>(s[r][c] - t, p, w, g);
        const bool keep = key <= row && row < T;
        Wt[(ty + 16 * r) * (XB + 1) + tx + 16 * c] = keep ? w : 0.0f;
        At[(ty + 16 * r) * (XB + 1) + tx + 16 * c] = keep ? dp[r][c] * g : 0.0f;
      }
    }
    __syncthreads();
    accum_wx<D>(Wt, Os, ty, tx, adv);
    accum_wx<D>(At, Qs, ty, tx, adk);
  }
  store_rows<D>(dk + base, n * XB, T, ty, tx, adk);
  store_rows<D>(dv + base, n * XB, T, ty, tx, adv);
}

template <int D, int PC>
int launch_bwd(const float* q, const float* k, const float* v, const float* dout, float* dq, float* dk, float* dv,
               int BH, int T, float beta, float p, cudaStream_t stream) {
  constexpr int QS = D + 1;
  constexpr size_t smem_dq = sizeof(float) * (4 * XB * QS + XB * (XB + 1));
  constexpr size_t smem_dkdv = sizeof(float) * (4 * XB * QS + 2 * XB * (XB + 1));
  auto kq = tra_f32_bwd_dq_kernel<D, PC>;
  auto kk = tra_f32_bwd_dkdv_kernel<D, PC>;
  if (cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_dq)) !=
          cudaSuccess ||
      cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_dkdv)) !=
          cudaSuccess)
    return ERR_LAUNCH;
  const int nM = (T + XB - 1) / XB;
  const long long grid = static_cast<long long>(nM) * BH;
  if (grid > 0x7fffffffLL) return ERR_SHAPE;
  kq<<<static_cast<unsigned>(grid), XTHREADS, smem_dq, stream>>>(q, k, v, dout, dq, BH, T, nM, beta, p);
  if (cudaGetLastError() != cudaSuccess) return ERR_LAUNCH;
  kk<<<static_cast<unsigned>(grid), XTHREADS, smem_dkdv, stream>>>(q, k, v, dout, dk, dv, BH, T, nM, beta, p);
  return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
}

// ----------------------------------------------------------- differential

// r[row] = 1 / max(||row||, 1e-12) for the 64 rows of a smem tile (one
// thread per row; `t` = the thread's index among the participating threads).
template <int D>
__device__ __forceinline__ void row_inv_norms(const float* X, float* r, int t) {
  constexpr int QS = D + 1;
  float ss = 0.0f;
#pragma unroll 8
  for (int d = 0; d < D; ++d) ss = fmaf(X[t * QS + d], X[t * QS + d], ss);
  r[t] = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
}

template <int D, int PC, bool NORM>
__global__ void __launch_bounds__(XTHREADS) tra_f32_diff_kernel(const float* __restrict__ q1,
                                                                const float* __restrict__ q2,
                                                                const float* __restrict__ k1,
                                                                const float* __restrict__ k2,
                                                                const float* __restrict__ v,
                                                                float* __restrict__ out, int BH, int T, int nM,
                                                                float beta, float p, float lam) {
  constexpr int QS = D + 1;
  extern __shared__ float xsm[];
  float* Q1 = xsm;              // [64][QS]
  float* Q2 = Q1 + XB * QS;
  float* K1 = Q2 + XB * QS;
  float* K2 = K1 + XB * QS;
  float* Vs = K2 + XB * QS;
  float* Ws = Vs + XB * QS;     // [64][65]
  float* rn = Ws + XB * (XB + 1);  // rq1[64] | rq2[64] | rk1[64] | rk2[64]
  const int m = nM - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int tid = static_cast<int>(threadIdx.x);
  const int ty = tid >> 4, tx = tid & 15;
  const size_t base = static_cast<size_t>(bh) * T * D;
  const float lc = fminf(fmaxf(lam, 0.0f), 1.0f);
  load_rows<D>(Q1, q1 + base, m * XB, T);
  load_rows<D>(Q2, q2 + base, m * XB, T);
  if constexpr (NORM) {
    __syncthreads();
    if (tid < XB) row_inv_norms<D>(Q1, rn, tid);
    else if (tid < 2 * XB) row_inv_norms<D>(Q2, rn + XB, tid - XB);
  }
  float tau[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) tau[r] = tau_f32(m * XB + ty + 16 * r, beta, D);
  float acc[4][D / 16];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < D / 16; ++c) acc[r][c] = 0.0f;

  for (int n = 0; n <= m; ++n) {
    __syncthreads();
    load_rows<D>(K1, k1 + base, n * XB, T);
    load_rows<D>(K2, k2 + base, n * XB, T);
    load_rows<D>(Vs, v + base, n * XB, T);
    __syncthreads();
    if constexpr (NORM) {
      if (tid < XB) row_inv_norms<D>(K1, rn + 2 * XB, tid);
      else if (tid < 2 * XB) row_inv_norms<D>(K2, rn + 3 * XB, tid - XB);
      __syncthreads();
    }
    float s1[4][4], s2[4][4];
    dot4x4<D>(Q1, K1, ty, tx, s1);
    dot4x4<D>(Q2, K2, ty, tx, s2);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int row = m * XB + ty + 16 * r;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int key = n * XB + tx + 16 * c;
        float a = s1[r][c], b = s2[r][c];
        if constexpr (NORM) {
          a *= rn[ty + 16 * r] * rn[2 * XB + tx + 16 * c];
          b *= rn[XB + ty + 16 * r] * rn[3 * XB + tx + 16 * c];
        }
        const float w = relu_pow<PC>(a - tau[r], p) - lc * relu_pow<PC>(b - tau[r], p);
        Ws[(ty + 16 * r) * (XB + 1) + tx + 16 * c] = key <= row ? w : 0.0f;
      }
    }
    __syncthreads();
    accum_wx<D>(Ws, Vs, ty, tx, acc);
  }
  store_rows<D>(out + base, m * XB, T, ty, tx, acc);
}

template <int D, int PC, bool NORM>
int launch_diff(const float* q1, const float* q2, const float* k1, const float* k2, const float* v, float* out,
                int BH, int T, float beta, float p, float lam, cudaStream_t stream) {
  constexpr int QS = D + 1;
  constexpr size_t smem = sizeof(float) * (5 * XB * QS + XB * (XB + 1) + 4 * XB);
  auto kern = tra_f32_diff_kernel<D, PC, NORM>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return ERR_LAUNCH;
  const int nM = (T + XB - 1) / XB;
  const long long grid = static_cast<long long>(nM) * BH;
  if (grid > 0x7fffffffLL) return ERR_SHAPE;
  kern<<<static_cast<unsigned>(grid), XTHREADS, smem, stream>>>(q1, q2, k1, k2, v, out, BH, T, nM, beta, p, lam);
  return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
}

template <int D, bool NORM>
int diff_pc(const float* q1, const float* q2, const float* k1, const float* k2, const float* v, float* out, int BH,
            int T, float beta, float p, float lam, cudaStream_t stream) {
  const int pc = power_class(p);
  if (pc == POW_TWO) return launch_diff<D, POW_TWO, NORM>(q1, q2, k1, k2, v, out, BH, T, beta, p, lam, stream);
  if (pc == POW_ONE) return launch_diff<D, POW_ONE, NORM>(q1, q2, k1, k2, v, out, BH, T, beta, p, lam, stream);
  return launch_diff<D, POW_GENERAL, NORM>(q1, q2, k1, k2, v, out, BH, T, beta, p, lam, stream);
}

}  // namespace

namespace {

template <int D>
int bwd_pc(const float* q, const float* k, const float* v, const float* dout, float* dq, float* dk, float* dv, int BH,
           int T, float beta, float p, cudaStream_t stream) {
  const int pc = power_class(p);
  if (pc == POW_TWO) return launch_bwd<D, POW_TWO>(q, k, v, dout, dq, dk, dv, BH, T, beta, p, stream);
  if (pc == POW_ONE) return launch_bwd<D, POW_ONE>(q, k, v, dout, dq, dk, dv, BH, T, beta, p, stream);
  return launch_bwd<D, POW_GENERAL>(q, k, v, dout, dq, dk, dv, BH, T, beta, p, stream);
}

template <int D>
int diff_norm(const float* q1, const float* q2, const float* k1, const float* k2, const float* v, float* out, int BH,
              int T, float beta, float p, float lam, bool normalize, cudaStream_t stream) {
  return normalize ? diff_pc<D, true>(q1, q2, k1, k2, v, out, BH, T, beta, p, lam, stream)
                   : diff_pc<D, false>(q1, q2, k1, k2, v, out, BH, T, beta, p, lam, stream);
}

}  // namespace

int launch_tra_bwd_f32(const float* q, const float* k, const float* v, const float* dout, float* dq, float* dk,
                       float* dv, int B, int H, int T, int D, float beta, float p, cudaStream_t stream) {
  const int BH = B * H;
  switch (D) {
    case 16: return bwd_pc<16>(q, k, v, dout, dq, dk, dv, BH, T, beta, p, stream);
    case 32: return bwd_pc<32>(q, k, v, dout, dq, dk, dv, BH, T, beta, p, stream);
    case 48: return bwd_pc<48>(q, k, v, dout, dq, dk, dv, BH, T, beta, p, stream);
    case 64: return bwd_pc<64>(q, k, v, dout, dq, dk, dv, BH, T, beta, p, stream);
    case 80: return bwd_pc<80>(q, k, v, dout, dq, dk, dv, BH, T, beta, p, stream);
    case 96: return bwd_pc<96>(q, k, v, dout, dq, dk, dv, BH, T, beta, p, stream);
    case 112: return bwd_pc<112>(q, k, v, dout, dq, dk, dv, BH, T, beta, p, stream);
    case 128: return bwd_pc<128>(q, k, v, dout, dq, dk, dv, BH, T, beta, p, stream);
    default: return ERR_UNSUPPORTED;
  }
}

int launch_tra_diff_f32(const float* q1, const float* q2, const float* k1, const float* k2, const float* v,
                        float* out, int B, int H, int T, int D, float beta, float lam, float p, bool normalize,
                        cudaStream_t stream) {
  const int BH = B * H;
  switch (D) {
    case 16: return diff_norm<16>(q1, q2, k1, k2, v, out, BH, T, beta, p, lam, normalize, stream);
    case 32: return diff_norm<32>(q1, q2, k1, k2, v, out, BH, T, beta, p, lam, normalize, stream);
    case 48: return diff_norm<48>(q1, q2, k1, k2, v, out, BH, T, beta, p, lam, normalize, stream);
    case 64: return diff_norm<64>(q1, q2, k1, k2, v, out, BH, T, beta, p, lam, normalize, stream);
    case 80: return diff_norm<80>(q1, q2, k1, k2, v, out, BH, T, beta, p, lam, normalize, stream);
    case 96: return diff_norm<96>(q1, q2, k1, k2, v, out, BH, T, beta, p, lam, normalize, stream);
    case 112: return diff_norm<112>(q1, q2, k1, k2, v, out, BH, T, beta, p, lam, normalize, stream);
    case 128: return diff_norm<128>(q1, q2, k1, k2, v, out, BH, T, beta, p, lam, normalize, stream);
    default: return ERR_UNSUPPORTED;
  }
}

}  // namespace bsa
