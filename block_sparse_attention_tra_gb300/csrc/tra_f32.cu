// tra_f32.cu -- threshold rectified attention forward in fp32 on the CUDA
// cores (FFMA throughout; TF32 tensor cores would miss a 1e-4 relative bar).
//
// Method: page "triton_threshold_attention.py" (module docstring formula and
// _threshold_rela_fwd_kernel): out_i = sum_{j<=i} ReLU(q_i.k_j - tau(i))^p v_j
// with tau(i) = beta sqrt(2 ln(i+1)/D), causal, unnormalised.
//
// One CTA (256 threads) owns a 64-row query tile of one (b, h) and walks the
// key tiles 0..m (64 keys each).  Thread (ty, tx) computes scores for rows
// ty + 16a and keys tx + 16c (a, c < 4), writes the weights to shared memory,
// then accumulates output rows ty + 16a, columns tx + 16c (c < D/16).
#include "kernels.h"
#include "ptx.cuh"

namespace bsa {
namespace {

constexpr int FBM = 64;
constexpr int FBN = 64;
constexpr int FTHREADS = 256;

template <int PC>
__device__ __forceinline__ float relu_pow_f32(float x, float p) {
  const float r = fmaxf(x, 0.0f);
  if constexpr (PC == POW_ONE) {
    return r;
  } else if constexpr (PC == POW_TWO) {
    return r * r;
  } else {
    return r > 0.0f ? exp2f(p * log2f(r)) : 0.0f;
  }
}

template <int D, int PC>
__global__ void __launch_bounds__(FTHREADS) tra_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                                                          const float* __restrict__ v, float* __restrict__ out,
                                                          int BH, int T, int nM, float beta, float p) {
  constexpr int QS = D + 1;  // padded row stride (bank-conflict free column reads)
  extern __shared__ float fsm[];
  float* Qs = fsm;               // [FBM][QS]
  float* Ks = Qs + FBM * QS;     // [FBN][QS]
  float* Vs = Ks + FBN * QS;     // [FBN][D]
  float* Ws = Vs + FBN * D;      // [FBM][FBN + 1]

  const int m = nM - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const size_t base = static_cast<size_t>(bh) * T * D;

  for (int e = tid; e < FBM * D; e += FTHREADS) {
    const int r = e / D, d = e % D;
    const int row = m * FBM + r;
    Qs[r * QS + d] = row < T ? q[base + static_cast<size_t>(row) * D + d] : 0.0f;
  }

  float tau[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int row = m * FBM + ty + 16 * a;
    tau[a] = beta * sqrtf(2.0f * logf(static_cast<float>(row + 1)) / static_cast<float>(D));
  }

  float acc[4][D / 16];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < D / 16; ++c) acc[a][c] = 0.0f;

  for (int n = 0; n <= m; ++n) {
    __syncthreads();
    for (int e = tid; e < FBN * D; e += FTHREADS) {
      const int r = e / D, d = e % D;
      const int key = n * FBN + r;
      const bool in = key < T;
      Ks[r * QS + d] = in ? k[base + static_cast<size_t>(key) * D + d] : 0.0f;
      Vs[r * D + d] = in ? v[base + static_cast<size_t>(key) * D + d] : 0.0f;
    }
    __syncthreads();

    float s[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[a][c] = 0.0f;
#pragma unroll 8
    for (int d = 0; d < D; ++d) {
      float qa[4], kc[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) qa[a] = Qs[(ty + 16 * a) * QS + d];
#pragma unroll
      for (int c = 0; c < 4; ++c) kc[c] = Ks[(tx + 16 * c) * QS + d];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[a][c] = fmaf(qa[a], kc[c], s[a][c]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int row = m * FBM + ty + 16 * a;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int key = n * FBN + tx + 16 * c;
        float w = relu_pow_f32<PC>(s[a][c] - tau[a], p);
        if (key > row) w = 0.0f;  // causal: keys j <= i only
        Ws[(ty + 16 * a) * (FBN + 1) + tx + 16 * c] = w;
      }
    }
    __syncthreads();

#pragma unroll 4
    for (int j = 0; j < FBN; ++j) {
      float wa[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) wa[a] = Ws[(ty + 16 * a) * (FBN + 1) + j];
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {
        const float vv = Vs[j * D + tx + 16 * c];
#pragma unroll
        for (int a = 0; a < 4; ++a) acc[a][c] = fmaf(wa[a], vv, acc[a][c]);
      }
    }
  }

#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int row = m * FBM + ty + 16 * a;
    if (row < T) {
#pragma unroll
      for (int c = 0; c < D / 16; ++c) out[base + static_cast<size_t>(row) * D + tx + 16 * c] = acc[a][c];
    }
  }
}

template <int D, int PC>
int launch(const float* q, const float* k, const float* v, float* out, int BH, int T, float beta, float p,
           cudaStream_t stream) {
  constexpr int QS = D + 1;
  constexpr size_t smem = sizeof(float) * (FBM * QS + FBN * QS + FBN * D + FBM * (FBN + 1));
  auto kern = tra_f32_kernel<D, PC>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return ERR_LAUNCH;
  const int nM = (T + FBM - 1) / FBM;
  const long long grid = static_cast<long long>(nM) * BH;
  if (grid > 0x7fffffffLL) return ERR_SHAPE;
  kern<<<static_cast<unsigned>(grid), FTHREADS, smem, stream>>>(q, k, v, out, BH, T, nM, beta, p);
  return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
}

template <int D>
int launch_d(const float* q, const float* k, const float* v, float* out, int BH, int T, float beta, float p,
             cudaStream_t stream) {
  const int pc = power_class(p);
  if (pc == POW_TWO) return launch<D, POW_TWO>(q, k, v, out, BH, T, beta, p, stream);
  if (pc == POW_ONE) return launch<D, POW_ONE>(q, k, v, out, BH, T, beta, p, stream);
  return launch<D, POW_GENERAL>(q, k, v, out, BH, T, beta, p, stream);
}

}  // namespace

int launch_tra_f32(const float* q, const float* k, const float* v, float* out, int B, int H, int T, int D,
                   float beta, float p, cudaStream_t stream) {
  const int BH = B * H;
  switch (D) {
    case 16: return launch_d<16>(q, k, v, out, BH, T, beta, p, stream);
    case 32: return launch_d<32>(q, k, v, out, BH, T, beta, p, stream);
    case 48: return launch_d<48>(q, k, v, out, BH, T, beta, p, stream);
    case 64: return launch_d<64>(q, k, v, out, BH, T, beta, p, stream);
    case 80: return launch_d<80>(q, k, v, out, BH, T, beta, p, stream);
    case 96: return launch_d<96>(q, k, v, out, BH, T, beta, p, stream);
    case 112: return launch_d<112>(q, k, v, out, BH, T, beta, p, stream);
    case 128: return launch_d<128>(q, k, v, out, BH, T, beta, p, stream);
    default: return ERR_UNSUPPORTED;
  }
}

unsigned int tra_f32_device_error() { return read_and_clear_device_error(); }

}  // namespace bsa
