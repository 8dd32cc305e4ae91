// tra_diff_bwd.cu -- gradients of the threshold differential attention.
//
// Method: page "triton_threshold_attention.py", differential_threshold_rela_triton
// (differentiated through its normalisation, its two ThresholdRelaFunction
// calls and the clamp of lambda):
//     out = TRA(a1, b1, v) - c TRA(a2, b2, v),  c = clamp(lambda, 0, 1),
//     a = n(q), b = n(k) with n(x) = x / max(||x||, 1e-12) row by row
//     (torch.nn.functional.normalize), or the identity without normalize.
// TRA's gradients are linear in the upstream gradient, so both paths run the
// threshold-attention backward with dout itself and path 2's are scaled by
// -c afterwards:
//     dv = dv1 - c dv2,  da1, db1 from path 1, da2 = -c da2', db2 = -c db2',
//     dx = (g - n(x) (n(x) . g)) / ||x||  through the normalisation
//     (g / 1e-12 for rows whose norm is at most 1e-12),
//     dlambda = -sum(dout * TRA(a2, b2, v)) for 0 < lambda < 1, else 0.
// With TRA(a2, b2, v) = W2 v and path 2's unscaled dv2 = W2^T dout, that sum
// is sum_ij dout_i W2_ij v_j = sum(v * dv2): dlambda comes from a dot product
// over gradients the backward passes already made, with no forward pass.
// The normalised rows go to the backward kernels as copies in the input
// dtype; the gradients through the normalisation are taken in fp32 from the
// inputs and their inverse norms.  Glue kernels here: the normalisation and
// the combination (16-byte accesses, the lanes of a row summing by shuffles;
// the combination also sums v * dv2 for dlambda); the two backward passes are
// the library's own kernels.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bsa {
namespace {

constexpr float NORM_EPS = 1e-12f;

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// Rows are handled by L lanes each (L = the power of two >= D / V, V = 16 /
// sizeof(T) elements per 16-byte access), 32 / L rows per warp; lane j of a
// row holds columns V j .. V j + V - 1 (none past D).  Sums over a row's
// lanes use the xor-shuffle within its aligned group of L lanes.
template <typename T>
struct Vec {
  static constexpr int V = 16 / sizeof(T);
  float f[V];
  __device__ __forceinline__ void load(const T* p) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    if constexpr (sizeof(T) == 4) {
      f[0] = __uint_as_float(u.x), f[1] = __uint_as_float(u.y), f[2] = __uint_as_float(u.z),
      f[3] = __uint_as_float(u.w);
    } else {
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      }
    }
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < V; ++i) f[i] = 0.0f;
  }
  __device__ __forceinline__ void store(T* p) const {
    uint4 u;
    if constexpr (sizeof(T) == 4) {
      u = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
    } else {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
      u = make_uint4(w[0], w[1], w[2], w[3]);
    }
    *reinterpret_cast<uint4*>(p) = u;
  }
};

__device__ __forceinline__ float group_sum(float s, int L) {
  for (int o = L >> 1; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// Rows of q1, q2, k1, k2 (rows each, D columns): xn = x / max(||x||, eps) in
// T, and inv = 1 / max(||x||, eps), for the four inputs laid end to end
// (row w of input i is row i * rows + w).
template <typename T>
__global__ void __launch_bounds__(256) diff_bwd_normalize_kernel(const T* __restrict__ x0, const T* __restrict__ x1,
                                                                 const T* __restrict__ x2, const T* __restrict__ x3,
                                                                 T* __restrict__ xn, float* __restrict__ inv,
                                                                 long long rows, int D, int L) {
  constexpr int V = Vec<T>::V;
  const int lane = threadIdx.x & 31, j = lane % L;
  const long long rpw = 32 / L;  // rows per warp
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const bool has = j * V < D;
  // two rows per lane group and pass, both loads issued before either is used
  for (long long w0 = ((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * rpw; w0 < 4 * rows;
       w0 += 2 * nw * rpw) {
    long long w[2];
    bool live[2];
    Vec<T> x[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      w[u] = w0 + u * nw * rpw + lane / L;
      live[u] = w[u] < 4 * rows && has;
      x[u].zero();
      if (live[u]) {
        // which input (no 64-bit division: this kernel is otherwise a copy)
        const int which = (w[u] >= rows) + (w[u] >= 2 * rows) + (w[u] >= 3 * rows);
        const long long r = w[u] - which * rows;
        x[u].load((which == 0 ? x0 : which == 1 ? x1 : which == 2 ? x2 : x3) + r * D + j * V);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float s = 0.0f;
#pragma unroll
      for (int i = 0; i < V; ++i) s += x[u].f[i] * x[u].f[i];
      const float iv = 1.0f / fmaxf(sqrtf(group_sum(s, L)), NORM_EPS);
      if (live[u]) {
#pragma unroll
        for (int i = 0; i < V; ++i) x[u].f[i] *= iv;
        x[u].store(xn + w[u] * D + j * V);
        if (j == 0) inv[w[u]] = iv;
      }
    }
  }
}

struct DiffGrads {
  const float *da1, *da2;                // the two passes' query gradients, fp32 (path 2 unscaled)
  const void *db1, *db2, *dv1, *dv2;     // their key and value gradients, in T (path 2 unscaled)
  void *dq1, *dq2, *dk1, *dk2, *dv;      // outputs
};

// V consecutive fp32 values (V = 4 or 8, 16-byte aligned).
template <int V>
__device__ __forceinline__ void load_f32(const float* p, float (&f)[V]) {
#pragma unroll
  for (int h = 0; h < V / 4; ++h) {
    const float4 u = reinterpret_cast<const float4*>(p)[h];
    f[4 * h] = u.x, f[4 * h + 1] = u.y, f[4 * h + 2] = u.z, f[4 * h + 3] = u.w;
  }
}

// dv = dv1 - c dv2, and for q1, q2, k1, k2 the gradient g (path 2 scaled by
// -c) taken back through the normalisation when inv is given (inv: 4 * rows
// factors in the order q1, q2, k1, k2); rows laid out as in the
// normalisation kernel.  With dlam (zeroed before): *dlam -= sum(v * dv2),
// block sums added with one fp32 atomic per block.
template <typename T>
__global__ void __launch_bounds__(256) diff_bwd_combine_kernel(const T* __restrict__ q1, const T* __restrict__ q2,
                                                               const T* __restrict__ k1, const T* __restrict__ k2,
                                                               const T* __restrict__ v, const float* __restrict__ inv,
                                                               DiffGrads g, float c, long long rows, int D, int L,
                                                               float* dlam) {
  __shared__ float part[8];
  float sl = 0.0f;  // this thread's share of sum(v * dv2)
  constexpr int V = Vec<T>::V;
  const int lane = threadIdx.x & 31, j = lane % L;
  const long long rpw = 32 / L;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const bool has = j * V < D;
  for (long long r0 = ((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * rpw; r0 < rows;
       r0 += nw * rpw) {
    const long long r = r0 + lane / L;
    const bool live = r < rows && has;
    const long long off = r * D + j * V;
    // every load of the row first (dv1, dv2, v, the four gradients and their
    // inputs), then the arithmetic and the stores
    Vec<T> a, b, vv, gv[4], xv[4];
    float iv[4];
#pragma unroll
    for (int which = 0; which < 4; ++which) {
      gv[which].zero();
      xv[which].zero();
      iv[which] = inv != nullptr && r < rows ? inv[which * rows + r] : 1.0f;
    }
    if (live) {
      a.load(static_cast<const T*>(g.dv1) + off);
      b.load(static_cast<const T*>(g.dv2) + off);
      if (dlam != nullptr) vv.load(v + off);
#pragma unroll
      for (int which = 0; which < 4; ++which) {
        if (which < 2)
          load_f32<V>((which == 0 ? g.da1 : g.da2) + off, gv[which].f);
        else
          gv[which].load(static_cast<const T*>(which == 2 ? g.db1 : g.db2) + off);
        if (inv != nullptr) xv[which].load((which == 0 ? q1 : which == 1 ? q2 : which == 2 ? k1 : k2) + off);
      }
      if (dlam != nullptr) {
#pragma unroll
        for (int i = 0; i < V; ++i) sl += vv.f[i] * b.f[i];
      }
#pragma unroll
      for (int i = 0; i < V; ++i) a.f[i] -= c * b.f[i];
      a.store(static_cast<T*>(g.dv) + off);
    }
#pragma unroll
    for (int which = 0; which < 4; ++which) {
      const float scale = (which & 1) ? -c : 1.0f;  // path 2 (q2, k2) carries -c
      float dot = 0.0f;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        gv[which].f[i] *= scale;
        xv[which].f[i] *= iv[which];
        dot += xv[which].f[i] * gv[which].f[i];
      }
      dot = group_sum(dot, L);
      // rows with a norm above eps: (g - xn (xn . g)) / ||x||; else g / eps
      const bool proj = iv[which] < 1.0f / NORM_EPS;
      if (live) {
        if (inv != nullptr) {
#pragma unroll
          for (int i = 0; i < V; ++i)
            gv[which].f[i] = (proj ? gv[which].f[i] - xv[which].f[i] * dot : gv[which].f[i]) * iv[which];
        }
        gv[which].store(static_cast<T*>(which == 0 ? g.dq1 : which == 1 ? g.dq2 : which == 2 ? g.dk1 : g.dk2) + off);
      }
    }
  }
  if (dlam != nullptr) {  // uniform across the launch: every thread reaches the barrier
    sl = warp_sum(sl);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = sl;
    __syncthreads();
    if (threadIdx.x < 32) {
      sl = threadIdx.x < (blockDim.x >> 5) ? part[threadIdx.x] : 0.0f;
      sl = warp_sum(sl);
      if (threadIdx.x == 0) atomicAdd(dlam, -sl);
    }
  }
}

size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

// Lanes per row: the power of two >= D / V.
int lanes_per_row(int D, int V) {
  int L = 1;
  while (L * V < D) L <<= 1;
  return L;
}

unsigned grid_for(long long warps_needed) {
  const int sms = sm_count();
  const long long cap = 16LL * (sms > 0 ? sms : 148);
  const long long blocks = (warps_needed + 7) / 8;  // 8 warps per 256-thread block
  return static_cast<unsigned>(blocks < 1 ? 1 : blocks < cap ? blocks : cap);
}

}  // namespace

size_t tra_diff_bwd_scratch_bytes(int B, int H, int T, int D, bool f32, bool normalize, bool dlam) {
  const size_t n = static_cast<size_t>(B) * H * T * D, rows = static_cast<size_t>(B) * H * T;
  const size_t el = f32 ? 4 : 2;
  // da1, da2 in fp32 (for bf16 the fused backward's dq accumulators, read
  // without a conversion), db1, db2, dv1, dv2 in the input dtype
  size_t b = 2 * align256(n * sizeof(float)) + 4 * align256(n * el);
  if (normalize) b += align256(4 * n * el) + align256(4 * rows * sizeof(float));
  (void)dlam;  // dlambda needs no temporary: it is summed from v and dv2
  return b;
}

int launch_tra_diff_bwd(const void* q1, const void* q2, const void* k1, const void* k2, const void* v,
                        const void* dout, void* dq1, void* dq2, void* dk1, void* dk2, void* dv, float* dlam, int B,
                        int H, int T, int D, float beta, float lam, float p, bool normalize, bool f32, void* scratch,
                        cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * H * T;
  const size_t n = static_cast<size_t>(rows) * D, el = f32 ? 4 : 2;
  const float c = fminf(fmaxf(lam, 0.0f), 1.0f);
  const bool want_dlam = dlam != nullptr && lam > 0.0f && lam < 1.0f;
  uint8_t* s = static_cast<uint8_t*>(scratch);
  auto take = [&](size_t bytes) {
    uint8_t* r = s;
    s += align256(bytes);
    return static_cast<void*>(r);
  };
  void* gr[6];  // da1, da2 (fp32), db1, db2, dv1, dv2 (input dtype)
  for (int i = 0; i < 6; ++i) gr[i] = take(n * (i < 2 ? sizeof(float) : el));
  const void *a1 = q1, *a2 = q2, *b1 = k1, *b2 = k2;
  float* inv = nullptr;
  if (normalize) {
    // the four normalised copies back to back (the kernel's row w of input i
    // is row i * rows + w); n * el is a multiple of 32 bytes, so each copy
    // starts 16-byte aligned as the tensor maps need
    uint8_t* xn = static_cast<uint8_t*>(take(4 * n * el));
    const void* cp[4] = {xn, xn + n * el, xn + 2 * n * el, xn + 3 * n * el};
    inv = static_cast<float*>(take(4 * static_cast<size_t>(rows) * sizeof(float)));
    a1 = cp[0], a2 = cp[1], b1 = cp[2], b2 = cp[3];
    const int L = lanes_per_row(D, f32 ? 4 : 8);
    const unsigned grid = grid_for((4 * rows * L + 31) / 32);
    if (f32)
      diff_bwd_normalize_kernel<float><<<grid, 256, 0, stream>>>(
          static_cast<const float*>(q1), static_cast<const float*>(q2), static_cast<const float*>(k1),
          static_cast<const float*>(k2), reinterpret_cast<float*>(xn), inv, rows, D, L);
    else
      diff_bwd_normalize_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(q1), static_cast<const __nv_bfloat16*>(q2),
          static_cast<const __nv_bfloat16*>(k1), static_cast<const __nv_bfloat16*>(k2),
          reinterpret_cast<__nv_bfloat16*>(xn), inv, rows, D, L);
    if (cudaGetLastError() != cudaSuccess) return ERR_LAUNCH;
  }
  // the two threshold-attention backward passes, both with dout
  int st;
  if (f32) {
    st = launch_tra_bwd_f32(static_cast<const float*>(a1), static_cast<const float*>(b1), static_cast<const float*>(v),
                            static_cast<const float*>(dout), static_cast<float*>(gr[0]), static_cast<float*>(gr[2]),
                            static_cast<float*>(gr[4]), B, H, T, D, beta, p, stream);
    if (st == OK)
      st = launch_tra_bwd_f32(static_cast<const float*>(a2), static_cast<const float*>(b2),
                              static_cast<const float*>(v), static_cast<const float*>(dout), static_cast<float*>(gr[1]),
                              static_cast<float*>(gr[3]), static_cast<float*>(gr[5]), B, H, T, D, beta, p, stream);
  } else {
    // each pass leaves its dq in its own fp32 accumulator (no conversion)
    st = launch_tra_bwd_fused_bf16(a1, b1, v, dout, nullptr, gr[2], gr[4], B, H, T, D, beta, p,
                                   static_cast<float*>(gr[0]), stream);
    if (st == OK)
      st = launch_tra_bwd_fused_bf16(a2, b2, v, dout, nullptr, gr[3], gr[5], B, H, T, D, beta, p,
                                     static_cast<float*>(gr[1]), stream);
  }
  if (st != OK) return st;
  if (dlam != nullptr && cudaMemsetAsync(dlam, 0, sizeof(float), stream) != cudaSuccess) return ERR_LAUNCH;
  float* dl = want_dlam ? dlam : nullptr;
  const DiffGrads g{static_cast<const float*>(gr[0]), static_cast<const float*>(gr[1]), gr[2], gr[3], gr[4], gr[5],
                    dq1, dq2, dk1, dk2, dv};
  const int L = lanes_per_row(D, f32 ? 4 : 8);
  const unsigned grid = grid_for((rows * L + 31) / 32);
  if (f32)
    diff_bwd_combine_kernel<float><<<grid, 256, 0, stream>>>(
        static_cast<const float*>(q1), static_cast<const float*>(q2), static_cast<const float*>(k1),
        static_cast<const float*>(k2), static_cast<const float*>(v), inv, g, c, rows, D, L, dl);
  else
    diff_bwd_combine_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(q1), static_cast<const __nv_bfloat16*>(q2),
        static_cast<const __nv_bfloat16*>(k1), static_cast<const __nv_bfloat16*>(k2),
        static_cast<const __nv_bfloat16*>(v), inv, g, c, rows, D, L, dl);
  if (cudaGetLastError() != cudaSuccess) return ERR_LAUNCH;
  return OK;
}

}  // namespace bsa
