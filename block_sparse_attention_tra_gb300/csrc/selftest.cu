// selftest.cu -- self-test entry points of the library: they exercise device
// code paths that the attention calls reach only in rare conditions, so that
// tests can check them on the GPU without faulting or hanging it.
//
//  * the expiry branch of the bounded mbarrier wait that every kernel uses
//    (ptx.cuh, mbar_wait_bounded): one thread waits, with a short limit, on an
//    mbarrier that nothing arrives on; no TMA copy or tcgen05 operation is in
//    flight, so the kernel simply records the timeout code and returns;
//  * the FMA-pipe log2 and exp2 of the general-power epilogue (tra_math.cuh,
//    p_log2_fma and exp2_fma2), evaluated beside CUDA's own log2f and exp2f
//    on the same inputs.
#include "kernels.h"
#include "ptx.cuh"
#include "tra_math.cuh"

namespace bsa {
namespace {

__global__ void wait_timeout_kernel(long long limit_cycles, int* result) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Phase 0 never completes: the single expected arrival never comes.
    const bool ok = mbar_wait_bounded(&bar, 0, limit_cycles);
    *result = ok ? 1 : 0;
  }
}

// y_fma[i] = log2(x[i]) from the epilogue's FMA-pipe evaluation (p = 1);
// y_ref[i] = CUDA's log2f(x[i]).
__global__ void log2_compare_kernel(const float* __restrict__ x, float* __restrict__ y_fma,
                                    float* __restrict__ y_ref, int n) {
  const PowParams w = pow_params(0.0f, 1.0f);
  for (int i2 = 2 * (blockIdx.x * blockDim.x + threadIdx.x); i2 < n; i2 += 2 * gridDim.x * blockDim.x) {
    const float x0 = x[i2], x1 = (i2 + 1 < n) ? x[i2 + 1] : 1.0f;
    float y0, y1;
    f2_unpack(p_log2_fma(x0, x1, w), y0, y1);
    y_fma[i2] = y0;
    y_ref[i2] = log2f(x0);
    if (i2 + 1 < n) {
      y_fma[i2 + 1] = y1;
      y_ref[i2 + 1] = log2f(x1);
    }
  }
}

// w_fma[i] = exp2(y[i]) from the epilogue's FMA-pipe evaluation (before its
// bf16 rounding); w_ref[i] = CUDA's exp2f(y[i]).
__global__ void exp2_compare_kernel(const float* __restrict__ y, float* __restrict__ w_fma,
                                    float* __restrict__ w_ref, int n) {
  for (int i2 = 2 * (blockIdx.x * blockDim.x + threadIdx.x); i2 < n; i2 += 2 * gridDim.x * blockDim.x) {
    const float y0 = y[i2], y1 = (i2 + 1 < n) ? y[i2 + 1] : 0.0f;
    float w0, w1;
    f2_unpack(exp2_fma2(f2_pack(y0, y1)), w0, w1);
    w_fma[i2] = w0;
    w_ref[i2] = exp2f(y0);
    if (i2 + 1 < n) {
      w_fma[i2 + 1] = w1;
      w_ref[i2 + 1] = exp2f(y1);
    }
  }
}

// Streaming read of `n16` 16-byte words, `reps` times, with loads that skip
// L1 (ld.global.cg): on a buffer the L2 already holds, the rate is the L2 read
// bandwidth that the NSA gathers are served from.  The XOR of everything read
// goes to *sink so that no load can be dropped.
__global__ void __launch_bounds__(512) read_probe_kernel(const uint4* __restrict__ buf, long long n16, int reps,
                                                         unsigned int* sink) {
  uint32_t x = 0;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (int r = 0; r < reps; ++r) {
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < n16; e += 4 * stride) {
      uint4 a[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const long long f = e + u * stride;
        if (f < n16)
          asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(a[u].x), "=r"(a[u].y), "=r"(a[u].z), "=r"(a[u].w)
                       : "l"(buf + f));
        else
          a[u] = make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) x ^= a[u].x ^ a[u].y ^ a[u].z ^ a[u].w;
    }
  }
  x = __reduce_xor_sync(0xffffffffu, x);
  if ((threadIdx.x & 31) == 0) atomicXor(sink, x);
}

}  // namespace

int launch_read_probe(const void* buf, long long bytes, int reps, unsigned int* sink, cudaStream_t stream) {
  const int sms = sm_count();
  if (sms <= 0) return ERR_DEVICE;
  read_probe_kernel<<<4 * sms, 512, 0, stream>>>(static_cast<const uint4*>(buf), bytes / 16, reps, sink);
  return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
}

int launch_selftest_wait_timeout(long long limit_cycles, int* result, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_cycles, result);
  return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
}

int launch_selftest_log2(const float* x, float* y_fma, float* y_ref, int n, cudaStream_t stream) {
  const int threads = 256;
  const int blocks = static_cast<int>(((n + 1) / 2 + threads - 1) / threads);
  log2_compare_kernel<<<blocks < 1024 ? (blocks > 0 ? blocks : 1) : 1024, threads, 0, stream>>>(x, y_fma, y_ref, n);
  return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
}

int launch_selftest_exp2(const float* y, float* w_fma, float* w_ref, int n, cudaStream_t stream) {
  const int threads = 256;
  const int blocks = static_cast<int>(((n + 1) / 2 + threads - 1) / threads);
  exp2_compare_kernel<<<blocks < 1024 ? (blocks > 0 ? blocks : 1) : 1024, threads, 0, stream>>>(y, w_fma, w_ref, n);
  return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
}

unsigned int selftest_device_error() { return read_and_clear_device_error(); }

}  // namespace bsa
