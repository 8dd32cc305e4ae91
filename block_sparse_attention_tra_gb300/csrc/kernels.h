// kernels.h -- host-side launchers shared between the C ABI (api.cu) and the
// kernel translation units.  Internal to libbsa.so; not installed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bsa {

// Status codes mirror bsa_status in include/bsa.h.
enum Status : int {
  OK = 0,
  ERR_NULLPTR = 1,
  ERR_SHAPE = 2,
  ERR_DTYPE = 3,
  ERR_UNSUPPORTED = 4,
  ERR_LAUNCH = 5,
  ERR_DEVICE = 6,
  ERR_ALIGN = 7,
  ERR_MEMORY = 8,
  ERR_SCRATCH_LIMIT = 9,
};

// Encode a rank-3 bf16 (or other 2-byte) tensor map with 128-byte swizzle.
// dims / box are innermost first; strides are byte strides of dims 1 and 2.
int encode_tmap_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                   uint32_t box2);
// Rank-2 fp32 tensor map (d0 innermost), 128-byte swizzle: used for TMA
// stores of fp32 rows from shared memory.
int encode_tmap_2d_f32(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t stride1_bytes,
                      uint32_t box0, uint32_t box1);
// Rank-3 fp32 tensor map, 128-byte swizzle (TMA reduce-adds of fp32 boxes).
int encode_tmap_3d_f32(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1, uint32_t box2);

// Streaming multiprocessors of the current device (cached per device; 0 if
// the query fails).  Persistent kernels size their grids with it, the
// head-grouped block orders their group sizes.
int sm_count();

// Threshold rectified attention, fp32 CUDA-core kernel.
int launch_tra_f32(const float* q, const float* k, const float* v, float* out, int B, int H, int T, int D,
                   float beta, float p, cudaStream_t stream);

// Threshold rectified attention, bf16 tcgen05 kernel.  sqrt_half_powers:
// p = k + 1/2 (k = 0..3) runs as x^k sqrt(x) instead of exp2(p log2 x).
int launch_tra_bf16(const void* q, const void* k, const void* v, void* out, int B, int H, int T, int D,
                    float beta, float p, bool sqrt_half_powers, cudaStream_t stream);

// Threshold rectified attention backward (dq, dk, dv), bf16 tcgen05 kernels.
int launch_tra_bwd_bf16(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk, void* dv,
                        int B, int H, int T, int D, float beta, float p, cudaStream_t stream);

// The same backward as one fused kernel: the scores and dP of each (key tile,
// query tile) pair are computed once, dk and dv accumulate in tensor memory
// and each pair's dq partial is added into dq_acc (fp32, B*H*T*D elements,
// 16-byte aligned), which this call zeroes first and converts into dq last.
// The order of those fp32 additions varies from run to run.  dq may be null:
// dQ is then left in dq_acc (fp32) and not converted.
int launch_tra_bwd_fused_bf16(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk,
                              void* dv, int B, int H, int T, int D, float beta, float p, float* dq_acc,
                              cudaStream_t stream);

// Gradients of the threshold differential attention (tra_diff_bwd.cu): the
// normalisation, both paths' backward passes, their combination and dlam
// (nullable; written, 0 outside 0 < lam < 1).  scratch: 256-byte aligned, at
// least tra_diff_bwd_scratch_bytes(B, H, T, D, f32, normalize, dlam != null).
size_t tra_diff_bwd_scratch_bytes(int B, int H, int T, int D, bool f32, bool normalize, bool dlam);
int launch_tra_diff_bwd(const void* q1, const void* q2, const void* k1, const void* k2, const void* v,
                        const void* dout, void* dq1, void* dq2, void* dk1, void* dk2, void* dv, float* dlam, int B,
                        int H, int T, int D, float beta, float lam, float p, bool normalize, bool f32, void* scratch,
                        cudaStream_t stream);

// fp32 forms of the backward and of the differential forward (CUDA-core FFMA
// kernels, tra_f32_ext.cu); the differential one needs no scratch memory.
int launch_tra_bwd_f32(const float* q, const float* k, const float* v, const float* dout, float* dq, float* dk,
                       float* dv, int B, int H, int T, int D, float beta, float p, cudaStream_t stream);
int launch_tra_diff_f32(const float* q1, const float* q2, const float* k1, const float* k2, const float* v,
                        float* out, int B, int H, int T, int D, float beta, float lam, float p, bool normalize,
                        cudaStream_t stream);

// Threshold differential attention (fused two-stream kernel).  inv_norm is a
// float scratch buffer of tra_diff_scratch_bytes(B, H, T) bytes (256-byte
// aligned) for the row normalisation factors, or null to skip the
// normalisation.  knorm (16-byte aligned, 2*B*H*T*D bf16) or null: where the
// pre-pass writes normalised copies of k1 and k2 for the kernel to read; the
// kernel then takes the query rows' factors from its Q tiles and inv_norm is
// not used (it may be null).  Without knorm (and with inv_norm) the kernel
// scales every score by both rows' factors from inv_norm.
size_t tra_diff_scratch_bytes(int B, int H, int T);
int launch_tra_diff_bf16(const void* q1, const void* q2, const void* k1, const void* k2, const void* v, void* out,
                         int B, int H, int T, int D, float beta, float lam, float p, float* inv_norm, void* knorm,
                         cudaStream_t stream);

// Allocation-free variant: the normalisation factors go to a fixed device
// array of TRA_DIFF_NOALLOC_MAX_ROWS rows per input (see tra_diff.cu).
constexpr long long TRA_DIFF_NOALLOC_MAX_ROWS = 1LL << 20;
bool tra_diff_noalloc_fits(int B, int H, int T);
int launch_tra_diff_noalloc_bf16(const void* q1, const void* q2, const void* k1, const void* k2, const void* v,
                                 void* out, int B, int H, int T, int D, float beta, float lam, float p,
                                 bool normalize, cudaStream_t stream);

// NSA selection attention, bf16 kernel.
int launch_nsa_select(const void* q, const void* k, const void* v, const int32_t* block_idx, void* out,
                      float* lse, int B, int Hq, int Hkv, int T, int D, int block_size, int S,
                      cudaStream_t stream);

// NSA selection attention for any accepted head dim and block size (cp.async
// + mma.sync kernel); launch_nsa_select hands other shapes to it.
int launch_nsa_general(const void* q, const void* k, const void* v, const int32_t* block_idx, void* out, float* lse,
                       int B, int Hq, int Hkv, int T, int D, int block_size, int S, cudaStream_t stream);

// NSA selection attention, block-outer split-K form with a log-sum-exp
// combine (nsa_fsa.cu).  `workspace` holds nsa_fsa_workspace_bytes(...) bytes,
// 256-byte aligned; block_size is 64.
size_t nsa_fsa_workspace_bytes(int B, int Hq, int Hkv, int T, int D, int S);

// Threshold attention on host-resident tensors, streamed through the GPU in
// chunks of heads with overlapped copies (tra_host.cu).  `workspace` holds
// tra_host_workspace_bytes(...) bytes of 256-byte aligned device memory.
int tra_host_chunk_heads(long long BH);
size_t tra_host_workspace_bytes(long long BH, int T, int D, int elsize);
int launch_tra_host(const void* q, const void* k, const void* v, void* out, int B, int H, int T, int D, float beta,
                    float p, bool f32, void* workspace, cudaStream_t stream);
int launch_nsa_fsa(const void* q, const void* k, const void* v, const int32_t* block_idx, void* out, float* lse,
                   int B, int Hq, int Hkv, int T, int D, int S, void* workspace, cudaStream_t stream);

// Self tests (selftest.cu): the bounded wait's expiry branch (result = 0 when
// the wait gave up, 1 if it unexpectedly completed) and the FMA-pipe log2
// beside CUDA's log2f.
int launch_selftest_wait_timeout(long long limit_cycles, int* result, cudaStream_t stream);
int launch_selftest_log2(const float* x, float* y_fma, float* y_ref, int n, cudaStream_t stream);
int launch_selftest_exp2(const float* y, float* w_fma, float* w_ref, int n, cudaStream_t stream);
// Streaming read of a device buffer `reps` times (L2 / HBM read-rate probe).
int launch_read_probe(const void* buf, long long bytes, int reps, unsigned int* sink, cudaStream_t stream);

// Read-and-clear of each kernel file's device error word (0 = none,
// 1 = a bounded wait timed out; 0xffffffff = the read itself failed).
unsigned int tra_bf16_device_error();
unsigned int tra_f32_device_error();
unsigned int nsa_device_error();
unsigned int tra_bwd_device_error();
unsigned int tra_diff_device_error();
unsigned int nsa_fsa_device_error();
unsigned int selftest_device_error();

// Power class of the TRA epilogue: p == 1, p == 2, or the general exp2/log2
// path; and, on request only, p = k + 1/2 (k = 0..3) as x^k sqrt(x).
// POW_GENERAL_MIX is the general path with part of the log2 evaluations on
// the FMA pipe instead of the MUFU unit (tra_math.cuh); it serves
// 1 <= p <= POW_MIX_MAX_P, where its exact zeros and its accuracy hold.
enum PowerClass : int { POW_GENERAL = 0, POW_ONE = 1, POW_TWO = 2, POW_HALF0 = 3, POW_HALF3 = 6, POW_GENERAL_MIX = 7 };
constexpr float POW_MIX_MAX_P = 64.0f;

inline int power_class(float p) {
  if (p == 1.0f) return POW_ONE;
  if (p == 2.0f) return POW_TWO;
  return (p >= 1.0f && p <= POW_MIX_MAX_P) ? POW_GENERAL_MIX : POW_GENERAL;
}

// Head dims of the threshold-attention entry points: multiples of 16 up to
// 128.  The bf16 kernels run tile width 64 (D <= 64) or 128 on the tensor
// maps' zero-filled columns past D; the fp32 kernels are built per D.
inline bool tra_head_dim_supported(int D) { return D >= 16 && D <= 128 && D % 16 == 0; }

// POW_HALF0 + k for p = k + 1/2 with k in 0..3, else -1.
inline int half_power_class(float p) {
  for (int k = 0; k <= POW_HALF3 - POW_HALF0; ++k)
    if (p == static_cast<float>(k) + 0.5f) return POW_HALF0 + k;
  return -1;
}

}  // namespace bsa
