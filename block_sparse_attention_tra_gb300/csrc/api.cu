// api.cu -- the C ABI of libbsa.so (declared in include/bsa.h): argument
// validation, dtype / head-dim dispatch and launch on the caller's stream.
// Validation happens on the host before any CUDA call, so a bad argument
// returns an error without touching the device.
#include <math.h>

#include <atomic>
#include <mutex>

#include "../../include/bsa.h"
#include "kernels.h"
#include "ptx.cuh"

namespace bsa {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The library's own stream-ordered memory pool on `dev`, created on first use.
// Its release threshold keeps freed temporaries mapped, so repeated calls
// recycle the same memory instead of mapping it again each time; the
// caller's default pool is left untouched.
cudaMemPool_t scratch_pool(int dev) {
  constexpr int MAX_DEVICES = 64;
  static std::mutex mu;
  static cudaMemPool_t pools[MAX_DEVICES] = {};
  if (dev < 0 || dev >= MAX_DEVICES) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (pools[dev] == nullptr) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
    uint64_t keep = 1ull << 30;  // keep up to 1 GiB of freed temporaries mapped
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    pools[dev] = pool;
  }
  return pools[dev];
}

// Sizes and parameters of the NSA selection entry points (pointers aside).
int check_nsa_shape(int B, int Hq, int Hkv, int T, int D, int block_size, int S) {
  if (B < 1 || Hq < 1 || Hkv < 1 || T < 1 || D < 1 || block_size < 1 || S < 1) return BSA_ERR_SHAPE;
  if (Hq % Hkv != 0) return BSA_ERR_SHAPE;
  if (T % block_size != 0) return BSA_ERR_SHAPE;
  if (S > 32) return BSA_ERR_SHAPE;
  if (static_cast<long long>(B) * Hq * T * D >= (1LL << 40)) return BSA_ERR_SHAPE;
  if (static_cast<long long>(B) * Hq > 0x7fffffffLL || static_cast<long long>(B) * Hkv * T * S >= (1LL << 40))
    return BSA_ERR_SHAPE;
  if (D != 16 && D != 32 && D != 64 && D != 128) return BSA_ERR_UNSUPPORTED;
  if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128) return BSA_ERR_UNSUPPORTED;
  if (Hq / Hkv > 16) return BSA_ERR_UNSUPPORTED;
  return BSA_OK;
}

// The split-K form is built for 64-token blocks of 64 or 128 dims.
bool fsa_shape_supported(int D, int block_size) { return block_size == 64 && (D == 64 || D == 128); }

int check_nsa_args(const void* q, const void* k, const void* v, const int32_t* block_idx, const void* out,
                   const float* lse, int B, int Hq, int Hkv, int T, int D, int block_size, int S) {
  if (q == nullptr || k == nullptr || v == nullptr || block_idx == nullptr || out == nullptr)
    return BSA_ERR_NULLPTR;
  const int sh = check_nsa_shape(B, Hq, Hkv, T, D, block_size, S);
  if (sh != BSA_OK) return sh;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_idx) & 3u) != 0 || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return BSA_ERR_ALIGN;
  return BSA_OK;
}

// The kernels are built for sm_103a only; refuse other devices up front
// instead of failing inside the launch.
int check_device() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ERR_DEVICE;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return ERR_DEVICE;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return ERR_DEVICE;
  if (major != 10 || minor != 3) return ERR_DEVICE;
  return OK;
}

}  // namespace

int encode_tmap_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1, uint32_t box2) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return ERR_DEVICE;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {box0, box1, box2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? OK : ERR_SHAPE;
}

int encode_tmap_2d_f32(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t stride1_bytes,
                      uint32_t box0, uint32_t box1) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return ERR_DEVICE;
  const cuuint64_t dims[2] = {d0, d1};
  const cuuint64_t strides[1] = {stride1_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? OK : ERR_SHAPE;
}

int encode_tmap_3d_f32(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1, uint32_t box2) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return ERR_DEVICE;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {box0, box1, box2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? OK : ERR_SHAPE;
}

int sm_count() {
  constexpr int MAX_DEVICES = 64;
  static std::atomic<int> counts[MAX_DEVICES] = {};  // 0 = not read yet; callers may race, all store one value
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return 0;
  int n = counts[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    counts[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace bsa

using namespace bsa;

extern "C" {

int tra_forward(const void* q, const void* k, const void* v, void* out, int B, int H, int T, int D, float beta,
                float p, int dtype, cudaStream_t stream) {
  return tra_forward_ex(q, k, v, out, B, H, T, D, beta, p, dtype, 0, stream);
}

int tra_forward_ex(const void* q, const void* k, const void* v, void* out, int B, int H, int T, int D, float beta,
                   float p, int dtype, int flags, cudaStream_t stream) {
  if ((flags & ~BSA_TRA_SQRT_HALF_POWERS) != 0) return BSA_ERR_UNSUPPORTED;
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) return BSA_ERR_NULLPTR;
  if (dtype != BSA_F32 && dtype != BSA_BF16) return BSA_ERR_DTYPE;
  if (B < 1 || H < 1 || T < 1 || D < 1) return BSA_ERR_SHAPE;
  if (static_cast<long long>(B) * H > 0x7fffffffLL) return BSA_ERR_SHAPE;
  if (static_cast<long long>(B) * H * T * D >= (1LL << 40)) return BSA_ERR_SHAPE;
  if (!tra_head_dim_supported(D)) return BSA_ERR_UNSUPPORTED;
  if (!isfinite(beta) || !isfinite(p) || !(p > 0.0f)) return BSA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return BSA_ERR_ALIGN;
  const int dv = check_device();
  if (dv != OK) return dv;
  if (dtype == BSA_F32)
    return launch_tra_f32(static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
                          static_cast<float*>(out), B, H, T, D, beta, p, stream);
  return launch_tra_bf16(q, k, v, out, B, H, T, D, beta, p, (flags & BSA_TRA_SQRT_HALF_POWERS) != 0, stream);
}

size_t tra_forward_host_workspace_size(int B, int H, int T, int D, int dtype) {
  if (dtype != BSA_F32 && dtype != BSA_BF16) return 0;
  if (B < 1 || H < 1 || T < 1 || !tra_head_dim_supported(D)) return 0;
  if (static_cast<long long>(B) * H > 0x7fffffffLL || static_cast<long long>(B) * H * T * D >= (1LL << 40)) return 0;
  return tra_host_workspace_bytes(static_cast<long long>(B) * H, T, D, dtype == BSA_F32 ? 4 : 2);
}

int tra_forward_host(const void* q, const void* k, const void* v, void* out, int B, int H, int T, int D, float beta,
                     float p, int dtype, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || workspace == nullptr) return BSA_ERR_NULLPTR;
  if (dtype != BSA_F32 && dtype != BSA_BF16) return BSA_ERR_DTYPE;
  if (B < 1 || H < 1 || T < 1 || D < 1) return BSA_ERR_SHAPE;
  if (static_cast<long long>(B) * H > 0x7fffffffLL) return BSA_ERR_SHAPE;
  if (static_cast<long long>(B) * H * T * D >= (1LL << 40)) return BSA_ERR_SHAPE;
  if (!tra_head_dim_supported(D)) return BSA_ERR_UNSUPPORTED;
  if (!isfinite(beta) || !isfinite(p) || !(p > 0.0f)) return BSA_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return BSA_ERR_ALIGN;
  if (workspace_bytes < tra_forward_host_workspace_size(B, H, T, D, dtype)) return BSA_ERR_SCRATCH_LIMIT;
  const int dv = check_device();
  if (dv != OK) return dv;
  return launch_tra_host(q, k, v, out, B, H, T, D, beta, p, dtype == BSA_F32, workspace, stream);
}

int tra_backward_ex(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk, void* dv,
                    int B, int H, int T, int D, float beta, float p, int dtype, int flags, cudaStream_t stream) {
  if (q == nullptr || k == nullptr || v == nullptr || dout == nullptr || dq == nullptr || dk == nullptr ||
      dv == nullptr)
    return BSA_ERR_NULLPTR;
  if (dtype != BSA_F32 && dtype != BSA_BF16) return BSA_ERR_DTYPE;
  if (B < 1 || H < 1 || T < 1 || D < 1) return BSA_ERR_SHAPE;
  if (static_cast<long long>(B) * H > 0x7fffffffLL) return BSA_ERR_SHAPE;
  if (static_cast<long long>(B) * H * T * D >= (1LL << 40)) return BSA_ERR_SHAPE;
  if (!tra_head_dim_supported(D)) return BSA_ERR_UNSUPPORTED;
  if (!isfinite(beta) || !isfinite(p) || !(p > 0.0f)) return BSA_ERR_UNSUPPORTED;
  if ((flags & ~BSA_TRA_BWD_DETERMINISTIC) != 0) return BSA_ERR_UNSUPPORTED;
  const void* ptrs[7] = {q, k, v, dout, dq, dk, dv};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return BSA_ERR_ALIGN;
  const int dvs = check_device();
  if (dvs != OK) return dvs;
  if (dtype == BSA_F32)
    return launch_tra_bwd_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                              static_cast<const float*>(v), static_cast<const float*>(dout), static_cast<float*>(dq),
                              static_cast<float*>(dk), static_cast<float*>(dv), B, H, T, D, beta, p, stream);
  if (flags & BSA_TRA_BWD_DETERMINISTIC)
    return launch_tra_bwd_bf16(q, k, v, dout, dq, dk, dv, B, H, T, D, beta, p, stream);
  // fp32 dq accumulator: a stream-ordered temporary, released on the same stream.
  float* acc = nullptr;
  const size_t bytes = static_cast<size_t>(B) * H * T * D * sizeof(float);
  int dev = 0;
  cudaMemPool_t pool = cudaGetDevice(&dev) == cudaSuccess ? scratch_pool(dev) : nullptr;
  if (pool == nullptr) return BSA_ERR_MEMORY;
  if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&acc), bytes, pool, stream) != cudaSuccess)
    return BSA_ERR_MEMORY;
  const int st = launch_tra_bwd_fused_bf16(q, k, v, dout, dq, dk, dv, B, H, T, D, beta, p, acc, stream);
  if (cudaFreeAsync(acc, stream) != cudaSuccess && st == OK) return BSA_ERR_MEMORY;
  return st;
}

int tra_backward(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk, void* dv, int B,
                 int H, int T, int D, float beta, float p, int dtype, cudaStream_t stream) {
  return tra_backward_ex(q, k, v, dout, dq, dk, dv, B, H, T, D, beta, p, dtype, 0, stream);
}

// Argument checks of tra_diff_forward and tra_diff_forward_noalloc.
static int check_diff_args(const void* q1, const void* q2, const void* k1, const void* k2, const void* v,
                           const void* out, int B, int H, int T, int D, float beta, float lambda, float p,
                           int dtype) {
  if (q1 == nullptr || q2 == nullptr || k1 == nullptr || k2 == nullptr || v == nullptr || out == nullptr)
    return BSA_ERR_NULLPTR;
  if (dtype != BSA_F32 && dtype != BSA_BF16) return BSA_ERR_DTYPE;
  if (B < 1 || H < 1 || T < 1 || D < 1) return BSA_ERR_SHAPE;
  if (static_cast<long long>(B) * H > 0x7fffffffLL) return BSA_ERR_SHAPE;
  if (static_cast<long long>(B) * H * T * D >= (1LL << 40)) return BSA_ERR_SHAPE;
  if (!tra_head_dim_supported(D)) return BSA_ERR_UNSUPPORTED;
  if (!isfinite(beta) || !isfinite(p) || !(p > 0.0f) || isnan(lambda)) return BSA_ERR_UNSUPPORTED;
  const void* ptrs[6] = {q1, q2, k1, k2, v, out};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return BSA_ERR_ALIGN;
  return BSA_OK;
}

int tra_diff_forward(const void* q1, const void* q2, const void* k1, const void* k2, const void* v, void* out, int B,
                     int H, int T, int D, float beta, float lambda, float p, int normalize, int dtype,
                     cudaStream_t stream) {
  const int chk = check_diff_args(q1, q2, k1, k2, v, out, B, H, T, D, beta, lambda, p, dtype);
  if (chk != BSA_OK) return chk;
  const int dvs = check_device();
  if (dvs != OK) return dvs;
  if (dtype == BSA_F32)  // no scratch: the fp32 kernel folds the normalisation into its scores
    return launch_tra_diff_f32(static_cast<const float*>(q1), static_cast<const float*>(q2),
                               static_cast<const float*>(k1), static_cast<const float*>(k2),
                               static_cast<const float*>(v), static_cast<float*>(out), B, H, T, D, beta, lambda, p,
                               normalize != 0, stream);
  if (!normalize)
    return launch_tra_diff_bf16(q1, q2, k1, k2, v, out, B, H, T, D, beta, lambda, p, nullptr, nullptr, stream);
  // Normalised copies of k1 and k2 (the kernel takes the query rows' factors
  // from its resident Q tiles): a stream-ordered temporary, released on the
  // same stream.
  void* kn = nullptr;
  const size_t bytes = 2 * sizeof(uint16_t) * static_cast<size_t>(B) * H * T * D;
  int dev = 0;
  cudaMemPool_t pool = cudaGetDevice(&dev) == cudaSuccess ? scratch_pool(dev) : nullptr;
  if (pool == nullptr) return BSA_ERR_MEMORY;
  if (cudaMallocFromPoolAsync(&kn, bytes, pool, stream) != cudaSuccess) return BSA_ERR_MEMORY;
  const int st = launch_tra_diff_bf16(q1, q2, k1, k2, v, out, B, H, T, D, beta, lambda, p, nullptr, kn, stream);
  if (cudaFreeAsync(kn, stream) != cudaSuccess && st == OK) return BSA_ERR_MEMORY;
  return st;
}

int tra_diff_backward(const void* q1, const void* q2, const void* k1, const void* k2, const void* v,
                      const void* dout, void* dq1, void* dq2, void* dk1, void* dk2, void* dv, float* dlambda, int B,
                      int H, int T, int D, float beta, float lambda, float p, int normalize, int dtype,
                      cudaStream_t stream) {
  const int chk = check_diff_args(q1, q2, k1, k2, v, dq1, B, H, T, D, beta, lambda, p, dtype);
  if (chk != BSA_OK) return chk;
  const void* more[5] = {dout, dq2, dk1, dk2, dv};
  for (const void* ptr : more) {
    if (ptr == nullptr) return BSA_ERR_NULLPTR;
    if (!aligned16(ptr)) return BSA_ERR_ALIGN;
  }
  if ((reinterpret_cast<uintptr_t>(dlambda) & 3u) != 0) return BSA_ERR_ALIGN;
  const int dvs = check_device();
  if (dvs != OK) return dvs;
  const bool f32 = dtype == BSA_F32;
  const size_t bytes = tra_diff_bwd_scratch_bytes(B, H, T, D, f32, normalize != 0, dlambda != nullptr);
  void* scratch = nullptr;
  int dev = 0;
  cudaMemPool_t pool = cudaGetDevice(&dev) == cudaSuccess ? scratch_pool(dev) : nullptr;
  if (pool == nullptr) return BSA_ERR_MEMORY;
  if (cudaMallocFromPoolAsync(&scratch, bytes, pool, stream) != cudaSuccess) return BSA_ERR_MEMORY;
  const int st = launch_tra_diff_bwd(q1, q2, k1, k2, v, dout, dq1, dq2, dk1, dk2, dv, dlambda, B, H, T, D, beta,
                                     lambda, p, normalize != 0, f32, scratch, stream);
  if (cudaFreeAsync(scratch, stream) != cudaSuccess && st == OK) return BSA_ERR_MEMORY;
  return st;
}

int tra_diff_forward_noalloc(const void* q1, const void* q2, const void* k1, const void* k2, const void* v,
                             void* out, int B, int H, int T, int D, float beta, float lambda, float p, int normalize,
                             int dtype, cudaStream_t stream) {
  const int chk = check_diff_args(q1, q2, k1, k2, v, out, B, H, T, D, beta, lambda, p, dtype);
  if (chk != BSA_OK) return chk;
  if (dtype == BSA_F32) {  // the fp32 kernel uses no scratch at all
    const int dvs = check_device();
    if (dvs != OK) return dvs;
    return launch_tra_diff_f32(static_cast<const float*>(q1), static_cast<const float*>(q2),
                               static_cast<const float*>(k1), static_cast<const float*>(k2),
                               static_cast<const float*>(v), static_cast<float*>(out), B, H, T, D, beta, lambda, p,
                               normalize != 0, stream);
  }
  if (normalize && !tra_diff_noalloc_fits(B, H, T)) return BSA_ERR_SCRATCH_LIMIT;
  const int dvs = check_device();
  if (dvs != OK) return dvs;
  return launch_tra_diff_noalloc_bf16(q1, q2, k1, k2, v, out, B, H, T, D, beta, lambda, p, normalize != 0, stream);
}

int nsa_select_forward(const void* q, const void* k, const void* v, const int32_t* block_idx, void* out, float* lse,
                       int B, int Hq, int Hkv, int T, int D, int block_size, int S, cudaStream_t stream) {
  const int chk = check_nsa_args(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, D, block_size, S);
  if (chk != BSA_OK) return chk;
  const int dv = check_device();
  if (dv != OK) return dv;
  return launch_nsa_select(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, D, block_size, S, stream);
}

size_t nsa_select_fsa_workspace_size(int B, int Hq, int Hkv, int T, int D, int block_size, int S) {
  if (check_nsa_shape(B, Hq, Hkv, T, D, block_size, S) != BSA_OK || !fsa_shape_supported(D, block_size)) return 0;
  // The partial rows are indexed with 32-bit integers inside the kernels.
  if (static_cast<long long>(B) * Hq * T * S >= (1LL << 31)) return 0;
  return nsa_fsa_workspace_bytes(B, Hq, Hkv, T, D, S);
}

int nsa_select_forward_fsa(const void* q, const void* k, const void* v, const int32_t* block_idx, void* out,
                           float* lse, int B, int Hq, int Hkv, int T, int D, int block_size, int S, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  const int chk = check_nsa_args(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, D, block_size, S);
  if (chk != BSA_OK) return chk;
  if (!fsa_shape_supported(D, block_size)) return BSA_ERR_UNSUPPORTED;
  if (workspace == nullptr) return BSA_ERR_NULLPTR;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return BSA_ERR_ALIGN;
  const size_t need = nsa_select_fsa_workspace_size(B, Hq, Hkv, T, D, block_size, S);
  if (need == 0) return BSA_ERR_SHAPE;
  if (workspace_bytes < need) return BSA_ERR_SCRATCH_LIMIT;
  const int dv = check_device();
  if (dv != OK) return dv;
  return launch_nsa_fsa(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, D, S, workspace, stream);
}

const char* bsa_status_string(int status) {
  switch (status) {
    case BSA_OK: return "success";
    case BSA_ERR_NULLPTR: return "a required pointer is NULL";
    case BSA_ERR_SHAPE: return "a size is out of range or inconsistent";
    case BSA_ERR_DTYPE: return "dtype is not a bsa_dtype value";
    case BSA_ERR_UNSUPPORTED: return "unsupported head dim, block size, group size or parameter value";
    case BSA_ERR_LAUNCH: return "CUDA kernel launch failed";
    case BSA_ERR_DEVICE: return "no usable sm_103 device or CUDA driver entry point";
    case BSA_ERR_ALIGN: return "a tensor pointer is not suitably aligned";
    case BSA_ERR_MEMORY: return "scratch memory could not be allocated or released";
    case BSA_ERR_SCRATCH_LIMIT:
      return "the problem needs more scratch than the fixed buffer or the caller's workspace holds";
    default: return "unknown bsa_status";
  }
}

int bsa_version(void) { return 100; }

int bsa_selftest_wait_timeout(long long limit_cycles, int* result, cudaStream_t stream) {
  if (result == nullptr) return BSA_ERR_NULLPTR;
  if (limit_cycles < 1 || limit_cycles > 100000000LL) return BSA_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(result) & 3u) != 0) return BSA_ERR_ALIGN;
  const int dv = check_device();
  if (dv != OK) return dv;
  return launch_selftest_wait_timeout(limit_cycles, result, stream);
}

int bsa_selftest_log2(const float* x, float* y_fma, float* y_ref, int n, cudaStream_t stream) {
  if (x == nullptr || y_fma == nullptr || y_ref == nullptr) return BSA_ERR_NULLPTR;
  if (n < 1) return BSA_ERR_SHAPE;
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y_fma) |
                         reinterpret_cast<uintptr_t>(y_ref)) & 3u;
  if (mis != 0) return BSA_ERR_ALIGN;
  const int dv = check_device();
  if (dv != OK) return dv;
  return launch_selftest_log2(x, y_fma, y_ref, n, stream);
}

int bsa_selftest_exp2(const float* y, float* w_fma, float* w_ref, int n, cudaStream_t stream) {
  if (y == nullptr || w_fma == nullptr || w_ref == nullptr) return BSA_ERR_NULLPTR;
  if (n < 1) return BSA_ERR_SHAPE;
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(w_fma) |
                         reinterpret_cast<uintptr_t>(w_ref)) & 3u;
  if (mis != 0) return BSA_ERR_ALIGN;
  const int dv = check_device();
  if (dv != OK) return dv;
  return launch_selftest_exp2(y, w_fma, w_ref, n, stream);
}

int bsa_read_probe(const void* buf, size_t bytes, int reps, unsigned int* sink, cudaStream_t stream) {
  if (buf == nullptr || sink == nullptr) return BSA_ERR_NULLPTR;
  if (bytes < 16 || bytes % 16 != 0 || bytes > (1ull << 40) || reps < 1 || reps > 100000) return BSA_ERR_SHAPE;
  if (!aligned16(buf) || (reinterpret_cast<uintptr_t>(sink) & 3u) != 0) return BSA_ERR_ALIGN;
  const int dv = check_device();
  if (dv != OK) return dv;
  return launch_read_probe(buf, static_cast<long long>(bytes), reps, sink, stream);
}

int bsa_device_error(void) {
  const unsigned codes[7] = {tra_bf16_device_error(), tra_f32_device_error(), nsa_device_error(),
                             tra_bwd_device_error(), tra_diff_device_error(), nsa_fsa_device_error(),
                             selftest_device_error()};
  unsigned worst = 0;
  for (unsigned c : codes) {
    if (c == 0xffffffffu) return -1;
    if (c > worst) worst = c;
  }
  return static_cast<int>(worst);
}

}  // extern "C"
