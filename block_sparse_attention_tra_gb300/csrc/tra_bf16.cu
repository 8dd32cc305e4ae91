// tra_bf16.cu -- threshold rectified attention forward, bf16 in / fp32
// accumulate, on the sm_100-family tensor cores (tcgen05 + TMEM + TMA).
//
// Method: page "triton_threshold_attention.py" (module docstring formula and
// _threshold_rela_fwd_kernel):
//     out_i = sum_{j <= i} ReLU(q_i . k_j - tau(i))^p v_j,
//     tau(i) = beta * sqrt(2 ln(i+1) / D),
// causal and unnormalised, no 1/sqrt(D) factor.  The page's kernel walks every
// key tile for every query tile; this one visits only key tiles n <= m (the
// rest are fully masked) and masks the diagonal tile per element.
//
// One CTA computes one 128-row query tile of one (b, h):
//   warp 4      TMA producer: Q tile once, then K and V tiles (128 keys x D)
//               into two separate smem rings (128-byte swizzled panels).
//   warp 5      MMA issuer (one thread): S_n = Q K_n^T into one of two TMEM
//               score buffers (fp32, 128 columns each), then O += P_{n-1} V_{n-1}
//               with P read straight from TMEM (the "A from TMEM" MMA form).
//   warps 0-3   epilogue: thread r owns query row r (TMEM lane r).  It loads
//               its 128 scores, applies the causal mask (diagonal tile only),
//               subtracts tau(i) in fp32, takes ReLU^p, rounds to bf16 and
//               writes P back over the consumed score columns.  At the end it
//               reads O (fp32, D columns) and stores it as bf16.
// TMEM: S0 at column 0, S1 at 128, O at 256 (512 columns allocated).
#include "kernels.h"
#include "ptx.cuh"

namespace bsa {
namespace {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per tile
constexpr int PANEL_BYTES = 128 * 128;  // 128 rows x 128 B (64 bf16) swizzle panel
constexpr int NUM_THREADS = 192;

template <int D>
struct Layout {
  static constexpr int NP = D / 64;                  // 64-column panels per tile
  static constexpr int TILE = NP * PANEL_BYTES;      // one 128 x D bf16 tile
  static constexpr int NS = (D == 128) ? 2 : 4;      // stages per K ring and per V ring
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + TILE;
  static constexpr int V_OFF = K_OFF + NS * TILE;
  static constexpr int BAR_OFF = V_OFF + NS * TILE;
  // barriers: q_full | k_full[NS] | k_empty[NS] | v_full[NS] | v_empty[NS] |
  //           s_full[2] | p_full[2] | o_full
  static constexpr int NBAR = 1 + 4 * NS + 2 + 2 + 1;
  static constexpr int TPTR_OFF = BAR_OFF + NBAR * 8;
  static constexpr int BYTES = TPTR_OFF + 16;
  static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024 B
};

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL0 = 0;
constexpr uint32_t O_COL = 256;

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

// ReLU(x)^p.  For the general class, lg2(0) = -inf and ex2(-inf) = 0 give the
// ReLU's zero for free once x is clamped at 0 (p > 0).
template <int PC>
__device__ __forceinline__ float relu_pow(float x, float p) {
  const float r = fmaxf(x, 0.0f);
  if constexpr (PC == POW_ONE) {
    return r;
  } else if constexpr (PC == POW_TWO) {
    return r * r;
  } else {
    return ex2_approx(p * lg2_approx(r));
  }
}

template <int D, int PC>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tra_bf16_tcgen05_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ out, int BH,
                            int T, int nM, float beta, float p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + L::NS;
  uint64_t* v_full = k_empty + L::NS;
  uint64_t* v_empty = v_full + L::NS;
  uint64_t* s_full = v_empty + L::NS;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = p_full + 2;
  uint32_t* tptr = reinterpret_cast<uint32_t*>(smem + L::TPTR_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Longest-first order: the first BH CTAs take the last (longest) row tile.
  const int m = nM - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int nN = m + 1;  // key tiles 0..m (BN == BM)

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < L::NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 4);
    }
    mbar_init(o_full, 1);
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(tptr, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tptr;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint8_t* sQ = smem + L::Q_OFF;
      mbar_arrive_expect_tx(q_full, L::TILE);
#pragma unroll
      for (int pnl = 0; pnl < L::NP; ++pnl) tma_load_3d(sQ + pnl * PANEL_BYTES, &tmQ, q_full, 64 * pnl, m * BM, bh);
      bool ok = true;
      int nk = 0, nv = 0;  // K / V tiles issued
      for (int n = 0; n < nN; ++n) {
        const int s = n % L::NS;
        const uint32_t ph = (n / L::NS) & 1;
        if (!(ok = mbar_wait(&k_empty[s], ph ^ 1))) break;
        uint8_t* sK = smem + L::K_OFF + s * L::TILE;
        mbar_arrive_expect_tx(&k_full[s], L::TILE);
#pragma unroll
        for (int pnl = 0; pnl < L::NP; ++pnl)
          tma_load_3d(sK + pnl * PANEL_BYTES, &tmK, &k_full[s], 64 * pnl, n * BN, bh);
        ++nk;
        if (!(ok = mbar_wait(&v_empty[s], ph ^ 1))) break;
        uint8_t* sV = smem + L::V_OFF + s * L::TILE;
        mbar_arrive_expect_tx(&v_full[s], L::TILE);
#pragma unroll
        for (int pnl = 0; pnl < L::NP; ++pnl)
          tma_load_3d(sV + pnl * PANEL_BYTES, &tmV, &v_full[s], 64 * pnl, n * BN, bh);
        ++nv;
      }
      if (!ok) {
        // Drain: never leave the CTA with a bulk copy still landing in its smem.
        mbar_wait(q_full, 0);
        for (int n = (nk > L::NS ? nk - L::NS : 0); n < nk; ++n) mbar_wait(&k_full[n % L::NS], (n / L::NS) & 1);
        for (int n = (nv > L::NS ? nv - L::NS : 0); n < nv; ++n) mbar_wait(&v_full[n % L::NS], (n / L::NS) & 1);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, 0, 0);  // Q, K both K-major
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, 0, 1);   // P (TMEM), V MN-major
      const uint32_t sQ = smem_u32(smem + L::Q_OFF);
      const uint32_t tO = tmem + O_COL;
      bool ok = mbar_wait(q_full, 0);

      auto issue_pv = [&](int j) -> bool {
        const int b = j & 1;
        const int s = j % L::NS;
        if (!mbar_wait(&p_full[b], (j >> 1) & 1)) return false;
        if (!mbar_wait(&v_full[s], (j / L::NS) & 1)) return false;
        tc_fence_after();
        const uint32_t sV = smem_u32(smem + L::V_OFF + s * L::TILE);
        const uint32_t tP = tmem + S_COL0 + b * BN;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // 16 keys = 16 rows of 128 B in every panel; panels are D-chunks.
          const uint64_t bdesc = smem_desc_sw128(sV + kk * 16 * 128, L::NP > 1 ? PANEL_BYTES : 1024, 1024);
          mma_ts(tO, tP + kk * 8, bdesc, IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&v_empty[s]);
        return true;
      };

      for (int n = 0; n < nN && ok; ++n) {
        const int s = n % L::NS;
        const int b = n & 1;
        ok = mbar_wait(&k_full[s], (n / L::NS) & 1);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sK = smem_u32(smem + L::K_OFF + s * L::TILE);
        const uint32_t tS = tmem + S_COL0 + b * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * PANEL_BYTES + (kk & 3) * 32;
          mma_ss(tS, smem_desc_sw128(sQ + off, 16, 1024), smem_desc_sw128(sK + off, 16, 1024), IDESC_QK,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[b]);
        mma_commit(&k_empty[s]);
        if (n > 0) ok = issue_pv(n - 1);
      }
      if (ok) ok = issue_pv(nN - 1);
      if (ok) mma_commit(o_full);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int r = warp * 32 + lane;
    const int row = m * BM + r;
    const float tau = beta * sqrtf(2.0f * logf(static_cast<float>(row + 1)) / static_cast<float>(D));
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    bool ok = true;
    for (int n = 0; n < nN; ++n) {
      const int b = n & 1;
      ok = mbar_wait(&s_full[b], (n >> 1) & 1);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tS = lane_base + S_COL0 + b * BN;
      const bool diag = (n == m);
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t sv[32];
        tmem_ld32(tS + c * 32, sv);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float w0 = relu_pow<PC>(__uint_as_float(sv[2 * e]) - tau, p);
          float w1 = relu_pow<PC>(__uint_as_float(sv[2 * e + 1]) - tau, p);
          if (diag) {
            const int key = n * BN + c * 32 + 2 * e;
            if (key > row) w0 = 0.0f;
            if (key + 1 > row) w1 = 0.0f;
          }
          pk[e] = pack_bf16x2(w0, w1);
        }
        tmem_st16(tS + c * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[b]);
    }
    if (ok) ok = mbar_wait(o_full, 0);
    if (ok) {
      tc_fence_after();
      __nv_bfloat16* orow = out + (static_cast<size_t>(bh) * T + row) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(lane_base + O_COL + c * 32, ov);
        tmem_wait_ld();
        if (row < T) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int vq = 0; vq < 4; ++vq) {
            uint4 u;
            u.x = pack_bf16x2(__uint_as_float(ov[8 * vq + 0]), __uint_as_float(ov[8 * vq + 1]));
            u.y = pack_bf16x2(__uint_as_float(ov[8 * vq + 2]), __uint_as_float(ov[8 * vq + 3]));
            u.z = pack_bf16x2(__uint_as_float(ov[8 * vq + 4]), __uint_as_float(ov[8 * vq + 5]));
            u.w = pack_bf16x2(__uint_as_float(ov[8 * vq + 6]), __uint_as_float(ov[8 * vq + 7]));
            dst[vq] = u;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int D, int PC>
int launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, void* out, int BH, int T,
           float beta, float p, cudaStream_t stream) {
  using L = Layout<D>;
  auto kern = tra_bf16_tcgen05_kernel<D, PC>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC) != cudaSuccess)
    return ERR_LAUNCH;
  const int nM = (T + BM - 1) / BM;
  const long long grid = static_cast<long long>(nM) * BH;
  if (grid > 0x7fffffffLL) return ERR_SHAPE;
  kern<<<static_cast<unsigned>(grid), NUM_THREADS, L::ALLOC, stream>>>(
      mq, mk, mv, static_cast<__nv_bfloat16*>(out), BH, T, nM, beta, p);
  return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
}

}  // namespace

int launch_tra_bf16(const void* q, const void* k, const void* v, void* out, int B, int H, int T, int D,
                    float beta, float p, cudaStream_t stream) {
  const int BH = B * H;
  CUtensorMap mq, mk, mv;
  const uint64_t rs = static_cast<uint64_t>(D) * 2;  // row stride in bytes
  const uint64_t hs = rs * T;                        // (b, h) stride in bytes
  int st = encode_tmap_3d(&mq, q, D, T, BH, rs, hs, 64, BM, 1);
  if (st == OK) st = encode_tmap_3d(&mk, k, D, T, BH, rs, hs, 64, BN, 1);
  if (st == OK) st = encode_tmap_3d(&mv, v, D, T, BH, rs, hs, 64, BN, 1);
  if (st != OK) return st;
  const int pc = power_class(p);
  if (D == 128) {
    if (pc == POW_TWO) return launch<128, POW_TWO>(mq, mk, mv, out, BH, T, beta, p, stream);
    if (pc == POW_ONE) return launch<128, POW_ONE>(mq, mk, mv, out, BH, T, beta, p, stream);
    return launch<128, POW_GENERAL>(mq, mk, mv, out, BH, T, beta, p, stream);
  }
  if (D == 64) {
    if (pc == POW_TWO) return launch<64, POW_TWO>(mq, mk, mv, out, BH, T, beta, p, stream);
    if (pc == POW_ONE) return launch<64, POW_ONE>(mq, mk, mv, out, BH, T, beta, p, stream);
    return launch<64, POW_GENERAL>(mq, mk, mv, out, BH, T, beta, p, stream);
  }
  return ERR_UNSUPPORTED;
}

unsigned int tra_bf16_device_error() { return read_and_clear_device_error(); }

}  // namespace bsa
