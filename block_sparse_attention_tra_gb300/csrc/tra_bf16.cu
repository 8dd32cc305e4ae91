// tra_bf16.cu -- threshold rectified attention forward, bf16 in / fp32
// accumulate, on the sm_100-family tensor cores (tcgen05 + TMEM + TMA).
//
// Method: page "triton_threshold_attention.py" (module docstring formula and
// _threshold_rela_fwd_kernel):
//     out_i = sum_{j <= i} ReLU(q_i . k_j - tau(i))^p v_j,
//     tau(i) = beta * sqrt(2 ln(i+1) / D),
// causal and unnormalised, no 1/sqrt(D) factor.  The page's kernel walks every
// key tile for every query tile; this one visits only key tiles at or below
// the diagonal and masks the diagonal tile per element.
//
// One CTA owns 256 query rows of one (b, h) as two 128-row tiles Q0, Q1 that
// share every K/V tile brought in by TMA:
//   warp 8      TMA producer: Q0, Q1 once, then K and V tiles (128 keys x D)
//               into two smem rings (128-byte swizzled 64-column panels).
//   warp 9      MMA issuer (one thread).  Per key tile n the tensor pipe runs
//                 ... PV0(n), QK0(n+1), PV1(n), QK1(n+1), PV0(n+1) ...
//               where QKt(n): S_t = Q_t K_n^T into TMEM (fp32, 128 columns),
//               PVt(n): O_t += P_t V_n with P_t read from TMEM.  Each epilogue
//               warpgroup therefore has two MMAs' time to turn S_t into P_t.
//   warps 0-3   epilogue of Q0, warps 4-7 epilogue of Q1: thread r owns query
//               row r (TMEM lane r).  It loads its 128 scores, masks the
//               diagonal tile, subtracts tau(i) in fp32, takes ReLU^p, rounds
//               to bf16 and writes P over the consumed score columns; at the
//               end it reads O_t (fp32) and stores it as bf16.
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
#include "kernels.h"
#include "ptx.cuh"

namespace bsa {
namespace {

constexpr int BM = 128;                 // query rows per tile
constexpr int BN = 128;                 // keys per tile
constexpr int PANEL_BYTES = 128 * 128;  // 128 rows x 128 B (64 bf16) swizzle panel
constexpr int NUM_THREADS = 320;        // 2 epilogue warpgroups + TMA warp + MMA warp
constexpr int TMA_WARP = 8;
constexpr int MMA_WARP = 9;

template <int D>
struct Layout {
  static constexpr int NP = D / 64;              // 64-column panels per tile
  static constexpr int TILE = NP * PANEL_BYTES;  // one 128 x D bf16 tile
  static constexpr int NS = (D == 128) ? 2 : 4;  // stages per K ring and per V ring
  static constexpr int Q_OFF = 0;                // Q0, Q1
  static constexpr int K_OFF = Q_OFF + 2 * TILE;
  static constexpr int V_OFF = K_OFF + NS * TILE;
  static constexpr int BAR_OFF = V_OFF + NS * TILE;
  // q_full | k_full[NS] | k_empty[NS] | v_full[NS] | v_empty[NS] | s_full[2] | p_full[2] | o_full[2]
  static constexpr int NBAR = 1 + 4 * NS + 6;
  static constexpr int TPTR_OFF = BAR_OFF + NBAR * 8;
  static constexpr int BYTES = TPTR_OFF + 16;
  static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024 B
};

constexpr uint32_t TMEM_COLS = 512;

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

// Weights of two adjacent keys from their scores: ReLU(s - tau)^p, bf16x2.
template <int PC>
__device__ __forceinline__ uint32_t weights2(float s0, float s1, float tau, float p) {
  const float x0 = s0 - tau, x1 = s1 - tau;
  if constexpr (PC == POW_ONE) {
    return relu_pack(x0, x1);
  } else if constexpr (PC == POW_TWO) {
    const uint32_t h = relu_pack(x0, x1);
    return mul_bf16x2(h, h);
  } else {
    // x^p = exp2(p log2 x); lg2(0) = -inf and ex2(-inf) = 0 give ReLU's zero.
    const float w0 = ex2_approx(p * lg2_approx(fmaxf(x0, 0.0f)));
    const float w1 = ex2_approx(p * lg2_approx(fmaxf(x1, 0.0f)));
    return pack_bf16x2(w0, w1);
  }
}

// Turn 64 scores (columns c0 .. c0+63 of the tile) into 32 packed weights and
// store them to TMEM columns c0/2 .. c0/2+31 of the same buffer.
template <int PC>
__device__ __forceinline__ void epilogue_half(const uint32_t (&s)[64], uint32_t tS, int c0, float tau, float p,
                                              bool diag, int key0, int row) {
  uint32_t pk[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    uint32_t w = weights2<PC>(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1]), tau, p);
    if (diag) {
      const int key = key0 + c0 + 2 * e;  // keys key, key + 1
      if (key > row) w = 0u;
      else if (key + 1 > row) w &= 0x0000ffffu;
    }
    pk[e] = w;
  }
  uint32_t lo[16], hi[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    lo[e] = pk[e];
    hi[e] = pk[16 + e];
  }
  tmem_st16(tS + c0 / 2, lo);
  tmem_st16(tS + c0 / 2 + 16, hi);
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
  tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
}

template <int D, int PC>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tra_bf16_tcgen05_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ out, int BH,
                            int T, int nQ, int nPair, float beta, float p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + L::NS;
  uint64_t* v_full = k_empty + L::NS;
  uint64_t* v_empty = v_full + L::NS;
  uint64_t* s_full = v_empty + L::NS;  // [2], one per query tile
  uint64_t* p_full = s_full + 2;       // [2]
  uint64_t* o_full = p_full + 2;       // [2]
  uint32_t* tptr = reinterpret_cast<uint32_t*>(smem + L::TPTR_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Longest-first order: the first BH CTAs take the last (longest) tile pair.
  const int t = nPair - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const bool has1 = (2 * t + 1) < nQ;     // second query tile exists
  const int nmax0 = 2 * t;                // last key tile of Q0 (its diagonal)
  const int nmax1 = has1 ? 2 * t + 1 : -1;
  const int nlast = has1 ? nmax1 : nmax0;

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
      mbar_init(&o_full[b], 1);
    }
    fence_barrier_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tptr, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tptr;

  if (warp == TMA_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(q_full, (has1 ? 2 : 1) * L::TILE);
      for (int qt = 0; qt < (has1 ? 2 : 1); ++qt) {
        uint8_t* sQ = smem + L::Q_OFF + qt * L::TILE;
#pragma unroll
        for (int pnl = 0; pnl < L::NP; ++pnl)
          tma_load_3d(sQ + pnl * PANEL_BYTES, &tmQ, q_full, 64 * pnl, (2 * t + qt) * BM, bh);
      }
      bool ok = true;
      int nk = 0, nv = 0;  // K / V tiles issued
      for (int n = 0; n <= nlast; ++n) {
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
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, 0, 0);  // Q, K both K-major
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, 0, 1);   // P (TMEM), V MN-major
      const uint32_t sQ0 = smem_u32(smem + L::Q_OFF);

      auto qk = [&](int qt, int n) {
        const uint32_t sQ = sQ0 + qt * L::TILE;
        const uint32_t sK = smem_u32(smem + L::K_OFF + (n % L::NS) * L::TILE);
        const uint32_t tS = tmem + qt * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * PANEL_BYTES + (kk & 3) * 32;
          mma_ss(tS, smem_desc_sw128(sQ + off, 16, 1024), smem_desc_sw128(sK + off, 16, 1024), IDESC_QK,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[qt]);
      };
      auto pv = [&](int qt, int n) {
        const uint32_t sV = smem_u32(smem + L::V_OFF + (n % L::NS) * L::TILE);
        const uint32_t tP = tmem + qt * BN;
        const uint32_t tO = tmem + 2 * BN + qt * D;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(sV + kk * 16 * 128, L::NP > 1 ? PANEL_BYTES : 1024, 1024);
          mma_ts(tO, tP + kk * 8, bdesc, IDESC_PV, (n > 0 || kk > 0) ? 1u : 0u);
        }
      };

      bool ok = mbar_wait(q_full, 0) && mbar_wait(&k_full[0], 0);
      if (ok) {
        tc_fence_after();
        qk(0, 0);
        if (has1) qk(1, 0);
        mma_commit(&k_empty[0]);
      }
      for (int n = 0; n <= nlast && ok; ++n) {
        const int s = n % L::NS;
        const uint32_t vph = (n / L::NS) & 1;
        const int n1 = n + 1;
        const bool next_k = n1 <= nlast;
        // tile 0: PV0(n), then QK0(n+1)
        if (n <= nmax0) {
          if (!(ok = mbar_wait(&p_full[0], n & 1) && mbar_wait(&v_full[s], vph))) break;
          tc_fence_after();
          pv(0, n);
          if (n == nmax0) mma_commit(&o_full[0]);
        }
        if (next_k) {
          if (!(ok = mbar_wait(&k_full[n1 % L::NS], (n1 / L::NS) & 1))) break;
          tc_fence_after();
          if (n1 <= nmax0) qk(0, n1);
        }
        // tile 1: PV1(n), then QK1(n+1)
        if (has1) {
          if (!(ok = mbar_wait(&p_full[1], n & 1) && mbar_wait(&v_full[s], vph))) break;
          tc_fence_after();
          pv(1, n);
          if (n == nmax1) mma_commit(&o_full[1]);
        }
        mma_commit(&v_empty[s]);
        if (next_k) {
          if (has1 && n1 <= nmax1) qk(1, n1);
          mma_commit(&k_empty[n1 % L::NS]);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int qt = warp >> 2;  // query tile of this warpgroup
    const int wq = warp & 3;   // TMEM lane quarter
    const int nmax = qt == 0 ? nmax0 : nmax1;
    const int r = wq * 32 + lane;
    const int row = (2 * t + qt) * BM + r;
    const float tau = beta * sqrtf(2.0f * logf(static_cast<float>(row + 1)) / static_cast<float>(D));
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t tS = lane_base + qt * BN;
    bool ok = true;
    for (int n = 0; n <= nmax; ++n) {
      if (!(ok = mbar_wait(&s_full[qt], n & 1))) break;
      tc_fence_after();
      const bool diag = (n == nmax);
      const int key0 = n * BN;
      uint32_t sa[64], sb[64];
      tmem_ld64(tS, sa);
      tmem_wait_ld();
      tmem_ld64(tS + 64, sb);
      epilogue_half<PC>(sa, tS, 0, tau, p, diag, key0, row);
      tmem_wait_ld();
      epilogue_half<PC>(sb, tS, 64, tau, p, diag, key0, row);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[qt]);
    }
    if (ok && nmax >= 0) ok = mbar_wait(&o_full[qt], 0);
    if (ok && nmax >= 0) {
      tc_fence_after();
      __nv_bfloat16* orow = out + (static_cast<size_t>(bh) * T + row) * D;
      const uint32_t tO = lane_base + 2 * BN + qt * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tO + c * 32, ov);
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
  if (warp == MMA_WARP) {
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
  const int nQ = (T + BM - 1) / BM;
  const int nPair = (nQ + 1) / 2;
  const long long grid = static_cast<long long>(nPair) * BH;
  if (grid > 0x7fffffffLL) return ERR_SHAPE;
  kern<<<static_cast<unsigned>(grid), NUM_THREADS, L::ALLOC, stream>>>(
      mq, mk, mv, static_cast<__nv_bfloat16*>(out), BH, T, nQ, nPair, beta, p);
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
