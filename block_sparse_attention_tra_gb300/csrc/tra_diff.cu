// tra_diff.cu -- threshold differential attention forward (bf16, tcgen05).
//
// Method: page "triton_threshold_attention.py", differential_threshold_rela_
// triton: optionally L2-normalise q1, k1, q2, k2 row by row, then
//     out = TRA(q1, k1, v) - clamp(lambda, 0, 1) * TRA(q2, k2, v)
// with both threshold-attention terms sharing beta, p and v.
//
// Fused: one CTA owns 128 query rows of one (b, h) and runs the two score
// streams side by side.  Stream t has its own Q_t (resident) and K_t tiles,
// both streams share each V tile (loaded once), and stream t accumulates
// P_t V into its own TMEM accumulator O_t; the store epilogue writes
// O_0 - clamp(lambda, 0, 1) O_1 from fp32.
//   warp 8      TMA producer (Q0, Q1 once; K0, K1 and V tiles in rings).
//   warp 9(+10) MMA issuer(s): per stream ... PV_t(n), QK_t(n+1) ...; at
//               D=64 with p = 1, 2 each stream has its own issuing warp (one
//               thread issues only about one tcgen05.mma per ~70 cycles);
//               otherwise warp 9 serves both streams in turn (at D=128 the
//               single-stage K1 ring keeps the streams in step anyway, and
//               two issuers measured slower).
//   warps 4t..  epilogue of stream t (thread = query row).
// TMEM: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
// The grid numbers its blocks in head groups (tile::head_group_item), so the
// CTAs resident at one time stream the K/V tiles of a few heads from L2.
//
// Normalisation does not rewrite q or k: with r(x) = 1 / max(||x||, 1e-12)
// the normalised score is s_ij r(q_i) r(k_j).  A pre-pass kernel writes r()
// of every row of q1, k1, q2, k2 into a float scratch buffer [4, B*H, Tp]
// (Tp = T rounded up to 128, zero past T); the producer copies the 2 x 128
// factors of each key tile (k1 and k2 rows) into a small shared-memory ring
// of its own (bulk copies), and the epilogue scales each score by
// r(q_i) r(k_j) before subtracting tau.
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"
#include "tc_tile.cuh"
#include "tra_math.cuh"

namespace bsa {
namespace {

using tile::PANEL_BYTES;
constexpr int BT = tile::ROWS;
constexpr int DIFF_TMA_WARP = 8;
constexpr int DIFF_MMA_WARP = 9;  // first MMA warp (allocates TMEM)
// General powers 1 <= p <= 64 with part of log2 on the FMA pipe (as the
// single-stream kernel does).
#ifndef BSA_DIFF_MIX
#define BSA_DIFF_MIX 1
#endif
template <int D, int PC>
struct DiffCfg {
  static constexpr int ISSUERS = (D == 64 && (PC == POW_ONE || PC == POW_TWO)) ? 2 : 1;
  static constexpr int THREADS = 256 + 32 + 32 * ISSUERS;
};

template <int D>
struct DiffLayout {
  static constexpr int NP = D / 64;
  static constexpr int TILE = NP * PANEL_BYTES;
  static constexpr int NSK0 = (D == 128) ? 2 : 3;  // K of stream 0 (needed first in each step)
  static constexpr int NSK1 = (D == 128) ? 1 : 3;  // K of stream 1
  static constexpr int NSV = (D == 128) ? 2 : 3;   // V (shared by both streams)
  static constexpr int NSR = 2;                    // key-factor ring (k1 and k2 rows of one key tile)
  static constexpr int RK_BYTES = BT * 4;
  static constexpr int Q_OFF = 0;                  // Q0, Q1
  static constexpr int K0_OFF = 2 * TILE;
  static constexpr int K1_OFF = K0_OFF + NSK0 * TILE;
  static constexpr int V_OFF = K1_OFF + NSK1 * TILE;
  static constexpr int RK_OFF = V_OFF + NSV * TILE;
  static constexpr int BAR_OFF = RK_OFF + NSR * 2 * RK_BYTES;
  // q_full | k0 full/empty | k1 full/empty | v full/empty | rk full/empty | s_full[2] | p_full[2] | o_full[2] |
  // mma_done[2]
  static constexpr int NBAR = 1 + 2 * (NSK0 + NSK1 + NSV + NSR) + 8;
  static constexpr int TPTR_OFF = BAR_OFF + NBAR * 8;
  static constexpr int ALLOC = TPTR_OFF + 16;  // the dynamic smem base is 1024-byte aligned
  static_assert(ALLOC <= 232448, "shared memory budget");
};

// A ring of NS single-tile stages with full/empty barriers.
struct Ring {
  uint64_t* full;
  uint64_t* empty;
  int off, ns;
  __device__ __forceinline__ int stage(int n) const { return n % ns; }
  __device__ __forceinline__ uint32_t phase(int n) const { return (n / ns) & 1; }
};

// 1 / max(||row||_2, 1e-12) for every row of the four inputs into
// inv[which][bh][Tp] (0 for the padding rows t >= T).  Eight threads per row,
// sixteen rows per warp and pass (four groups of four, whose 16-byte loads are
// all issued before any arithmetic), fp32 sums of the squared bf16 elements;
// the warps stride over the rows, and every lane takes part in every shuffle
// (rows past the end contribute zeros and store nothing).
__device__ __forceinline__ float sumsq_bf16x8(const uint4& u) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  float acc = 0.0f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
    acc = fmaf(lo, lo, acc);
    acc = fmaf(hi, hi, acc);
  }
  return acc;
}

constexpr int NORM_NG = 4;  // groups of four rows per warp and pass

// Row index -> (input, head, position).  Idx is 32-bit when the four inputs'
// padded rows fit (no 64-bit division), 64-bit otherwise.
template <typename Idx>
__device__ __forceinline__ void norm_row(long long row, long long rows_p, int Tp, int& which, long long& bh, int& t) {
  const Idx r = static_cast<Idx>(row), rp = static_cast<Idx>(rows_p);
  which = static_cast<int>(r / rp);
  const Idx rem = r - static_cast<Idx>(which) * rp;
  const Idx b = rem / static_cast<Idx>(Tp);
  bh = static_cast<long long>(b);
  t = static_cast<int>(rem - b * static_cast<Idx>(Tp));
}

// x * r rounded to bf16, for the eight bf16 of a 16-byte chunk.
__device__ __forceinline__ uint4 scale_bf16x8(const uint4& u, float r) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
    o[e] = pack_bf16x2(lo * r, hi * r);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// WRITE_K: only the k1 and k2 rows (inputs 1 and 3) are visited, and written
// normalised, x / max(||x||, 1e-12) rounded to bf16 -- the page normalises q
// and k before its kernel, in the input dtype -- into kn (k1 at kn, k2 at
// kn + B*H*T*D); no factors are written (inv unused).
template <int D, typename Idx, bool WRITE_K>
__global__ void __launch_bounds__(256) row_inv_norm_kernel(const __nv_bfloat16* __restrict__ a0,
                                                           const __nv_bfloat16* __restrict__ a1,
                                                           const __nv_bfloat16* __restrict__ a2,
                                                           const __nv_bfloat16* __restrict__ a3,
                                                           float* __restrict__ inv, __nv_bfloat16* __restrict__ kn,
                                                           int BH, int T, int Tp) {
  // Row of D bf16 = D / 8 chunks of 16 bytes over the eight lanes of a row:
  // lane `sub` takes chunks sub + 8c (none past the row for D = 16, 32).
  constexpr int CH = (D + 63) / 64;
  constexpr int NG = NORM_NG;
  const int lane = threadIdx.x & 31, sub = lane & 7;
  const long long rows_p = static_cast<long long>(BH) * Tp;
  const long long total = (WRITE_K ? 2 : 4) * rows_p;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long base = warp0 * 4 * NG; base < total; base += nwarps * 4 * NG) {
    long long row[NG];
    bool live[NG];
    int which_g[NG];
    long long src_off[NG];  // element offset of the row in its input
    uint4 u[NG][CH];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      row[g] = base + 4 * g + (lane >> 3);
      live[g] = false;
      which_g[g] = 0;
      src_off[g] = 0;
#pragma unroll
      for (int c = 0; c < CH; ++c) u[g][c] = make_uint4(0u, 0u, 0u, 0u);
      if (row[g] < total) {
        int which, t;
        long long bh;
        norm_row<Idx>(row[g], rows_p, Tp, which, bh, t);
        if constexpr (WRITE_K) which = 2 * which + 1;  // k1 or k2
        live[g] = t < T;
        which_g[g] = which;
        src_off[g] = (bh * T + t) * D;
        if (live[g]) {
          const __nv_bfloat16* src = which == 0 ? a0 : which == 1 ? a1 : which == 2 ? a2 : a3;
          const uint4* x = reinterpret_cast<const uint4*>(src + src_off[g]);
#pragma unroll
          for (int c = 0; c < CH; ++c)
            if (sub + 8 * c < D / 8) u[g][c] = x[sub + 8 * c];
        }
      }
    }
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      float acc = 0.0f;
#pragma unroll
      for (int c = 0; c < CH; ++c) acc += sumsq_bf16x8(u[g][c]);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      const float r = 1.0f / fmaxf(sqrtf(acc), 1e-12f);
      if constexpr (!WRITE_K) {
        if (sub == 0 && row[g] < total) inv[row[g]] = live[g] ? r : 0.0f;
      } else {
        if (live[g]) {
          uint4* y = reinterpret_cast<uint4*>(kn + (which_g[g] == 3 ? static_cast<long long>(BH) * T * D : 0LL) +
                                              src_off[g]);
#pragma unroll
          for (int c = 0; c < CH; ++c)
            if (sub + 8 * c < D / 8) y[sub + 8 * c] = scale_bf16x8(u[g][c], r);
        }
      }
    }
  }
}

// 32 scores of stream t -> 16 packed weights over the consumed score
// columns.  With NM = 1 the scores are scaled by rq * rk[col] (the normalisation
// of row and key): x = s (rq rk) - tau in one packed multiply and one packed
// fused multiply-add per key pair.
// DIAG (compile time): the tile holds the diagonal, mask keys after the row.
// POW_GENERAL_MIX: log2 of a share of the pairs on the FMA pipe, as in the
// single-stream kernel (tra_math.cuh, mix_mufu_pairs; PLAN its plan).
template <int PC, int NM, bool DIAG, int PLAN = 0>
__device__ __forceinline__ void diff_quarter(const uint32_t (&s)[32], uint32_t tS, int c0, const PowParams& wp,
                                             uint64_t rq2, uint64_t ntau2, const float (&rk)[32], int key0,
                                             int row) {
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const uint64_t s2 = f2_pack(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1]));
    uint64_t x2;
    if constexpr (NM == 1)
      x2 = f2_fma(s2, f2_mul(rq2, f2_pack(rk[2 * e], rk[2 * e + 1])), ntau2);
    else if constexpr (NM == 2)  // k already normalised: only the query's factor
      x2 = f2_fma(s2, rq2, ntau2);
    else
      x2 = f2_sub(s2, wp.tau2);
    uint32_t w = (PC == POW_GENERAL_MIX && mix_pair_on_fma<PLAN>(e)) ? weights2_x<PC, true>(x2, wp)
                                                                    : weights2_x<PC>(x2, wp);
    if constexpr (DIAG) {
      const int key = key0 + c0 + 2 * e;
      if (key > row) w = 0u;
      else if (key + 1 > row) w &= 0x0000ffffu;
    }
    pk[e] = w;
  }
  tmem_st16(tS + c0 / 2, pk);
}

template <int D, int PC, int NM>
__global__ void __launch_bounds__(DiffCfg<D, PC>::THREADS, 1)
    tra_diff_kernel(const __grid_constant__ CUtensorMap tmQ0, const __grid_constant__ CUtensorMap tmQ1,
                    const __grid_constant__ CUtensorMap tmK0, const __grid_constant__ CUtensorMap tmK1,
                    const __grid_constant__ CUtensorMap tmV, const float* __restrict__ inv_norm,
                    __nv_bfloat16* __restrict__ out, int BH, int T, int nQ, int G, float beta, float p, float lam,
                    int d_real) {
  const int Tp = nQ * BT;  // row stride of the normalisation buffer
  const int dr = d_real;  // head dim (the tile width D or less: zero-filled columns)
  using L = DiffLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  // The swizzled tiles need a 1024-byte aligned base (the layout has no slack
  // to round it up); refuse to run rather than compute garbage.
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) record_device_error(BSA_DEVERR_LAYOUT);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* b1 = bars + 1;
  const Ring rk0{b1, b1 + L::NSK0, L::K0_OFF, L::NSK0};
  b1 += 2 * L::NSK0;
  const Ring rk1{b1, b1 + L::NSK1, L::K1_OFF, L::NSK1};
  b1 += 2 * L::NSK1;
  const Ring rv{b1, b1 + L::NSV, L::V_OFF, L::NSV};
  b1 += 2 * L::NSV;
  const Ring rr{b1, b1 + L::NSR, L::RK_OFF, L::NSR};
  b1 += 2 * L::NSR;
  uint64_t* s_full = b1;  // [2]
  uint64_t* p_full = s_full + 2;                                    // [2]
  uint64_t* o_full = p_full + 2;                                    // [2]
  uint64_t* mma_done = o_full + 2;                                  // [2]
  uint32_t* tptr = reinterpret_cast<uint32_t*>(smem + L::TPTR_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tile::HeadItem item = tile::head_group_item(static_cast<int>(blockIdx.x), BH, nQ, G);
  const int m = nQ - 1 - item.rank;  // longest first
  const int bh = item.bh;
  const int nmax = m;
  constexpr uint32_t O_COL = 2 * BT;  // O0; O1 at O_COL + D

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2 * (L::NSK0 + L::NSK1 + L::NSV); ++i) mbar_init(bars + 1 + i, 1);
    for (int i = 0; i < L::NSV; ++i) mbar_init(&rv.empty[i], 2);  // released once per stream
    for (int i = 0; i < L::NSR; ++i) {
      mbar_init(&rr.full[i], 1);
      mbar_init(&rr.empty[i], 8);  // four warps of each stream's epilogue
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&o_full[b], 1);
      mbar_init(&mma_done[b], 1);
    }
    fence_barrier_init();
  }
  if (warp == DIFF_MMA_WARP) {
    tmem_alloc(tptr, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tptr;

  if (warp == DIFF_TMA_WARP) {
    if (lane == 0) {
      tma_prefetch_desc(&tmQ0);
      tma_prefetch_desc(&tmQ1);
      tma_prefetch_desc(&tmK0);
      tma_prefetch_desc(&tmK1);
      tma_prefetch_desc(&tmV);
      debug_check(m >= 0 && m * BT < T && bh >= 0 && bh < BH);
      mbar_arrive_expect_tx(q_full, 2 * L::TILE);
      tile::tma_tile<D>(smem + L::Q_OFF, &tmQ0, q_full, m * BT, bh);
      tile::tma_tile<D>(smem + L::Q_OFF + L::TILE, &tmQ1, q_full, m * BT, bh);
      bool ok = true;
      int issued[3] = {0, 0, 0};
      const Ring* rings[3] = {&rk0, &rk1, &rv};
      const CUtensorMap* maps[3] = {&tmK0, &tmK1, &tmV};
      int issued_rk = 0;
      for (int n = 0; n <= nmax && ok; ++n) {
        if constexpr (NM == 1) {  // key factors of the k1 and k2 rows of key tile n
          if (!(ok = mbar_wait(&rr.empty[rr.stage(n)], rr.phase(n) ^ 1))) break;
          mbar_arrive_expect_tx(&rr.full[rr.stage(n)], 2 * L::RK_BYTES);
          uint8_t* dst = smem + rr.off + rr.stage(n) * 2 * L::RK_BYTES;
          // inv_norm rows [q1 | k1 | q2 | k2]: k1 = 1, k2 = 3
          bulk_load(dst, inv_norm + (1LL * BH + bh) * Tp + n * BT, L::RK_BYTES, &rr.full[rr.stage(n)]);
          bulk_load(dst + L::RK_BYTES, inv_norm + (3LL * BH + bh) * Tp + n * BT, L::RK_BYTES, &rr.full[rr.stage(n)]);
          issued_rk = n + 1;
        }
        for (int r = 0; r < 3; ++r) {
          const Ring& R = *rings[r];
          if (!(ok = mbar_wait(&R.empty[R.stage(n)], R.phase(n) ^ 1))) break;
          mbar_arrive_expect_tx(&R.full[R.stage(n)], L::TILE);
          tile::tma_tile<D>(smem + R.off + R.stage(n) * L::TILE, maps[r], &R.full[R.stage(n)], n * BT, bh);
          issued[r] = n + 1;
        }
      }
      if (!ok) {  // drain: never leave with a bulk copy still landing
        mbar_wait(q_full, 0);
        for (int n = (issued_rk > L::NSR ? issued_rk - L::NSR : 0); n < issued_rk; ++n)
          mbar_wait(&rr.full[rr.stage(n)], rr.phase(n));
        for (int r = 0; r < 3; ++r) {
          const Ring& R = *rings[r];
          for (int n = (issued[r] > R.ns ? issued[r] - R.ns : 0); n < issued[r]; ++n)
            mbar_wait(&R.full[R.stage(n)], R.phase(n));
        }
      }
    }
  } else if (warp >= DIFF_MMA_WARP) {
    // Issuer j serves streams T0 .. T0 + NT - 1, per key tile n in the order
    // PV_t(n), QK_t(n+1).  Each V use is released once per stream, after the
    // stream's P V on it (and so after its wait for that V load).
    constexpr int NT = 3 - DiffCfg<D, PC>::ISSUERS;
    const int j = warp - DIFF_MMA_WARP;
    const int T0 = NT == 1 ? j : 0;
    // The whole warp walks the issue loop at D = 64 (short N = 64 P V
    // products; descriptors are then warp-uniform values) and one elected
    // lane issues; at D = 128 the elected lane walks it alone.
    const bool leader = elect_one();
    if (D == 64 || leader) {
      const uint32_t sQ = smem_u32(smem + L::Q_OFF);
      auto mma_commit = [&](uint64_t* bar) {
        if (leader) bsa::mma_commit(bar);
      };
      // QKt(n): S_t = Q_t K_t(n)^T, then release K_t(n).
      auto qk = [&](int t, int n) -> bool {
        const Ring& R = t == 0 ? rk0 : rk1;
        if (!mbar_wait(&R.full[R.stage(n)], R.phase(n))) return false;
        tc_fence_after();
        tile::mma_abt<D>(tmem + t * BT, sQ + t * L::TILE, smem_u32(smem + R.off + R.stage(n) * L::TILE), leader);
        mma_commit(&s_full[t]);
        mma_commit(&R.empty[R.stage(n)]);
        return true;
      };
      // PVt(n): O_t += P_t V(n), then release V(n) for this stream.
      auto pv = [&](int t, int n) -> bool {
        if (!mbar_wait(&p_full[t], n & 1) || !mbar_wait(&rv.full[rv.stage(n)], rv.phase(n))) return false;
        tc_fence_after();
        const uint32_t sV = smem_u32(smem + rv.off + rv.stage(n) * L::TILE);
        tile::mma_tmem_a<D>(tmem + O_COL + t * D, tmem + t * BT, sV, 0, BT / 16, n == 0, leader);
        mma_commit(&rv.empty[rv.stage(n)]);
        return true;
      };
      bool ok = mbar_wait(q_full, 0);
#pragma unroll
      for (int i = 0; i < NT; ++i) ok = ok && qk(T0 + i, 0);
      for (int n = 0; n <= nmax && ok; ++n) {
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          if (!(ok = pv(T0 + i, n) && (n == nmax || qk(T0 + i, n + 1)))) break;
        }
      }
      if (ok) {
#pragma unroll
        for (int i = 0; i < NT; ++i) mma_commit(&o_full[T0 + i]);
      }
      mma_commit(&mma_done[j]);
      mbar_wait(&mma_done[j], 0);
    }
  } else {
    const int t = warp >> 2, wq = warp & 3;
    const int row = m * BT + wq * 32 + lane;
    const float tau = tile::tau_of_row(row, beta, dr);
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t tS = lane_base + t * BT;
    const PowParams wp = pow_params(tau, p);
    const float lc = fminf(fmaxf(lam, 0.0f), 1.0f);
    // Query factor: NM = 1 reads it from inv_norm ([q1 | k1 | q2 | k2] x
    // [B*H] x [Tp], zero past T); NM = 2 sums the squares of this thread's row
    // of the resident Q_t tile (once, before the MMA stream), as the pre-pass
    // does for the keys.
    float rq = 1.0f;
    bool ok = true;
    if constexpr (NM == 1) rq = inv_norm[(static_cast<long long>(t == 0 ? 0 : 2) * BH + bh) * Tp + row];
    if constexpr (NM == 2) {
      ok = mbar_wait(q_full, 0);
      const int r = wq * 32 + lane;
      float acc = 0.0f;
#pragma unroll
      for (int pnl = 0; pnl < D / 64; ++pnl)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          acc += sumsq_bf16x8(*reinterpret_cast<const uint4*>(smem + L::Q_OFF + t * L::TILE + pnl * PANEL_BYTES +
                                                               r * 128 + ((k ^ (r & 7)) << 4)));
      rq = 1.0f / fmaxf(sqrtf(acc), 1e-12f);
    }
    const uint64_t rq2 = f2_pack(rq, rq), ntau2 = f2_pack(-tau, -tau);
    for (int n = 0; n <= nmax && ok; ++n) {
      if (!(ok = mbar_wait(&s_full[t], n & 1))) break;
      tc_fence_after();
      const bool diag = (n == nmax);
      // Key normalisation factors of this tile (stream t's half of the stage).
      const float* rk_tile =
          reinterpret_cast<const float*>(smem + rr.off + rr.stage(n) * 2 * L::RK_BYTES + t * L::RK_BYTES);
      if (NM == 1 && !(ok = mbar_wait(&rr.full[rr.stage(n)], rr.phase(n)))) break;
      // Four 32-column chunks; each chunk's scores are loaded while the
      // previous one is turned into weights (two buffers of 32 registers).
      auto quarter = [&](const uint32_t (&sv)[32], int c) {
        float rk[32];
        if constexpr (NM == 1) {
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 f = *reinterpret_cast<const float4*>(rk_tile + 32 * c + j);
            rk[j] = f.x;
            rk[j + 1] = f.y;
            rk[j + 2] = f.z;
            rk[j + 3] = f.w;
          }
        }
        if (diag)
          diff_quarter<PC, NM, true, mix_mufu_pairs<D>()>(sv, tS, 32 * c, wp, rq2, ntau2, rk, n * BT, row);
        else
          diff_quarter<PC, NM, false, mix_mufu_pairs<D>()>(sv, tS, 32 * c, wp, rq2, ntau2, rk, n * BT, row);
      };
      uint32_t sa[32], sb[32];
      tmem_ld32(tS, sa);
      tmem_wait_ld();
      tmem_ld32(tS + 32, sb);
      quarter(sa, 0);  // P of chunk c lands in columns 16c .., already read
      tmem_wait_ld();
      tmem_ld32(tS + 64, sa);
      quarter(sb, 1);
      tmem_wait_ld();
      tmem_ld32(tS + 96, sb);
      quarter(sa, 2);
      tmem_wait_ld();
      quarter(sb, 3);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&p_full[t]);
        if constexpr (NM == 1) mbar_arrive(&rr.empty[rr.stage(n)]);  // done with the key factors
      }
    }
    if (ok && mbar_wait(&o_full[0], 0) && mbar_wait(&o_full[1], 0)) {
      tc_fence_after();
      __nv_bfloat16* orow = out + (static_cast<size_t>(bh) * T + row) * dr;
      // out = O0 - clamp(lambda, 0, 1) O1; stream t's warpgroup writes every other 32-column chunk.
      for (int c = t; c < D / 32 && c * 32 < dr; c += 2) {
        uint32_t o0[32], o1[32];
        tmem_ld32(lane_base + O_COL + c * 32, o0);
        tmem_ld32(lane_base + O_COL + D + c * 32, o1);
        tmem_wait_ld();
        if (row < T) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
          const int nq = min(32, dr - c * 32) / 8;  // 16-byte stores of this chunk's real columns
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (q >= nq) break;
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = fmaf(-lc, __uint_as_float(o1[8 * q + e]), __uint_as_float(o0[8 * q + e]));
            dst[q] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                                pack_bf16x2(f[6], f[7]));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == DIFF_MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int PC, int NM>
int launch_diff_kernel(const CUtensorMap* maps, const float* inv, void* out, int BH, int T, float beta, float p,
                       float lam, int d_real, cudaStream_t stream) {
  using L = DiffLayout<D>;
  auto kern = tra_diff_kernel<D, PC, NM>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC) != cudaSuccess)
    return ERR_LAUNCH;
  const int nQ = (T + BT - 1) / BT;
  const long long grid = static_cast<long long>(nQ) * BH;
  if (grid > 0x7fffffffLL) return ERR_SHAPE;
  // K1, K2, V: three streamed bf16 tensors per head; one resident CTA per SM
  const int G = tile::head_groups(BH, nQ, 6LL * T * d_real, sm_count());
  kern<<<static_cast<unsigned>(grid), DiffCfg<D, PC>::THREADS, L::ALLOC, stream>>>(
      maps[0], maps[1], maps[2], maps[3], maps[4], inv, static_cast<__nv_bfloat16*>(out), BH, T, nQ, G, beta, p,
      lam, d_real);
  return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
}

template <int D, int NM>
int dispatch_pc(const CUtensorMap* maps, const float* inv, void* out, int BH, int T, float beta, float p, float lam,
                int d_real, cudaStream_t stream) {
  const int pc = power_class(p);
  if (pc == POW_TWO) return launch_diff_kernel<D, POW_TWO, NM>(maps, inv, out, BH, T, beta, p, lam, d_real, stream);
  if (pc == POW_ONE) return launch_diff_kernel<D, POW_ONE, NM>(maps, inv, out, BH, T, beta, p, lam, d_real, stream);
  if (pc == POW_GENERAL_MIX && BSA_DIFF_MIX)
    return launch_diff_kernel<D, POW_GENERAL_MIX, NM>(maps, inv, out, BH, T, beta, p, lam, d_real, stream);
  return launch_diff_kernel<D, POW_GENERAL, NM>(maps, inv, out, BH, T, beta, p, lam, d_real, stream);
}

// Row-norm pre-pass at the head dim D (the real one).
template <int D>
void launch_row_norms(unsigned blocks, const __nv_bfloat16* a0, const __nv_bfloat16* a1, const __nv_bfloat16* a2,
                      const __nv_bfloat16* a3, float* inv, __nv_bfloat16* kn, int BH, int T, int Tp, bool idx32,
                      cudaStream_t stream) {
  if (kn != nullptr) {
    if (idx32)
      row_inv_norm_kernel<D, uint32_t, true><<<blocks, 256, 0, stream>>>(a0, a1, a2, a3, inv, kn, BH, T, Tp);
    else
      row_inv_norm_kernel<D, unsigned long long, true><<<blocks, 256, 0, stream>>>(a0, a1, a2, a3, inv, kn, BH, T,
                                                                                  Tp);
  } else if (idx32) {
    row_inv_norm_kernel<D, uint32_t, false><<<blocks, 256, 0, stream>>>(a0, a1, a2, a3, inv, kn, BH, T, Tp);
  } else {
    row_inv_norm_kernel<D, unsigned long long, false><<<blocks, 256, 0, stream>>>(a0, a1, a2, a3, inv, kn, BH, T, Tp);
  }
}

}  // namespace

size_t tra_diff_scratch_bytes(int B, int H, int T) {
  const size_t Tp = ((static_cast<size_t>(T) + BT - 1) / BT) * BT;
  return 4 * sizeof(float) * static_cast<size_t>(B) * H * Tp;
}

int launch_tra_diff_bf16(const void* q1, const void* q2, const void* k1, const void* k2, const void* v, void* out,
                         int B, int H, int T, int D, float beta, float lam, float p, float* inv_norm, void* knorm,
                         cudaStream_t stream) {
  if (!tra_head_dim_supported(D)) return ERR_UNSUPPORTED;
  const int BH = B * H;
  CUtensorMap maps[5];
  const uint64_t rs = static_cast<uint64_t>(D) * 2, hs = rs * T;
  // with knorm, the kernel reads the normalised k copies the pre-pass writes there
  const bool kn = knorm != nullptr;
  auto* kn1 = static_cast<__nv_bfloat16*>(knorm);
  const void* src[5] = {q1, q2, kn ? static_cast<const void*>(kn1) : k1,
                        kn ? static_cast<const void*>(kn1 + static_cast<size_t>(BH) * T * D) : k2, v};
  for (int i = 0; i < 5; ++i) {
    const int st = encode_tmap_3d(&maps[i], src[i], D, T, BH, rs, hs, 64, BT, 1);
    if (st != OK) return st;
  }
  const bool norm = inv_norm != nullptr || kn;
  if (norm) {
    const int Tp = ((T + BT - 1) / BT) * BT;
    const long long rows = (kn ? 2LL : 4LL) * BH * Tp;  // 32 * NORM_NG rows per 256-thread block per pass
    const int sms = sm_count();
    if (sms <= 0) return ERR_DEVICE;
    const long long want = (rows + 32 * NORM_NG - 1) / (32 * NORM_NG), cap = 8LL * sms;
    const unsigned blocks = static_cast<unsigned>(want < cap ? want : cap);
    const auto* a0 = static_cast<const __nv_bfloat16*>(q1);
    const auto* a1 = static_cast<const __nv_bfloat16*>(k1);
    const auto* a2 = static_cast<const __nv_bfloat16*>(q2);
    const auto* a3 = static_cast<const __nv_bfloat16*>(k2);
    const bool idx32 = rows < (1LL << 32);  // every row index (and the division by Tp) fits 32 bits
    auto* kw = kn ? kn1 : nullptr;
    switch (D) {
#define BSA_ROW_NORMS(d) \
  case d: launch_row_norms<d>(blocks, a0, a1, a2, a3, inv_norm, kw, BH, T, Tp, idx32, stream); break;
      BSA_ROW_NORMS(16) BSA_ROW_NORMS(32) BSA_ROW_NORMS(48) BSA_ROW_NORMS(64)
      BSA_ROW_NORMS(80) BSA_ROW_NORMS(96) BSA_ROW_NORMS(112) BSA_ROW_NORMS(128)
#undef BSA_ROW_NORMS
      default: return ERR_UNSUPPORTED;
    }
    if (cudaGetLastError() != cudaSuccess) return ERR_LAUNCH;
  }
  const int nm = !norm ? 0 : kn ? 2 : 1;
  if (D > 64) {  // width 128 (80 .. 128 on zero-filled columns)
    if (nm == 2) return dispatch_pc<128, 2>(maps, inv_norm, out, BH, T, beta, p, lam, D, stream);
    if (nm == 1) return dispatch_pc<128, 1>(maps, inv_norm, out, BH, T, beta, p, lam, D, stream);
    return dispatch_pc<128, 0>(maps, inv_norm, out, BH, T, beta, p, lam, D, stream);
  }
  // width 64 (16 .. 48 on zero-filled columns)
  if (nm == 2) return dispatch_pc<64, 2>(maps, inv_norm, out, BH, T, beta, p, lam, D, stream);
  if (nm == 1) return dispatch_pc<64, 1>(maps, inv_norm, out, BH, T, beta, p, lam, D, stream);
  return dispatch_pc<64, 0>(maps, inv_norm, out, BH, T, beta, p, lam, D, stream);
}

// ------------------------------------------------ allocation-free entry point
//
// Fixed scratch for tra_diff_forward_noalloc: the normalisation factors of at
// most TRA_DIFF_NOALLOC_MAX_ROWS padded (b, h, t) rows of each of q1, k1, q2,
// k2 (16 MiB of device memory on every GPU that loads the library, held until
// the process exits).  In host code the name below is only a stand-in for the
// device symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) float g_noalloc_inv_norm[4 * TRA_DIFF_NOALLOC_MAX_ROWS];

namespace {
// Device address of g_noalloc_inv_norm on the current device, looked up once
// per device (with that device current) and cached.
int noalloc_scratch(float** out) {
  constexpr int MAX_DEVICES = 64;
  static std::mutex mu;
  static float* cache[MAX_DEVICES] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return ERR_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_inv_norm) != cudaSuccess || ptr == nullptr) return ERR_DEVICE;
    cache[dev] = static_cast<float*>(ptr);
  }
  *out = cache[dev];
  return OK;
}
}  // namespace

bool tra_diff_noalloc_fits(int B, int H, int T) {
  return tra_diff_scratch_bytes(B, H, T) <= sizeof(float) * 4 * static_cast<size_t>(TRA_DIFF_NOALLOC_MAX_ROWS);
}

int launch_tra_diff_noalloc_bf16(const void* q1, const void* q2, const void* k1, const void* k2, const void* v,
                                 void* out, int B, int H, int T, int D, float beta, float lam, float p,
                                 bool normalize, cudaStream_t stream) {
  if (!normalize)
    return launch_tra_diff_bf16(q1, q2, k1, k2, v, out, B, H, T, D, beta, lam, p, nullptr, nullptr, stream);
  if (!tra_diff_noalloc_fits(B, H, T)) return ERR_SCRATCH_LIMIT;
  float* scratch = nullptr;
  const int st = noalloc_scratch(&scratch);
  if (st != OK) return st;
  return launch_tra_diff_bf16(q1, q2, k1, k2, v, out, B, H, T, D, beta, lam, p, scratch, nullptr, stream);
}

unsigned int tra_diff_device_error() { return read_and_clear_device_error(); }

}  // namespace bsa
