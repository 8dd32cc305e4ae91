// tra_bwd.cu -- threshold rectified attention backward, bf16 in / fp32
// accumulate, on tcgen05 tensor cores.
//
// Method: page "triton_threshold_attention.py", ThresholdRelaFunction.backward
// with _threshold_rela_bwd_kernel_dq and _threshold_rela_bwd_kernel_dkv: with
// x_ij = q_i.k_j - tau(i) over the causal pairs j <= i,
//     W_ij  = ReLU(x_ij)^p                       dV_j = sum_i W_ij dO_i
//     dA_ij = (dO_i . v_j) p ReLU(x_ij)^(p-1)     dK_j = sum_i dA_ij q_i
//                                                dQ_i = sum_j dA_ij k_j
// (derivative 0 where x <= 0, as on the page; beta and p get no gradient).
// Like the page, two kernels: one per key tile for dK and dV, one per query
// tile for dQ; both recompute the scores instead of storing W.  This is the
// deterministic form (bit-repeatable, no scratch) behind
// BSA_TRA_BWD_DETERMINISTIC; the default bf16 backward is the fused kernel of
// tra_bwd_fused.cu, which produces the scores once per tile pair.  Head dims
// 16 and 32 run the width-64 kernels on zero-filled columns.
//
// dK/dV kernel, one CTA per 128-key tile n of one (b, h), looping over the
// query tiles m >= n: S^T = K_n Q_m^T and dP^T = V_n dO_m^T into TMEM; the
// epilogue (thread = key row, tau per query column from a shared table) turns
// them into W^T and dA^T (bf16, written over the consumed columns); then
// dV += W^T dO_m and dK += dA^T Q_m with the A operand read from TMEM.
// TMEM: S^T [0,128), dP^T [128,256), dV [256,256+D), dK [256+D,256+2D).
//
// dQ kernel, one CTA per 128-row query tile m, looping over key tiles n <= m:
// S = Q_m K_n^T and dP = dO_m V_n^T; the epilogue (thread = query row) forms
// dA; then dQ += dA K_n.  TMEM: S [0,128), dP [128,256), dQ [256,256+D).
//
// Both grids number their blocks in head groups (tile::head_group_item): the
// CTAs resident at one time stream the tiles of a few heads, which stay in L2.
//
// Both kernels produce each 128 x 128 score (and gradient) tile in two
// 64-column halves h that behave like two tiles: the epilogue turns half h
// into bf16 while the other half's products run, and the products that read
// half h (dV, dK; dQ) start as soon as it is done.  Two threads issue the
// MMAs (one thread sustains only about one tcgen05.mma per ~70 cycles):
//   dK/dV: warp 5 issues S^T_h and dV (its A operand, W^T, lives in S^T's
//          columns), warp 6 issues dP^T_h and dK (dA^T in dP^T's columns);
//   dQ:    warp 5 issues S_h and dQ (dA is written over S), warp 6 dP_h.
// Each issuer's own MMAs overwrite a half only after the products that read
// it (same thread, in order).  Warp 4 = TMA producer, warps 0-3 = epilogue;
// every wait is bounded.
#include "kernels.h"
#include "ptx.cuh"
#include "tc_tile.cuh"
#include "tra_bwd_common.cuh"

namespace bsa {
namespace {

using tile::PANEL_BYTES;
constexpr int BT = tile::ROWS;  // 128 rows per query tile and per key tile
// Epilogue warpgroups (1 or 2).  With two, warps w and w + 4 share a TMEM lane
// quarter and take the two 32-column chunks of each score half, so every
// SMSP runs two epilogue warps and one chunk's TMEM loads and arithmetic
// overlap the other's.  Measured: B2 H32 T8192 D64 p=2 2.19 -> 2.10 ms,
// p=1.5 3.69 -> 3.29 ms; B4 H16 T4096 D128 p=2 0.791 -> 0.816 ms (slower), so
// D = 128 with p = 1 or 2 keeps one.  BSA_BWD_EPI_WG forces 1 or 2 (0: that
// choice).
#ifndef BSA_BWD_EPI_WG
#define BSA_BWD_EPI_WG 0
#endif
#ifndef BSA_BWD_DQ_EPI_WG
#define BSA_BWD_DQ_EPI_WG BSA_BWD_EPI_WG
#endif
#ifndef BSA_BWD_DKDV_EPI_WG
#define BSA_BWD_DKDV_EPI_WG BSA_BWD_EPI_WG
#endif
template <int D, int PC, bool DQ>
struct BwdCfg {
  static constexpr bool LIGHT = (PC == POW_ONE || PC == POW_TWO) && D == 128;
  static constexpr int FORCED = DQ ? BSA_BWD_DQ_EPI_WG : BSA_BWD_DKDV_EPI_WG;
  static constexpr int EPI_WG = FORCED != 0 ? FORCED : (LIGHT ? 1 : 2);
  static constexpr int EPI_WARPS = 4 * EPI_WG;
  static constexpr int TMA_WARP = EPI_WARPS;
  static constexpr int MMA_WARP = EPI_WARPS + 1;  // first of the two MMA-issuing warps (allocates TMEM)
  static constexpr int THREADS = 32 * (EPI_WARPS + 3);
};
constexpr uint32_t TMEM_COLS = 512;

using bwd::weight_and_grad;

template <int D>
struct BwdLayout {
  static constexpr int NP = D / 64;
  static constexpr int TILE = NP * PANEL_BYTES;
  static constexpr int NS = (D == 128) ? 2 : 4;  // ring stages, each two tiles
  static constexpr int RES_OFF = 0;              // two resident tiles
  static constexpr int RING_OFF = 2 * TILE;
  static constexpr int TAU_OFF = RING_OFF + NS * 2 * TILE;  // float[2][128]
  static constexpr int BAR_OFF = TAU_OFF + 2 * BT * 4;
  // res_full | ring_full[NS] | ring_empty[NS] | s_full[2] | p_full[2] | acc_full | mma_done[2] | tau_full[2]
  static constexpr int NBAR = 1 + 2 * NS + 9;
  static constexpr int TPTR_OFF = BAR_OFF + NBAR * 8;
  static constexpr int ALLOC = TPTR_OFF + 16 + 1024;
};

struct BwdBars {
  uint64_t *res_full, *ring_full, *ring_empty, *s_full, *p_full, *acc_full, *mma_done, *tau_full;
};

template <int D>
__device__ __forceinline__ BwdBars bwd_bars(uint8_t* smem) {
  using L = BwdLayout<D>;
  uint64_t* b = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  BwdBars r;
  r.res_full = b;
  r.ring_full = b + 1;
  r.ring_empty = r.ring_full + L::NS;
  r.s_full = r.ring_empty + L::NS;  // [2], per half
  r.p_full = r.s_full + 2;          // [2], per half
  r.acc_full = r.p_full + 2;
  r.mma_done = r.acc_full + 1;      // [2], per issuer
  r.tau_full = r.mma_done + 2;      // [2], per tau buffer
  return r;
}

template <int D>
__device__ __forceinline__ void bwd_setup(uint8_t* smem, const BwdBars& B, uint32_t* tptr, int warp, int acc_count,
                                          int epi_warps, int mma_warp) {
  using L = BwdLayout<D>;
  if (threadIdx.x == 0) {
    mbar_init(B.res_full, 1);
    for (int s = 0; s < L::NS; ++s) {
      mbar_init(&B.ring_full[s], 1);
      mbar_init(&B.ring_empty[s], 2);  // one release per issuer
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&B.s_full[h], 2);  // both issuers' products of half h
      mbar_init(&B.p_full[h], epi_warps);
      mbar_init(&B.mma_done[h], 1);
      mbar_init(&B.tau_full[h], epi_warps);
    }
    mbar_init(B.acc_full, acc_count);
    fence_barrier_init();
  }
  if (warp == mma_warp) {
    tmem_alloc(tptr, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

__device__ __forceinline__ void bwd_teardown(uint32_t tmem, int warp, int mma_warp) {
  tc_fence_before();
  __syncthreads();
  if (warp == mma_warp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// C_tmem[128 x 64] = A[128 x D] B_h[64 x D]^T: the score half h of a tile,
// B_h being rows 64h .. 64h+63 of a K-major 128-row smem tile (8 KB into
// each 128-byte-swizzled panel, a whole number of swizzle atoms).
template <int D>
__device__ __forceinline__ void mma_abt_half(uint32_t tC, uint32_t sA, uint32_t sB, int h, bool leader) {
  constexpr uint32_t IDESC = idesc_bf16_f32(BT, 64, 0, 0);
  const uint32_t sBh = sB + static_cast<uint32_t>(h) * 64u * 128u;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * PANEL_BYTES + (kk & 3) * 32;
    const uint64_t a = smem_desc_sw128(sA + off, 16, 1024), b = smem_desc_sw128(sBh + off, 16, 1024);
    if (leader) mma_ss(tC, a, b, IDESC, kk > 0 ? 1u : 0u);
  }
}

// MMA issue: one elected lane issues.  At D = 64 the whole warp walks the
// issue loop with it (the descriptors are then warp-uniform values), which
// issues the short N = 64 products faster (B2 H32 T8192 D64 p=2: 2.38 ->
// 2.19 ms); at D = 128 that measured 5% slower than the elected lane
// walking it alone.  0: never, 1: D = 64 only, 2: always.
#ifndef BSA_BWD_CONVERGED_ISSUE
#define BSA_BWD_CONVERGED_ISSUE 1
#endif
template <int D>
constexpr bool bwd_converged_issue() {
  return BSA_BWD_CONVERGED_ISSUE == 2 || (BSA_BWD_CONVERGED_ISSUE == 1 && D == 64);
}

// Producer: two resident tiles (rows res_row of maps r0, r1), then for
// j = 0..count-1 two ring tiles (rows (first + j) * 128 of maps g0, g1).
template <int D>
__device__ __forceinline__ void bwd_produce(uint8_t* smem, const BwdBars& B, const CUtensorMap* r0,
                                            const CUtensorMap* r1, int res_row, const CUtensorMap* g0,
                                            const CUtensorMap* g1, int first, int count, int bh) {
  using L = BwdLayout<D>;
  tma_prefetch_desc(r0);
  tma_prefetch_desc(r1);
  tma_prefetch_desc(g0);
  tma_prefetch_desc(g1);
  debug_check(res_row >= 0 && first >= 0 && bh >= 0);
  mbar_arrive_expect_tx(B.res_full, 2 * L::TILE);
  tile::tma_tile<D>(smem + L::RES_OFF, r0, B.res_full, res_row, bh);
  tile::tma_tile<D>(smem + L::RES_OFF + L::TILE, r1, B.res_full, res_row, bh);
  int issued = 0;
  bool ok = true;
  for (int j = 0; j < count; ++j) {
    const int s = j % L::NS;
    if (!(ok = mbar_wait(&B.ring_empty[s], ((j / L::NS) & 1) ^ 1))) break;
    uint8_t* dst = smem + L::RING_OFF + s * 2 * L::TILE;
    mbar_arrive_expect_tx(&B.ring_full[s], 2 * L::TILE);
    tile::tma_tile<D>(dst, g0, &B.ring_full[s], (first + j) * BT, bh);
    tile::tma_tile<D>(dst + L::TILE, g1, &B.ring_full[s], (first + j) * BT, bh);
    issued = j + 1;
  }
  if (!ok) {  // drain what is still landing before the CTA may exit
    mbar_wait(B.res_full, 0);
    for (int j = (issued > L::NS ? issued - L::NS : 0); j < issued; ++j)
      mbar_wait(&B.ring_full[j % L::NS], (j / L::NS) & 1);
  }
}

// ---------------------------------------------------------------- dK / dV

// dK/dV work of block `blk` (key tile, head): the body of the dK/dV kernel.
template <int D, int PC>
__device__ __forceinline__ void bwd_dkdv_block(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                               const CUtensorMap& tmDO, __nv_bfloat16* __restrict__ dk,
                                               __nv_bfloat16* __restrict__ dv, int BH, int T, int nT, int G,
                                               float beta, float p, int blk, int d_real) {
  using L = BwdLayout<D>;
  const int dr = d_real;  // head dim (the tile width D or less: zero-filled columns)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const BwdBars B = bwd_bars<D>(smem);
  uint32_t* tptr = reinterpret_cast<uint32_t*>(smem + L::TPTR_OFF);
  float* tau_s = reinterpret_cast<float*>(smem + L::TAU_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tile::HeadItem item = tile::head_group_item(blk, BH, nT, G);
  const int n = item.rank;  // key tile; n = 0 has the most query tiles
  const int bh = item.bh;
  const int nq = nT - n;  // query tiles m = n .. nT-1
  constexpr uint32_t ST = 0, DPT = BT, DV = 2 * BT, DK = 2 * BT + D;

  using Cfg = BwdCfg<D, PC, false>;
  constexpr int EPI_WG = Cfg::EPI_WG, EPI_WARPS = Cfg::EPI_WARPS, TMA_WARP = Cfg::TMA_WARP, MMA_WARP = Cfg::MMA_WARP;
  bwd_setup<D>(smem, B, tptr, warp, 2, EPI_WARPS, MMA_WARP);
  const uint32_t tmem = *tptr;

  if (warp == TMA_WARP) {
    if (lane == 0) {
      debug_check(bh >= 0 && bh < BH && n * BT < T && (n + nq - 1) * BT < T);
      bwd_produce<D>(smem, B, &tmK, &tmV, n * BT, &tmQ, &tmDO, n, nq, bh);
    }
  } else if (warp == MMA_WARP || warp == MMA_WARP + 1) {
    // Issuer X (warp 5): S^T_h = K_n Q_m[h]^T and dV += W^T_h dO_m[h];
    // issuer Y (warp 6): dP^T_h = V_n dO_m[h]^T and dK += dA^T_h Q_m[h].
    // Per query tile j: acc(j, 0), score(j+1, 0), acc(j, 1), score(j+1, 1).
    const int is = warp - MMA_WARP;
    const bool leader = elect_one();
    if (bwd_converged_issue<D>() || leader) {
      const uint32_t sRes = smem_u32(smem + L::RES_OFF) + (is == 0 ? 0u : static_cast<uint32_t>(L::TILE));
      const uint32_t tScore = tmem + (is == 0 ? ST : DPT), tAcc = tmem + (is == 0 ? DV : DK);
      auto slot = [&](int j) { return smem_u32(smem + L::RING_OFF + (j % L::NS) * 2 * L::TILE); };  // Q_j | dO_j
      auto mma_commit = [&](uint64_t* bar) {
        if (leader) bsa::mma_commit(bar);
      };
      auto score = [&](int j, int h) {
        mma_abt_half<D>(tScore + 64 * h, sRes, slot(j) + (is == 0 ? 0u : static_cast<uint32_t>(L::TILE)), h,
                        leader);
        mma_commit(&B.s_full[h]);
      };
      auto acc = [&](int j, int h) {
        tile::mma_tmem_a<D>(tAcc, tScore + 32 * h, slot(j) + (is == 0 ? static_cast<uint32_t>(L::TILE) : 0u),
                            4 * h, 4 * h + 4, j == 0 && h == 0, leader);
      };
      bool ok = mbar_wait(B.res_full, 0) && mbar_wait(&B.ring_full[0], 0);
      if (ok) {
        tc_fence_after();
        score(0, 0);
        score(0, 1);
      }
      for (int j = 0; j < nq && ok; ++j) {
        const bool more = j + 1 < nq;
        for (int h = 0; h < 2; ++h) {
          if (!(ok = mbar_wait(&B.p_full[h], j & 1))) break;
          tc_fence_after();
          acc(j, h);
          if (h == 1) mma_commit(&B.ring_empty[j % L::NS]);  // Q_j, dO_j read by every product issued so far
          if (more) {
            if (h == 0 && !(ok = mbar_wait(&B.ring_full[(j + 1) % L::NS], ((j + 1) / L::NS) & 1))) break;
            tc_fence_after();
            score(j + 1, h);
          }
        }
      }
      if (ok) mma_commit(B.acc_full);
      mma_commit(&B.mma_done[is]);
      mbar_wait(&B.mma_done[is], 0);
    }
  } else if (warp < EPI_WARPS) {
    const int wq = warp & 3, grp = warp >> 2;  // TMEM lane quarter; chunk of each half (two warpgroups)
    const int r = wq * 32 + lane;              // key row within the tile
    const int key = n * BT + r;
    const float lp = log2f(p);
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    bool ok = true;
    for (int j = 0; j < nq && ok; ++j) {
      const int m = n + j;
      // Double-buffered tau table: a warp writes buffer j&1 for step j only
      // after every warp arrived for step j-1 (so all have finished step j-2,
      // the buffer's previous user); the barrier wait is bounded.
      float* tau_m = tau_s + (j & 1) * BT;
      tau_m[r] = tile::tau_of_row(m * BT + r, beta, dr);  // tau of query column r
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.tau_full[j & 1]);
      if (!(ok = mbar_wait(&B.tau_full[j & 1], (j >> 1) & 1))) break;
      const bool diag = (m == n);
      for (int h = 0; h < 2; ++h) {
        if (!(ok = mbar_wait(&B.s_full[h], j & 1))) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 2 * h + (EPI_WG == 2 ? grp : 0); c < 2 * h + 2; c += EPI_WG) {
          uint32_t sv[32], dp[32];
          tmem_ld32(lane_base + ST + 32 * c, sv);
          tmem_ld32(lane_base + DPT + 32 * c, dp);
          tmem_wait_ld();
          // Chunk 2h + 1 packs into chunk 2h's columns: with two warpgroups,
          // both chunks are loaded before either warp stores.
          if constexpr (EPI_WG == 2) asm volatile("bar.sync %0, 64;" ::"r"(1 + wq) : "memory");
          uint32_t wpk[16], apk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float w0, g0, w1, g1;
            const int i0 = 32 * c + 2 * e;  // query column within the tile
            weight_and_grad<PC>(__uint_as_float(sv[2 * e]) - tau_m[i0], p, lp, w0, g0);
            weight_and_grad<PC>(__uint_as_float(sv[2 * e + 1]) - tau_m[i0 + 1], p, lp, w1, g1);
            float a0 = __uint_as_float(dp[2 * e]) * g0, a1 = __uint_as_float(dp[2 * e + 1]) * g1;
            if (diag) {  // causal: key r <= query column
              if (i0 < r) w0 = a0 = 0.0f;
              if (i0 + 1 < r) w1 = a1 = 0.0f;
            }
            wpk[e] = pack_bf16x2(w0, w1);
            apk[e] = pack_bf16x2(a0, a1);
          }
          // half h packs into its own first 32 columns (already-consumed scores)
          const int pc = 64 * h + 16 * (c - 2 * h);
          tmem_st16(lane_base + ST + pc, wpk);
          tmem_st16(lane_base + DPT + pc, apk);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.p_full[h]);
      }
    }
    if (ok && mbar_wait(B.acc_full, 0)) {
      tc_fence_after();
      const size_t rowoff = (static_cast<size_t>(bh) * T + key) * dr;
      constexpr int CPW = D / 32 / EPI_WG;  // 32-column chunks of dK, dV this warp stores
#pragma unroll
      for (int c = grp * CPW; c < (grp + 1) * CPW; ++c) {
        if (dr == D) {
          tile::store_row_chunk(lane_base + DV, c, dv + rowoff, key < T);
          tile::store_row_chunk(lane_base + DK, c, dk + rowoff, key < T);
        } else if (c * 32 < dr) {
          tile::store_row_part(lane_base + DV, c, dv + rowoff, key < T, min(32, dr - c * 32));
          tile::store_row_part(lane_base + DK, c, dk + rowoff, key < T, min(32, dr - c * 32));
        }
      }
    }
  }
  bwd_teardown(tmem, warp, MMA_WARP);
}

// ---------------------------------------------------------------------- dQ

// dQ work of block `blk` (query tile, head): the body of the dQ kernel.
template <int D, int PC>
__device__ __forceinline__ void bwd_dq_block(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                             const CUtensorMap& tmDO, __nv_bfloat16* __restrict__ dq, int BH, int T,
                                             int nT, int G, float beta, float p, int blk, int d_real) {
  using L = BwdLayout<D>;
  const int dr = d_real;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const BwdBars B = bwd_bars<D>(smem);
  uint32_t* tptr = reinterpret_cast<uint32_t*>(smem + L::TPTR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tile::HeadItem item = tile::head_group_item(blk, BH, nT, G);
  const int m = nT - 1 - item.rank;  // longest first
  const int bh = item.bh;
  constexpr uint32_t S = 0, DP = BT, DQ = 2 * BT;

  using Cfg = BwdCfg<D, PC, true>;
  constexpr int EPI_WG = Cfg::EPI_WG, EPI_WARPS = Cfg::EPI_WARPS, TMA_WARP = Cfg::TMA_WARP, MMA_WARP = Cfg::MMA_WARP;
  bwd_setup<D>(smem, B, tptr, warp, 1, EPI_WARPS, MMA_WARP);
  const uint32_t tmem = *tptr;

  if (warp == TMA_WARP) {
    if (lane == 0) {
      debug_check(bh >= 0 && bh < BH && m * BT < T);
      bwd_produce<D>(smem, B, &tmQ, &tmDO, m * BT, &tmK, &tmV, 0, m + 1, bh);
    }
  } else if (warp == MMA_WARP || warp == MMA_WARP + 1) {
    // Issuer X (warp 5): S_h = Q_m K_n[h]^T and dQ += dA_h K_n[h] (dA over S);
    // issuer Y (warp 6): dP_h = dO_m V_n[h]^T, re-issued for the next key tile
    // once the epilogue has read half h.
    const int is = warp - MMA_WARP;
    const bool leader = elect_one();
    if (bwd_converged_issue<D>() || leader) {
      const uint32_t sRes = smem_u32(smem + L::RES_OFF) + (is == 0 ? 0u : static_cast<uint32_t>(L::TILE));
      const uint32_t tScore = tmem + (is == 0 ? S : DP);
      auto slot = [&](int j) { return smem_u32(smem + L::RING_OFF + (j % L::NS) * 2 * L::TILE); };  // K_j | V_j
      auto mma_commit = [&](uint64_t* bar) {
        if (leader) bsa::mma_commit(bar);
      };
      auto score = [&](int j, int h) {
        mma_abt_half<D>(tScore + 64 * h, sRes, slot(j) + (is == 0 ? 0u : static_cast<uint32_t>(L::TILE)), h,
                        leader);
        mma_commit(&B.s_full[h]);
      };
      bool ok = mbar_wait(B.res_full, 0) && mbar_wait(&B.ring_full[0], 0);
      if (ok) {
        tc_fence_after();
        score(0, 0);
        score(0, 1);
      }
      for (int j = 0; j <= m && ok; ++j) {
        const bool more = j < m;
        for (int h = 0; h < 2; ++h) {
          if (!(ok = mbar_wait(&B.p_full[h], j & 1))) break;
          tc_fence_after();
          if (is == 0)
            tile::mma_tmem_a<D>(tmem + DQ, tmem + S + 32 * h, slot(j), 4 * h, 4 * h + 4, j == 0 && h == 0, leader);
          if (h == 1) mma_commit(&B.ring_empty[j % L::NS]);  // K_j, V_j read by every product issued so far
          if (more) {
            if (h == 0 && !(ok = mbar_wait(&B.ring_full[(j + 1) % L::NS], ((j + 1) / L::NS) & 1))) break;
            tc_fence_after();
            score(j + 1, h);
          }
        }
      }
      if (ok && is == 0) mma_commit(B.acc_full);
      mma_commit(&B.mma_done[is]);
      mbar_wait(&B.mma_done[is], 0);
    }
  } else if (warp < EPI_WARPS) {
    const int wq = warp & 3, grp = warp >> 2;  // TMEM lane quarter; chunk of each half (two warpgroups)
    const int r = wq * 32 + lane;
    const int row = m * BT + r;
    const float tau = tile::tau_of_row(row, beta, dr);
    const float lp = log2f(p);
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    bool ok = true;
    for (int n = 0; n <= m && ok; ++n) {
      const bool diag = (n == m);
      for (int h = 0; h < 2; ++h) {
        if (!(ok = mbar_wait(&B.s_full[h], n & 1))) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 2 * h + (EPI_WG == 2 ? grp : 0); c < 2 * h + 2; c += EPI_WG) {
          uint32_t sv[32], dp[32];
          tmem_ld32(lane_base + S + 32 * c, sv);
          tmem_ld32(lane_base + DP + 32 * c, dp);
          tmem_wait_ld();
          // Chunk 2h + 1 packs into chunk 2h's columns (see the dK/dV kernel).
          if constexpr (EPI_WG == 2) asm volatile("bar.sync %0, 64;" ::"r"(1 + wq) : "memory");
          uint32_t apk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float w0, g0, w1, g1;
            weight_and_grad<PC>(__uint_as_float(sv[2 * e]) - tau, p, lp, w0, g0);
            weight_and_grad<PC>(__uint_as_float(sv[2 * e + 1]) - tau, p, lp, w1, g1);
            float a0 = __uint_as_float(dp[2 * e]) * g0, a1 = __uint_as_float(dp[2 * e + 1]) * g1;
            if (diag) {  // causal: key column <= query row r
              const int kc = 32 * c + 2 * e;
              if (kc > r) a0 = 0.0f;
              if (kc + 1 > r) a1 = 0.0f;
            }
            apk[e] = pack_bf16x2(a0, a1);
          }
          tmem_st16(lane_base + S + 64 * h + 16 * (c - 2 * h), apk);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.p_full[h]);
      }
    }
    if (ok && mbar_wait(B.acc_full, 0)) {
      tc_fence_after();
      __nv_bfloat16* dst = dq + (static_cast<size_t>(bh) * T + row) * dr;
      constexpr int CPW = D / 32 / EPI_WG;  // 32-column chunks of dQ this warp stores
#pragma unroll
      for (int c = grp * CPW; c < (grp + 1) * CPW; ++c) {
        if (dr == D)
          tile::store_row_chunk(lane_base + DQ, c, dst, row < T);
        else if (c * 32 < dr)
          tile::store_row_part(lane_base + DQ, c, dst, row < T, min(32, dr - c * 32));
      }
    }
  }
  bwd_teardown(tmem, warp, MMA_WARP);
}

template <int D, int PC>
__global__ void __launch_bounds__(BwdCfg<D, PC, false>::THREADS, 1)
    tra_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                        __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, int BH, int T, int nT,
                        int G, float beta, float p, int d_real) {
  bwd_dkdv_block<D, PC>(tmQ, tmK, tmV, tmDO, dk, dv, BH, T, nT, G, beta, p, static_cast<int>(blockIdx.x), d_real);
}

template <int D, int PC>
__global__ void __launch_bounds__(BwdCfg<D, PC, true>::THREADS, 1)
    tra_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                      __nv_bfloat16* __restrict__ dq, int BH, int T, int nT, int G, float beta, float p,
                      int d_real) {
  bwd_dq_block<D, PC>(tmQ, tmK, tmV, tmDO, dq, BH, T, nT, G, beta, p, static_cast<int>(blockIdx.x), d_real);
}

// Both kinds of block in one grid: the dK/dV blocks first, then the dQ
// blocks, which start on the SMs the dK/dV blocks' tail leaves free instead of
// after the whole first launch has drained.
template <int D, int PC>
__global__ void __launch_bounds__(BwdCfg<D, PC, false>::THREADS, 1)
    tra_bwd_both_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                        __nv_bfloat16* __restrict__ dq, __nv_bfloat16* __restrict__ dk,
                        __nv_bfloat16* __restrict__ dv, int BH, int T, int nT, int G, float beta, float p,
                        int d_real) {
  const int nk = nT * BH, b = static_cast<int>(blockIdx.x);
  if (b < nk)
    bwd_dkdv_block<D, PC>(tmQ, tmK, tmV, tmDO, dk, dv, BH, T, nT, G, beta, p, b, d_real);
  else
    bwd_dq_block<D, PC>(tmQ, tmK, tmV, tmDO, dq, BH, T, nT, G, beta, p, b - nk, d_real);
}

#ifndef BSA_BWD_ONE_GRID
#define BSA_BWD_ONE_GRID 1
#endif

template <int D, int PC>
int launch_bwd(const CUtensorMap* maps, void* dq, void* dk, void* dv, int BH, int T, float beta, float p,
               int d_real, cudaStream_t stream) {
  using L = BwdLayout<D>;
  const int nT = (T + BT - 1) / BT;
  const long long grid = static_cast<long long>(nT) * BH;
  if (2 * grid > 0x7fffffffLL) return ERR_SHAPE;
  // two streamed bf16 tensors of T x D per head; one resident CTA per SM
  const int G = tile::head_groups(BH, nT, 4LL * T * d_real, sm_count());
  constexpr bool ONE_GRID = BSA_BWD_ONE_GRID && BwdCfg<D, PC, false>::THREADS == BwdCfg<D, PC, true>::THREADS;
  if constexpr (ONE_GRID) {
    auto k = tra_bwd_both_kernel<D, PC>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC) != cudaSuccess)
      return ERR_LAUNCH;
    k<<<static_cast<unsigned>(2 * grid), BwdCfg<D, PC, false>::THREADS, L::ALLOC, stream>>>(
        maps[0], maps[1], maps[2], maps[3], static_cast<__nv_bfloat16*>(dq), static_cast<__nv_bfloat16*>(dk),
        static_cast<__nv_bfloat16*>(dv), BH, T, nT, G, beta, p, d_real);
    return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
  } else {
    auto k1 = tra_bwd_dkdv_kernel<D, PC>;
    auto k2 = tra_bwd_dq_kernel<D, PC>;
    if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC) != cudaSuccess ||
        cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC) != cudaSuccess)
      return ERR_LAUNCH;
    k1<<<static_cast<unsigned>(grid), BwdCfg<D, PC, false>::THREADS, L::ALLOC, stream>>>(
        maps[0], maps[1], maps[2], maps[3], static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), BH, T,
        nT, G, beta, p, d_real);
    if (cudaGetLastError() != cudaSuccess) return ERR_LAUNCH;
    k2<<<static_cast<unsigned>(grid), BwdCfg<D, PC, true>::THREADS, L::ALLOC, stream>>>(
        maps[0], maps[1], maps[2], maps[3], static_cast<__nv_bfloat16*>(dq), BH, T, nT, G, beta, p, d_real);
    return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
  }
}

}  // namespace

int launch_tra_bwd_bf16(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk, void* dv,
                        int B, int H, int T, int D, float beta, float p, cudaStream_t stream) {
  const int BH = B * H;
  CUtensorMap maps[4];
  const uint64_t rs = static_cast<uint64_t>(D) * 2, hs = rs * T;
  const void* src[4] = {q, k, v, dout};
  for (int i = 0; i < 4; ++i) {
    const int st = encode_tmap_3d(&maps[i], src[i], D, T, BH, rs, hs, 64, BT, 1);
    if (st != OK) return st;
  }
  const int pc = bwd::bwd_power_class(p);
  if (D > 64) {  // width 128 (head dims 80 .. 128 on zero-filled columns)
    if (pc == POW_TWO) return launch_bwd<128, POW_TWO>(maps, dq, dk, dv, BH, T, beta, p, D, stream);
    if (pc == POW_ONE) return launch_bwd<128, POW_ONE>(maps, dq, dk, dv, BH, T, beta, p, D, stream);
    if (pc == POW_GENERAL_MIX) return launch_bwd<128, POW_GENERAL_MIX>(maps, dq, dk, dv, BH, T, beta, p, D, stream);
    return launch_bwd<128, POW_GENERAL>(maps, dq, dk, dv, BH, T, beta, p, D, stream);
  }
  if (tra_head_dim_supported(D)) {  // width 64 (16 .. 48 on zero-filled columns)
    if (pc == POW_TWO) return launch_bwd<64, POW_TWO>(maps, dq, dk, dv, BH, T, beta, p, D, stream);
    if (pc == POW_ONE) return launch_bwd<64, POW_ONE>(maps, dq, dk, dv, BH, T, beta, p, D, stream);
    if (pc == POW_GENERAL_MIX) return launch_bwd<64, POW_GENERAL_MIX>(maps, dq, dk, dv, BH, T, beta, p, D, stream);
    return launch_bwd<64, POW_GENERAL>(maps, dq, dk, dv, BH, T, beta, p, D, stream);
  }
  return ERR_UNSUPPORTED;
}

unsigned int tra_bwd_device_error() { return read_and_clear_device_error(); }

}  // namespace bsa
