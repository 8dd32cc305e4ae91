// tra_bwd_fused.cu -- threshold rectified attention backward as one fused
// kernel: bf16 in, fp32 accumulate, tcgen05 tensor cores.
//
// Method: page "triton_threshold_attention.py", ThresholdRelaFunction.backward
// (W and dA as in tra_bwd_common.cuh):
//     dV_j = sum_i W_ij dO_i,   dK_j = sum_i dA_ij q_i,   dQ_i = sum_j dA_ij k_j.
// The page (and tra_bwd.cu) computes dK/dV and dQ in two kernels that both
// produce the scores and dP; here each (key tile n, query tile m) pair
// produces them once: 10 D tensor FLOPs per causal pair instead of 14 D.
//
// One CTA per 128-key tile n of one (b, h), looping over the query tiles
// m >= n (j = m - n).  Per step, all MMAs 128 x 128 (full tensor rate):
//   S^T  = K_n Q_m^T          -> TMEM S   (fp32; the epilogue packs W^T over it)
//   dP^T = V_n dO_m^T         -> TMEM P   (fp32)
//   dV  += W^T dO_m           (A from TMEM)
//   dQ_m = dA K_n             (A = the dA^T tile in shared memory read MN-major)
//   dK  += dA^T Q_m           (A = the same tile read K-major)
// and the dQ partial leaves TMEM through four drain warps that stage it in
// shared memory and add it into an fp32 accumulator with TMA reduce-adds (the
// L2 performs the additions).  A last small kernel converts the accumulator
// to bf16 (and a first one zeroes it).
//
// The epilogue (thread = key row, two warpgroups, one per 64-query half)
// works in two parts: from S^T alone it forms W^T (for dV) and keeps
// g = p ReLU(x)^(p-1) in registers; from dP^T it then forms dA^T = dP^T g.
// The issue order per step, dP^T(j) dV(j) S^T(j+1) dQ(j) dK(j), lets the
// tensor pipe run dP^T under the first part, dV and the next S^T under the
// second, and dQ / dK under the next step's first part; dQ goes before dK so
// that the drain of dQ's TMEM overlaps dK.
//
// TMEM (512 columns): S [0,128), P [128,256), dV [256,256+D), dK [256+D,
// 256+2D); dQ reuses P at D = 128 (the MMA issuer waits for the drain before
// the next dP^T) and has [384,448) of its own at D = 64.  A trace of one CTA
// (clock64 at every wait and arrive) showed the order S^T dP^T dV dK dQ --
// every product of a step behind the epilogue of the same step -- running at
// ~5000 cycles per step against 2560 of tensor work.
// Shared memory (D = 128): K_n, V_n resident; Q in two slots; dO in one slot
// (dO_m's last reader, dV, finishes ~1500 tensor cycles before the next dP^T
// needs dO_{m+1}); the dA^T operand; 32 KB of staging for the dQ boxes.  At
// D = 64, Q and dO have two slots each.  A trace there shows the MMA issuer
// waiting ~2000 cycles per step for dO, but three or four slots measured
// slower (B2 H32 T8192 p=2: 1.50 / 1.59 / 1.63 ms for 2 / 3 / 4): the wait is
// the L2 serving the loads beside the dQ reduce-adds, not prefetch depth.
//
// Warps: 0-7 epilogue, 8-11 dQ drain, 12 TMA producer, 13 MMA issuer.  Every
// mbarrier wait is bounded; the drain warps take each go/no-go decision
// together (bar.red) so a timeout never leaves one of them at a named barrier.
#include "kernels.h"
#include "ptx.cuh"
#include "tc_tile.cuh"
#include "tra_bwd_common.cuh"
#include "tra_math.cuh"

namespace bsa {
namespace {

using tile::PANEL_BYTES;
constexpr int BT = tile::ROWS;
constexpr uint32_t TMEM_COLS = 512;

constexpr int EPI_WARPS = 8;
constexpr int DRAIN_WARP = 8;  // four warps, one per TMEM lane quarter
constexpr int TMA_WARP = 12;
constexpr int MMA_WARP = 13;
constexpr int THREADS = 14 * 32;
constexpr int DRAIN_BAR = 1;  // named barrier of the drain warps

#ifndef BSA_FBWD_SLOTS_D64
#define BSA_FBWD_SLOTS_D64 2  // Q and dO slots at D = 64
#endif

template <int D>
struct FusedLayout {
  static constexpr int TILE = D / 64 * PANEL_BYTES;
  static constexpr int Q_SLOTS = D == 128 ? 2 : BSA_FBWD_SLOTS_D64;
  static constexpr int DO_SLOTS = D == 128 ? 1 : BSA_FBWD_SLOTS_D64;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TILE;
  static constexpr int Q_OFF = 2 * TILE;                    // Q_SLOTS slots
  static constexpr int DO_OFF = Q_OFF + Q_SLOTS * TILE;     // DO_SLOTS slots
  static constexpr int DA_OFF = DO_OFF + DO_SLOTS * TILE;   // dA^T: 128 keys x 128 queries bf16, two panels
  static constexpr int STG_OFF = DA_OFF + 2 * PANEL_BYTES;  // two fp32 boxes of 128 rows x 32 columns
  static constexpr int BOX_BYTES = BT * 32 * 4;
  static constexpr int TAU_OFF = STG_OFF + 2 * BOX_BYTES;   // float[2][128]
  static constexpr int BAR_OFF = TAU_OFF + 2 * BT * 4;
  // kv_full | q_full[QS] | q_empty[QS] | do_full[S] | do_empty[S] | s_full | p_full | w_ready | a_ready |
  // dq_full | dq_empty | da_free | tau_full[2] | acc_full | mma_done
  static constexpr int NBAR = 1 + 2 * Q_SLOTS + 2 * DO_SLOTS + 7 + 2 + 2;
  static constexpr int TPTR_OFF = BAR_OFF + NBAR * 8;
  static constexpr int ALLOC = TPTR_OFF + 16 + 1024;
  static_assert(ALLOC <= 232448, "shared memory");
  // TMEM columns
  static constexpr uint32_t TS = 0, TP = BT, TDV = 2 * BT, TDK = 2 * BT + D;
  static constexpr uint32_t TDQ = D == 128 ? TP : 2 * BT + 2 * D;
};

struct FusedBars {
  uint64_t *kv_full, *q_full, *q_empty, *do_full, *do_empty, *s_full, *p_full, *w_ready, *a_ready, *dq_full,
      *dq_empty, *da_free, *tau_full, *acc_full, *mma_done;
};

template <int D>
__device__ __forceinline__ FusedBars fused_bars(uint8_t* smem) {
  using L = FusedLayout<D>;
  uint64_t* b = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  FusedBars r;
  r.kv_full = b;
  r.q_full = b + 1;
  r.q_empty = r.q_full + L::Q_SLOTS;
  r.do_full = r.q_empty + L::Q_SLOTS;
  r.do_empty = r.do_full + L::DO_SLOTS;
  r.s_full = r.do_empty + L::DO_SLOTS;
  r.p_full = r.s_full + 1;
  r.w_ready = r.p_full + 1;
  r.a_ready = r.w_ready + 1;
  r.dq_full = r.a_ready + 1;
  r.dq_empty = r.dq_full + 1;
  r.da_free = r.dq_empty + 1;
  r.tau_full = r.da_free + 1;  // [2]
  r.acc_full = r.tau_full + 2;
  r.mma_done = r.acc_full + 1;
  return r;
}

// dQ_m[128 x D] = dA[128 x 128] K_n[128 x D]: A = the dA^T tile in shared
// memory read MN-major (queries along M, 64 per panel; keys along K), B = K_n
// read MN-major (D along N, keys along K).
template <int D>
__device__ __forceinline__ void mma_dq(uint32_t tC, uint32_t sDA, uint32_t sK, bool leader) {
  constexpr uint32_t IDESC = idesc_bf16_f32(BT, D, 1, 1);
  constexpr int NP = D / 64;
#pragma unroll
  for (int kk = 0; kk < BT / 16; ++kk) {
    const uint64_t a = smem_desc_sw128(sDA + kk * 16 * 128, PANEL_BYTES, 1024);
    const uint64_t b = smem_desc_sw128(sK + kk * 16 * 128, NP > 1 ? PANEL_BYTES : 1024, 1024);
    if (leader) mma_ss(tC, a, b, IDESC, kk > 0 ? 1u : 0u);
  }
}

// dK += dA^T[128 x 128] Q_m[128 x D]: A = the dA^T tile read K-major (keys
// along M, queries along K, 64 per panel), B = Q_m read MN-major.
template <int D>
__device__ __forceinline__ void mma_dk(uint32_t tC, uint32_t sDA, uint32_t sQ, bool first, bool leader) {
  constexpr uint32_t IDESC = idesc_bf16_f32(BT, D, 0, 1);
  constexpr int NP = D / 64;
#pragma unroll
  for (int kk = 0; kk < BT / 16; ++kk) {
    const uint64_t a = smem_desc_sw128(sDA + (kk >> 2) * PANEL_BYTES + (kk & 3) * 32, 16, 1024);
    const uint64_t b = smem_desc_sw128(sQ + kk * 16 * 128, NP > 1 ? PANEL_BYTES : 1024, 1024);
    if (leader) mma_ss(tC, a, b, IDESC, (!first || kk > 0) ? 1u : 0u);
  }
}

// 32 fp32 columns of this thread's row r -> row r of a 128-row x 32-column
// fp32 box in the 128-byte-swizzled layout a TMA copy of that box uses.
__device__ __forceinline__ void stage_box(uint8_t* box, int r, const uint32_t (&v)[32]) {
#pragma unroll
  for (int k = 0; k < 8; ++k)
    *reinterpret_cast<uint4*>(box + r * 128 + ((k ^ (r & 7)) << 4)) =
        make_uint4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
}

// tau(i) = beta sqrt(2 ln(i+1) / d) from the MUFU lg2 and sqrt approximations
// (k2 = 2 ln 2 / d): within ~1e-7 relative of the correctly rounded value, at
// a few instructions instead of the dozens of logf, a divide and sqrtf.
// BSA_FBWD_FAST_TAU = 0 uses tile::tau_of_row instead.
#ifndef BSA_FBWD_FAST_TAU
#define BSA_FBWD_FAST_TAU 1
#endif
__device__ __forceinline__ float tau_fast(int row, float beta, float k2, int d) {
#if BSA_FBWD_FAST_TAU
  (void)d;
  return beta * sqrt_approx(lg2_approx(static_cast<float>(row + 1)) * k2);
#else
  (void)k2;
  return tile::tau_of_row(row, beta, d);
#endif
}

// W and g = p ReLU(x)^(p-1) of two scores at once for p = 1 and p = 2 on
// packed f32x2 arithmetic (x = s - tau in one packed subtract; W = r r and
// g = r + r in one packed multiply and add for p = 2), bit-identical to
// bwd::weight_and_grad; other powers take the scalar form.
template <int PC>
__device__ __forceinline__ void weight_and_grad2(float s0, float s1, float t0, float t1, float p, float lp,
                                                 float& w0, float& w1, uint64_t& g) {
  if constexpr (PC == POW_GENERAL_MIX) {
    // p > 1: the exponents p l and (p - 1) l + log2 p of one score in one
    // packed multiply-add, the same roundings as the scalar form
    float x0, x1;
    f2_unpack(f2_sub(f2_pack(s0, s1), f2_pack(t0, t1)), x0, x1);
    const float l0 = bwd::lg2a(fmaxf(x0, 0.0f)), l1 = bwd::lg2a(fmaxf(x1, 0.0f));
    const uint64_t pq = f2_pack(p, p - 1.0f), z = f2_pack(0.0f, lp);
    float a0, b0, a1, b1;
    f2_unpack(f2_fma(f2_pack(l0, l0), pq, z), a0, b0);
    f2_unpack(f2_fma(f2_pack(l1, l1), pq, z), a1, b1);
    w0 = bwd::ex2a(a0);
    w1 = bwd::ex2a(a1);
    g = f2_pack(bwd::ex2a(b0), bwd::ex2a(b1));
  } else if constexpr (PC == POW_TWO || PC == POW_ONE) {
    float x0, x1;
    f2_unpack(f2_sub(f2_pack(s0, s1), f2_pack(t0, t1)), x0, x1);
    const float r0 = fmaxf(x0, 0.0f), r1 = fmaxf(x1, 0.0f);
    const uint64_t r = f2_pack(r0, r1);
    if constexpr (PC == POW_TWO) {
      f2_unpack(f2_mul(r, r), w0, w1);
      g = f2_add(r, r);
    } else {
      w0 = r0;
      w1 = r1;
      g = f2_pack(x0 > 0.0f ? 1.0f : 0.0f, x1 > 0.0f ? 1.0f : 0.0f);
    }
  } else {
    float g0, g1;
    bwd::weight_and_grad<PC>(s0 - t0, p, lp, w0, g0);
    bwd::weight_and_grad<PC>(s1 - t1, p, lp, w1, g1);
    g = f2_pack(g0, g1);
  }
}

// Who fills the epilogue's tau table: the drain warps at D = 64, two steps
// ahead; at D = 128 (where the drain warps sit on the path to the next dP^T
// and the change measured 1-3% slower) the epilogue warps, per step.
#ifndef BSA_FBWD_DRAIN_TAU
#define BSA_FBWD_DRAIN_TAU 1  // 1: D = 64 only; 2: every D
#endif
template <int D>
constexpr bool drain_fills_tau() {
  return BSA_FBWD_DRAIN_TAU == 2 || (BSA_FBWD_DRAIN_TAU == 1 && D == 64);
}

// MMA issue: a converged warp with an elected issuing lane (at D = 128 the
// elected lane alone was 0.5-1% slower).
#ifndef BSA_FBWD_CONVERGED_ISSUE
#define BSA_FBWD_CONVERGED_ISSUE 2  // 1: D = 64 only; 2: every D (D = 128 measured 0.5-1% faster)
#endif
template <int D>
constexpr bool fused_converged_issue() {
  return BSA_FBWD_CONVERGED_ISSUE == 2 || (BSA_FBWD_CONVERGED_ISSUE == 1 && D == 64);
}

template <int D, int PC>
__global__ void __launch_bounds__(THREADS, 1)
    tra_bwd_fused_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                         const __grid_constant__ CUtensorMap tmDQ, __nv_bfloat16* __restrict__ dk,
                         __nv_bfloat16* __restrict__ dv, int BH, int T, int nT, int G, float beta, float p,
                         int d_real) {
  using L = FusedLayout<D>;
  // Head dims below the tile width run on zero-filled columns (the tensor
  // maps cover the real d_real columns).
  const int dr = d_real;
  const float k2 = 2.0f * 0.6931471805599453f / static_cast<float>(dr);  // 2 ln 2 / d
  const float lp = log2f(p);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const FusedBars B = fused_bars<D>(smem);
  uint32_t* tptr = reinterpret_cast<uint32_t*>(smem + L::TPTR_OFF);
  float* tau_s = reinterpret_cast<float*>(smem + L::TAU_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const tile::HeadItem item = tile::head_group_item(static_cast<int>(blockIdx.x), BH, nT, G);
  const int n = item.rank;  // key tile; n = 0 has the most query tiles
  const int bh = item.bh;
  const int nq = nT - n;  // query tiles m = n .. nT-1

  if (threadIdx.x == 0) {
    mbar_init(B.kv_full, 1);
    for (int s = 0; s < L::Q_SLOTS; ++s) {
      mbar_init(&B.q_full[s], 1);
      mbar_init(&B.q_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) mbar_init(&B.tau_full[s], drain_fills_tau<D>() ? 4 : EPI_WARPS);
    for (int s = 0; s < L::DO_SLOTS; ++s) {
      mbar_init(&B.do_full[s], 1);
      mbar_init(&B.do_empty[s], 1);
    }
    mbar_init(B.s_full, 1);
    mbar_init(B.p_full, 1);
    mbar_init(B.w_ready, EPI_WARPS);
    mbar_init(B.a_ready, EPI_WARPS);
    mbar_init(B.dq_full, 1);
    mbar_init(B.dq_empty, 4);
    mbar_init(B.da_free, 1);
    mbar_init(B.acc_full, 1);
    mbar_init(B.mma_done, 1);
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
    if (lane == 0) {
      debug_check(bh >= 0 && bh < BH && n * BT < T && (n + nq - 1) * BT < T);
      bwd::produce<D, L::Q_SLOTS, L::DO_SLOTS>(smem + L::K_OFF, smem + L::V_OFF, B.kv_full, smem + L::Q_OFF, B.q_full,
                                      B.q_empty, smem + L::DO_OFF, B.do_full, B.do_empty, &tmK, &tmV, n * BT, &tmQ,
                                      &tmDO, n, nq, bh);
    }
  } else if (warp == MMA_WARP) {
    const bool leader = elect_one();
    if (fused_converged_issue<D>() || leader) {
      auto commit = [&](uint64_t* bar) {
        if (leader) mma_commit(bar);
      };
      const uint32_t sK = smem_u32(smem + L::K_OFF), sV = smem_u32(smem + L::V_OFF);
      const uint32_t sDA = smem_u32(smem + L::DA_OFF);
      auto q_slot = [&](int j) { return smem_u32(smem + L::Q_OFF + (j % L::Q_SLOTS) * L::TILE); };
      // S^T = K_n Q_m^T of step j (into S, whose W^T of step j-1 dV has read, in issue order)
      auto scores = [&](int j) -> bool {
        if (!mbar_wait(&B.q_full[j % L::Q_SLOTS], (j / L::Q_SLOTS) & 1)) return false;
        tc_fence_after();
        tile::mma_abt<D>(tmem + L::TS, sK, q_slot(j), leader);
        commit(B.s_full);
        return true;
      };
      bool ok = mbar_wait(B.kv_full, 0) && scores(0);
      for (int j = 0; j < nq && ok; ++j) {
        const int ds = j % L::DO_SLOTS;
        const uint32_t sQ = q_slot(j);
        const uint32_t sDO = smem_u32(smem + L::DO_OFF + ds * L::TILE);
        // dP^T = V_n dO_m^T: P is free once step j-1's second part has read it
        // (waited below, before its dQ) and, at D = 128, its dQ was drained.
        if (!(ok = mbar_wait(&B.do_full[ds], (j / L::DO_SLOTS) & 1))) break;
        if (D == 128 && j > 0 && !(ok = mbar_wait(B.dq_empty, (j - 1) & 1))) break;
        tc_fence_after();
        tile::mma_abt<D>(tmem + L::TP, sV, sDO, leader);
        commit(B.p_full);
        // dV += W^T dO_m; W^T of query half h packed into S columns [64h, 64h+32)
        if (!(ok = mbar_wait(B.w_ready, j & 1))) break;
        tc_fence_after();
        tile::mma_tmem_a<D>(tmem + L::TDV, tmem + L::TS, sDO, 0, 4, j == 0, leader);
        tile::mma_tmem_a<D>(tmem + L::TDV, tmem + L::TS + 32, sDO, 4, 8, false, leader);
        commit(&B.do_empty[ds]);
        if (j + 1 < nq && !(ok = scores(j + 1))) break;
        // dQ_m = dA K_n, then dK += dA^T Q_m, both from the dA^T tile
        if (!(ok = mbar_wait(B.a_ready, j & 1))) break;
        if (D == 64 && j > 0 && !(ok = mbar_wait(B.dq_empty, (j - 1) & 1))) break;
        tc_fence_after();
        mma_dq<D>(tmem + L::TDQ, sDA, sK, leader);
        commit(B.dq_full);
        mma_dk<D>(tmem + L::TDK, sDA, sQ, j == 0, leader);
        commit(&B.q_empty[j % L::Q_SLOTS]);
        commit(B.da_free);
      }
      if (ok) commit(B.acc_full);
      commit(B.mma_done);
      mbar_wait(B.mma_done, 0);
    }
  } else if (warp >= DRAIN_WARP) {
    // dQ drain: thread = query row of the tile; the partial leaves TMEM as
    // soon as it is loaded, then goes out box by box through the staging.
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    uint8_t* stg = smem + L::STG_OFF;
    const uint32_t sStg = smem_u32(stg);
    const bool issuer = warp == DRAIN_WARP && lane == 0;
    // At D = 64 the drain warps also fill the epilogue's double-buffered tau table
    // (tau(i) of the step's 128 query columns): steps 0 and 1 up front, step
    // j + 2 once dQ of step j is done (the epilogue finished reading buffer
    // j & 1 before it produced the dA of step j) and its TMEM released.  This
    // keeps the tau evaluation (log, divide, square root) and a barrier of
    // all eight epilogue warps off the epilogue's path (B2 H32 T8192 D64:
    // p=2 1.50 -> 1.45 ms, p=1.5 2.17 -> 2.07 ms).
    auto fill_tau = [&](int jj) {
      if constexpr (drain_fills_tau<D>()) {
        tau_s[(jj & 1) * BT + r] = tau_fast((n + jj) * BT + r, beta, k2, dr);
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.tau_full[jj & 1]);
      }
    };
    fill_tau(0);
    if (nq > 1) fill_tau(1);
    bool ok = true;
    for (int j = 0; j < nq; ++j) {
      const int m = n + j;
      ok = bar_and(DRAIN_BAR, 128, mbar_wait(B.dq_full, j & 1));
      if (!ok) break;
      tc_fence_after();
      uint32_t v0[32], v1[32];
      tmem_ld32(lane_base + L::TDQ, v0);
      tmem_ld32(lane_base + L::TDQ + 32, v1);
      tmem_wait_ld();
      if constexpr (D == 64) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(B.dq_empty);
      }
      stage_box(stg, r, v0);
      stage_box(stg + L::BOX_BYTES, r, v1);
      if constexpr (D == 128) {
        tmem_ld32(lane_base + L::TDQ + 64, v0);
        tmem_ld32(lane_base + L::TDQ + 96, v1);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(B.dq_empty);
      }
      // (after dQ's TMEM is released: at D = 128 the next dP^T waits for it)
      if (j + 2 < nq) fill_tau(j + 2);
      fence_proxy_async_smem();
      bar_sync(DRAIN_BAR, 128);
      if (issuer) {
        tma_reduce_add_3d(&tmDQ, sStg, 0, m * BT, bh);
        if (dr > 32) tma_reduce_add_3d(&tmDQ, sStg + L::BOX_BYTES, 32, m * BT, bh);
        bulk_commit();
        bulk_wait_read<0>();
      }
      bar_sync(DRAIN_BAR, 128);
      if constexpr (D == 128) {
        stage_box(stg, r, v0);
        stage_box(stg + L::BOX_BYTES, r, v1);
        fence_proxy_async_smem();
        bar_sync(DRAIN_BAR, 128);
        if (issuer) {
          tma_reduce_add_3d(&tmDQ, sStg, 64, m * BT, bh);  // dr > 64 at width 128
          if (dr > 96) tma_reduce_add_3d(&tmDQ, sStg + L::BOX_BYTES, 96, m * BT, bh);
          bulk_commit();
          bulk_wait_read<0>();
        }
        bar_sync(DRAIN_BAR, 128);
      }
    }
    if (issuer) bulk_wait_all();
  } else {
    // Epilogue: thread = key row r of TMEM lane quarter wq; warpgroup h takes
    // the query columns [64h, 64h+64) of every score tile.
    const int wq = warp & 3, h = warp >> 2;
    const int r = wq * 32 + lane;
    const int key = n * BT + r;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    uint8_t* da_panel = smem + L::DA_OFF + h * PANEL_BYTES;
    bool ok = true;
    for (int j = 0; j < nq && ok; ++j) {
      const int m = n + j;
      // Double-buffered tau table (a warp writes buffer j & 1 for step j only
      // after every warp arrived for step j - 1, i.e. finished step j - 2).
      float* tau_m = tau_s + (j & 1) * BT;
      if constexpr (!drain_fills_tau<D>()) {
        tau_m[r] = tau_fast(m * BT + r, beta, k2, dr);
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.tau_full[j & 1]);
      }
      if (!(ok = mbar_wait(&B.tau_full[j & 1], (j >> 1) & 1))) break;
      const bool diag = (m == n);
      // Part 1: W^T and g from S^T.
      if (!(ok = mbar_wait(B.s_full, j & 1))) break;
      tc_fence_after();
      uint64_t g[32];  // g of this warp's 64 query columns, two per register pair
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int q0 = 64 * h + 32 * c;
        uint32_t sv[32];
        tmem_ld32(lane_base + L::TS + q0, sv);
        tmem_wait_ld();
        uint32_t wpk[16];
        float4 t4;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int i0 = q0 + 2 * e;  // query column within the tile
          if ((e & 1) == 0) t4 = *reinterpret_cast<const float4*>(tau_m + i0);  // tau of columns i0 .. i0+3
          const float ta = (e & 1) ? t4.z : t4.x, tb = (e & 1) ? t4.w : t4.y;
          float w0, w1;
          uint64_t g2;
          weight_and_grad2<PC>(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1]), ta, tb, p, lp, w0, w1,
                               g2);
          if (diag) {  // causal: key r <= query column
            float g0, g1;
            f2_unpack(g2, g0, g1);
            if (i0 < r) w0 = g0 = 0.0f;
            if (i0 + 1 < r) w1 = g1 = 0.0f;
            g2 = f2_pack(g0, g1);
          }
          wpk[e] = pack_bf16x2(w0, w1);
          g[16 * c + e] = g2;
        }
        // packs into the half's own first 32 columns (already-consumed scores)
        tmem_st16(lane_base + L::TS + 64 * h + 16 * c, wpk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B.w_ready);
      // Part 2: dA^T = dP^T g into the shared-memory tile (for dQ and dK),
      // once step j-1's dQ and dK have read the previous one.
      if (!(ok = mbar_wait(B.p_full, j & 1))) break;
      if (j > 0 && !(ok = mbar_wait(B.da_free, (j - 1) & 1))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int q0 = 64 * h + 32 * c;
        uint32_t dp[32];
        tmem_ld32(lane_base + L::TP + q0, dp);
        tmem_wait_ld();
        uint32_t apk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float a0, a1;
          f2_unpack(f2_mul(f2_pack(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])), g[16 * c + e]), a0, a1);
          apk[e] = pack_bf16x2(a0, a1);
        }
        // row r, query columns q0 .. q0+31 = 16-byte chunks 4c .. 4c+3 of panel h
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int k = 4 * c + i;
          *reinterpret_cast<uint4*>(da_panel + r * 128 + ((k ^ (r & 7)) << 4)) =
              make_uint4(apk[4 * i], apk[4 * i + 1], apk[4 * i + 2], apk[4 * i + 3]);
        }
      }
      fence_proxy_async_smem();  // the dA^T stores are read by the tensor core
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B.a_ready);
    }
    if (ok && mbar_wait(B.acc_full, 0)) {
      tc_fence_after();
      const size_t rowoff = (static_cast<size_t>(bh) * T + key) * dr;
      constexpr int CPW = D / 32 / 2;  // 32-column chunks of dK, dV this warp stores
#pragma unroll
      for (int c = h * CPW; c < (h + 1) * CPW; ++c) {
        if (dr == D) {
          tile::store_row_chunk(lane_base + L::TDV, c, dv + rowoff, key < T);
          tile::store_row_chunk(lane_base + L::TDK, c, dk + rowoff, key < T);
        } else if (c * 32 < dr) {  // head dim below the tile width: only its columns
          tile::store_row_part(lane_base + L::TDV, c, dv + rowoff, key < T, min(32, dr - c * 32));
          tile::store_row_part(lane_base + L::TDK, c, dk + rowoff, key < T, min(32, dr - c * 32));
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

// dq_acc = 0, sixteen bytes per thread and step.
__global__ void __launch_bounds__(256) tra_bwd_dq_zero_kernel(uint4* __restrict__ acc, size_t n16) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride)
    acc[i] = make_uint4(0u, 0u, 0u, 0u);
}

// dq (bf16) = dq_acc (fp32), eight elements per thread and step.
__global__ void __launch_bounds__(256) tra_bwd_dq_convert_kernel(const float* __restrict__ acc,
                                                                 __nv_bfloat16* __restrict__ dq, size_t n8) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    reinterpret_cast<uint4*>(dq)[i] =
        make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
  }
}

template <int D, int PC>
int launch_fused(const CUtensorMap* maps, const CUtensorMap& mdq, void* dk, void* dv, int BH, int T, float beta,
                 float p, int d_real, cudaStream_t stream) {
  using L = FusedLayout<D>;
  const int nT = (T + BT - 1) / BT;
  const long long grid = static_cast<long long>(nT) * BH;
  if (grid > 0x7fffffffLL) return ERR_SHAPE;
  // streamed per head: q and dO (bf16) and the dq accumulator (fp32)
  const int G = tile::head_groups(BH, nT, 8LL * T * d_real, sm_count());
  auto k = tra_bwd_fused_kernel<D, PC>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC) != cudaSuccess)
    return ERR_LAUNCH;
  k<<<static_cast<unsigned>(grid), THREADS, L::ALLOC, stream>>>(maps[0], maps[1], maps[2], maps[3], mdq,
                                                                static_cast<__nv_bfloat16*>(dk),
                                                                static_cast<__nv_bfloat16*>(dv), BH, T, nT, G, beta, p,
                                                                d_real);
  return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
}

template <int D>
int launch_fused_pc(const CUtensorMap* maps, const CUtensorMap& mdq, void* dk, void* dv, int BH, int T, float beta,
                    float p, int d_real, cudaStream_t stream) {
  const int pc = bwd::bwd_power_class(p);
  if (pc == POW_TWO) return launch_fused<D, POW_TWO>(maps, mdq, dk, dv, BH, T, beta, p, d_real, stream);
  if (pc == POW_ONE) return launch_fused<D, POW_ONE>(maps, mdq, dk, dv, BH, T, beta, p, d_real, stream);
  if (pc == POW_GENERAL_MIX)
    return launch_fused<D, POW_GENERAL_MIX>(maps, mdq, dk, dv, BH, T, beta, p, d_real, stream);
  return launch_fused<D, POW_GENERAL>(maps, mdq, dk, dv, BH, T, beta, p, d_real, stream);
}

}  // namespace

int launch_tra_bwd_fused_bf16(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk,
                              void* dv, int B, int H, int T, int D, float beta, float p, float* dq_acc,
                              cudaStream_t stream) {
  if (!tra_head_dim_supported(D)) return ERR_UNSUPPORTED;
  const int BH = B * H;
  CUtensorMap maps[4], mdq;
  const uint64_t rs = static_cast<uint64_t>(D) * 2, hs = rs * T;
  const void* src[4] = {q, k, v, dout};
  for (int i = 0; i < 4; ++i) {
    const int st = encode_tmap_3d(&maps[i], src[i], D, T, BH, rs, hs, 64, BT, 1);
    if (st != OK) return st;
  }
  const int st = encode_tmap_3d_f32(&mdq, dq_acc, D, T, BH, static_cast<uint64_t>(D) * 4,
                                    static_cast<uint64_t>(D) * 4 * T, 32, BT, 1);
  if (st != OK) return st;
  const size_t elems = static_cast<size_t>(BH) * T * D;  // a multiple of 16 (D is)
  const size_t n8 = elems / 8;
  const int sms = sm_count();
  size_t blocks = (n8 + 255) / 256;
  const size_t cap = static_cast<size_t>(sms > 0 ? sms : 148) * 8;
  if (blocks > cap) blocks = cap;
  tra_bwd_dq_zero_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(reinterpret_cast<uint4*>(dq_acc),
                                                                             elems / 4);
  if (cudaGetLastError() != cudaSuccess) return ERR_LAUNCH;
  const int rc = D > 64 ? launch_fused_pc<128>(maps, mdq, dk, dv, BH, T, beta, p, D, stream)
                          : launch_fused_pc<64>(maps, mdq, dk, dv, BH, T, beta, p, D, stream);
  if (rc != OK) return rc;
  if (dq == nullptr) return OK;  // the caller reads dQ from dq_acc (fp32)
  tra_bwd_dq_convert_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      dq_acc, static_cast<__nv_bfloat16*>(dq), n8);
  return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
}

}  // namespace bsa
