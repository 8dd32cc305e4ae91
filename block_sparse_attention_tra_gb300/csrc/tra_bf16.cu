// tra_bf16.cu -- threshold rectified attention forward, bf16 in / fp32
// accumulate, on the sm_100-family tensor cores (tcgen05 + TMEM + TMA).
//
// Method: page "triton_threshold_attention.py" (module docstring formula and
// _threshold_rela_fwd_kernel):
//     out_i = sum_{j <= i} ReLU(q_i . k_j - tau(i))^p v_j,
//     tau(i) = beta * sqrt(2 ln(i+1) / D),
// causal and unnormalised, no 1/sqrt(D) factor.  The page's kernel walks every
// key tile for every query tile; these visit only key tiles at or below the
// diagonal and mask the diagonal tile per element.
//
// Q/K/V tiles (128 rows x D, 128-byte swizzled 64-column panels) arrive by
// TMA; S = Q K^T (M=128, N=128, K=D; both operands K-major in smem) and
// O += P V (M=128, N=D, K=128; P read straight from TMEM, V an MN-major smem
// operand) run on tcgen05 with fp32 TMEM accumulators, each tile's MMAs
// issued by a single thread; an epilogue thread owns one query row
// (one TMEM lane): it loads its scores, subtracts tau(i) in fp32, applies
// ReLU^p, masks the diagonal tile, rounds to bf16 and writes P over the
// consumed score columns in two halves, so the P V MMA can start on the
// first 64 keys while the second half is still being computed.
//
// One organisation for every power class, the persistent "pair" kernel: a
// work item is 256 query rows of one (b, h) as two 128-row tiles Q0, Q1
// sharing every K/V tile (half the K/V smem traffic per FLOP); one CTA per SM
// walks a list of items.  For each tile t the tensor pipe runs
//     ... PV_t(n), QK_t(n+1), PV_t(n+1) ...
// and epilogue warpgroup t (warps 4t..4t+3) turns S_t into P_t.  For p = 1
// and p = 2 each tile has its own MMA-issuing thread; for the other powers
// one thread issues both tiles' MMAs in turn (PairCfg).  TMEM: S0, S1, O0,
// O1.  The power class
// (p = 1, p = 2, general p through exp2(p log2 x), or on request a half
// power as x^k sqrt(x)) only changes the epilogue arithmetic.
#include "kernels.h"
#include "ptx.cuh"
#include "tc_tile.cuh"
#include "tra_math.cuh"

namespace bsa {
namespace {

using tile::PANEL_BYTES;                // 128 rows x 128 B (64 bf16) swizzle panel
constexpr int BM = tile::ROWS;          // query rows per tile
constexpr int BN = tile::ROWS;          // keys per tile
constexpr uint32_t TMEM_COLS = 512;

// The weights of pair e (0 .. 15) of a quarter, two raw fp32 scores: the
// units each pair's log2 and exp2 run on are fixed at compile time by the
// plan (the loops that call this are unrolled).
template <int PC, int PLAN>
__device__ __forceinline__ uint32_t mix_weights2(int e, uint32_t s0, uint32_t s1, const PowParams& wp) {
  if (PC == POW_GENERAL_MIX && mix_pair_on_fma<PLAN>(e))
    return weights2<PC, true>(__uint_as_float(s0), __uint_as_float(s1), wp);
  if (PC == POW_GENERAL_MIX && mix_exp_on_fma<PLAN>(e))
    return weights2<PC, false, true>(__uint_as_float(s0), __uint_as_float(s1), wp);
  return weights2<PC, false>(__uint_as_float(s0), __uint_as_float(s1), wp);
}

// 32 scores (tile columns c0 .. c0+31) -> 16 packed weights, stored to TMEM
// columns c0/2 .. c0/2+15 of the same buffer (already-consumed scores).
// DIAG: the tile holds the diagonal, mask keys after the row (a compile-time
// flag, so that the other tiles carry no masking instructions at all).
template <int PC, bool DIAG, int MUFU_PAIRS>
__device__ __forceinline__ void epilogue_quarter(const uint32_t (&s)[32], uint32_t tS, int c0, const PowParams& wp,
                                                 int key0, int row) {
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    // (unrolled: the choice of log2 unit per pair is made at compile time)
    uint32_t w = mix_weights2<PC, MUFU_PAIRS>(e, s[2 * e], s[2 * e + 1], wp);
    if constexpr (DIAG) {
      const int key = key0 + c0 + 2 * e;  // keys key, key + 1
      if (key > row) w = 0u;
      else if (key + 1 > row) w &= 0x0000ffffu;
    }
    pk[e] = w;
  }
  tmem_st16(tS + c0 / 2, pk);
}

// Half of a quarter: 16 scores of this thread's row, keys key0 + c0 ..
// key0 + c0 + 15 (c0 a multiple of 16), into 8 packed P columns at tS +
// c0 / 2.  Pair e of the half is pair e0 + e of its quarter (for the choice
// of log2 unit).
template <int PC, bool DIAG, int MUFU_PAIRS>
__device__ __forceinline__ void epilogue_eighth(const uint32_t (&s)[16], uint32_t tS, int c0, int e0,
                                                const PowParams& wp, int key0, int row) {
  uint32_t pk[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    uint32_t w = mix_weights2<PC, MUFU_PAIRS>(e0 + e, s[2 * e], s[2 * e + 1], wp);
    if constexpr (DIAG) {
      const int key = key0 + c0 + 2 * e;
      if (key > row) w = 0u;
      else if (key + 1 > row) w &= 0x0000ffffu;
    }
    pk[e] = w;
  }
  tmem_st8(tS + c0 / 2, pk);
}

// One 128-key score tile of this thread's row -> P, in four software-
// pipelined quarters; arrives on p_half after keys 0..63 and on p_full after
// all 128 (one arrival per warp).
template <int PC, bool SPLIT, bool DIAG, int MP>
__device__ __forceinline__ void epilogue_tile(uint32_t tS, const PowParams& wp, int key0, int row, int lane,
                                              uint64_t* p_half, uint64_t* p_full) {
  uint32_t a[32], b[32];
  tmem_ld32(tS, a);
  tmem_wait_ld();
  tmem_ld32(tS + 32, b);
  epilogue_quarter<PC, DIAG, MP>(a, tS, 0, wp, key0, row);
  tmem_wait_ld();
  tmem_ld32(tS + 64, a);
  epilogue_quarter<PC, DIAG, MP>(b, tS, 32, wp, key0, row);
  if constexpr (SPLIT) {
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(p_half);
  }
  tmem_wait_ld();
  tmem_ld32(tS + 96, b);
  epilogue_quarter<PC, DIAG, MP>(a, tS, 64, wp, key0, row);
  tmem_wait_ld();
  epilogue_quarter<PC, DIAG, MP>(b, tS, 96, wp, key0, row);
  tmem_wait_st();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(p_full);
}

// Two of a tile's four score quarters (q = half and half + 2) for one of the
// two warps that share a TMEM lane quarter.  P of quarter q lands in TMEM
// columns 16q .. 16q+15, inside quarter q / 2's scores, which may belong to
// the other warp: both warps load their first quarter before either stores
// (named barrier `bar_id`, 64 threads).  Quarters 0 and 1 make up P's first
// half (p_half: one arrival per warp), all four the whole of it (p_full).
//
//
// Half loads: each quarter is loaded in two 16-column halves, and the next
// half's load is issued before the current half is turned into P, so its
// latency overlaps that work (same 32 registers of scores).  Measured at
// T=8192 D=64 p=1.5: 0.739 -> 0.715 ms; at D=128 p=1.5 1% slower, so
// BSA_PAIR_HALF_LOADS = 1 (default) uses them at D = 64 only (0: never,
// 2: always).
#ifndef BSA_PAIR_HALF_LOADS
#define BSA_PAIR_HALF_LOADS 1
#endif
template <int D>
constexpr bool pair_half_loads() {
  return BSA_PAIR_HALF_LOADS == 2 || (BSA_PAIR_HALF_LOADS == 1 && D == 64);
}
template <int PC, bool DIAG, int MP, bool HALF_LOADS>
__device__ __forceinline__ void epilogue_two_quarters(uint32_t tS, const PowParams& wp, int key0, int row, int lane,
                                                      int half, int bar_id, uint64_t* p_half, uint64_t* p_full) {
  if constexpr (HALF_LOADS) {
    const int c1 = 32 * half, c2 = 32 * (half + 2);  // this warp's quarters
    uint32_t a[16], b[16];
    tmem_ld16(tS + c1, a);
    tmem_ld16(tS + c1 + 16, b);
    tmem_wait_ld();
    asm volatile("bar.sync %0, 64;" ::"r"(bar_id) : "memory");
    epilogue_eighth<PC, DIAG, MP>(a, tS, c1, 0, wp, key0, row);
    tmem_ld16(tS + c2, a);  // P above went to columns c1 / 2 .., never c2 ..
    epilogue_eighth<PC, DIAG, MP>(b, tS, c1 + 16, 8, wp, key0, row);
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(p_half);
    tmem_wait_ld();
    tmem_ld16(tS + c2 + 16, b);
    epilogue_eighth<PC, DIAG, MP>(a, tS, c2, 0, wp, key0, row);
    tmem_wait_ld();
    epilogue_eighth<PC, DIAG, MP>(b, tS, c2 + 16, 8, wp, key0, row);
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(p_full);
  } else {
    uint32_t a[32];
    tmem_ld32(tS + 32 * half, a);
    tmem_wait_ld();
    asm volatile("bar.sync %0, 64;" ::"r"(bar_id) : "memory");
    epilogue_quarter<PC, DIAG, MP>(a, tS, 32 * half, wp, key0, row);
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(p_half);
    tmem_ld32(tS + 32 * (half + 2), a);
    tmem_wait_ld();
    epilogue_quarter<PC, DIAG, MP>(a, tS, 32 * (half + 2), wp, key0, row);
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(p_full);
  }
}

// ============================================================ pair kernel (p = 1, 2)
//
// Persistent: grid = min(items, SMs).  An item is one (pair index t, bh): the
// query tiles 2t and 2t+1 of head bh.  Items are numbered longest first and
// CTA c of G takes, in round r, item r*G + c (r even) or r*G + G-1-c (r odd);
// this snake order spreads the causal load within ~1% of even for the
// benchmark shapes.  Every role walks the same item sequence, so no queue is
// needed; barrier phases are running counts across items, and the next
// item's Q, K and V loads and QK products overlap the current item's tail.

template <int D>
struct PairLayout {
  static constexpr int NP = D / 64;
  static constexpr int TILE = NP * PANEL_BYTES;
  static constexpr int NS = (D == 128) ? 2 : 4;
  static constexpr int Q_OFF = 0;  // Q0, Q1
  static constexpr int K_OFF = Q_OFF + 2 * TILE;
  static constexpr int V_OFF = K_OFF + NS * TILE;
  static constexpr int BAR_OFF = V_OFF + NS * TILE;
  // q_full[2] | q_empty[2] | k_full[NS] | k_empty[NS] | v_full[NS] | v_empty[NS] | s_full[2] | p_half[2] |
  // p_full[2] | o_full[2] | o_empty[2] | mma_done[2]
  static constexpr int NBAR = 4 + 4 * NS + 10 + 2;
  static constexpr int TPTR_OFF = BAR_OFF + NBAR * 8;
  static constexpr int ALLOC = TPTR_OFF + 16 + 1024;
};
// MMA issuers: a single thread sustains only about one tcgen05.mma per ~70
// cycles whatever N is (measured), which cannot keep the tensor pipe fed
// when the epilogue is light (p = 1, 2): there each query tile gets its own
// issuing warp.  With a heavy epilogue (general and half powers) one issuer
// serving both tiles in turn is faster: it keeps the two epilogue
// warpgroups half a step apart, so one of them is always computing.
#ifndef BSA_PAIR_GENERAL_ISSUERS
#define BSA_PAIR_GENERAL_ISSUERS 1
#endif
// Epilogue warpgroups per query tile for the general powers (1 or 2).  With
// two, warps w and w + 8 share a TMEM lane quarter of one tile and take its
// score quarters {0, 2} and {1, 3}: four epilogue warps per SMSP instead of
// two hide more of the MUFU and TMEM-load latency (B2 H32 T8192 D64 p=1.5
// 0.803 -> 0.783 ms, and 0.733 ms with more of log2 on the FMA pipe; B4 H16
// T4096 D128 p=1.5 0.239 -> 0.229 ms), at 80-96 registers per thread.
#ifndef BSA_PAIR_GENERAL_EPI_WG
#define BSA_PAIR_GENERAL_EPI_WG 2
#endif
template <int PC>
struct PairCfg {
  static constexpr bool GENERAL = !(PC == POW_ONE || PC == POW_TWO);
  static constexpr int ISSUERS = GENERAL ? BSA_PAIR_GENERAL_ISSUERS : 2;
  static constexpr int EPI_WG = GENERAL ? BSA_PAIR_GENERAL_EPI_WG : 1;
  static constexpr int TMA_WARP = 8 * EPI_WG;
  static constexpr int MMA_WARP = TMA_WARP + 1;  // first MMA warp (allocates TMEM)
  static constexpr int THREADS = 256 * EPI_WG + 32 + 32 * ISSUERS;  // epilogue warpgroups, TMA warp, MMA warp(s)
};
#ifndef BSA_PAIR_SPLIT_P
#define BSA_PAIR_SPLIT_P 1
#endif
constexpr bool PAIR_SPLIT_P = BSA_PAIR_SPLIT_P;  // hand P over in two halves
// MMA issue: with a converged warp walking the issue loop (one elected lane
// issuing), tcgen05.mma issues every ~32 cycles against ~48 for a lone
// thread that builds its own descriptors (measured); that matters where the
// MMAs are short (the N = 64 P V products of D = 64) and measured slower at
// D = 128, where every MMA already runs 64 cycles.  0: never, 1: D = 64
// only, 2: always.
#ifndef BSA_PAIR_CONVERGED_ISSUE
#define BSA_PAIR_CONVERGED_ISSUE 1
#endif
template <int D>
constexpr bool pair_converged_issue() {
  return BSA_PAIR_CONVERGED_ISSUE == 2 || (BSA_PAIR_CONVERGED_ISSUE == 1 && D == 64);
}

// Item of round r for this CTA (false once the CTA has no more items).
struct PairItem {
  int t, bh, nmax0, nmax1, nlast;
  bool has1;
};
__device__ __forceinline__ bool pair_item(int r, int nItems, int BH, int nPair, int nQ, PairItem& it) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const long long k = static_cast<long long>(r) * G + ((r & 1) ? G - 1 - c : c);
  if (k >= nItems) return false;
  it.t = nPair - 1 - static_cast<int>(k / BH);
  it.bh = static_cast<int>(k % BH);
  it.has1 = (2 * it.t + 1) < nQ;  // second query tile exists
  it.nmax0 = 2 * it.t;            // last key tile of Q0 (its diagonal)
  it.nmax1 = it.has1 ? 2 * it.t + 1 : -1;
  it.nlast = it.has1 ? it.nmax1 : it.nmax0;
  return true;
}

template <int D, int PC>
__global__ void __launch_bounds__(PairCfg<PC>::THREADS, 1)
    tra_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ out, int BH, int T,
                         int nQ, int nPair, int nItems, float beta, float p, int d_real) {
  using L = PairLayout<D>;
  using Cfg = PairCfg<PC>;
  constexpr int PAIR_TMA_WARP = Cfg::TMA_WARP;
  const int dr = d_real;  // head dim (the tile width D or less: zero-filled columns)
  constexpr int PAIR_MMA_WARP = Cfg::MMA_WARP;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bars;               // [2], one per query tile
  uint64_t* q_empty = q_full + 2;        // [2]
  uint64_t* k_full = q_empty + 2;
  uint64_t* k_empty = k_full + L::NS;
  uint64_t* v_full = k_empty + L::NS;
  uint64_t* v_empty = v_full + L::NS;
  uint64_t* s_full = v_empty + L::NS;    // [2]
  uint64_t* p_half = s_full + 2;         // [2]
  uint64_t* p_full = p_half + 2;         // [2]
  uint64_t* o_full = p_full + 2;         // [2]
  uint64_t* o_empty = o_full + 2;        // [2]
  uint64_t* mma_done = o_empty + 2;     // [2]
  uint32_t* tptr = reinterpret_cast<uint32_t*>(smem + L::TPTR_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], 1);
      mbar_init(&s_full[b], 1);
      mbar_init(&p_half[b], 4 * Cfg::EPI_WG);
      mbar_init(&p_full[b], 4 * Cfg::EPI_WG);
      mbar_init(&o_full[b], 1);
      mbar_init(&o_empty[b], 4 * Cfg::EPI_WG);
    }
    for (int s = 0; s < L::NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], PairCfg<PC>::ISSUERS);  // one release per issuer per use
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], PairCfg<PC>::ISSUERS);
    }
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    fence_barrier_init();
  }
  if (warp == PAIR_MMA_WARP) {
    tmem_alloc(tptr, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tptr;
  PairItem it;

  if (warp == PAIR_TMA_WARP) {
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      bool ok = true;
      int g = 0;                // K/V tiles issued so far (ring position)
      int uq[2] = {0, 0};       // items so far that used query tile qt
      int nk = 0, nv = 0;
      for (int r = 0; ok && pair_item(r, nItems, BH, nPair, nQ, it); ++r) {
        for (int qt = 0; qt < (it.has1 ? 2 : 1); ++qt) {
          // The previous user of this Q buffer has finished its last QK.
          if (uq[qt] > 0 && !(ok = mbar_wait(&q_empty[qt], (uq[qt] - 1) & 1))) break;
          debug_check((2 * it.t + qt) < nQ && it.bh >= 0 && it.bh < BH);
          mbar_arrive_expect_tx(&q_full[qt], L::TILE);
#pragma unroll
          for (int pnl = 0; pnl < L::NP; ++pnl)
            tma_load_3d(smem + L::Q_OFF + qt * L::TILE + pnl * PANEL_BYTES, &tmQ, &q_full[qt], 64 * pnl,
                        (2 * it.t + qt) * BM, it.bh);
          ++uq[qt];
        }
        for (int n = 0; ok && n <= it.nlast; ++n, ++g) {
          const int s = g % L::NS;
          const uint32_t ph = (g / L::NS) & 1;
          if (!(ok = mbar_wait(&k_empty[s], ph ^ 1))) break;
          debug_check(n >= 0 && n < nQ && n <= it.nlast);
          mbar_arrive_expect_tx(&k_full[s], L::TILE);
#pragma unroll
          for (int pnl = 0; pnl < L::NP; ++pnl)
            tma_load_3d(smem + L::K_OFF + s * L::TILE + pnl * PANEL_BYTES, &tmK, &k_full[s], 64 * pnl, n * BN,
                        it.bh);
          nk = g + 1;
          if (!(ok = mbar_wait(&v_empty[s], ph ^ 1))) break;
          mbar_arrive_expect_tx(&v_full[s], L::TILE);
#pragma unroll
          for (int pnl = 0; pnl < L::NP; ++pnl)
            tma_load_3d(smem + L::V_OFF + s * L::TILE + pnl * PANEL_BYTES, &tmV, &v_full[s], 64 * pnl, n * BN,
                        it.bh);
          nv = g + 1;
        }
      }
      if (!ok) {
        // Drain: never leave the CTA with a bulk copy still landing in its smem.
        for (int qt = 0; qt < 2; ++qt)
          if (uq[qt] > 0) mbar_wait(&q_full[qt], (uq[qt] - 1) & 1);
        for (int n = (nk > L::NS ? nk - L::NS : 0); n < nk; ++n) mbar_wait(&k_full[n % L::NS], (n / L::NS) & 1);
        for (int n = (nv > L::NS ? nv - L::NS : 0); n < nv; ++n) mbar_wait(&v_full[n % L::NS], (n / L::NS) & 1);
      }
    }
  } else if (warp >= PAIR_MMA_WARP && PairCfg<PC>::ISSUERS == 2) {
    // Issuer qt serves query tile qt: per key tile n, P V(n) and then
    // QK(n+1), on the items and K/V ring positions the producer walks.  Every
    // ring use takes two arrivals on k_empty / v_empty: one commit from each
    // issuer, or two from the one issuer whose tile alone reads that key tile
    // (Q1's diagonal tile; every key tile of an item without Q1).  An issuer
    // arrives for a use only after waiting for that use's load, so an arrival
    // can never count toward the previous phase.  The whole warp walks the
    // loop (or only the elected lane, see pair_converged_issue); one elected
    // lane issues the MMAs and commits.  Every lane waits on its own, so the
    // lanes can part only when a wait gives up, and nothing after that needs
    // them together.
    const int qt = warp - PAIR_MMA_WARP;
    const bool leader = elect_one();
    if (pair_converged_issue<D>() || leader) {
      const uint32_t sQ = smem_u32(smem + L::Q_OFF + qt * L::TILE);
      const uint32_t tS = tmem + qt * BN, tO = tmem + 2 * BN + qt * D;
      int g = 0;   // K/V ring position of the item's key tile 0
      int cs = 0;  // score tiles so far (s_full / p_half / p_full phase)
      int uq = 0;  // items so far for this query tile (q_full / o_full / o_empty phase)
      bool ok = true;
      for (int r = 0; ok && pair_item(r, nItems, BH, nPair, nQ, it); ++r) {
        if (qt == 1 && !it.has1) {
          g += it.nlast + 1;
          continue;
        }
        const int nmax = qt == 0 ? it.nmax0 : it.nmax1;
        const bool alone_all = !it.has1;  // Q0 alone reads every key tile of the item
        auto release = [&](uint64_t* empty, int n) {
          if (leader) {
            mma_commit(empty);
            if (alone_all || (qt == 1 && n == it.nlast)) mma_commit(empty);
          }
        };
        auto qk = [&](int n) -> bool {
          const int gi = g + n;
          if (!mbar_wait(&k_full[gi % L::NS], (gi / L::NS) & 1)) return false;
          tc_fence_after();
          tile::mma_abt<D>(tS, sQ, smem_u32(smem + L::K_OFF + (gi % L::NS) * L::TILE), leader);
          if (leader) mma_commit(&s_full[qt]);
          release(&k_empty[gi % L::NS], n);
          if (leader && n == nmax) mma_commit(&q_empty[qt]);
          return true;
        };
        if (!(ok = mbar_wait(&q_full[qt], uq & 1) && qk(0))) break;
        for (int n = 0; n <= nmax; ++n, ++cs) {
          // P V(n) in two halves: keys 0..63 as soon as that half of P is there.
          const int gi = g + n;
          const uint32_t sV = smem_u32(smem + L::V_OFF + (gi % L::NS) * L::TILE);
          const uint32_t ph = cs & 1;
          // V(n) has usually landed long before P: then only the P barrier
          // sits between the epilogue and the P V issue.  With p = 1 (the
          // lightest epilogue) and with the four-stage D = 64 ring V is
          // waited for first (measured fastest there); otherwise, if V has
          // not landed yet (two-stage D = 128 ring), P is waited for first.
          constexpr bool V_FIRST = PC == POW_ONE || D == 64;
          uint64_t* vb = &v_full[gi % L::NS];
          const uint32_t vph = (gi / L::NS) & 1;
          const bool v_in = V_FIRST ? mbar_wait(vb, vph) : mbar_test(vb, vph);
          if (V_FIRST && !(ok = v_in)) break;
          if (!(ok = mbar_wait(PAIR_SPLIT_P ? &p_half[qt] : &p_full[qt], ph) &&
                     (v_in || mbar_wait(vb, vph))))
            break;
          // The first P V of an item overwrites O: the epilogue has read the last one.
          if (n == 0 && uq > 0 && !(ok = mbar_wait(&o_empty[qt], (uq - 1) & 1))) break;
          tc_fence_after();
          tile::mma_tmem_a<D>(tO, tS, sV, 0, BN / 32, n == 0, leader);
          if (!(ok = mbar_wait(&p_full[qt], ph))) break;
          tc_fence_after();
          tile::mma_tmem_a<D>(tO, tS, sV, BN / 32, BN / 16, false, leader);
          release(&v_empty[gi % L::NS], n);
          if (n == nmax) {
            if (leader) mma_commit(&o_full[qt]);
          } else if (!(ok = qk(n + 1))) {
            break;
          }
        }
        g += it.nlast + 1;
        ++uq;
      }
      // Commits arrive in issue order: once this one has landed, every
      // barrier arrival of this thread's MMAs has too, and smem may be released.
      if (leader) mma_commit(&mma_done[qt]);
      mbar_wait(&mma_done[qt], 0);
    }
  } else if (warp == PAIR_MMA_WARP) {
    // One issuer for both tiles, in the order PV0(n), QK0(n+1), PV1(n),
    // QK1(n+1); each ring use is released by one commit once both tiles'
    // products on it have been issued.  The whole warp walks the loop (or
    // only the elected lane, see pair_converged_issue); one elected lane
    // issues and commits.
    const bool leader = elect_one();
    if (pair_converged_issue<D>() || leader) {
      const uint32_t sQ0 = smem_u32(smem + L::Q_OFF);
      int g = 0;               // K/V ring position of the item's key tile 0
      int cs[2] = {0, 0};      // score tiles so far per query tile (s_full / p_half / p_full phase)
      int uq[2] = {0, 0};      // items so far per query tile (q_full / o_full / o_empty phase)
      bool ok = true;
      auto commit = [&](uint64_t* bar) {
        if (leader) mma_commit(bar);
      };
      auto qk = [&](int qt, int gi) {
        tile::mma_abt<D>(tmem + qt * BN, sQ0 + qt * L::TILE, smem_u32(smem + L::K_OFF + (gi % L::NS) * L::TILE),
                         leader);
        commit(&s_full[qt]);
      };
      // PVt(n) in two halves: keys 0..63 as soon as that half of P is there.
      auto pv = [&](int qt, int n, int gi) -> bool {
        const uint32_t sV = smem_u32(smem + L::V_OFF + (gi % L::NS) * L::TILE);
        const uint32_t tP = tmem + qt * BN, tO = tmem + 2 * BN + qt * D;
        const uint32_t ph = cs[qt] & 1;
        uint64_t* vb = &v_full[gi % L::NS];  // V usually landed long before P (see the per-tile issuer)
        const uint32_t vph = (gi / L::NS) & 1;
        const bool v_in = mbar_test(vb, vph);
        if (!mbar_wait(PAIR_SPLIT_P ? &p_half[qt] : &p_full[qt], ph) || !(v_in || mbar_wait(vb, vph)))
          return false;
        // The first P V of an item overwrites O: the epilogue has read the last one.
        if (n == 0 && uq[qt] > 0 && !mbar_wait(&o_empty[qt], (uq[qt] - 1) & 1)) return false;
        tc_fence_after();
        tile::mma_tmem_a<D>(tO, tP, sV, 0, BN / 32, n == 0, leader);
        if (!mbar_wait(&p_full[qt], ph)) return false;
        tc_fence_after();
        tile::mma_tmem_a<D>(tO, tP, sV, BN / 32, BN / 16, false, leader);
        ++cs[qt];
        return true;
      };

      for (int r = 0; ok && pair_item(r, nItems, BH, nPair, nQ, it); ++r) {
        if (!(ok = mbar_wait(&k_full[g % L::NS], (g / L::NS) & 1) && mbar_wait(&q_full[0], uq[0] & 1)))
          break;
        tc_fence_after();
        qk(0, g);
        if (it.nmax0 == 0) commit(&q_empty[0]);
        if (it.has1) {
          if (!(ok = mbar_wait(&q_full[1], uq[1] & 1))) break;
          tc_fence_after();
          qk(1, g);
        }
        commit(&k_empty[g % L::NS]);
        for (int n = 0; n <= it.nlast && ok; ++n) {
          const int n1 = n + 1, gn = g + n, gn1 = g + n1;
          const bool next_k = n1 <= it.nlast;
          // tile 0: PV0(n), then QK0(n+1)
          if (n <= it.nmax0) {
            if (!(ok = pv(0, n, gn))) break;
            if (n == it.nmax0) commit(&o_full[0]);
          }
          if (next_k) {
            if (!(ok = mbar_wait(&k_full[gn1 % L::NS], (gn1 / L::NS) & 1))) break;
            tc_fence_after();
            if (n1 <= it.nmax0) {
              qk(0, gn1);
              if (n1 == it.nmax0) commit(&q_empty[0]);
            }
          }
          // tile 1: PV1(n), then QK1(n+1)
          if (it.has1) {
            if (!(ok = pv(1, n, gn))) break;
            if (n == it.nmax1) commit(&o_full[1]);
          }
          commit(&v_empty[gn % L::NS]);
          if (next_k) {
            if (it.has1 && n1 <= it.nmax1) {
              qk(1, gn1);
              if (n1 == it.nmax1) commit(&q_empty[1]);
            }
            commit(&k_empty[gn1 % L::NS]);
          }
        }
        g += it.nlast + 1;
        ++uq[0];
        if (it.has1) ++uq[1];
      }
      // Commits arrive in issue order: once this one has landed, every
      // barrier arrival of this CTA's MMAs has too, and smem may be released.
      commit(&mma_done[0]);
      mbar_wait(&mma_done[0], 0);
    }
  } else {
    const int qt = (warp >> 2) & 1;  // query tile of this warpgroup
    const int wq = warp & 3;         // TMEM lane quarter
    const int half = warp >> 3;      // with two warpgroups per tile: score quarters {0, 2} or {1, 3}
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t tS = lane_base + qt * BN;
    int cs = 0, uq = 0;
    bool ok = true;
    for (int r = 0; ok && pair_item(r, nItems, BH, nPair, nQ, it); ++r) {
      if (qt == 1 && !it.has1) continue;
      const int nmax = qt == 0 ? it.nmax0 : it.nmax1;
      const int row = (2 * it.t + qt) * BM + wq * 32 + lane;
      const PowParams wp = pow_params(tile::tau_of_row(row, beta, dr), p);
      for (int n = 0; n <= nmax; ++n, ++cs) {
        if (!(ok = mbar_wait(&s_full[qt], cs & 1))) break;
        tc_fence_after();
        constexpr int MP = mix_mufu_pairs<D>();
        if constexpr (Cfg::EPI_WG == 2) {
          const int bar_id = 1 + qt * 4 + wq;  // the two warps sharing this lane quarter
          constexpr bool HL = pair_half_loads<D>();
          if (n == nmax)
            epilogue_two_quarters<PC, true, MP, HL>(tS, wp, n * BN, row, lane, half, bar_id, &p_half[qt],
                                                    &p_full[qt]);
          else
            epilogue_two_quarters<PC, false, MP, HL>(tS, wp, n * BN, row, lane, half, bar_id, &p_half[qt],
                                                     &p_full[qt]);
        } else {
          if (n == nmax)
            epilogue_tile<PC, PAIR_SPLIT_P, true, MP>(tS, wp, n * BN, row, lane, &p_half[qt], &p_full[qt]);
          else
            epilogue_tile<PC, PAIR_SPLIT_P, false, MP>(tS, wp, n * BN, row, lane, &p_half[qt], &p_full[qt]);
        }
      }
      if (!ok || !(ok = mbar_wait(&o_full[qt], uq & 1))) break;
      tc_fence_after();
      __nv_bfloat16* orow = out + (static_cast<size_t>(it.bh) * T + row) * dr;
      constexpr int CPW = D / 32 / Cfg::EPI_WG;  // 32-column chunks of O this warp stores
#pragma unroll
      for (int c = 0; c < CPW; ++c) {
        const int cc = half * CPW + c;
        if (dr == D)
          tile::store_row_chunk(lane_base + 2 * BN + qt * D, cc, orow, row < T);
        else if (cc * 32 < dr)  // head dim below the tile width: only its columns
          tile::store_row_part(lane_base + 2 * BN + qt * D, cc, orow, row < T, min(32, dr - cc * 32));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_empty[qt]);
      ++uq;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == PAIR_MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int D, int PC>
int launch_pair(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, void* out, int BH, int T,
                float beta, float p, cudaStream_t stream, int d_real = D) {
  using L = PairLayout<D>;
  auto kern = tra_bf16_pair_kernel<D, PC>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC) != cudaSuccess)
    return ERR_LAUNCH;
  const int nQ = (T + BM - 1) / BM;
  const int nPair = (nQ + 1) / 2;
  const long long items = static_cast<long long>(nPair) * BH;
  if (items > 0x7fffffffLL) return ERR_SHAPE;
  const int sms = sm_count();
  if (sms <= 0) return ERR_DEVICE;
  const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
  kern<<<grid, PairCfg<PC>::THREADS, L::ALLOC, stream>>>(mq, mk, mv, static_cast<__nv_bfloat16*>(out), BH, T, nQ, nPair,
                                                 static_cast<int>(items), beta, p, d_real);
  return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
}

// Half powers (on request).
template <int D>
int launch_half(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, void* out, int BH, int T,
                float beta, float p, int hc, cudaStream_t stream, int d_real) {
  switch (hc) {
    case POW_HALF0: return launch_pair<D, POW_HALF0>(mq, mk, mv, out, BH, T, beta, p, stream, d_real);
    case POW_HALF0 + 1: return launch_pair<D, POW_HALF0 + 1>(mq, mk, mv, out, BH, T, beta, p, stream, d_real);
    case POW_HALF0 + 2: return launch_pair<D, POW_HALF0 + 2>(mq, mk, mv, out, BH, T, beta, p, stream, d_real);
    case POW_HALF3: return launch_pair<D, POW_HALF3>(mq, mk, mv, out, BH, T, beta, p, stream, d_real);
    default: return ERR_UNSUPPORTED;
  }
}

// Every power class at tile width D for a head dim d_real <= D.
template <int D>
int launch_width(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, void* out, int BH, int T,
                 float beta, float p, int pc, cudaStream_t stream, int d_real) {
  if (pc == POW_TWO) return launch_pair<D, POW_TWO>(mq, mk, mv, out, BH, T, beta, p, stream, d_real);
  if (pc == POW_ONE) return launch_pair<D, POW_ONE>(mq, mk, mv, out, BH, T, beta, p, stream, d_real);
  if (pc == POW_GENERAL_MIX) return launch_pair<D, POW_GENERAL_MIX>(mq, mk, mv, out, BH, T, beta, p, stream, d_real);
  return launch_pair<D, POW_GENERAL>(mq, mk, mv, out, BH, T, beta, p, stream, d_real);
}

}  // namespace

int launch_tra_bf16(const void* q, const void* k, const void* v, void* out, int B, int H, int T, int D,
                    float beta, float p, bool sqrt_half_powers, cudaStream_t stream) {
  const int BH = B * H;
  if (!tra_head_dim_supported(D)) return ERR_UNSUPPORTED;
  CUtensorMap mq, mk, mv;
  const uint64_t rs = static_cast<uint64_t>(D) * 2;  // row stride in bytes
  const uint64_t hs = rs * T;                        // (b, h) stride in bytes
  int st = encode_tmap_3d(&mq, q, D, T, BH, rs, hs, 64, BM, 1);
  if (st == OK) st = encode_tmap_3d(&mk, k, D, T, BH, rs, hs, 64, BN, 1);
  if (st == OK) st = encode_tmap_3d(&mv, v, D, T, BH, rs, hs, 64, BN, 1);
  if (st != OK) return st;
  const int pc = power_class(p);
  const int hc = sqrt_half_powers ? half_power_class(p) : -1;
  // Head dims below the tile width (64 for D <= 64, else 128): the TMA boxes
  // of 64 columns read zeros past the tensor's D columns, which change neither
  // q.k nor P V, and only the D real columns of O are stored.
  const int width = D <= 64 ? 64 : 128;
  if (hc >= 0)
    return width == 128 ? launch_half<128>(mq, mk, mv, out, BH, T, beta, p, hc, stream, D)
                        : launch_half<64>(mq, mk, mv, out, BH, T, beta, p, hc, stream, D);
  return width == 128 ? launch_width<128>(mq, mk, mv, out, BH, T, beta, p, pc, stream, D)
                      : launch_width<64>(mq, mk, mv, out, BH, T, beta, p, pc, stream, D);
}

unsigned int tra_bf16_device_error() { return read_and_clear_device_error(); }

}  // namespace bsa
