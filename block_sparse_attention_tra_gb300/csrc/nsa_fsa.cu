// nsa_fsa.cu -- NSA selection forward in the block-outer split-K form: one
// pass over the selected key blocks that loads each block's K/V once, then a
// log-sum-exp combine.
//
// Method: page "nsa_selection_kernel.py", FSA forward section
// (_selection_fwd_blockouter_kernel and selection_forward_fsa).  For every
// (query i, selected block j) pair and head g of the group the first pass
// writes the block's softmax partial over its tokens t <= i:
//     m = max_t s_t,  l = sum_t exp(s_t - m),  acc = sum_t exp(s_t - m) v_t,
//     s_t = q_i . k_t * D^-0.5;
// the combine merges a query's partials into one softmax over the union:
//     M = max_j m_j,  w_j = exp(m_j - M),  o = sum_j w_j acc_j / sum_j w_j l_j,
//     lse = M + ln sum_j w_j l_j   (o = 0, lse = -1e9 with no pair).
//
// Launches, all on the caller's stream, scratch in the caller's workspace:
//   1. fsa_zero          clear the per-block counters
//   2. fsa_pairs<count>  count the pairs of every (b, kv head, block)
//   3. fsa_scan          exclusive scan -> list offsets; cut every block's
//                        list into work items of at most ITEM_TILES M tiles
//   4. fsa_pairs<fill>   write the inverted lists (packed i * 32 + slot)
//   5. fsa_blockouter    one CTA per work item: K/V of the block by TMA, once;
//                        M tiles of 128 rows = 128 / G queries x G heads
//                        gathered by cp.async; S = Q K^T (N = 64) and
//                        acc = P V on tcgen05; the softmax partial per row in
//                        registers; partials out
//   6. fsa_combine       one warp per (b, query head, i): the log-sum-exp merge
//
// A pair (i, j) exists for every live slot of row i: 0 <= j < T / 64 and
// j * 64 <= i (the rule of the query-outer kernel), so both paths agree on
// which blocks a query reads.  Partials live at the slot they came from,
// [(b, hkv, i, slot), g, D], which lets the combine read them in row order
// without a second index.  Within a list the order of the pairs depends on
// atomics, but every row of an M tile is computed independently, so the
// results do not.
#include <algorithm>

#include "kernels.h"
#include "nsa_slots.cuh"
#include "ptx.cuh"

namespace bsa {
namespace {

constexpr int FSA_BS = 64;             // tokens per block
constexpr int FSA_M = 128;             // rows per M tile (queries x heads)
constexpr int FSA_ITEM_TILES = 32;     // M tiles per work item at most
constexpr int FSA_NQS = 3;             // Q stages
constexpr int FSA_EPI_WARPS = 8;       // two epilogue warpgroups (ping-pong tiles)
constexpr int FSA_PROD_WARP0 = 8;      // warps 8..11 gather Q
constexpr int FSA_MMA_WARP = 12;
constexpr int FSA_THREADS = 13 * 32;
constexpr int FSA_STG_STRIDE = 272;    // staging row: 64 floats + 16 bytes of skew
constexpr int FSA_STG_WARP = 32 * FSA_STG_STRIDE;
constexpr int FSA_TSTG_BUF = 32 * 128;  // TMA-store stage: 32 rows x 32 floats, 128-byte swizzled
constexpr int FSA_TSTG_WARP = 2 * FSA_TSTG_BUF;  // two stages per warp (8 KB, 1 KB aligned)
static_assert(FSA_TSTG_WARP <= FSA_STG_WARP, "the TMA-store stages reuse the staging area");
constexpr int PANEL = 128 * 128;       // 128 rows x 128 B swizzle panel

template <int D>
struct FsaLayout {
  static constexpr int NP = D / 64;
  static constexpr int KV_PANEL = FSA_BS * 128;  // 64 tokens x 128 B
  static constexpr int KV_TILE = NP * KV_PANEL;
  static constexpr int Q_TILE = NP * PANEL;      // 128 rows x D
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KV_TILE;
  static constexpr int Q_OFF = V_OFF + KV_TILE;
  static constexpr int STG_OFF = Q_OFF + FSA_NQS * Q_TILE;
  static constexpr int BAR_OFF = STG_OFF + FSA_EPI_WARPS * FSA_STG_WARP;
  // kv_full | q_full[NQS] | q_empty[NQS] | s_full[2] | p_full[2] | o_full[2] | o_empty[2] | mma_done
  static constexpr int NBAR = 1 + 2 * FSA_NQS + 8 + 1;
  static constexpr int TPTR_OFF = BAR_OFF + NBAR * 8;
  static constexpr int ALLOC = TPTR_OFF + 16 + 1024;
  // TMEM columns: S0 | S1 | O0 | O1
  static constexpr uint32_t S_COL = 0, O_COL = 2 * FSA_BS;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(O_COL + 2 * D <= TMEM_COLS, "TMEM budget");
};

// ------------------------------------------------------------------ CSR build

__global__ void fsa_zero_kernel(int* __restrict__ counts, int n, int* __restrict__ meta) {
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n; e += gridDim.x * blockDim.x) counts[e] = 0;
  if (blockIdx.x == 0 && threadIdx.x < 4) meta[threadIdx.x] = 0;
}

// FILL = false: counts[bh, j] += 1 per live slot.  FILL = true: append the
// pair (packed i * 32 + slot) at the block's cursor.  One warp per index row
// (lane s takes slot s): the live slots, de-duplicated under the set reading
// of the row, come from nsa_live_slots as in the query-outer kernels.
template <bool FILL>
__global__ void fsa_pairs_kernel(const int32_t* __restrict__ block_idx, int* __restrict__ counter,
                                 int* __restrict__ list, long long n_rows, int T, int S, int n_blk) {
  const int lane = static_cast<int>(threadIdx.x & 31u);
  const long long n_warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long row = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5; row < n_rows;
       row += n_warps) {  // warp-uniform: the whole warp takes a row
    const int i = static_cast<int>(row % T);
    const long long bh = row / T;
    const SlotRow r = nsa_live_slots(block_idx + row * S, S, i, n_blk, FSA_BS);
    if ((r.live >> lane) & 1u) {
      int* c = counter + bh * n_blk + r.blk_lane;
      if constexpr (FILL) {
        const int pos = debug_index(atomicAdd(c, 1), 0, static_cast<int>(n_rows * S));
        list[pos] = i * 32 + lane;
      } else {
        atomicAdd(c, 1);
      }
    }
  }
}

// Single CTA.  counts[NB] -> off[NB + 1] (exclusive scan; counts become the
// fill cursors) and the work items {bh * n_blk + j, first list index, pairs}.
constexpr int SCAN_THREADS = 1024;
__global__ void __launch_bounds__(SCAN_THREADS) fsa_scan_kernel(int* __restrict__ counts, int* __restrict__ off,
                                                                int4* __restrict__ items, int* __restrict__ meta,
                                                                int NB, int qch) {
  __shared__ int warp_pairs[32], warp_items[32];
  const int per = (NB + SCAN_THREADS - 1) / SCAN_THREADS;
  const int lo = min(NB, static_cast<int>(threadIdx.x) * per), hi = min(NB, lo + per);
  int np = 0, ni = 0;
  for (int e = lo; e < hi; ++e) {
    np += counts[e];
    ni += (counts[e] + qch - 1) / qch;
  }
  // Block-wide exclusive scan of (np, ni).
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int sp = np, si = ni;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, sp, d), b = __shfl_up_sync(0xffffffffu, si, d);
    if (lane >= d) { sp += a; si += b; }
  }
  if (lane == 31) { warp_pairs[warp] = sp; warp_items[warp] = si; }
  __syncthreads();
  if (warp == 0) {
    int wp = warp_pairs[lane], wi = warp_items[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, wp, d), b = __shfl_up_sync(0xffffffffu, wi, d);
      if (lane >= d) { wp += a; wi += b; }
    }
    warp_pairs[lane] = wp;
    warp_items[lane] = wi;
  }
  __syncthreads();
  int pbase = sp - np + (warp > 0 ? warp_pairs[warp - 1] : 0);
  int ibase = si - ni + (warp > 0 ? warp_items[warp - 1] : 0);
  for (int e = lo; e < hi; ++e) {
    const int c = counts[e];
    off[e] = pbase;
    counts[e] = pbase;  // fill cursor
    for (int s = 0; s < c; s += qch) items[ibase++] = make_int4(e, pbase + s, min(qch, c - s), 0);
    pbase += c;
  }
  if (threadIdx.x == SCAN_THREADS - 1) {
    off[NB] = pbase;
    meta[0] = ibase;  // work items
    meta[1] = pbase;  // pairs
  }
}

// ------------------------------------------------------------- block-outer pass

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// TMA_OUT (G = 8 or 16): the acc rows of each query (G consecutive partial
// rows) leave through a 128-byte-swizzled shared-memory stage and one TMA
// tensor store per query and 32-column chunk (tmAcc: fp32 [rows, D], box
// 32 x G); otherwise through the skewed staging area and 16-byte stores.
template <int D, bool TMA_OUT>
__global__ void __launch_bounds__(FSA_THREADS, 1)
    fsa_blockouter_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ CUtensorMap tmAcc,
                          const __nv_bfloat16* __restrict__ q, const int* __restrict__ list,
                          const int4* __restrict__ items, const int* __restrict__ meta, float* __restrict__ acc,
                          float* __restrict__ pm, float* __restrict__ pl, int G, int Hq, int Hkv, int T, int S,
                          int n_blk, float scale) {
  using L = FsaLayout<D>;
  if (static_cast<int>(blockIdx.x) >= meta[0]) return;  // fewer items than the launch bound
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;              // [NQS]
  uint64_t* q_empty = q_full + FSA_NQS;     // [NQS]
  uint64_t* s_full = q_empty + FSA_NQS;     // [2]
  uint64_t* p_full = s_full + 2;            // [2]
  uint64_t* o_full = p_full + 2;            // [2]
  uint64_t* o_empty = o_full + 2;           // [2]
  uint64_t* mma_done = o_empty + 2;
  uint32_t* tptr = reinterpret_cast<uint32_t*>(smem + L::TPTR_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int4 item = items[blockIdx.x];
  const int bh = item.x / n_blk, j = item.x % n_blk;
  const int b = bh / Hkv, hkv = bh % Hkv;
  const int first = item.y, npairs = item.z;
  const int qpt = FSA_M / G;                    // queries per M tile
  const int nt = (npairs + qpt - 1) / qpt;      // M tiles of this item

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < FSA_NQS; ++s) {
      mbar_init(&q_full[s], 4 * 32);
      mbar_init(&q_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 4);
      mbar_init(&o_full[x], 1);
      mbar_init(&o_empty[x], 4);
    }
    mbar_init(mma_done, 1);
    fence_barrier_init();
  }
  if (warp == FSA_MMA_WARP) {
    tmem_alloc(tptr, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tptr;

  if (warp >= FSA_PROD_WARP0 && warp < FSA_MMA_WARP) {
    // ---- Q gather.  Thread r resolves row r (query r / G, head r % G) of each
    // tile; the copies go row by row, CPR consecutive lanes taking the 16-byte
    // chunks of one row, so that a warp instruction reads whole rows (two at
    // D = 128, four at D = 64) instead of one chunk of 32 different rows.
    constexpr int CPR = D / 8;      // 16-byte chunks per row
    constexpr int RPI = 32 / CPR;   // rows per warp instruction
    const int r = threadIdx.x - FSA_PROD_WARP0 * 32;
    const int qi = r / G, g = r % G;
    const int row0 = r & ~31;       // first row of this warp
    const int c = lane % CPR;       // this lane's chunk of every row it copies
    const size_t head_row0 = (static_cast<size_t>(b) * Hq + static_cast<size_t>(hkv) * G + g) * T;
    bool ok = true;
    int issued = 0;
    for (int t = 0; t < nt; ++t) {
      const int st = t % FSA_NQS;
      if (t >= FSA_NQS && !(ok = mbar_wait(&q_empty[st], ((t / FSA_NQS) - 1) & 1))) break;
      const int slot = t * qpt + qi;
      const bool valid = qi < qpt && slot < npairs;
      const int i = valid ? debug_index(list[first + slot] >> 5, 0, T) : 0;
      const unsigned long long src = reinterpret_cast<unsigned long long>(q + (head_row0 + i) * D);
      const uint32_t tile = smem_u32(smem + L::Q_OFF + st * L::Q_TILE);
#pragma unroll
      for (int k = 0; k < 32 / RPI; ++k) {
        const int from = k * RPI + lane / CPR;  // lane holding the row copied now
        const int rr = row0 + from;
        const unsigned long long rsrc = __shfl_sync(0xffffffffu, src, from);
        const bool rvalid = __shfl_sync(0xffffffffu, valid, from);
        const uint32_t dst = tile + rr * 128 + (c >> 3) * PANEL + (((c & 7) ^ (rr & 7)) << 4);
        cp_async16(dst, reinterpret_cast<const __nv_bfloat16*>(rsrc) + c * 8, rvalid ? 16u : 0u);
      }
      cp_async_commit();
      issued = t + 1;
      if (t >= 1) {
        cp_async_wait<1>();
        fence_proxy_async_smem();
        mbar_arrive(&q_full[(t - 1) % FSA_NQS]);
      }
    }
    cp_async_wait<0>();  // never leave a copy landing in a finished CTA
    if (ok && issued > 0) {
      fence_proxy_async_smem();
      mbar_arrive(&q_full[(issued - 1) % FSA_NQS]);
    }
  } else if (warp == FSA_MMA_WARP) {
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      debug_check(j >= 0 && j < n_blk);
      mbar_arrive_expect_tx(kv_full, 2 * L::KV_TILE);
#pragma unroll
      for (int pnl = 0; pnl < L::NP; ++pnl) {
        tma_load_3d(smem + L::K_OFF + pnl * L::KV_PANEL, &tmK, kv_full, 64 * pnl, j * FSA_BS, bh);
        tma_load_3d(smem + L::V_OFF + pnl * L::KV_PANEL, &tmV, kv_full, 64 * pnl, j * FSA_BS, bh);
      }
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(FSA_M, FSA_BS, 0, 0);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(FSA_M, D, 0, 1);
      const uint32_t sK = smem_u32(smem + L::K_OFF), sV = smem_u32(smem + L::V_OFF);
      bool ok = mbar_wait(kv_full, 0);
      for (int t = 0; t <= nt && ok; ++t) {
        if (t < nt) {  // S_t = Q_t K^T into S[t & 1]
          const int st = t % FSA_NQS;
          if (!(ok = mbar_wait(&q_full[st], (t / FSA_NQS) & 1))) break;
          tc_fence_after();
          const uint32_t sQ = smem_u32(smem + L::Q_OFF + st * L::Q_TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ko = (kk & 3) * 32;
            mma_ss(tmem + L::S_COL + (t & 1) * FSA_BS,
                   smem_desc_sw128(sQ + (kk >> 2) * PANEL + ko, 16, 1024),
                   smem_desc_sw128(sK + (kk >> 2) * L::KV_PANEL + ko, 16, 1024), IDESC_QK, kk > 0 ? 1u : 0u);
          }
          mma_commit(&s_full[t & 1]);
          mma_commit(&q_empty[st]);
        }
        if (t >= 1) {  // acc_u = P_u V into O[u & 1]
          const int u = t - 1, x = u & 1;
          if (!(ok = mbar_wait(&p_full[x], (u >> 1) & 1))) break;
          if (u >= 2 && !(ok = mbar_wait(&o_empty[x], ((u >> 1) - 1) & 1))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < FSA_BS / 16; ++kk)
            mma_ts(tmem + L::O_COL + x * D, tmem + L::S_COL + x * FSA_BS + kk * 8,
                   smem_desc_sw128(sV + kk * 16 * 128, L::NP > 1 ? L::KV_PANEL : 1024, 1024), IDESC_PV,
                   kk > 0 ? 1u : 0u);
          mma_commit(&o_full[x]);
        }
      }
      mma_commit(mma_done);
      mbar_wait(mma_done, 0);
    }
  } else {
    // ---- epilogue warpgroup w: tiles t = w, w + 2, ...; thread = TMEM lane = tile row.
    const int w = warp >> 2, wq = warp & 3;
    const int r = wq * 32 + lane;
    const int qi = r / G, g = r % G;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t tS = lane_base + L::S_COL + w * FSA_BS, tO = lane_base + L::O_COL + w * D;
    const float sl2 = scale * 1.4426950408889634f;  // scale * log2(e)
    const uint32_t stg_u = smem_u32(smem + L::STG_OFF + warp * FSA_STG_WARP);
    const uint32_t tstg = smem_u32(smem + L::STG_OFF + warp * FSA_TSTG_WARP);  // 1 KB aligned (TMA_OUT)
    int tsc = 0;  // 32-column chunks staged so far (TMA_OUT: selects the stage)
    for (int t = w, n = 0; t < nt; t += 2, ++n) {
      const int slot = t * qpt + qi;
      const bool valid = qi < qpt && slot < npairs;
      const int e = valid ? list[first + slot] : 0;
      const int i = e >> 5, s = e & 31;
      const int lim = valid ? i - j * FSA_BS : -1;  // tokens c <= lim are causal
      // Partial row index (b, hkv, i, slot, g); -1 = no row.
      const int prow = valid ? ((bh * T + i) * S + s) * G + g : -1;
      if (!mbar_wait(&s_full[w], n & 1)) break;
      tc_fence_after();
      uint32_t sa[32], sb[32];
      tmem_ld32(tS, sa);
      tmem_ld32(tS + 32, sb);
      tmem_wait_ld();
      float m = -INFINITY;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        if (c <= lim) m = fmaxf(m, __uint_as_float(sa[c]));
        if (c + 32 <= lim) m = fmaxf(m, __uint_as_float(sb[c]));
      }
      const float mb = m * sl2;
      float l = 0.0f;
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float p0 = (2 * c <= lim) ? ex2f(fmaf(__uint_as_float(sa[2 * c]), sl2, -mb)) : 0.0f;
        const float p1 = (2 * c + 1 <= lim) ? ex2f(fmaf(__uint_as_float(sa[2 * c + 1]), sl2, -mb)) : 0.0f;
        l += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      tmem_st16(tS, pk);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float p0 = (2 * c + 32 <= lim) ? ex2f(fmaf(__uint_as_float(sb[2 * c]), sl2, -mb)) : 0.0f;
        const float p1 = (2 * c + 33 <= lim) ? ex2f(fmaf(__uint_as_float(sb[2 * c + 1]), sl2, -mb)) : 0.0f;
        l += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      tmem_st16(tS + 16, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[w]);
      if (prow >= 0) {
        pm[prow] = m * scale;  // local max of the scaled scores
        pl[prow] = l;
      }
      if (!mbar_wait(&o_full[w], n & 1)) break;
      tc_fence_after();
      if constexpr (TMA_OUT) {
        // First partial row of each query of this warp (lanes k * G), or -1.
        int qrow[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) qrow[k] = __shfl_sync(0xffffffffu, prow, (k * G) & 31);
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c, ++tsc) {
          const uint32_t buf = tstg + (tsc & 1) * FSA_TSTG_BUF;
          // The store issued two chunks ago read this stage: let it finish reading.
          if (tsc >= 2 && lane == 0) bulk_wait_read<1>();
          __syncwarp();
          uint32_t ov[32];
          tmem_ld32(tO + c * 32, ov);
          tmem_wait_ld();
          if (c == D / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_empty[w]);
          }
#pragma unroll
          for (int x = 0; x < 8; ++x)
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(buf + lane * 128 + ((x ^ (lane & 7)) << 4)),
                         "r"(ov[4 * x]), "r"(ov[4 * x + 1]), "r"(ov[4 * x + 2]), "r"(ov[4 * x + 3])
                         : "memory");
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (k * G < 32 && qrow[k] >= 0) tma_store_2d(&tmAcc, buf + k * G * 128, c * 32, qrow[k]);
            bulk_commit();
          }
        }
      } else {
        // acc row -> HBM, 64 columns at a time through a skewed staging area so
        // that every global store instruction writes two contiguous 256-byte rows.
#pragma unroll 1
        for (int h = 0; h < D / 64; ++h) {
          uint32_t oa[32], ob[32];
          tmem_ld32(tO + h * 64, oa);
          tmem_ld32(tO + h * 64 + 32, ob);
          tmem_wait_ld();
          if (h == D / 64 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_empty[w]);
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t a = stg_u + lane * FSA_STG_STRIDE + c * 16;
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(oa[4 * c]), "r"(oa[4 * c + 1]),
                         "r"(oa[4 * c + 2]), "r"(oa[4 * c + 3]) : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(a + 128), "r"(ob[4 * c]), "r"(ob[4 * c + 1]),
                         "r"(ob[4 * c + 2]), "r"(ob[4 * c + 3]) : "memory");
          }
          __syncwarp();
#pragma unroll 4
          for (int k = 0; k < 16; ++k) {
            const int rr = 2 * k + (lane >> 4), ch = lane & 15;
            const int orow = __shfl_sync(0xffffffffu, prow, rr);
            uint4 v4;
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(v4.x), "=r"(v4.y), "=r"(v4.z), "=r"(v4.w)
                         : "r"(stg_u + rr * FSA_STG_STRIDE + ch * 16));
            if (orow >= 0)
              *reinterpret_cast<uint4*>(acc + static_cast<size_t>(orow) * D + h * 64 + ch * 4) = v4;
          }
          __syncwarp();
        }
      }
    }
    // Never leave the CTA while a tensor store still reads its stage.
    if constexpr (TMA_OUT) {
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == FSA_MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

// ----------------------------------------------------------------- combine

// One warp per output row (b, hkv * G + g, i); G fastest so that the warps of
// one query read adjacent partial rows.
template <int D>
__global__ void __launch_bounds__(256) fsa_combine_kernel(const int32_t* __restrict__ block_idx,
                                                          const float* __restrict__ acc,
                                                          const float* __restrict__ pm,
                                                          const float* __restrict__ pl,
                                                          __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                                          long long n_rows, int G, int Hkv, int T, int S,
                                                          int n_blk) {
  constexpr int V = D / 32;  // floats per lane
  const long long wid = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= n_rows) return;
  const int g = static_cast<int>(wid % G);
  const int i = static_cast<int>((wid / G) % T);
  const long long bh = wid / (static_cast<long long>(G) * T);
  const long long srow = (bh * T + i) * S;  // first slot of (b, hkv, i)
  // The slots that formed a pair (the first occurrence of each causal block).
  const unsigned mask = nsa_live_slots(block_idx + srow, S, i, n_blk, FSA_BS).live;
  const bool live = (mask >> lane) & 1u;
  float m = -INFINITY, l = 0.0f;
  if (live) {
    m = pm[(srow + lane) * G + g];
    l = pl[(srow + lane) * G + g];
  }
  float M = m;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, d));
  const float wgt = live ? ex2f((m - M) * 1.4426950408889634f) : 0.0f;
  float Lsum = wgt * l;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, d);
  float o[V];
#pragma unroll
  for (int x = 0; x < V; ++x) o[x] = 0.0f;
  for (unsigned mm = mask; mm != 0u; mm &= mm - 1u) {
    const int s = __ffs(mm) - 1;
    const float ws = __shfl_sync(0xffffffffu, wgt, s);
    const float* a = acc + ((srow + s) * G + g) * D + lane * V;
    if constexpr (V == 4) {
      const float4 v = *reinterpret_cast<const float4*>(a);
      o[0] = fmaf(ws, v.x, o[0]);
      o[1] = fmaf(ws, v.y, o[1]);
      o[2] = fmaf(ws, v.z, o[2]);
      o[3] = fmaf(ws, v.w, o[3]);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(a);
      o[0] = fmaf(ws, v.x, o[0]);
      o[1] = fmaf(ws, v.y, o[1]);
    }
  }
  const float inv = mask != 0u ? 1.0f / Lsum : 0.0f;
  const long long b = bh / Hkv, hkv = bh % Hkv;
  const long long orow = ((b * Hkv + hkv) * G + g) * T + i;  // [B, Hq, T] with hq = hkv * G + g
  __nv_bfloat16* dst = out + orow * D + lane * V;
  if constexpr (V == 4) {
    uint2 u;
    u.x = pack_bf16x2(o[0] * inv, o[1] * inv);
    u.y = pack_bf16x2(o[2] * inv, o[3] * inv);
    *reinterpret_cast<uint2*>(dst) = u;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(o[0] * inv, o[1] * inv);
  }
  if (lse != nullptr && lane == 0) lse[orow] = mask != 0u ? M + logf(Lsum) : -1.0e9f;
}

// ------------------------------------------------------------ workspace plan

struct FsaPlan {
  long long slots, rows;  // B*Hkv*T*S partial slots; rows = slots * G
  long long NB;           // B*Hkv*n_blk blocks
  long long max_items;
  int qch;                // queries per work item
  size_t acc_off, pm_off, pl_off, list_off, off_off, cnt_off, item_off, meta_off, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

FsaPlan fsa_plan(int B, int Hq, int Hkv, int T, int D, int S) {
  FsaPlan p{};
  const int G = Hq / Hkv;
  p.slots = static_cast<long long>(B) * Hkv * T * S;
  p.rows = p.slots * G;
  p.NB = static_cast<long long>(B) * Hkv * (T / FSA_BS);
  p.qch = FSA_ITEM_TILES * (FSA_M / G);
  p.max_items = (p.slots + p.qch - 1) / p.qch + p.NB;
  size_t o = 0;
  p.acc_off = o;  o = align256(o + static_cast<size_t>(p.rows) * D * sizeof(float));
  p.pm_off = o;   o = align256(o + static_cast<size_t>(p.rows) * sizeof(float));
  p.pl_off = o;   o = align256(o + static_cast<size_t>(p.rows) * sizeof(float));
  p.list_off = o; o = align256(o + static_cast<size_t>(p.slots) * sizeof(int));
  p.off_off = o;  o = align256(o + static_cast<size_t>(p.NB + 1) * sizeof(int));
  p.cnt_off = o;  o = align256(o + static_cast<size_t>(p.NB) * sizeof(int));
  p.item_off = o; o = align256(o + static_cast<size_t>(p.max_items) * sizeof(int4));
  p.meta_off = o; o = align256(o + 4 * sizeof(int));
  p.total = o;
  return p;
}

template <int D>
int launch_fsa(const void* q, const void* k, const void* v, const int32_t* block_idx, void* out, float* lse,
               int B, int Hq, int Hkv, int T, int S, uint8_t* ws, cudaStream_t stream) {
  using L = FsaLayout<D>;
  const FsaPlan pl = fsa_plan(B, Hq, Hkv, T, D, S);
  const int G = Hq / Hkv, n_blk = T / FSA_BS;
  float* acc = reinterpret_cast<float*>(ws + pl.acc_off);
  float* pmv = reinterpret_cast<float*>(ws + pl.pm_off);
  float* plv = reinterpret_cast<float*>(ws + pl.pl_off);
  int* list = reinterpret_cast<int*>(ws + pl.list_off);
  int* off = reinterpret_cast<int*>(ws + pl.off_off);
  int* cnt = reinterpret_cast<int*>(ws + pl.cnt_off);
  int4* items = reinterpret_cast<int4*>(ws + pl.item_off);
  int* meta = reinterpret_cast<int*>(ws + pl.meta_off);

  CUtensorMap mk, mv;
  const uint64_t rs = static_cast<uint64_t>(D) * 2, hs = rs * T;
  int st = encode_tmap_3d(&mk, k, D, T, static_cast<uint64_t>(B) * Hkv, rs, hs, 64, FSA_BS, 1);
  if (st == OK) st = encode_tmap_3d(&mv, v, D, T, static_cast<uint64_t>(B) * Hkv, rs, hs, 64, FSA_BS, 1);
  if (st != OK) return st;

  auto grid_for = [](long long n, int threads) {
    return static_cast<unsigned>(std::min<long long>((n + threads - 1) / threads, 148LL * 64));
  };
  fsa_zero_kernel<<<grid_for(pl.NB, 256), 256, 0, stream>>>(cnt, static_cast<int>(pl.NB), meta);
  const long long idx_rows = pl.slots / S;  // one warp per index row
  fsa_pairs_kernel<false><<<grid_for(idx_rows * 32, 256), 256, 0, stream>>>(block_idx, cnt, list, idx_rows, T, S,
                                                                             n_blk);
  fsa_scan_kernel<<<1, SCAN_THREADS, 0, stream>>>(cnt, off, items, meta, static_cast<int>(pl.NB), pl.qch);
  fsa_pairs_kernel<true><<<grid_for(idx_rows * 32, 256), 256, 0, stream>>>(block_idx, cnt, list, idx_rows, T, S,
                                                                            n_blk);

  // G = 8 or 16: each query's G partial rows are contiguous, so they leave by
  // TMA tensor stores (fp32 [rows, D] map, 32 x G boxes).
  const bool tma_out = G == 8 || G == 16;
  CUtensorMap macc = mk;  // unused unless tma_out
  if (tma_out) {
    st = encode_tmap_2d_f32(&macc, acc, D, static_cast<uint64_t>(pl.rows), static_cast<uint64_t>(D) * 4, 32,
                            static_cast<uint32_t>(G));
    if (st != OK) return st;
  }
  auto kern = tma_out ? fsa_blockouter_kernel<D, true> : fsa_blockouter_kernel<D, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC) != cudaSuccess)
    return ERR_LAUNCH;
  if (pl.max_items > 0x7fffffffLL) return ERR_SHAPE;
  kern<<<static_cast<unsigned>(pl.max_items), FSA_THREADS, L::ALLOC, stream>>>(
      mk, mv, macc, static_cast<const __nv_bfloat16*>(q), list, items, meta, acc, pmv, plv, G, Hq, Hkv, T, S,
      n_blk, 1.0f / sqrtf(static_cast<float>(D)));

  const long long warps = static_cast<long long>(B) * Hq * T;
  const long long blocks = (warps * 32 + 255) / 256;
  if (blocks > 0x7fffffffLL) return ERR_SHAPE;
  fsa_combine_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      block_idx, acc, pmv, plv, static_cast<__nv_bfloat16*>(out), lse, warps, G, Hkv, T, S, n_blk);
  return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
}

}  // namespace

size_t nsa_fsa_workspace_bytes(int B, int Hq, int Hkv, int T, int D, int S) {
  return fsa_plan(B, Hq, Hkv, T, D, S).total;
}

int launch_nsa_fsa(const void* q, const void* k, const void* v, const int32_t* block_idx, void* out, float* lse,
                   int B, int Hq, int Hkv, int T, int D, int S, void* workspace, cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (D == 128) return launch_fsa<128>(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, S, ws, stream);
  if (D == 64) return launch_fsa<64>(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, S, ws, stream);
  return ERR_UNSUPPORTED;
}

unsigned int nsa_fsa_device_error() { return read_and_clear_device_error(); }

}  // namespace bsa
