// nsa_select.cu -- NSA selection-branch attention forward (bf16 in, fp32
// softmax state, bf16 out, fp32 lse).
//
// Method: page "nsa_selection_kernel.py" (module docstring "The operation",
// selection_forward_reference, _selection_fwd_kernel): for query i of kv
// group (b, hkv), the G query heads attend to the tokens j <= i of the blocks
// listed in block_idx[b, hkv, i, :] (-1 = padding), softmax with scale
// D^-0.5; no valid token -> out 0 and lse -1e9; lse = m + ln l.
//
// Gather, not scan: each selected block is fetched as one 64-token K tile and
// one V tile by TMA (box 64 x 64 of a [B*Hkv, T, D] tensor map, 128-byte
// swizzle) into a 2-stage ring per CTA.  The G heads of the group are the 16
// rows of mma.sync.m16n8k16 (rows >= G are zero).  Four consumer warps split
// every 64-token block into 16-token slices, each keeping its own online-
// softmax state (running max m, partial sum l, 16 x D accumulator); at the end
// of a query the four states are merged through shared memory.  A fifth warp
// is the TMA producer.  The grid is persistent with two CTAs per SM: CTA c
// takes query groups c, c + gridDim.x, ...
#include "kernels.h"
#include "mma_sync.cuh"
#include "nsa_slots.cuh"
#include "ptx.cuh"

namespace bsa {
namespace {

constexpr int NSA_BS = 64;        // tokens per selected block
constexpr int NSA_CONSUMERS = 4;  // consumer warps (16 tokens each)
constexpr int NSA_THREADS = (NSA_CONSUMERS + 1) * 32;
constexpr int NSA_NS = 2;         // K/V stages per CTA (two CTAs per SM)
constexpr int NSA_NQ = 2;         // Q stages

template <int D>
struct NsaLayout {
  static constexpr int NP = D / 64;
  static constexpr int KV_PANEL = NSA_BS * 128;        // 64 tokens x 128 B
  static constexpr int KV_TILE = NP * KV_PANEL;        // one K (or V) block
  static constexpr int Q_PANEL = 16 * 128;             // 16 rows x 128 B
  static constexpr int Q_TILE = NP * Q_PANEL;
  static constexpr int CST = D + 8;                    // combine row stride (floats)
  static constexpr int KV_OFF = 0;
  static constexpr int Q_OFF = KV_OFF + NSA_NS * 2 * KV_TILE;
  static constexpr int C_OFF = Q_OFF + NSA_NQ * Q_TILE;           // fp32 [4][16][CST]
  static constexpr int ML_OFF = C_OFF + NSA_CONSUMERS * 16 * CST * 4;  // fp32 [4][16][2]
  static constexpr int BAR_OFF = ML_OFF + NSA_CONSUMERS * 16 * 2 * 4;
  static constexpr int NBAR = 2 * NSA_NS + 2 * NSA_NQ;
  static constexpr int BYTES = BAR_OFF + NBAR * 8;
  static constexpr int ALLOC = BYTES + 1024;
};

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(NSA_CONSUMERS * 32)); }

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a panel of
// 128-byte rows written by TMA with 128-byte swizzle (1024-byte aligned).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(NSA_THREADS, 2)
    nsa_select_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const int32_t* __restrict__ block_idx,
                      __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int Hq, int Hkv, int G, int T,
                      int S, long long n_queries, float scale_log2) {
  using L = NsaLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* kv_empty = kv_full + NSA_NS;
  uint64_t* q_full = kv_empty + NSA_NS;
  uint64_t* q_empty = q_full + NSA_NQ;
  float* comb = reinterpret_cast<float*>(smem + L::C_OFF);
  float* ml = reinterpret_cast<float*>(smem + L::ML_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_blk = T / NSA_BS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSA_NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], NSA_CONSUMERS);
    }
    for (int s = 0; s < NSA_NQ; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], NSA_CONSUMERS);
    }
    fence_barrier_init();
  }
  // Rows G..15 of every Q stage stay zero (TMA writes rows 0..G-1 only).
  for (int e = threadIdx.x; e < NSA_NQ * L::Q_TILE / 16; e += blockDim.x)
    reinterpret_cast<uint4*>(smem + L::Q_OFF)[e] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  __syncthreads();

  if (warp == NSA_CONSUMERS) {
    // ---------------------------------------------------------------- producer
    // The whole warp walks the queries (it computes each row's live slots
    // together); lane 0 waits on the ring and issues the copies.
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    int kv_it = 0, q_it = 0;
    bool ok = true;
    for (long long qg = blockIdx.x; qg < n_queries && ok; qg += gridDim.x) {
      const int i = static_cast<int>(qg % T);
      const long long bg = qg / T;  // b * Hkv + hkv
      const int b = static_cast<int>(bg / Hkv), hkv = static_cast<int>(bg % Hkv);
      const int qs = q_it % NSA_NQ;
      if (lane == 0 && (ok = mbar_wait(&q_empty[qs], ((q_it / NSA_NQ) & 1) ^ 1))) {
        debug_check(i >= 0 && i < T && bg >= 0 && bg < n_queries / T);
        mbar_arrive_expect_tx(&q_full[qs], static_cast<uint32_t>(L::NP * G * 128));
        uint8_t* sQ = smem + L::Q_OFF + qs * L::Q_TILE;
#pragma unroll
        for (int pnl = 0; pnl < L::NP; ++pnl)
          tma_load_3d(sQ + pnl * L::Q_PANEL, &tmQ, &q_full[qs], 64 * pnl, i, b * Hq + hkv * G);
      }
      if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;
      ++q_it;
      const SlotRow row = nsa_live_slots(block_idx + qg * S, S, i, n_blk, NSA_BS);
      for (uint32_t m = row.live; m != 0u && ok; m &= m - 1u) {
        const int blk = nsa_slot_block(row, __ffs(m) - 1);
        const int st = kv_it % NSA_NS;
        if (lane == 0 && (ok = mbar_wait(&kv_empty[st], ((kv_it / NSA_NS) & 1) ^ 1))) {
          debug_check(blk >= 0 && blk < n_blk && blk * NSA_BS <= i);
          mbar_arrive_expect_tx(&kv_full[st], 2 * L::KV_TILE);
          uint8_t* sK = smem + L::KV_OFF + st * 2 * L::KV_TILE;
          uint8_t* sV = sK + L::KV_TILE;
#pragma unroll
          for (int pnl = 0; pnl < L::NP; ++pnl) {
            tma_load_3d(sK + pnl * L::KV_PANEL, &tmK, &kv_full[st], 64 * pnl, blk * NSA_BS, static_cast<int>(bg));
            tma_load_3d(sV + pnl * L::KV_PANEL, &tmV, &kv_full[st], 64 * pnl, blk * NSA_BS, static_cast<int>(bg));
          }
        }
        if ((ok = __shfl_sync(0xffffffffu, ok, 0))) ++kv_it;
      }
    }
    // Drain whatever is still landing before the CTA may exit.
    if (lane == 0) {
      for (int n = (kv_it > NSA_NS ? kv_it - NSA_NS : 0); n < kv_it; ++n)
        mbar_wait(&kv_full[n % NSA_NS], (n / NSA_NS) & 1);
      for (int n = (q_it > NSA_NQ ? q_it - NSA_NQ : 0); n < q_it; ++n) mbar_wait(&q_full[n % NSA_NQ], (n / NSA_NQ) & 1);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int g = lane >> 2;  // fragment row (and row + 8)
  const int t = lane & 3;   // fragment column pair
  const int mat = lane >> 3, mrow = lane & 7;
  int kv_it = 0, q_it = 0;
  bool ok = true;
  for (long long qg = blockIdx.x; qg < n_queries; qg += gridDim.x) {
    const int i = static_cast<int>(qg % T);
    const long long bg = qg / T;
    const int b = static_cast<int>(bg / Hkv), hkv = static_cast<int>(bg % Hkv);

    // Q fragments (A operand) for all D/16 k-steps.
    const int qs = q_it % NSA_NQ;
    if (ok) ok = mbar_wait(&q_full[qs], (q_it / NSA_NQ) & 1);
    uint32_t qa[D / 16][4];
    {
      const uint32_t sQ = smem_u32(smem + L::Q_OFF + qs * L::Q_TILE);
      const int row = mrow + 8 * (mat & 1);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int chunk = 2 * (ks & 3) + (mat >> 1);
        ldsm_x4(sQ + (ks >> 2) * L::Q_PANEL + swz(row, chunk), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&q_empty[qs]);
    ++q_it;

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    float acc[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;

    const SlotRow row = nsa_live_slots(block_idx + qg * S, S, i, n_blk, NSA_BS);
    for (uint32_t msk = row.live; msk != 0u; msk &= msk - 1u) {
      const int blk = nsa_slot_block(row, __ffs(msk) - 1);
      const int st = kv_it % NSA_NS;
      if (ok) ok = mbar_wait(&kv_full[st], (kv_it / NSA_NS) & 1);
      ++kv_it;
      const int tok0 = blk * NSA_BS + 16 * warp;  // first token of this warp's slice
      if (ok && tok0 <= i) {
        const uint32_t sK = smem_u32(smem + L::KV_OFF + st * 2 * L::KV_TILE);
        const uint32_t sV = sK + L::KV_TILE;
        // ---- S = Q K^T for tokens tok0 .. tok0+15 (two n8 tiles)
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          const int trow = 16 * warp + 8 * (mat >> 1) + mrow;  // token row in the block
          // Even and odd k-steps accumulate into separate fragments (two
          // independent mma.sync chains per tile instead of one; measured 8%
          // faster on both selection workloads), summed at the end.
          float sd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t b00, b01, b10, b11;
            const int chunk = 2 * (ks & 3) + (mat & 1);
            ldsm_x4(sK + (ks >> 2) * L::KV_PANEL + swz(trow, chunk), b00, b01, b10, b11);
            if (ks & 1) {
              mma16816(sd[0], qa[ks], b00, b01);
              mma16816(sd[1], qa[ks], b10, b11);
            } else {
              mma16816(sc[0], qa[ks], b00, b01);
              mma16816(sc[1], qa[ks], b10, b11);
            }
          }
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[j][e] += sd[j][e];
        }
        // ---- scale (log2 domain), causal mask, online softmax
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = tok0 + 8 * j + 2 * t + e;
            const bool ok_key = key <= i;
            sc[j][e] = ok_key ? sc[j][e] * scale_log2 : -INFINITY;
            sc[j][2 + e] = ok_key ? sc[j][2 + e] * scale_log2 : -INFINITY;
            mx0 = fmaxf(mx0, sc[j][e]);
            mx1 = fmaxf(mx1, sc[j][2 + e]);
          }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        // Lazy rescale: keep the running max unless a new score exceeds it
        // by more than 8 (log2 units) in some row of the warp; exp2(s - m)
        // then stays below 2^8 and the accumulator is rescaled only rarely.
        // The first live slice always rescales (m = -inf).
        if (__any_sync(0xffffffffu, mx0 > m0 + 8.0f || mx1 > m1 + 8.0f)) {
          const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);  // finite: tok0 <= i
          const float al0 = ex2f(m0 - mn0), al1 = ex2f(m1 - mn1);
          m0 = mn0;
          m1 = mn1;
          l0 *= al0;
          l1 *= al1;
#pragma unroll
          for (int j = 0; j < D / 8; ++j) {
            acc[j][0] *= al0;
            acc[j][1] *= al0;
            acc[j][2] *= al1;
            acc[j][3] *= al1;
          }
        }
        uint32_t pa[4];
        float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float p0 = ex2f(sc[j][0] - m0), p1 = ex2f(sc[j][1] - m0);
          const float p2 = ex2f(sc[j][2] - m1), p3 = ex2f(sc[j][3] - m1);
          rs0 += p0 + p1;
          rs1 += p2 + p3;
          pa[2 * j + 0] = pack_bf16x2(p0, p1);  // row g,     k = 8j + 2t
          pa[2 * j + 1] = pack_bf16x2(p2, p3);  // row g + 8, k = 8j + 2t
        }
        l0 += rs0;
        l1 += rs1;
        // ---- O += P V over this slice (k = 16 tokens)
        {
          const int vrow = 16 * warp + 8 * (mat & 1) + mrow;  // token row
#pragma unroll
          for (int jj = 0; jj < D / 16; ++jj) {
            const int d0 = 16 * jj + 8 * (mat >> 1);
            uint32_t v0, v1, v2, v3;
            ldsm_x4_t(sV + (d0 >> 6) * L::KV_PANEL + swz(vrow, (d0 & 63) >> 3), v0, v1, v2, v3);
            mma16816(acc[2 * jj], pa, v0, v1);
            mma16816(acc[2 * jj + 1], pa, v2, v3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&kv_empty[st]);
    }

    // ---- merge the four warps' states and write out / lse
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    float* cw = comb + warp * 16 * L::CST;
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      *reinterpret_cast<float2*>(cw + g * L::CST + 8 * j + 2 * t) = make_float2(acc[j][0], acc[j][1]);
      *reinterpret_cast<float2*>(cw + (g + 8) * L::CST + 8 * j + 2 * t) = make_float2(acc[j][2], acc[j][3]);
    }
    if (t == 0) {
      ml[(warp * 16 + g) * 2 + 0] = m0;
      ml[(warp * 16 + g) * 2 + 1] = l0;
      ml[(warp * 16 + g + 8) * 2 + 0] = m1;
      ml[(warp * 16 + g + 8) * 2 + 1] = l1;
    }
    consumer_sync();
    {
      constexpr int PER = D / 8;  // output elements per thread
      const int ctid = threadIdx.x;  // 0..127
      const int row = ctid >> 3;     // head within the group
      const int d0 = (ctid & 7) * PER;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NSA_CONSUMERS; ++w) M = fmaxf(M, ml[(w * 16 + row) * 2]);
      float wsum = 0.0f, wt[NSA_CONSUMERS];
#pragma unroll
      for (int w = 0; w < NSA_CONSUMERS; ++w) {
        const float mw = ml[(w * 16 + row) * 2];
        wt[w] = (M == -INFINITY) ? 0.0f : ex2f(mw - M);
        wsum += wt[w] * ml[(w * 16 + row) * 2 + 1];
      }
      const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
      if (row < G) {
        const int h = hkv * G + row;
        uint32_t pk[PER / 2];
#pragma unroll
        for (int e = 0; e < PER; e += 2) {
          float o0 = 0.f, o1 = 0.f;
#pragma unroll
          for (int w = 0; w < NSA_CONSUMERS; ++w) {
            o0 += wt[w] * comb[(w * 16 + row) * L::CST + d0 + e];
            o1 += wt[w] * comb[(w * 16 + row) * L::CST + d0 + e + 1];
          }
          pk[e / 2] = pack_bf16x2(o0 * inv, o1 * inv);
        }
        __nv_bfloat16* dst = out + ((static_cast<size_t>(b) * Hq + h) * T + i) * D + d0;
#pragma unroll
        for (int e = 0; e < PER / 8; ++e)
          reinterpret_cast<uint4*>(dst)[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        if (lse != nullptr && (ctid & 7) == 0) {
          lse[(static_cast<size_t>(b) * Hq + h) * T + i] =
              wsum > 0.0f ? (M + __log2f(wsum)) * 0.69314718055994531f : -1.0e9f;
        }
      }
    }
    consumer_sync();
  }
}

template <int D>
int launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const int32_t* idx, void* out,
           float* lse, int B, int Hq, int Hkv, int T, int S, cudaStream_t stream) {
  using L = NsaLayout<D>;
  auto kern = nsa_select_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC) != cudaSuccess)
    return ERR_LAUNCH;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ERR_DEVICE;
  const long long nq = static_cast<long long>(B) * Hkv * T;
  const long long grid = nq < 2 * sms ? nq : 2 * sms;  // two CTAs per SM
  const float scale_log2 = (1.0f / sqrtf(static_cast<float>(D))) * 1.4426950408889634f;
  kern<<<static_cast<unsigned>(grid), NSA_THREADS, L::ALLOC, stream>>>(
      mq, mk, mv, idx, static_cast<__nv_bfloat16*>(out), lse, Hq, Hkv, Hq / Hkv, T, S, nq, scale_log2);
  return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
}

}  // namespace

int launch_nsa_select(const void* q, const void* k, const void* v, const int32_t* block_idx, void* out, float* lse,
                      int B, int Hq, int Hkv, int T, int D, int block_size, int S, cudaStream_t stream) {
  // The TMA kernel serves 64-token blocks of 64 or 128 dims; every other
  // accepted shape runs the general kernel.
  if (block_size != NSA_BS || (D != 64 && D != 128))
    return launch_nsa_general(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, D, block_size, S, stream);
  const int G = Hq / Hkv;
  if (G < 1 || G > 16) return ERR_UNSUPPORTED;
  CUtensorMap mq, mk, mv;
  const uint64_t rs = static_cast<uint64_t>(D) * 2;
  const uint64_t hs = rs * T;
  int st = encode_tmap_3d(&mq, q, D, T, static_cast<uint64_t>(B) * Hq, rs, hs, 64, 1, G);
  if (st == OK) st = encode_tmap_3d(&mk, k, D, T, static_cast<uint64_t>(B) * Hkv, rs, hs, 64, NSA_BS, 1);
  if (st == OK) st = encode_tmap_3d(&mv, v, D, T, static_cast<uint64_t>(B) * Hkv, rs, hs, 64, NSA_BS, 1);
  if (st != OK) return st;
  if (D == 128) return launch<128>(mq, mk, mv, block_idx, out, lse, B, Hq, Hkv, T, S, stream);
  if (D == 64) return launch<64>(mq, mk, mv, block_idx, out, lse, B, Hq, Hkv, T, S, stream);
  return ERR_UNSUPPORTED;
}

unsigned int nsa_device_error() { return read_and_clear_device_error(); }

}  // namespace bsa
