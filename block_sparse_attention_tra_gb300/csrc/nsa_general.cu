// nsa_general.cu -- NSA selection-branch attention forward for every head
// dim and block size the page accepts (D in {16, 32, 64, 128}, block_size in
// {16, 32, 64, 128}); the TMA kernel of nsa_select.cu serves block_size 64
// with D in {64, 128}.
//
// Method: page "nsa_selection_kernel.py" (module docstring "The operation",
// selection_forward_reference, _selection_fwd_kernel): for query i of kv
// group (b, hkv), the G query heads attend to the tokens j <= i of the blocks
// listed in block_idx[b, hkv, i, :] (-1 = padding), softmax with scale
// D^-0.5; no valid token -> out 0 and lse -1e9; lse = m + ln l.
//
// One warp per query group at a time (persistent grid of four-warp CTAs,
// each warp on its own groups).  The group's G heads are the 16 rows of
// mma.sync.m16n8k16 (rows >= G zero).  The causal tokens of its live blocks
// are cut into 16-token chunks (32 at D <= 32 when the block size is a
// multiple of 32; a chunk never straddles two blocks); the warp brings each
// chunk's K and V rows into its own double-buffered shared memory with
// cp.async, computes S = Q K^T, an online softmax with lazy rescaling and
// O += P V in registers, and normalises and stores its rows from registers.  Rows are padded to D + 8
// elements so that ldmatrix reads are free of bank conflicts.  (Measured
// against four warps per group with a merge through shared memory: faster
// at every head dim and block size; deeper cp.async rings are slower: the
// shared memory they take costs more resident warps than the extra chunks in
// flight give back.)
#include "kernels.h"
#include "mma_sync.cuh"
#include "nsa_slots.cuh"
#include "ptx.cuh"

namespace bsa {
namespace {

#ifndef BSA_NSA_GEN_C32
#define BSA_NSA_GEN_C32 1  // 32-token chunks for D <= 32 where block_size allows (see launch_nsa_general)
#endif
constexpr int GEN_WARPS = 4;  // warps per CTA, each on its own query groups
constexpr int GEN_THREADS = GEN_WARPS * 32;
constexpr int GEN_CHUNK = 16;  // tokens per chunk (32 for D <= 32 where block_size allows)

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Walks the C-token chunks of one query's live blocks (nsa_slots.cuh) in
// slot order; `tok0` is the chunk's first token.  Every lane of the warp
// steps it alike.
template <int C>
struct ChunkIter {
  SlotRow row;
  int i, bs;
  int s, c, nc;  // slot, chunk in block, chunks of that block (causal part only)
  int tok0;
  bool valid;

  __device__ __forceinline__ void seek_slot() {  // from slot s onwards, c = 0
    const uint32_t rest = s < 32 ? row.live & ~((1u << s) - 1u) : 0u;
    if (rest != 0u) {
      s = __ffs(rest) - 1;
      const int blk = nsa_slot_block(row, s);
      const int first = blk * bs;
      const int last = min(first + bs - 1, i);
      nc = (last - first) / C + 1;
      tok0 = first;
      c = 0;
      valid = true;
      return;
    }
    valid = false;
  }
  __device__ __forceinline__ void step() {
    if (++c < nc) {
      tok0 += C;
    } else {
      ++s;
      seek_slot();
    }
  }
};

// Per-warp shared memory: the group's Q rows and a ring of NB chunks.
template <int D, int NB, int C>
struct GenLayout {
  static constexpr int RS = D + 8;                  // padded row (bf16 elements)
  static constexpr int RB = RS * 2;                 // padded row in bytes
  static constexpr int Q_BYTES = 16 * RB;           // [16][RS] bf16, rows >= G zero
  static constexpr int STAGE = 2 * C * RB;          // K rows, then V rows, of one chunk
  static constexpr int WARP_BYTES = Q_BYTES + NB * STAGE;
  static constexpr int BYTES = GEN_WARPS * WARP_BYTES;
};

// The minimum CTAs per SM are what each form's shared memory and registers
// allow at once; without them the compiler takes more registers than that
// occupancy leaves (139 instead of 64 at D = 16).
template <int D, int C>
constexpr int gen_min_ctas() {
  if constexpr (C == 32) return D == 16 ? 6 : 4;
  return D == 16 ? 8 : D == 32 ? 7 : D == 64 ? 4 : 2;
}

template <int D, int NB, int C>
__global__ void __launch_bounds__(GEN_THREADS, gen_min_ctas<D, C>())
    nsa_general_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                       const __nv_bfloat16* __restrict__ v, const int32_t* __restrict__ block_idx,
                       __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int Hq, int Hkv, int G, int T,
                       int S, int bs, long long n_queries, float scale_log2) {
  using L = GenLayout<D, NB, C>;
  static_assert(NB >= 2, "at least double buffering");
  static_assert(C == 16 || C == 32, "16 or 32 tokens per chunk");
  constexpr int NT = C / 8;  // n8 tiles of a chunk's scores
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;  // fragment row (and row + 8) / column pair
  const int mat = lane >> 3, mrow = lane & 7;
  const int n_blk = T / bs;
  uint8_t* wq = smem + warp * L::WARP_BYTES;
  const uint32_t sQ = smem_u32(wq), sKV = sQ + L::Q_BYTES;
  constexpr int CPR = D / 8;  // 16-byte pieces per row

  for (int e = lane; e < L::Q_BYTES / 16; e += 32) reinterpret_cast<uint4*>(wq)[e] = make_uint4(0, 0, 0, 0);
  __syncwarp();

  const long long stride = static_cast<long long>(gridDim.x) * GEN_WARPS;
  for (long long qg = static_cast<long long>(blockIdx.x) * GEN_WARPS + warp; qg < n_queries; qg += stride) {
    const int i = static_cast<int>(qg % T);
    const long long bg = qg / T;  // b * Hkv + hkv
    const int b = static_cast<int>(bg / Hkv), hkv = static_cast<int>(bg % Hkv);
    const __nv_bfloat16* kb = k + static_cast<size_t>(bg) * T * D;
    const __nv_bfloat16* vb = v + static_cast<size_t>(bg) * T * D;

    // K and V rows of one chunk into ring slot `buf`.
    auto load_chunk = [&](int tok0, int buf) {
      const uint32_t dk = sKV + buf * L::STAGE, dv = dk + C * L::RB;
      for (int e = lane; e < C * CPR; e += 32) {
        const int r = e / CPR, c = e % CPR;
        const size_t off = static_cast<size_t>(debug_index(tok0 + r, 0, T)) * D + c * 8;
        cp_async16(dk + r * L::RB + c * 16, kb + off);
        cp_async16(dv + r * L::RB + c * 16, vb + off);
      }
    };
    ChunkIter<C> cur{nsa_live_slots(block_idx + qg * S, S, i, n_blk, bs), i, bs, 0, 0, 0, 0, false};
    cur.seek_slot();
    ChunkIter<C> pf = cur;  // the next chunk to load
#pragma unroll
    for (int st = 0; st < NB - 1; ++st) {
      if (pf.valid) {
        load_chunk(pf.tok0, st);
        pf.step();
      }
      cp_async_commit();
    }

    // ---- Q rows of the group (row r = head hkv * G + r), under the first loads
    for (int e = lane; e < G * CPR; e += 32) {
      const int r = e / CPR, c = e % CPR;
      const int hq = debug_index(hkv * G + r, 0, Hq);
      const uint4 val = *reinterpret_cast<const uint4*>(
          q + ((static_cast<size_t>(b) * Hq + hq) * T + debug_index(i, 0, T)) * D + c * 8);
      *reinterpret_cast<uint4*>(wq + r * L::RB + c * 16) = val;
    }
    __syncwarp();
    uint32_t qa[D / 16][4];
    {
      const int row = mrow + 8 * (mat & 1);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        ldsm_x4(sQ + row * L::RB + (16 * ks + 8 * (mat >> 1)) * 2, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
    }

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    float acc[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;

    for (int it = 0; cur.valid; ++it) {
      if (pf.valid) {
        load_chunk(pf.tok0, (it + NB - 1) % NB);
        pf.step();
      }
      cp_async_commit();
      cp_async_wait<NB - 1>();  // this chunk's copies have landed
      __syncwarp();
      const uint32_t sK = sKV + (it % NB) * L::STAGE, sV = sK + C * L::RB;
      const int tok0 = cur.tok0;

      // ---- S = Q K^T for tokens tok0 .. tok0+C-1 (NT n8 tiles, 16 tokens per ldmatrix group)
      float sc[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
      {
        // From D = 64 on, even and odd k-steps go to two independent mma.sync
        // chains, summed at the end (8% faster at D = 128 in the 64-token-block
        // kernel; at D = 32 the two k-steps gain nothing from it).
        constexpr bool SPLIT = D >= 64;
#pragma unroll
        for (int hh = 0; hh < C / 16; ++hh) {
          const int trow = 16 * hh + 8 * (mat >> 1) + mrow;
          float sd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t b00, b01, b10, b11;
            ldsm_x4(sK + trow * L::RB + (16 * ks + 8 * (mat & 1)) * 2, b00, b01, b10, b11);
            if (SPLIT && (ks & 1)) {
              mma16816(sd[0], qa[ks], b00, b01);
              mma16816(sd[1], qa[ks], b10, b11);
            } else {
              mma16816(sc[2 * hh], qa[ks], b00, b01);
              mma16816(sc[2 * hh + 1], qa[ks], b10, b11);
            }
          }
          if constexpr (SPLIT) {
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int e = 0; e < 4; ++e) sc[2 * hh + j][e] += sd[j][e];
          }
        }
      }
      // ---- scale (log2 domain), causal mask on the chunk holding token i, online softmax
      float mx0 = -INFINITY, mx1 = -INFINITY;
      const bool full = tok0 + C - 1 <= i;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool ok_key = full || tok0 + 8 * j + 2 * t + e <= i;
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
      // lazy rescale: keep the running max unless a new score exceeds it by 8
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
      uint32_t pa[C / 16][4];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const float p0 = ex2f(sc[j][0] - m0), p1 = ex2f(sc[j][1] - m0);
        const float p2 = ex2f(sc[j][2] - m1), p3 = ex2f(sc[j][3] - m1);
        l0 += p0 + p1;
        l1 += p2 + p3;
        pa[j >> 1][2 * (j & 1) + 0] = pack_bf16x2(p0, p1);  // row g,     k = 8j + 2t
        pa[j >> 1][2 * (j & 1) + 1] = pack_bf16x2(p2, p3);  // row g + 8, k = 8j + 2t
      }
      // ---- O += P V over this chunk (k-steps of 16 tokens)
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk) {
        const int vrow = 16 * kk + 8 * (mat & 1) + mrow;
#pragma unroll
        for (int jj = 0; jj < D / 16; ++jj) {
          uint32_t v0, v1, v2, v3;
          ldsm_x4_t(sV + vrow * L::RB + (16 * jj + 8 * (mat >> 1)) * 2, v0, v1, v2, v3);
          mma16816(acc[2 * jj], pa[kk], v0, v1);
          mma16816(acc[2 * jj + 1], pa[kk], v2, v3);
        }
      }
      __syncwarp();  // this ring slot is refilled by the next iteration's load
      cur.step();
    }
    cp_async_wait<0>();

    // ---- normalise and store rows g and g + 8 (heads hkv * G + row, rows < G)
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = l0 > 0.0f ? 1.0f / l0 : 0.0f, inv1 = l1 > 0.0f ? 1.0f / l1 : 0.0f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int row = g + 8 * half;
      if (row < G) {
        const int h = hkv * G + row;
        const size_t ro = (static_cast<size_t>(b) * Hq + h) * T + i;
        uint32_t* dst = reinterpret_cast<uint32_t*>(out + ro * D);
        const float inv = half ? inv1 : inv0;
#pragma unroll
        for (int j = 0; j < D / 8; ++j)
          dst[4 * j + t] = pack_bf16x2(acc[j][2 * half] * inv, acc[j][2 * half + 1] * inv);
        if (lse != nullptr && t == 0) {
          const float l = half ? l1 : l0, m = half ? m1 : m0;
          lse[ro] = l > 0.0f ? (m + __log2f(l)) * 0.69314718055994531f : -1.0e9f;
        }
      }
    }
    __syncwarp();  // Q rows are rewritten by the next query group
  }
}

template <int D, int NB, int C = GEN_CHUNK>
int launch_general(const void* q, const void* k, const void* v, const int32_t* idx, void* out, float* lse, int B,
                   int Hq, int Hkv, int T, int bs, int S, cudaStream_t stream) {
  using L = GenLayout<D, NB, C>;
  auto kern = nsa_general_kernel<D, NB, C>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES) != cudaSuccess)
    return ERR_LAUNCH;
  const int sms = sm_count();
  if (sms <= 0) return ERR_DEVICE;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, GEN_THREADS, L::BYTES) != cudaSuccess ||
      per_sm < 1)
    return ERR_LAUNCH;
  const long long nq = static_cast<long long>(B) * Hkv * T;
  const long long cap = static_cast<long long>(sms) * per_sm;
  const long long need = (nq + GEN_WARPS - 1) / GEN_WARPS;
  const long long grid = need < cap ? need : cap;
  const float scale_log2 = (1.0f / sqrtf(static_cast<float>(D))) * 1.4426950408889634f;
  kern<<<static_cast<unsigned>(grid), GEN_THREADS, L::BYTES, stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), idx, static_cast<__nv_bfloat16*>(out), lse, Hq, Hkv, Hq / Hkv, T, S, bs,
      nq, scale_log2);
  return cudaGetLastError() == cudaSuccess ? OK : ERR_LAUNCH;
}

}  // namespace

int launch_nsa_general(const void* q, const void* k, const void* v, const int32_t* block_idx, void* out, float* lse,
                       int B, int Hq, int Hkv, int T, int D, int block_size, int S, cudaStream_t stream) {
  const int G = Hq / Hkv;
  if (G < 1 || G > 16 || block_size < GEN_CHUNK || block_size % GEN_CHUNK != 0) return ERR_UNSUPPORTED;
  // D <= 32 with block_size a multiple of 32: 32-token chunks, half the
  // per-chunk work (slot walk, masks, rescale test) per token (measured 3-4%
  // faster; at D = 64 the doubled ring costs half the resident warps).
  const bool c32 = BSA_NSA_GEN_C32 && block_size % 32 == 0;
  switch (D) {
    case 16:
      return c32 ? launch_general<16, 2, 32>(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, block_size, S, stream)
                 : launch_general<16, 2>(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, block_size, S, stream);
    case 32:
      return c32 ? launch_general<32, 2, 32>(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, block_size, S, stream)
                 : launch_general<32, 2>(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, block_size, S, stream);
    case 64: return launch_general<64, 2>(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, block_size, S, stream);
    case 128: return launch_general<128, 2>(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, block_size, S, stream);
    default: return ERR_UNSUPPORTED;
  }
}

}  // namespace bsa
