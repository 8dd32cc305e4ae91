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
// One CTA of four warps per query group at a time (persistent grid).  The
// group's G heads are the 16 rows of mma.sync.m16n8k16 (rows >= G zero).  The
// causal tokens of its live blocks are cut into 16-token chunks (block sizes
// are multiples of 16, so a chunk never straddles two blocks) and dealt to
// the warps round-robin.  Each warp brings its chunks' K and V rows into its
// own double-buffered shared memory with cp.async (deeper rings measured
// slower: the shared memory they take costs more resident CTAs per SM than the
// extra chunks in flight give back), computes S = Q K^T, an
// online softmax with lazy rescaling and O += P V in registers; the four
// states are merged through shared memory at the end of the query.  Rows are
// padded to D + 8 elements so that ldmatrix reads are free of bank conflicts.
#include "kernels.h"
#include "mma_sync.cuh"
#include "nsa_slots.cuh"
#include "ptx.cuh"

namespace bsa {
namespace {

constexpr int GEN_WARPS = 4;
constexpr int GEN_THREADS = GEN_WARPS * 32;
constexpr int GEN_CHUNK = 16;  // tokens per chunk

template <int D>
struct GenLayout {
  static constexpr int RS = D + 8;                       // padded row (bf16 elements)
  static constexpr int RB = RS * 2;                      // padded row in bytes
  static constexpr int Q_OFF = 0;                        // [16][RS] bf16
  static constexpr int KV_OFF = Q_OFF + 16 * RB;         // [warp][buf][K|V][16][RS]
  static constexpr int KV_WARP = 2 * 2 * 16 * RB;
  static constexpr int CST = D + 4;                      // combine row stride (floats)
  static constexpr int C_OFF = KV_OFF + GEN_WARPS * KV_WARP;             // fp32 [4][16][CST]
  static constexpr int ML_OFF = C_OFF + GEN_WARPS * 16 * CST * 4;        // fp32 [4][16][2]
  static constexpr int BYTES = ML_OFF + GEN_WARPS * 16 * 2 * 4;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void gen_sync() { asm volatile("bar.sync 1, %0;" ::"n"(GEN_THREADS)); }

// Walks the 16-token chunks of one query's live blocks (nsa_slots.cuh) in
// slot order.  A warp takes chunks warp, warp + 4, ...; `tok0` is the chunk's
// first token.  Every lane of the warp steps it alike.
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
      nc = (last - first) / GEN_CHUNK + 1;
      tok0 = first;
      c = 0;
      valid = true;
      return;
    }
    valid = false;
  }
  __device__ __forceinline__ void step() {
    if (++c < nc) {
      tok0 += GEN_CHUNK;
    } else {
      ++s;
      seek_slot();
    }
  }
  // n steps at once: whole blocks are skipped instead of walked chunk by chunk.
  __device__ __forceinline__ void advance(int n) {
    while (valid) {
      const int left = nc - c;  // chunks of this block from c on
      if (n < left) {
        c += n;
        tok0 += n * GEN_CHUNK;
        return;
      }
      n -= left;
      ++s;
      seek_slot();
      if (n == 0) return;
    }
  }
};

template <int D>
__global__ void __launch_bounds__(GEN_THREADS)
    nsa_general_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                       const __nv_bfloat16* __restrict__ v, const int32_t* __restrict__ block_idx,
                       __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int Hq, int Hkv, int G, int T,
                       int S, int bs, long long n_queries, float scale_log2) {
  using L = GenLayout<D>;
  extern __shared__ __align__(16) uint8_t smem[];
  float* comb = reinterpret_cast<float*>(smem + L::C_OFF);
  float* ml = reinterpret_cast<float*>(smem + L::ML_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;  // fragment row (and row + 8) / column pair
  const int mat = lane >> 3, mrow = lane & 7;
  const int n_blk = T / bs;
  const uint32_t sQ = smem_u32(smem + L::Q_OFF);
  const uint32_t sKV = smem_u32(smem + L::KV_OFF + warp * L::KV_WARP);
  constexpr int CPR = D / 8;  // 16-byte pieces per row

  // Q rows G..15 stay zero for the whole kernel.
  for (int e = threadIdx.x; e < 16 * L::RB / 16; e += GEN_THREADS)
    reinterpret_cast<uint4*>(smem + L::Q_OFF)[e] = make_uint4(0, 0, 0, 0);
  gen_sync();

  for (long long qg = blockIdx.x; qg < n_queries; qg += gridDim.x) {
    const int i = static_cast<int>(qg % T);
    const long long bg = qg / T;  // b * Hkv + hkv
    const int b = static_cast<int>(bg / Hkv), hkv = static_cast<int>(bg % Hkv);
    const __nv_bfloat16* kb = k + static_cast<size_t>(bg) * T * D;
    const __nv_bfloat16* vb = v + static_cast<size_t>(bg) * T * D;

    // ---- Q rows of the group into smem (row r = head hkv * G + r)
    for (int e = threadIdx.x; e < G * CPR; e += GEN_THREADS) {
      const int r = e / CPR, c = e % CPR;
      const int hq = debug_index(hkv * G + r, 0, Hq);
      const uint4 val = *reinterpret_cast<const uint4*>(
          q + ((static_cast<size_t>(b) * Hq + hq) * T + debug_index(i, 0, T)) * D + c * 8);
      *reinterpret_cast<uint4*>(smem + L::Q_OFF + r * L::RB + c * 16) = val;
    }
    gen_sync();
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

    // K and V rows of one chunk into buffer `buf` of this warp.
    auto load_chunk = [&](int tok0, int buf) {
      const uint32_t dk = sKV + buf * 2 * 16 * L::RB, dv = dk + 16 * L::RB;
      for (int e = lane; e < 16 * CPR; e += 32) {
        const int r = e / CPR, c = e % CPR;
        const size_t off = static_cast<size_t>(debug_index(tok0 + r, 0, T)) * D + c * 8;
        cp_async16(dk + r * L::RB + c * 16, kb + off);
        cp_async16(dv + r * L::RB + c * 16, vb + off);
      }
    };

    ChunkIter cur{nsa_live_slots(block_idx + qg * S, S, i, n_blk, bs), i, bs, 0, 0, 0, 0, false};
    cur.seek_slot();
    cur.advance(warp);
    ChunkIter nxt = cur;
    nxt.advance(GEN_WARPS);
    if (cur.valid) load_chunk(cur.tok0, 0);
    cp_async_commit();
    for (int it = 0; cur.valid; ++it) {
      if (nxt.valid) load_chunk(nxt.tok0, (it + 1) & 1);
      cp_async_commit();
      cp_async_wait<1>();  // this chunk's copies have landed
      __syncwarp();
      const uint32_t sK = sKV + (it & 1) * 2 * 16 * L::RB, sV = sK + 16 * L::RB;
      const int tok0 = cur.tok0;

      // ---- S = Q K^T for tokens tok0 .. tok0+15 (two n8 tiles)
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int trow = 8 * (mat >> 1) + mrow;
        // From D = 64 on, even and odd k-steps go to two independent mma.sync
        // chains, summed at the end (as in the 64-token-block kernel, where it
        // measured 8% faster at D = 128; at D = 32 the two k-steps gain
        // nothing from it and it measured 3% slower).
        constexpr bool SPLIT = D >= 64;
        float sd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t b00, b01, b10, b11;
          ldsm_x4(sK + trow * L::RB + (16 * ks + 8 * (mat & 1)) * 2, b00, b01, b10, b11);
          if (SPLIT && (ks & 1)) {
            mma16816(sd[0], qa[ks], b00, b01);
            mma16816(sd[1], qa[ks], b10, b11);
          } else {
            mma16816(sc[0], qa[ks], b00, b01);
            mma16816(sc[1], qa[ks], b10, b11);
          }
        }
        if constexpr (SPLIT) {
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[j][e] += sd[j][e];
        }
      }
      // ---- scale (log2 domain), causal mask, online softmax.  Only the chunk
      // holding token i has keys after it (a warp-uniform test).
      float mx0 = -INFINITY, mx1 = -INFINITY;
      if (tok0 + GEN_CHUNK - 1 <= i) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            sc[j][e] *= scale_log2;
            sc[j][2 + e] *= scale_log2;
            mx0 = fmaxf(mx0, sc[j][e]);
            mx1 = fmaxf(mx1, sc[j][2 + e]);
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const bool ok_key = tok0 + 8 * j + 2 * t + e <= i;
            sc[j][e] = ok_key ? sc[j][e] * scale_log2 : -INFINITY;
            sc[j][2 + e] = ok_key ? sc[j][2 + e] * scale_log2 : -INFINITY;
            mx0 = fmaxf(mx0, sc[j][e]);
            mx1 = fmaxf(mx1, sc[j][2 + e]);
          }
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      // Keep the running max unless a new score exceeds it by more than 8
      // (log2 units) in some row of the warp: exp2(s - m) stays below 2^8.
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
      // ---- O += P V over this chunk (k = 16 tokens)
      {
        const int vrow = 8 * (mat & 1) + mrow;
#pragma unroll
        for (int jj = 0; jj < D / 16; ++jj) {
          uint32_t v0, v1, v2, v3;
          ldsm_x4_t(sV + vrow * L::RB + (16 * jj + 8 * (mat >> 1)) * 2, v0, v1, v2, v3);
          mma16816(acc[2 * jj], pa, v0, v1);
          mma16816(acc[2 * jj + 1], pa, v2, v3);
        }
      }
      __syncwarp();  // the buffer is refilled two chunks later
      cur = nxt;
      nxt.advance(GEN_WARPS);
    }
    cp_async_wait<0>();

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
    gen_sync();
    {
      constexpr int PER = D / 8;  // output elements per thread: 8 threads per head row
      const int row = threadIdx.x >> 3;
      const int d0 = (threadIdx.x & 7) * PER;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < GEN_WARPS; ++w) M = fmaxf(M, ml[(w * 16 + row) * 2]);
      float wsum = 0.0f, wt[GEN_WARPS];
#pragma unroll
      for (int w = 0; w < GEN_WARPS; ++w) {
        wt[w] = (M == -INFINITY) ? 0.0f : ex2f(ml[(w * 16 + row) * 2] - M);
        wsum += wt[w] * ml[(w * 16 + row) * 2 + 1];
      }
      const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
      if (row < G) {
        const int h = hkv * G + row;
        uint32_t* dst = reinterpret_cast<uint32_t*>(out + ((static_cast<size_t>(b) * Hq + h) * T + i) * D + d0);
#pragma unroll
        for (int e = 0; e < PER; e += 2) {
          float o0 = 0.f, o1 = 0.f;
#pragma unroll
          for (int w = 0; w < GEN_WARPS; ++w) {
            o0 += wt[w] * comb[(w * 16 + row) * L::CST + d0 + e];
            o1 += wt[w] * comb[(w * 16 + row) * L::CST + d0 + e + 1];
          }
          dst[e / 2] = pack_bf16x2(o0 * inv, o1 * inv);
        }
        if (lse != nullptr && (threadIdx.x & 7) == 0)
          lse[(static_cast<size_t>(b) * Hq + h) * T + i] =
              wsum > 0.0f ? (M + __log2f(wsum)) * 0.69314718055994531f : -1.0e9f;
      }
    }
    gen_sync();  // Q buffer and combine area are reused by the next query
  }
}

template <int D>
int launch_general(const void* q, const void* k, const void* v, const int32_t* idx, void* out, float* lse, int B,
                   int Hq, int Hkv, int T, int bs, int S, cudaStream_t stream) {
  using L = GenLayout<D>;
  auto kern = nsa_general_kernel<D>;
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
  const long long grid = nq < cap ? nq : cap;
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
  switch (D) {
    case 16: return launch_general<16>(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, block_size, S, stream);
    case 32: return launch_general<32>(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, block_size, S, stream);
    case 64: return launch_general<64>(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, block_size, S, stream);
    case 128: return launch_general<128>(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, block_size, S, stream);
    default: return ERR_UNSUPPORTED;
  }
}

}  // namespace bsa
