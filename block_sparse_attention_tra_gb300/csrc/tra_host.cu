// tra_host.cu -- threshold rectified attention forward on host-resident
// tensors: the (b, h) heads stream through the GPU in chunks, so that the
// host-to-device copies of one chunk, the kernel of the previous one and the
// device-to-host copy of the one before that run at the same time.
//
// Pipeline (chunk i uses workspace stage s = i mod 3):
//   copy-in stream : wait free[s]  -> q, k, v chunk i host -> stage s -> in[s]
//   compute stream : wait in[s]    -> TRA kernel on stage s          -> done[s]
//   copy-out stream: wait done[s]  -> out chunk i stage s -> host    -> free[s]
// The caller's stream is ordered before the first copy and after the last.
// The three streams and their events are created once per device and kept
// for the life of the process; a per-device mutex serialises the enqueueing
// of concurrent calls (each call's waits capture the event records made by
// that call, so calls sharing the streams stay correct).
#include <mutex>

#include "kernels.h"

namespace bsa {
namespace {

constexpr int HOST_STAGES = 3;
#ifndef BSA_HOST_CHUNKS
#define BSA_HOST_CHUNKS 8
#endif
constexpr int HOST_CHUNKS = BSA_HOST_CHUNKS;  // target number of chunks per call
constexpr int MAX_HOST_DEVICES = 64;

struct HostPipe {
  std::mutex m;
  bool ready = false;
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t entry = nullptr, in_ev[HOST_STAGES] = {}, done[HOST_STAGES] = {}, free_ev[HOST_STAGES] = {};
  cudaEvent_t tail[3] = {};
};
HostPipe g_pipes[MAX_HOST_DEVICES];

bool pipe_init(HostPipe& P) {
  if (P.ready) return true;
  const unsigned sf = cudaStreamNonBlocking, ef = cudaEventDisableTiming;
  if (cudaStreamCreateWithFlags(&P.in, sf) != cudaSuccess || cudaStreamCreateWithFlags(&P.comp, sf) != cudaSuccess ||
      cudaStreamCreateWithFlags(&P.out, sf) != cudaSuccess || cudaEventCreateWithFlags(&P.entry, ef) != cudaSuccess)
    return false;
  for (int s = 0; s < HOST_STAGES; ++s)
    if (cudaEventCreateWithFlags(&P.in_ev[s], ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&P.done[s], ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&P.free_ev[s], ef) != cudaSuccess)
      return false;
  for (int t = 0; t < 3; ++t)
    if (cudaEventCreateWithFlags(&P.tail[t], ef) != cudaSuccess) return false;
  P.ready = true;
  return true;
}

size_t round256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

}  // namespace

int tra_host_chunk_heads(long long BH) {
  const long long c = (BH + HOST_CHUNKS - 1) / HOST_CHUNKS;
  return static_cast<int>(c < 1 ? 1 : c);
}

size_t tra_host_workspace_bytes(long long BH, int T, int D, int elsize) {
  const size_t chunk = round256(static_cast<size_t>(tra_host_chunk_heads(BH)) * T * D * elsize);
  return static_cast<size_t>(HOST_STAGES) * 4 * chunk;
}

int launch_tra_host(const void* q, const void* k, const void* v, void* out, int B, int H, int T, int D, float beta,
                    float p, bool f32, void* workspace, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_HOST_DEVICES) return ERR_DEVICE;
  HostPipe& P = g_pipes[dev];
  std::lock_guard<std::mutex> lock(P.m);
  if (!pipe_init(P)) return ERR_LAUNCH;

  const long long BH = static_cast<long long>(B) * H;
  const int el = f32 ? 4 : 2;
  const int C = tra_host_chunk_heads(BH);
  const size_t head_bytes = static_cast<size_t>(T) * D * el;
  const size_t chunk = round256(static_cast<size_t>(C) * head_bytes);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const long long nchunks = (BH + C - 1) / C;

  bool ok = cudaEventRecord(P.entry, stream) == cudaSuccess && cudaStreamWaitEvent(P.in, P.entry, 0) == cudaSuccess;
  int st = OK;
  for (long long i = 0; ok && i < nchunks; ++i) {
    const int s = static_cast<int>(i % HOST_STAGES);
    const long long h0 = i * C;
    const int hc = static_cast<int>(BH - h0 < C ? BH - h0 : C);
    const size_t off = static_cast<size_t>(h0) * head_bytes, bytes = static_cast<size_t>(hc) * head_bytes;
    uint8_t* sq = ws + (static_cast<size_t>(s) * 4 + 0) * chunk;
    uint8_t* sk = sq + chunk;
    uint8_t* sv = sk + chunk;
    uint8_t* so = sv + chunk;
    // copy-in: the stage's previous chunk (this call's or the last call's) has left it
    ok = cudaStreamWaitEvent(P.in, P.free_ev[s], 0) == cudaSuccess &&
         cudaMemcpyAsync(sq, static_cast<const uint8_t*>(q) + off, bytes, cudaMemcpyHostToDevice, P.in) == cudaSuccess &&
         cudaMemcpyAsync(sk, static_cast<const uint8_t*>(k) + off, bytes, cudaMemcpyHostToDevice, P.in) == cudaSuccess &&
         cudaMemcpyAsync(sv, static_cast<const uint8_t*>(v) + off, bytes, cudaMemcpyHostToDevice, P.in) == cudaSuccess &&
         cudaEventRecord(P.in_ev[s], P.in) == cudaSuccess;
    if (!ok) break;
    // compute: the chunk's heads as one (1, hc) batch
    if (cudaStreamWaitEvent(P.comp, P.in_ev[s], 0) != cudaSuccess) {
      ok = false;
      break;
    }
    st = f32 ? launch_tra_f32(reinterpret_cast<const float*>(sq), reinterpret_cast<const float*>(sk),
                              reinterpret_cast<const float*>(sv), reinterpret_cast<float*>(so), 1, hc, T, D, beta, p,
                              P.comp)
             : launch_tra_bf16(sq, sk, sv, so, 1, hc, T, D, beta, p, false, P.comp);
    if (st != OK) break;
    // copy-out
    ok = cudaEventRecord(P.done[s], P.comp) == cudaSuccess && cudaStreamWaitEvent(P.out, P.done[s], 0) == cudaSuccess &&
         cudaMemcpyAsync(static_cast<uint8_t*>(out) + off, so, bytes, cudaMemcpyDeviceToHost, P.out) == cudaSuccess &&
         cudaEventRecord(P.free_ev[s], P.out) == cudaSuccess;
  }
  // The caller's stream waits for everything enqueued on the three streams
  // (also after a failure, so that the caller may release its buffers once
  // its stream has drained).
  cudaStream_t ss[3] = {P.in, P.comp, P.out};
  bool tail_ok = true;
  for (int t = 0; t < 3; ++t)
    tail_ok = tail_ok && cudaEventRecord(P.tail[t], ss[t]) == cudaSuccess &&
              cudaStreamWaitEvent(stream, P.tail[t], 0) == cudaSuccess;
  if (st != OK) return st;
  return ok && tail_ok ? OK : ERR_LAUNCH;
}

}  // namespace bsa
