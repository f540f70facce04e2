// attn_fwd_from_host: the forward for inputs and outputs in host memory, with
// the copies to and from the device overlapped with the kernels.  The heads
// (B*H slices) are cut into chunks; chunk c's Q, K, V go up on one copy stream
// while the kernel runs on chunk c - 1 on the caller's stream and chunk c - 2's
// O and LSE come back on a second copy stream.  Events order the three streams;
// the caller's stream ends waiting on the last copy back, so synchronising it
// (or anything ordered after it) covers the whole call.  The device buffers are
// the caller's; the two copy streams and the events are created once per device
// and reused.  Included by attn_fwd.cu (one translation unit).
#pragma once

namespace {

// Chunks of heads per call.  A chunk's kernel lasts at least as long as its
// longest unit (all key tiles of two query tiles: ~1.55 us per key tile at
// D = 128, ~0.8 at D <= 64, measured on GB300), so more chunks only help while
// each chunk's upload (~200 GB/s over the host link, measured both for the copy
// engines and for SM loads) still takes longer than that; at most 8 (measured:
// the bench shape, 32-key-tile units, is best at 8; causal N = 16384, 128-tile
// units, at 4 -- 816 against 620 TFLOP/s end to end at 8).  attn_set_tuning
// overrides the choice (tuning).
int pipe_chunks(uint64_t in_bytes, int64_t n_ktiles, int64_t D) {
  const int x = g_tune_chunks.load(std::memory_order_relaxed);
  if (x >= 1 && x <= kPipeChunksMax) return x;
  const double unit_us = double(n_ktiles) * (D <= 64 ? 0.8 : 1.55);
  const double upload_us = double(in_bytes) / 200e3;  // 200 GB/s = 200e3 bytes per us
  const double n = upload_us / unit_us;
  return n >= 8.0 ? 8 : (n >= 1.0 ? int(n) : 1);
}

struct HostPipe {
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t in[kPipeChunksMax] = {}, out[kPipeChunksMax] = {};
  bool ready = false;
};
HostPipe g_pipe[kMaxDevices];
// Held while a call enqueues its work: the shared events are recorded and waited
// on in pairs, which must not interleave with another thread's call.
std::mutex g_pipe_mutex;

attn_status_t pipe_ready(int dev) {
  HostPipe& hp = g_pipe[dev];
  if (hp.ready) return ATTN_OK;
  const unsigned ev = cudaEventDisableTiming;
  if (cudaStreamCreateWithFlags(&hp.up, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&hp.down, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&hp.start, ev) != cudaSuccess || cudaEventCreateWithFlags(&hp.done, ev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  for (int c = 0; c < kPipeChunksMax; ++c)
    if (cudaEventCreateWithFlags(&hp.in[c], ev) != cudaSuccess || cudaEventCreateWithFlags(&hp.out[c], ev) != cudaSuccess)
      return ATTN_ERR_CUDA;
  hp.ready = true;
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status_t attn_fwd_from_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                                            float* lse_host, void* q, void* k, void* v, void* o, float* lse, int64_t B,
                                            int64_t H, int64_t Nq, int64_t Nk, int64_t D, int causal, float scale,
                                            void* stream) {
  const bool empty = B >= 0 && H >= 0 && Nq >= 0 && (B == 0 || H == 0 || Nq == 0);
  if (!empty && (!q_host || !k_host || !v_host || !o_host || !lse_host)) return ATTN_ERR_INVALID_ARG;
  // Device-side arguments, sizes and the device are checked as attn_fwd_qk does.
  const attn_status_t chk = launch_fwd(q, k, v, o, lse, B, H, Nq, Nk, D, causal, scale, stream, true);
  if (chk != ATTN_OK || empty) return chk;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;

  std::lock_guard<std::mutex> lock(g_pipe_mutex);
  if (pipe_ready(dev) != ATTN_OK) return ATTN_ERR_CUDA;
  HostPipe& hp = g_pipe[dev];
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t BH = B * H;
  const uint64_t q_row = uint64_t(Nq) * uint64_t(D) * 2u, kv_row = uint64_t(Nk) * uint64_t(D) * 2u;
  const int chunks = pipe_chunks(uint64_t(BH) * (q_row + 2u * kv_row), (Nk + attn::BN - 1) / attn::BN, D);
  const int n = int(BH < chunks ? BH : chunks);
  const uint64_t l_row = uint64_t(Nq) * 4u;
  auto at = [](const void* p, uint64_t off) { return static_cast<const uint8_t*>(p) + off; };
  auto atw = [](void* p, uint64_t off) { return static_cast<uint8_t*>(p) + off; };

  // Nothing of this call may start before the work already on the caller's stream.
  if (cudaEventRecord(hp.start, st) != cudaSuccess || cudaStreamWaitEvent(hp.up, hp.start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp.down, hp.start, 0) != cudaSuccess)
    return ATTN_ERR_CUDA;
  for (int c = 0; c < n; ++c) {
    const int64_t h0 = BH * c / n, h1 = BH * (c + 1) / n, nh = h1 - h0;
    const uint64_t qo = uint64_t(h0) * q_row, kvo = uint64_t(h0) * kv_row, lo = uint64_t(h0) * l_row;
    if (cudaMemcpyAsync(atw(q, qo), at(q_host, qo), uint64_t(nh) * q_row, cudaMemcpyDefault, hp.up) != cudaSuccess ||
        cudaMemcpyAsync(atw(k, kvo), at(k_host, kvo), uint64_t(nh) * kv_row, cudaMemcpyDefault, hp.up) != cudaSuccess ||
        cudaMemcpyAsync(atw(v, kvo), at(v_host, kvo), uint64_t(nh) * kv_row, cudaMemcpyDefault, hp.up) != cudaSuccess ||
        cudaEventRecord(hp.in[c], hp.up) != cudaSuccess || cudaStreamWaitEvent(st, hp.in[c], 0) != cudaSuccess)
      return ATTN_ERR_CUDA;
    const attn_status_t ls = launch_fwd(atw(q, qo), atw(k, kvo), atw(v, kvo), atw(o, qo),
                                        reinterpret_cast<float*>(atw(lse, lo)), 1, nh, Nq, Nk, D, causal, scale, stream);
    if (ls != ATTN_OK) return ls;
    if (cudaEventRecord(hp.out[c], st) != cudaSuccess || cudaStreamWaitEvent(hp.down, hp.out[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(atw(o_host, qo), at(o, qo), uint64_t(nh) * q_row, cudaMemcpyDefault, hp.down) != cudaSuccess ||
        cudaMemcpyAsync(atw(lse_host, lo), at(lse, lo), uint64_t(nh) * l_row, cudaMemcpyDefault, hp.down) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  if (cudaEventRecord(hp.done, hp.down) != cudaSuccess || cudaStreamWaitEvent(st, hp.done, 0) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}
