// attn_fwd_from_host_static: the forward for inputs and outputs in host memory,
// staged through a fixed device array compiled into this library instead of
// device buffers the caller allocates.  It serves callers that have host data
// and a stream but must not allocate device memory themselves: a plain C host
// program that links only this library and has no device allocator of its own,
// or code running beside a caching allocator that already holds the free device
// memory (where a cudaMalloc of its own would fail, or would stall the device
// while it synchronises).  Included by attn_fwd.cu (one translation unit).
#pragma once

namespace {

// The staging array: ATTN_STATIC_STAGING_BYTES bytes in the library's device
// image.  Every device that loads the library's device code holds it until the
// process exits, and it keeps whatever the last call left in it.  In host code
// the name is only a stand-in for the array; its device address comes from
// cudaGetSymbolAddress, once per device.
constexpr uint64_t kStagingBytes = uint64_t(ATTN_STATIC_STAGING_BYTES);
static __device__ __align__(256) uint8_t g_attn_staging[kStagingBytes];

uint8_t* g_staging_dev[kMaxDevices];
std::mutex g_staging_mutex;

// The array's address on device `dev`, which must be the current device.  The
// first call on a device looks it up (this may load the library's device code
// there); later calls read the cached address.
attn_status_t staging_ptr(int dev, uint8_t** out) {
  std::lock_guard<std::mutex> lock(g_staging_mutex);
  if (!g_staging_dev[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_staging) != cudaSuccess || !p) return ATTN_ERR_CUDA;
    g_staging_dev[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_staging_dev[dev];
  return ATTN_OK;
}

constexpr uint64_t align256(uint64_t x) { return (x + 255u) & ~uint64_t(255); }

}  // namespace

extern "C" attn_status_t attn_fwd_from_host_static(const void* q_host, const void* k_host, const void* v_host,
                                                   void* o_host, float* lse_host, int64_t B, int64_t H, int64_t Nq,
                                                   int64_t Nk, int64_t D, int causal, float scale, void* stream) {
  // attn_fwd_qk's argument rules, as far as the staging sizes depend on them.
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (D > 256 || D % 8 != 0) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || Nq == 0) return ATTN_OK;  // nothing is read or written
  if (!q_host || !k_host || !v_host || !o_host || !lse_host) return ATTN_ERR_INVALID_ARG;
  constexpr int64_t kI32 = 2147483647;
  if (B > kI32 || H > kI32 || B * H > kI32 || Nq > kI32 || Nk > kI32) return ATTN_ERR_INVALID_ARG;

  // Q, K, V, O, LSE one after another, each starting on a 256-byte boundary.
  // Rows of at least 16 bytes, so more than kStagingBytes rows cannot fit (and
  // bounding the row counts first keeps the byte counts below 2^64).
  const uint64_t BH = uint64_t(B) * uint64_t(H);
  if (BH * uint64_t(Nq) > kStagingBytes || BH * uint64_t(Nk) > kStagingBytes) return ATTN_ERR_UNSUPPORTED;
  const uint64_t q_bytes = BH * uint64_t(Nq) * uint64_t(D) * 2u, kv_bytes = BH * uint64_t(Nk) * uint64_t(D) * 2u;
  const uint64_t lse_bytes = BH * uint64_t(Nq) * 4u;
  const uint64_t off_k = align256(q_bytes), off_v = off_k + align256(kv_bytes), off_o = off_v + align256(kv_bytes);
  const uint64_t off_l = off_o + align256(q_bytes);
  if (off_l + lse_bytes > kStagingBytes) return ATTN_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  uint8_t* base = nullptr;
  const attn_status_t sp = staging_ptr(dev, &base);
  if (sp != ATTN_OK) return sp;
  uint8_t *q = base, *k = base + off_k, *v = base + off_v, *o = base + off_o;
  float* lse = reinterpret_cast<float*>(base + off_l);
  // The rest of attn_fwd_qk's rules (lengths, masks, the device) on the staged layout.
  const attn_status_t chk = launch_fwd(q, k, v, o, lse, B, H, Nq, Nk, D, causal, scale, stream, true);
  if (chk != ATTN_OK) return chk;

  // All of it on the caller's stream, in order: inputs up, the kernel, results
  // down.  Every byte the kernel reads is written by the copies just before it.
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(q, q_host, q_bytes, cudaMemcpyDefault, st) != cudaSuccess ||
      cudaMemcpyAsync(k, k_host, kv_bytes, cudaMemcpyDefault, st) != cudaSuccess ||
      cudaMemcpyAsync(v, v_host, kv_bytes, cudaMemcpyDefault, st) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const attn_status_t ls = launch_fwd(q, k, v, o, lse, B, H, Nq, Nk, D, causal, scale, stream);
  if (ls != ATTN_OK) return ls;
  if (cudaMemcpyAsync(o_host, o, q_bytes, cudaMemcpyDefault, st) != cudaSuccess ||
      cudaMemcpyAsync(lse_host, lse, lse_bytes, cudaMemcpyDefault, st) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}
