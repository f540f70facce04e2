// Host side of attn_based_fwd: validation, tensor maps and the launch of the
// Based linear-attention kernel (one CTA per (batch, head) sequence).
// Included by attn_fwd.cu so it shares the device preparation and status word.
#pragma once
#include "based_fwd_kernel.cuh"

namespace {

std::atomic<int> g_based_ready[kMaxDevices];

attn_status_t prepare_based(int dev) {
  if (g_based_ready[dev].load(std::memory_order_acquire) == 1) return ATTN_OK;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_based_ready[dev].load(std::memory_order_relaxed) == 1) return ATTN_OK;
  if (cudaFuncSetAttribute(based::based_fwd_sm103, cudaFuncAttributeMaxDynamicSharedMemorySize, int(based::SMEM)) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  g_based_ready[dev].store(1, std::memory_order_release);
  return ATTN_OK;
}

// q or k [B*H, N, F] bf16 as a 3-D tensor {F, N, B*H}: boxes of 8 x 128 x 1
// (128 rows of 16 bytes, no swizzle: the unswizzled K-major MMA layout); a tile
// is two boxes at features 0 and 8; features past F and rows past N read as zero.
bool encode_feature_map(EncodeTiledFn enc, CUtensorMap* map, const void* ptr, int64_t F, int64_t N, int64_t BH) {
  const cuuint64_t dims[3] = {cuuint64_t(F), cuuint64_t(N), cuuint64_t(BH)};
  const cuuint64_t strides[2] = {cuuint64_t(F) * 2u, cuuint64_t(N) * cuuint64_t(F) * 2u};
  const cuuint32_t box[3] = {8u, 128u, 1u};
  const cuuint32_t estride[3] = {1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

attn_status_t attn_based_fwd(const void* q, const void* k, const void* v, void* y, float* z, int64_t B, int64_t H,
                             int64_t N, int64_t F, int64_t D, float scale, void* stream) {
  if (B < 0 || H < 0 || N < 0 || F <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (F > 16 || F % 8 != 0 || D > 64 || D % 8 != 0) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;  // nothing is read or written
  if (!q || !k || !v || !y || !z) return ATTN_ERR_INVALID_ARG;
  constexpr int64_t kI32 = 2147483647;
  if (B > kI32 || H > kI32 || B * H > kI32 || N > kI32 - 256) return ATTN_ERR_INVALID_ARG;
  const int64_t BH = B * H;
  if (BH > (int64_t(1) << 62) / (N * 64 * 2)) return ATTN_ERR_INVALID_ARG;  // byte sizes
  const uint64_t qk_bytes = uint64_t(BH) * uint64_t(N) * uint64_t(F) * 2u;
  const uint64_t v_bytes = uint64_t(BH) * uint64_t(N) * uint64_t(D) * 2u;
  const uint64_t z_bytes = uint64_t(BH) * uint64_t(N) * 4u;
  const auto mis16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
  if (mis16(q) || mis16(k) || mis16(v) || mis16(y) || (reinterpret_cast<uintptr_t>(z) & 3u) != 0)
    return ATTN_ERR_INVALID_ARG;
  if (ranges_overlap(y, v_bytes, q, qk_bytes) || ranges_overlap(y, v_bytes, k, qk_bytes) ||
      ranges_overlap(y, v_bytes, v, v_bytes) || ranges_overlap(y, v_bytes, z, z_bytes) ||
      ranges_overlap(z, z_bytes, q, qk_bytes) || ranges_overlap(z, z_bytes, k, qk_bytes) ||
      ranges_overlap(z, z_bytes, v, v_bytes))
    return ATTN_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  attn_status_t ready = prepare_device(dev);
  if (ready != ATTN_OK) return ready;
  if ((ready = prepare_based(dev)) != ATTN_OK) return ready;
  const EncodeTiledFn enc = encode_fn();
  if (!enc) return ATTN_ERR_CUDA;
  based::BasedParams prm{};
  if (!encode_feature_map(enc, &prm.tq, q, F, N, BH) || !encode_feature_map(enc, &prm.tk, k, F, N, BH) ||
      !encode_qkv_map(enc, &prm.tv, v, D, N, BH) || !encode_qkv_map(enc, &prm.ty, y, D, N, BH))
    return ATTN_ERR_CUDA;
  prm.z = z;
  prm.N = int(N);
  prm.n_chunks = int((N + based::C - 1) / based::C);
  prm.scale = scale;
  prm.timeout_cycles = timeout_cycles();
  based::based_fwd_sm103<<<dim3(unsigned(BH)), dim3(based::kThreads), based::SMEM, static_cast<cudaStream_t>(stream)>>>(
      prm);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

double attn_based_fwd_flops(int64_t B, int64_t H, int64_t N, int64_t F, int64_t D) {
  // The linear (running-state) form per token: the state update and the
  // readout, each 2 * Fs * (D + 1) with Fs = 1 + F + F (F + 1) / 2 features of
  // the symmetric second-order Taylor map and D + 1 value columns (values and
  // the normaliser).
  const double fs = 1.0 + double(F) + 0.5 * double(F) * double(F + 1);
  return 4.0 * fs * double(D + 1) * double(B) * double(H) * double(N);
}

}  // extern "C"
