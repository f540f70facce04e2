// Host side of the backward entry points (attn_bwd, attn_bwd_qk): validation,
// tensor maps, launch of the dQ kernel and then the dK/dV kernel on one stream.
// Included by attn_fwd.cu so both passes share one module (one status word).
#pragma once
#include "attn_bwd_kernel.cuh"

namespace {

template <int D, bool CAUSAL>
cudaError_t opt_in_bwd_smem() {
  cudaError_t e = cudaFuncSetAttribute(attn::attn_bwd_dq_sm103<D, CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(attn::CfgDq<D>::SMEM));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attn::attn_bwd_dkdv_sm103<D, CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(attn::CfgDkv<D>::SMEM));
}

std::atomic<int> g_bwd_ready[kMaxDevices];

// Causal order of the dQ kernel's query tiles (BwdParams::lpt).  Each tile
// reads every K and V tile it sees, so the order decides how often K and V
// come from HBM.  Tiles of about equal key ranges (the first at least 3/4 of
// the last: a short query block against a long key cache) run with a head's
// tiles adjacent (0) when all heads' K and V exceed half of L2 (64 MB): with
// the heads interleaved, a 512-query block against an 8192-key cache read
// every K and V once per query tile (backward 793 -> 751 us, CUDA events,
// L2 flushed; 1024 queries against 4096 keys 709 -> 666).  When they fit,
// heaviest first over all heads (BH), which measured 1.3 % faster than
// head-adjacent there (b2h16, 1024 queries against 8192 keys, D = 64).  Tiles
// of very different key ranges (the square causal case): heaviest first
// within bands of heads whose K and V take at most half of L2.
int dq_lpt_band(int64_t BH, int64_t Nq, int64_t Nk, int64_t ld) {
  const int64_t n_kt = (Nk + attn::BN - 1) / attn::BN;
  const int64_t light = (Nq < attn::BM ? Nq : attn::BM) - 1 + (Nk - Nq);  // last key the first tile sees
  int64_t nk_light = light / attn::BN + 1;
  if (nk_light > n_kt) nk_light = n_kt;
  const int64_t kv_head = 4 * Nk * ld;  // bytes of one head's K and V
  const int64_t half_l2 = int64_t(64) << 20;
  if (4 * nk_light >= 3 * n_kt) return half_l2 / kv_head < BH ? 0 : int(BH);  // (no overflow)
  const int64_t band = half_l2 / kv_head;
  return int(band < 1 ? 1 : (band > BH ? BH : band));
}

attn_status_t prepare_bwd(int dev) {
  if (g_bwd_ready[dev].load(std::memory_order_acquire) == 1) return ATTN_OK;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_bwd_ready[dev].load(std::memory_order_relaxed) == 1) return ATTN_OK;
  if (opt_in_bwd_smem<64, false>() != cudaSuccess || opt_in_bwd_smem<64, true>() != cudaSuccess ||
      opt_in_bwd_smem<128, false>() != cudaSuccess || opt_in_bwd_smem<128, true>() != cudaSuccess ||
      opt_in_bwd_smem<256, false>() != cudaSuccess || opt_in_bwd_smem<256, true>() != cudaSuccess)
    return ATTN_ERR_CUDA;
  g_bwd_ready[dev].store(1, std::memory_order_release);
  return ATTN_OK;
}

// prm_dq, prm_dkv: the same problem; they differ only in the box heights of
// the load maps (D = 256: 64-key K/V boxes for dQ, 32-query Q/dO boxes for dK/dV).
// The dK/dV kernel runs one CTA per SM walking the key tiles (D <= 128) or one
// CTA per key tile and column half (D = 256).
template <int D, bool CAUSAL>
cudaError_t launch_bwd_kernels(const attn::BwdParams& prm_dq, const attn::BwdParams& prm_dkv, int64_t sms,
                               cudaStream_t st) {
  attn::attn_bwd_dq_sm103<D, CAUSAL><<<dim3(unsigned(int64_t(prm_dq.n_qtiles) * prm_dq.bh)), dim3(attn::kBwdThreads),
                                       attn::CfgDq<D>::SMEM, st>>>(prm_dq);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t units = int64_t(prm_dkv.n_ktiles) * prm_dkv.bh * attn::CfgDkv<D>::NHALF;
  const int64_t ctas = attn::CfgDkv<D>::PERSIST && units > sms ? sms : units;
  attn::attn_bwd_dkdv_sm103<D, CAUSAL>
      <<<dim3(unsigned(ctas)), dim3(attn::kBwdThreads), attn::CfgDkv<D>::SMEM, st>>>(prm_dkv);
  return cudaGetLastError();
}

// ld: row stride in elements of every [.., N, D] tensor (0 = contiguous, ld = D).
attn_status_t launch_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv, float* delta, int64_t B, int64_t H,
                         int64_t Nq, int64_t Nk, int64_t D, int causal, float scale, void* stream, int64_t ld = 0) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (D > 256) return ATTN_ERR_UNSUPPORTED;
  if (ld == 0) {
    if (D % 8 != 0) return ATTN_ERR_UNSUPPORTED;  // contiguous rows must be 16-byte multiples (TMA)
    ld = D;
  } else {
    // Padded rows: the kernels use the first roundup8(D) columns (see launch_fwd).
    D = (D + 7) & ~int64_t(7);
    if (ld < D || ld % 8 != 0 || ld > (int64_t(1) << 20)) return ATTN_ERR_INVALID_ARG;
  }
  if (B == 0 || H == 0 || (Nq == 0 && Nk == 0)) return ATTN_OK;  // nothing is read or written
  // Nq = 0 leaves dK = dV = 0 and Nk = 0 leaves rows without keys: neither is
  // produced by these kernels.
  if (Nq == 0 || Nk == 0 || (causal && Nq > Nk)) return ATTN_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !delta) return ATTN_ERR_INVALID_ARG;
  constexpr int64_t kI32 = 2147483647;
  if (B > kI32 || H > kI32 || B * H > kI32 || Nq > kI32 - 256 || Nk > kI32 - 256) return ATTN_ERR_INVALID_ARG;
  const int64_t BH = B * H;
  const int64_t n_qtiles = (Nq + attn::BM - 1) / attn::BM, n_ktiles = (Nk + attn::BN - 1) / attn::BN;
  // Grids: n_qtiles * BH dQ CTAs; n_ktiles * BH (two per key tile at D > 128) dK/dV units, whose
  // persistent walk runs up to two grid sizes past the last one: all in int32.
  if (BH > (kI32 - 4096) / (n_qtiles > 2 * n_ktiles ? n_qtiles : 2 * n_ktiles)) return ATTN_ERR_INVALID_ARG;
  const int64_t Nmax = Nq > Nk ? Nq : Nk;
  if (BH > (int64_t(1) << 62) / (Nmax * ld * 2)) return ATTN_ERR_INVALID_ARG;
  const uint64_t qb = uint64_t(BH) * uint64_t(Nq) * uint64_t(ld) * 2u, kb = uint64_t(BH) * uint64_t(Nk) * uint64_t(ld) * 2u;
  const uint64_t vb4 = uint64_t(BH) * uint64_t(Nq) * 4u;
  const auto mis16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
  const auto mis4 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) != 0; };
  if (mis16(q) || mis16(k) || mis16(v) || mis16(o) || mis16(dout) || mis16(dq) || mis16(dk) || mis16(dv) || mis4(lse) ||
      mis4(delta))
    return ATTN_ERR_INVALID_ARG;
  // Outputs must not overlap each other or any input.
  const struct { const void* p; uint64_t n; } outs[4] = {{dq, qb}, {dk, kb}, {dv, kb}, {delta, vb4}};
  const struct { const void* p; uint64_t n; } ins[6] = {{q, qb}, {k, kb}, {v, kb}, {o, qb}, {lse, vb4}, {dout, qb}};
  for (int a = 0; a < 4; ++a) {
    for (int b = 0; b < 6; ++b)
      if (ranges_overlap(outs[a].p, outs[a].n, ins[b].p, ins[b].n)) return ATTN_ERR_INVALID_ARG;
    for (int b = a + 1; b < 4; ++b)
      if (ranges_overlap(outs[a].p, outs[a].n, outs[b].p, outs[b].n)) return ATTN_ERR_INVALID_ARG;
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  attn_status_t ready = prepare_device(dev);
  if (ready != ATTN_OK) return ready;
  if ((ready = prepare_bwd(dev)) != ATTN_OK) return ready;
  const EncodeTiledFn enc = encode_fn();
  if (!enc) return ATTN_ERR_CUDA;
  attn::BwdParams prm{};
  if (!encode_qkv_map(enc, &prm.tq, q, D, Nq, BH, ld) || !encode_qkv_map(enc, &prm.tdo, dout, D, Nq, BH, ld) ||
      !encode_qkv_map(enc, &prm.tk, k, D, Nk, BH, ld) || !encode_qkv_map(enc, &prm.tv, v, D, Nk, BH, ld) ||
      !encode_qkv_map(enc, &prm.tdq, dq, D, Nq, BH, ld) || !encode_qkv_map(enc, &prm.tdk, dk, D, Nk, BH, ld) ||
      !encode_qkv_map(enc, &prm.tdv, dv, D, Nk, BH, ld))
    return ATTN_ERR_CUDA;
  prm.o = static_cast<const __nv_bfloat16*>(o);
  prm.dout = static_cast<const __nv_bfloat16*>(dout);
  prm.lse = lse;
  prm.delta = delta;
  prm.Nq = int(Nq);
  prm.Nk = int(Nk);
  prm.kv_off = int(Nk - Nq);
  prm.bh = int(BH);
  prm.n_qtiles = int(n_qtiles);
  prm.n_ktiles = int(n_ktiles);
  prm.d = int(D);
  prm.ld = int(ld);
  prm.scale = scale;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.timeout_cycles = timeout_cycles();
  prm.lpt = causal ? dq_lpt_band(BH, Nq, Nk, ld) : 0;
  // D > 128 (the D = 256 kernels): the dQ kernel loads K, V in 64-key boxes,
  // the dK/dV kernel Q, dO in 32-query boxes.
  attn::BwdParams prm_dq = prm, prm_dkv = prm;
  if (D > 128 && (!encode_qkv_map(enc, &prm_dq.tk, k, D, Nk, BH, ld, attn::CfgDq<256>::BNK) ||
                  !encode_qkv_map(enc, &prm_dq.tv, v, D, Nk, BH, ld, attn::CfgDq<256>::BNK) ||
                  !encode_qkv_map(enc, &prm_dkv.tq, q, D, Nq, BH, ld, attn::CfgDkv<256>::SQ) ||
                  !encode_qkv_map(enc, &prm_dkv.tdo, dout, D, Nq, BH, ld, attn::CfgDkv<256>::SQ)))
    return ATTN_ERR_CUDA;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t sms = g_dev_sms[dev] > 0 ? g_dev_sms[dev] : 1;
  cudaError_t err;
  if (D <= 64)  // padded to 64, 128 or 256 as in the forward
    err = causal ? launch_bwd_kernels<64, true>(prm_dq, prm_dkv, sms, st) : launch_bwd_kernels<64, false>(prm_dq, prm_dkv, sms, st);
  else if (D <= 128)
    err = causal ? launch_bwd_kernels<128, true>(prm_dq, prm_dkv, sms, st) : launch_bwd_kernels<128, false>(prm_dq, prm_dkv, sms, st);
  else
    err = causal ? launch_bwd_kernels<256, true>(prm_dq, prm_dkv, sms, st) : launch_bwd_kernels<256, false>(prm_dq, prm_dkv, sms, st);
  return err == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                       void* dq, void* dk, void* dv, float* delta, int64_t B, int64_t H, int64_t N, int64_t D,
                       int causal, float scale, void* stream) {
  return launch_bwd(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, N, N, D, causal, scale, stream);
}

attn_status_t attn_bwd_qk(const void* q, const void* k, const void* v, const void* o, const float* lse,
                          const void* dout, void* dq, void* dk, void* dv, float* delta, int64_t B, int64_t H,
                          int64_t Nq, int64_t Nk, int64_t D, int causal, float scale, void* stream) {
  return launch_bwd(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, Nq, Nk, D, causal, scale, stream);
}

attn_status_t attn_bwd_ld(const void* q, const void* k, const void* v, const void* o, const float* lse,
                          const void* dout, void* dq, void* dk, void* dv, float* delta, int64_t B, int64_t H,
                          int64_t Nq, int64_t Nk, int64_t D, int64_t ld, int causal, float scale, void* stream) {
  if (ld <= 0) return ATTN_ERR_INVALID_ARG;
  return launch_bwd(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, Nq, Nk, D, causal, scale, stream, ld);
}

}  // extern "C"
