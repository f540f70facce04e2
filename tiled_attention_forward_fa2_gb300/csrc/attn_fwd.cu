// Host side of the C ABI declared in include/attn.h: argument validation,
// TMA tensor maps, grid shape and launch of the sm_103a kernels, and the
// device status word.  Nothing here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "attn.h"
#include "attn_fwd_kernel.cuh"
#include "attn_fwd_short_kernel.cuh"
#ifdef ATTN_TEST_HOOKS
#include "attn_test_hooks.h"
#endif

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library does not link libcuda directly and loads on machines without a GPU.
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// [B*H, N, D] bf16 with rows ld elements apart (ld = D when contiguous) viewed
// as a 3-D tensor {D, N, B*H}; boxes of 64 x box_rows x 1 (64 bf16 = one 128-byte
// swizzle span); columns past D and rows past N read as zero and are never written.
bool encode_qkv_map(EncodeTiledFn enc, CUtensorMap* map, const void* ptr, int64_t D, int64_t N, int64_t BH,
                    int64_t ld = 0, uint32_t box_rows = 128) {
  if (ld == 0) ld = D;
  const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(N), cuuint64_t(BH)};
  const cuuint64_t strides[2] = {cuuint64_t(ld) * 2u, cuuint64_t(N) * cuuint64_t(ld) * 2u};
  const cuuint32_t box[3] = {64u, box_rows, 1u};
  const cuuint32_t estride[3] = {1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-device one-time state: architecture check, SM count and the shared-memory
// opt-in of every kernel instance.  0 = not yet, 1 = ready, 2 = unsupported, 3 = error.
constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_state[kMaxDevices];
int g_dev_sms[kMaxDevices];
std::mutex g_dev_mutex;

template <int D, bool CAUSAL>
cudaError_t opt_in_smem() {
  cudaError_t e = cudaFuncSetAttribute(attn::attn_fwd_sm103<D, CAUSAL, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(attn::Cfg<D>::SMEM));
  if (e != cudaSuccess) return e;
  if constexpr (D == 64) {
    e = cudaFuncSetAttribute(attn::attn_fwd_sm103<64, CAUSAL, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(attn::Cfg<64>::SMEM));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn::attn_fwd_short_sm103<CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(attn::CfgShort::SMEM));
    if (e != cudaSuccess) return e;
  }
  if constexpr (attn::Cfg<D>::STAGE_IN_Q) return cudaSuccess;  // one-unit grid only
  else
    return cudaFuncSetAttribute(attn::attn_fwd_sm103<D, CAUSAL, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(attn::Cfg<D>::SMEM));
}

attn_status_t prepare_device(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  int st = g_dev_state[dev].load(std::memory_order_acquire);
  if (st == 0) {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    st = g_dev_state[dev].load(std::memory_order_relaxed);
    if (st == 0) {
      int major = 0, minor = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&g_dev_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        st = 3;
      } else if (major != 10 || minor != 3) {
        st = 2;
      } else if (opt_in_smem<64, false>() != cudaSuccess || opt_in_smem<64, true>() != cudaSuccess ||
                 opt_in_smem<128, false>() != cudaSuccess || opt_in_smem<128, true>() != cudaSuccess ||
                 opt_in_smem<256, false>() != cudaSuccess || opt_in_smem<256, true>() != cudaSuccess) {
        st = 3;
      } else {
        st = 1;
      }
      if (st != 3) g_dev_state[dev].store(st, std::memory_order_release);
    }
  }
  if (st == 1) return ATTN_OK;
  return st == 2 ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_CUDA;
}

bool ranges_overlap(const void* a, uint64_t na, const void* b, uint64_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Key tiles (of 128) up to which the persistent grid is used.  It saves about
// 3.5 us of launch, Q load and epilogue per unit and costs about 6 % of the
// key loop's speed (1.55 us per key tile of a two-tile unit at D = 128): even
// at about 38 tiles; measured on GB300, 32 tiles (N = 4096) still gains and
// 128 (N = 16384) loses 6 %.
constexpr int64_t kPersistMaxKeyTiles = 32;
// Causal: up to 16.  The one-unit grid hands P over in two halves (split P),
// which only it does: causal b4h16n4096d128 1383 against 1286 TFLOP/s
// persistent; b8h16n2048d128 1075 against 1070; b16h16n1024d128 726 against
// 760 (CUDA events, L2 flushed, mean of 60).
constexpr int64_t kPersistMaxKeyTilesCausal = 16;

// Process-wide overrides set by attn_set_tuning (0 = the launcher's own choice).
// Read once per call with relaxed loads: a call sees either the old or the new value.
std::atomic<int> g_tune_unit{0};          // 1 or 2 query tiles per unit, 3 key split, 4 short kernel
std::atomic<int> g_tune_grid{0};          // 1 one CTA per unit, 2 persistent
std::atomic<int> g_tune_chunks{0};        // chunks of heads in attn_fwd_from_host
constexpr int kPipeChunksMax = 32;        // chunks at most (events held per device)
std::atomic<long long> g_tune_wait{0};    // bound of every pipeline wait (SM cycles)
std::atomic<unsigned> g_status_slot{0};   // next result slot of attn_last_status
#ifdef ATTN_TEST_HOOKS
std::atomic<int> g_test_withhold_kv{0};   // test build only: issue no K/V loads
#endif

long long timeout_cycles() {
  // About two seconds at the GB300 clock; no legitimate wait comes near it.
  const long long x = g_tune_wait.load(std::memory_order_relaxed);
  return x > 0 ? x : (1LL << 32);
}

template <int D, bool CAUSAL>
cudaError_t launch(const attn::FwdParams& prm, int64_t ctas, bool persist, bool split, cudaStream_t stream,
                   bool shortk = false) {
  if constexpr (D == 64) {
    if (shortk) {  // two CTAs per SM, each walking single-tile units
      attn::attn_fwd_short_sm103<CAUSAL><<<dim3(unsigned(ctas)), dim3(attn::kShortThreads), attn::CfgShort::SMEM,
                                           stream>>>(prm);
      return cudaGetLastError();
    }
    if (split) {  // the key-split kernel walks its units like the persistent one
      attn::attn_fwd_sm103<64, CAUSAL, true, true><<<dim3(unsigned(ctas)), dim3(attn::kThreads), attn::Cfg<64>::SMEM,
                                                     stream>>>(prm);
      return cudaGetLastError();
    }
  }
  if constexpr (!attn::Cfg<D>::STAGE_IN_Q) {
    if (persist) {
      attn::attn_fwd_sm103<D, CAUSAL, true><<<dim3(unsigned(ctas)), dim3(attn::kThreads), attn::Cfg<D>::SMEM,
                                               stream>>>(prm);
      return cudaGetLastError();
    }
  }
  attn::attn_fwd_sm103<D, CAUSAL, false><<<dim3(unsigned(ctas)), dim3(attn::kThreads), attn::Cfg<D>::SMEM, stream>>>(prm);
  return cudaGetLastError();
}

// The launcher's choices for one problem: query tiles per unit, key split,
// short-unit kernel, grid, causal order.  attn_set_tuning overrides some.
struct FwdPlan {
  int T = 1;              // query tiles per unit
  bool split = false;     // key split (D <= 64)
  bool shortk = false;    // short-unit kernel (D <= 64)
  bool persist = false;   // persistent grid
  int lpt = 0;            // causal: heads per longest-first band (0: a head's units adjacent)
  int64_t n_work = 0;     // units of the whole problem
  int64_t ctas = 0;       // grid size
};

FwdPlan plan_fwd(int64_t BH, int64_t Nq, int64_t Nk, int64_t D, bool causal, int64_t sms) {
  FwdPlan pl;
  const int64_t n_qtiles = (Nq + attn::BM - 1) / attn::BM;
  const int64_t n_ktiles = (Nk + attn::BN - 1) / attn::BN;
  // Two query tiles per CTA share every K/V tile and let two softmax warpgroups
  // take turns on the tensor core: one key step of both tiles costs about 3100
  // SM cycles, against about 2500 for one tile alone (no partner to overlap
  // with).  Pick the tiling whose waves of CTAs finish first:
  //   waves(T=2) * 3100 <= waves(T=1) * 2500, i.e. about 5 * waves2 <= 4 * waves1.
  // attn_set_tuning overrides the choice (testing and tuning).
  const int64_t waves2 = ((n_qtiles + 1) / 2 * BH + sms - 1) / sms;
  const int64_t waves1 = (n_qtiles * BH + sms - 1) / sms;
  int T = 5 * waves2 <= 4 * waves1 ? 2 : 1;
  // Key split (D <= 64): one query tile per unit, its key tiles shared out
  // between the two softmax warpgroups.  It halves a unit's chain of key steps
  // at the same tensor-core throughput per CTA as two tiles per unit, so it
  // wins when the single-tile units fit in one wave of CTAs (then every CTA's
  // time is one unit's chain; b2h8n1024d64: 128 tiles on 152 SMs).  Beyond a
  // wave its extra per-unit cost (Q load, merge) loses to two tiles per unit.
  bool split = D <= 64 && n_ktiles >= 2 && n_qtiles * BH <= sms;
  // Short-unit kernel (D <= 64, two CTAs per SM, one tile per unit): short
  // rows, where unit boundaries come every few key steps (and, causal, the two
  // tiles of a unit differ in length), with at least a full wave of its grid.
  // Measured (CUDA events, L2 flushed, mean of 50-150): causal b16h32n512d64
  // 43.7 against 54.9 us, b32h32n256d64 35.5 against 44.5, b8h16n1024d64
  // 35.5 against 40.5, b4h32n2048d64 100.3 against 99.9; full rows up to 8
  // key tiles b16h32n512d64 50.3 against 51.4, b8h16n1024d64 49.9 against
  // 51.9.  It loses on longer full rows (b4h16n4096d64 300 against 285: the
  // two-tile unit's shared K/V stream), on a short query block against 4096
  // keys and below a wave (b2h8n1024d64 causal 17.3 against 16.7).
  bool shortk = D <= 64 && n_qtiles >= 2 && n_qtiles * BH >= 2 * sms && n_ktiles <= (causal ? 16 : 8);
  if (shortk) split = false;
  if (const int u = g_tune_unit.load(std::memory_order_relaxed)) {
    T = u >= 3 ? 1 : u;
    split = u == 3 && D <= 64;
    shortk = u == 4 && D <= 64;
  }
  if (split || shortk) T = 1;
  if (D > 128) T = 1;  // the D = 256 kernel holds one query tile (TMEM)
  pl.T = T;
  pl.split = split;
  pl.shortk = shortk;
  pl.n_work = (n_qtiles + T - 1) / T * BH;
  // Causal order: longest first over all heads when the units' key ranges
  // differ a lot (lightest below 3/4 of the heaviest: the square causal case);
  // when they are about equal (a short query block against a long key cache)
  // a head's units stay adjacent instead, so its K and V are read from HBM
  // once (the longest-first order read them twice there: 976 against 553 MB).
  // The short-unit kernel keeps a head's units adjacent whatever their
  // lengths: its units are at most 16 key tiles, so the longest-first order
  // gains little balance, and it sent every head's first (longest) unit out
  // in the first quarter of the launch, all reading their K and V from HBM at
  // once (causal b16h32n512d64 45.7 -> 43.7 us, b32h32n256d64 37.5 -> 35.5;
  // CUDA events, L2 flushed, median of 100).
  if (causal && !shortk) {
    const int64_t last_row_light = (T == 2 ? 2 * attn::BM : attn::BM) - 1;  // unit 0's last query row
    const int64_t light_row = last_row_light < Nq - 1 ? last_row_light : Nq - 1;
    int64_t nk_light = (light_row + (Nk - Nq)) / attn::BN + 1;
    if (nk_light > n_ktiles) nk_light = n_ktiles;
    if (4 * nk_light < 3 * n_ktiles) {
      // Bands of heads whose K and V together take at most half of L2 (64 MB):
      // over all 16 heads of causal N = 16384 (8 MB each) the longest-first
      // order read 552 MB from HBM for 201 MB of K, V and Q.
      const int64_t kv_head = 4 * Nk * D;
      const int64_t band = (int64_t(64) << 20) / kv_head;
      pl.lpt = int(band < 1 ? 1 : (band > BH ? BH : band));
    }
  }
  // Short key ranges: a persistent grid (one CTA per SM taking every gridDim-th
  // unit) overlaps each unit's Q load and epilogue with the previous unit's
  // work.  Long ones: one CTA per unit, whose key loop runs faster (see the
  // kernel) and whose launch cost is small beside the unit.
  // attn_set_tuning forces the choice (testing and tuning).
  // At D <= 64 a key step costs about half as much, so the persistent grid wins
  // at every length measured (N = 4096: +6 %, 16384: +2.5 %).
  bool persist = D <= 64 || n_ktiles <= (causal ? kPersistMaxKeyTilesCausal : kPersistMaxKeyTiles);
  if (const int g = g_tune_grid.load(std::memory_order_relaxed)) persist = g == 2;
  if (D > 128) persist = false;  // the D = 256 kernel stages O in its Q buffer
  int64_t ctas = persist && pl.n_work > sms ? sms : pl.n_work;
  if (shortk) ctas = pl.n_work > 2 * sms ? 2 * sms : pl.n_work;  // two CTAs per SM
  pl.persist = persist;
  pl.ctas = ctas;
  return pl;
}

// Shared launcher of attn_fwd and attn_fwd_qk: Q, O [B*H, Nq, D]; K, V [B*H, Nk, D].
// With check_only it validates the arguments and the device and returns.
// ld: row stride in elements of q, k, v, o (0 = contiguous, ld = D).
attn_status_t launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                         int64_t Nq, int64_t Nk, int64_t D, int causal, float scale, void* stream,
                         bool check_only = false, int64_t ld = 0) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (D > 256) return ATTN_ERR_UNSUPPORTED;
  if (ld == 0) {
    if (D % 8 != 0) return ATTN_ERR_UNSUPPORTED;  // contiguous rows must be 16-byte multiples (TMA)
    ld = D;
  } else {
    // Padded rows: the kernels use the first roundup8(D) columns (the tensor
    // copies move whole 16-byte groups); columns D.. of that group are zeros.
    D = (D + 7) & ~int64_t(7);
    if (ld < D || ld % 8 != 0 || ld > (int64_t(1) << 20)) return ATTN_ERR_INVALID_ARG;
  }
  if (B == 0 || H == 0 || Nq == 0) return ATTN_OK;  // nothing is read or written
  // Query rows that see no key at all (Nk = 0, or causal with Nq > Nk) are not
  // produced by the kernel.
  if (Nk == 0 || (causal && Nq > Nk)) return ATTN_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  constexpr int64_t kI32 = 2147483647;
  if (B > kI32 || H > kI32 || B * H > kI32 || Nq > kI32 - 256 || Nk > kI32 - 256) return ATTN_ERR_INVALID_ARG;
  const int64_t BH = B * H;
  const int64_t n_qtiles = (Nq + attn::BM - 1) / attn::BM;
  const int64_t n_ktiles = (Nk + attn::BN - 1) / attn::BN;
  // Units of work (at most one per query tile) and the persistent grid's unit
  // index, which runs up to two grid sizes past the last unit, stay in int32.
  if (BH > (kI32 - 4096) / n_qtiles) return ATTN_ERR_INVALID_ARG;
  const int64_t Nmax = Nq > Nk ? Nq : Nk;
  if (BH > (int64_t(1) << 62) / (Nmax * ld * 2)) return ATTN_ERR_INVALID_ARG;  // byte sizes
  const uint64_t q_bytes = uint64_t(BH) * uint64_t(Nq) * uint64_t(ld) * 2u;
  const uint64_t kv_bytes = uint64_t(BH) * uint64_t(Nk) * uint64_t(ld) * 2u;
  const uint64_t lse_bytes = uint64_t(BH) * uint64_t(Nq) * 4u;
  const auto mis16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
  if (mis16(q) || mis16(k) || mis16(v) || mis16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return ATTN_ERR_INVALID_ARG;
  if (ranges_overlap(o, q_bytes, q, q_bytes) || ranges_overlap(o, q_bytes, k, kv_bytes) ||
      ranges_overlap(o, q_bytes, v, kv_bytes) || ranges_overlap(o, q_bytes, lse, lse_bytes) ||
      ranges_overlap(lse, lse_bytes, q, q_bytes) || ranges_overlap(lse, lse_bytes, k, kv_bytes) ||
      ranges_overlap(lse, lse_bytes, v, kv_bytes))
    return ATTN_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  const attn_status_t ready = prepare_device(dev);
  if (ready != ATTN_OK || check_only) return ready;
  const EncodeTiledFn enc = encode_fn();
  if (!enc) return ATTN_ERR_CUDA;

  attn::FwdParams prm{};
  if (!encode_qkv_map(enc, &prm.tq, q, D, Nq, BH, ld) || !encode_qkv_map(enc, &prm.tk, k, D, Nk, BH, ld) ||
      !encode_qkv_map(enc, &prm.tv, v, D, Nk, BH, ld) || !encode_qkv_map(enc, &prm.to, o, D, Nq, BH, ld))
    return ATTN_ERR_CUDA;
  const int64_t sms = g_dev_sms[dev] > 0 ? g_dev_sms[dev] : 1;
  const FwdPlan pl = plan_fwd(BH, Nq, Nk, D, causal != 0, sms);
  const int T = pl.T;
  prm.lse = lse;
  prm.Nq = int(Nq);
  prm.Nk = int(Nk);
  prm.kv_off = int(Nk - Nq);
  prm.bh = int(BH);
  prm.n_qtiles = int(n_qtiles);
  prm.n_ktiles = int(n_ktiles);
  prm.tiles_per_cta = T;
  prm.n_units = int((n_qtiles + T - 1) / T);
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.timeout_cycles = timeout_cycles();
#ifdef ATTN_TEST_HOOKS
  // Test build only: the kernel issues no K/V loads, so its pipeline waits run
  // out and it reports ATTN_ERR_TIMEOUT (used with a lowered wait bound).
  prm.withhold_kv = g_test_withhold_kv.load(std::memory_order_relaxed);
#endif

  prm.n_work = int(pl.n_work);
  prm.lpt = pl.lpt;
  const bool persist = pl.persist, split = pl.split, shortk = pl.shortk;
  const int64_t ctas = pl.ctas;
  if (shortk && !encode_qkv_map(enc, &prm.to32, o, D, Nq, BH, ld, 32)) return ATTN_ERR_CUDA;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t err;
  // Head dims below 64, 128 or 256 run on that kernel: the tensor maps carry the true
  // D, so TMA fills the missing columns with zeros on load (they add nothing to
  // Q K^T, and P V gives zeros there) and leaves them out on store.
  if (D <= 64)
    err = causal ? launch<64, true>(prm, ctas, persist, split, st, shortk)
                 : launch<64, false>(prm, ctas, persist, split, st, shortk);
  else if (D <= 128)
    err = causal ? launch<128, true>(prm, ctas, persist, false, st) : launch<128, false>(prm, ctas, persist, false, st);
  else
    err = causal ? launch<256, true>(prm, ctas, persist, false, st) : launch<256, false>(prm, ctas, persist, false, st);
  return err == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* attn_fwd_kernel_name(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, int causal) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || D <= 0 || D > 256) return nullptr;
  constexpr int64_t kI32 = 2147483647;
  if (B > kI32 || H > kI32 || B * H > kI32 || Nq > kI32 - 256 || Nk > kI32 - 256) return nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || prepare_device(dev) != ATTN_OK) return nullptr;
  const int64_t D8 = (D + 7) & ~int64_t(7);
  const FwdPlan pl = plan_fwd(B * H, Nq, Nk, D8, causal != 0, g_dev_sms[dev] > 0 ? g_dev_sms[dev] : 1);
  const int dk = D8 <= 64 ? 64 : (D8 <= 128 ? 128 : 256);
  const char* mask = causal ? "causal" : "full";
  thread_local char name[96];
  if (pl.shortk)
    std::snprintf(name, sizeof(name), "attn_fwd_short_sm103<%s>", mask);
  else if (pl.split)
    std::snprintf(name, sizeof(name), "attn_fwd_sm103<64,%s,persistent,key split>", mask);
  else
    std::snprintf(name, sizeof(name), "attn_fwd_sm103<%d,%s,%s,%d tile%s/unit>", dk, mask,
                  pl.persist ? "persistent" : "one unit per CTA", pl.T, pl.T > 1 ? "s" : "");
  return name;
}

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                       int64_t N, int64_t D, int causal, float scale, void* stream) {
  return launch_fwd(q, k, v, o, lse, B, H, N, N, D, causal, scale, stream);
}

attn_status_t attn_fwd_qk(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                          int64_t Nq, int64_t Nk, int64_t D, int causal, float scale, void* stream) {
  return launch_fwd(q, k, v, o, lse, B, H, Nq, Nk, D, causal, scale, stream);
}

attn_status_t attn_fwd_ld(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                          int64_t Nq, int64_t Nk, int64_t D, int64_t ld, int causal, float scale, void* stream) {
  if (ld <= 0) return ATTN_ERR_INVALID_ARG;
  return launch_fwd(q, k, v, o, lse, B, H, Nq, Nk, D, causal, scale, stream, false, ld);
}

attn_status_t attn_last_status(void* stream) {
  // The status word is taken and cleared in one atomic exchange on the device,
  // behind the work already on `stream`, so a timeout recorded concurrently by
  // a kernel on another stream is never lost.  Each call uses its own result
  // slot (round robin), so concurrent callers do not overwrite each other.
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int slot = int(g_status_slot.fetch_add(1, std::memory_order_relaxed) % unsigned(attn::kStatusSlots));
  attn::status_take<<<1, 1, 0, st>>>(slot);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  int word = 0;
  if (cudaMemcpyFromSymbolAsync(&word, attn::g_status_taken, sizeof(int), size_t(slot) * sizeof(int),
                                cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return ATTN_ERR_CUDA;
  return word == 0 ? ATTN_OK : ATTN_ERR_TIMEOUT;
}

attn_status_t attn_set_tuning(int unit, int grid, int pipe_chunks, int64_t wait_limit_cycles) {
  if (unit < 0 || unit > 4 || grid < 0 || grid > 2 || pipe_chunks < 0 || pipe_chunks > kPipeChunksMax ||
      wait_limit_cycles < 0)
    return ATTN_ERR_INVALID_ARG;
  g_tune_unit.store(unit, std::memory_order_relaxed);
  g_tune_grid.store(grid, std::memory_order_relaxed);
  g_tune_chunks.store(pipe_chunks, std::memory_order_relaxed);
  g_tune_wait.store(wait_limit_cycles, std::memory_order_relaxed);
  return ATTN_OK;
}

#ifdef ATTN_TEST_HOOKS
attn_status_t attn_test_withhold_kv(int on) {
  g_test_withhold_kv.store(on ? 1 : 0, std::memory_order_relaxed);
  return ATTN_OK;
}
#endif

const char* attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
  }
  return "ATTN_ERR_UNKNOWN";
}

double attn_fwd_flops(int64_t B, int64_t H, int64_t N, int64_t D, int causal) {
  const double f = 4.0 * double(B) * double(H) * double(N) * double(N) * double(D);
  return causal ? 0.5 * f : f;
}

double attn_bwd_qk_flops(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, int causal);

double attn_fwd_qk_flops(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, int causal) {
  // Visible (query, key) pairs: Nq * Nk, or for the bottom-right causal mask
  // (Nk >= Nq) sum over i of (i + 1 + Nk - Nq) = Nq * (Nk - Nq) + Nq (Nq + 1) / 2,
  // taken as Nq * (Nk - Nq) + Nq^2 / 2 so that Nq = Nk gives exactly half.
  const double nq = double(Nq), nk = double(Nk);
  const double pairs = causal ? nq * (nk - nq) + 0.5 * nq * nq : nq * nk;
  return 4.0 * double(B) * double(H) * pairs * double(D);
}

}  // extern "C"
#include "attn_bwd_host.cuh"
#include "attn_host_pipeline.cuh"
#include "attn_host_static.cuh"
#include "based_fwd_host.cuh"

extern "C" double attn_bwd_qk_flops(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, int causal) {
  return 2.5 * attn_fwd_qk_flops(B, H, Nq, Nk, D, causal);
}
