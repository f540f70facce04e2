// Fused attention forward for sm_103a (GB300): one CTA per 128-row query tile.
//
// What it computes ("[GPU] Deep Learning for HPC", bkkhyunn.github.io, section
// "Flash Attention"): S = Q K^T, a row softmax, O = softmax(S) V, tiled so the
// score matrix only ever lives on chip.  The running-max / running-sum form of
// the softmax is the one the FlashAttention-2 forward returns `Lse` for
// (null-ptr.tistory.com "development", the Triton `_fwd_kernel` post); the
// safe-softmax step (subtract the row max before exp) follows the softmax post
// on the same site ("Original softmax").
//
// Hardware mapping (the pages' H100 design is prior art: "GPUの爆発的な性能向上",
// ja.news.hada.io topic 14783, sections "WGMMA", "Shared memoryとbank conflict",
// "アドレス生成とTMA"):
//   warp 4   : TMA producer.  Q tile once, then K_j and V_j into NS-deep rings of
//              128-byte-swizzled shared-memory tiles, completion on mbarriers.
//   warp 5   : allocates 512 TMEM columns, then one thread issues tcgen05.mma:
//              S_j = Q K_j^T into one of two TMEM score buffers, and
//              O += P_j V_j with P_j read from TMEM (bf16, written over S_j).
//              It issues S_{j+1} before waiting for P_j, so the tensor core
//              computes the next scores while the softmax warps work.
//   warps 0-3: one thread per query row (= TMEM lane).  Per key tile: load the
//              score row from TMEM, mask (causal diagonal, keys past N), update
//              the running max m and sum l in base 2, write P as bf16 into TMEM,
//              rescale the O accumulator in TMEM when m grew, signal the MMA
//              warp.  Epilogue: O / l -> bf16, LSE = ln2 * (m + log2 l).
// Every barrier wait is bounded: on expiry the kernel records a timeout in a
// device status word, the other roles see a shared abort flag, in-flight TMA
// copies and MMAs are drained, TMEM is freed and the CTA returns.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace attn {

constexpr int BM = 128;                   // query rows per CTA (= TMEM lanes)
constexpr int BN = 128;                   // keys per tile
constexpr int kThreads = 192;             // 4 softmax warps + TMA warp + MMA warp
constexpr int kLoadWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kSubTile = 128u * 128u;  // 128 rows x 64 bf16 (one 128-B swizzle span)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;            // two score buffers: columns [0,128) and [128,256)
constexpr uint32_t kTmemO = 256;          // O accumulator: columns [256, 256 + D)
constexpr int kStatusTimeout = 4;         // value of ATTN_ERR_TIMEOUT

struct FwdParams {
  CUtensorMap tq, tk, tv;  // 3-D maps {D, N, B*H}, box {64, 128, 1}, 128-B swizzle, zero fill
  __nv_bfloat16* o;        // [B*H, N, D]
  float* lse;              // [B*H, N]
  int N;
  int bh;                  // B*H
  int n_tiles;             // ceil(N / 128), for queries and keys alike
  float scale_log2;        // scale * log2(e)
  long long timeout_cycles;
};

template <int D>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int KB = D / 64;                      // 64-column sub-tiles per tile
  static constexpr int NS = D == 128 ? 3 : 4;            // K and V ring depth
  static constexpr uint32_t TILE = KB * kSubTile;        // bytes of one 128 x D bf16 tile
  static constexpr uint32_t OFF_Q = 1024;                // first 1 KB: barriers and flags
  static constexpr uint32_t OFF_K = OFF_Q + TILE;
  static constexpr uint32_t OFF_V = OFF_K + NS * TILE;
  static constexpr uint32_t USED = OFF_V + NS * TILE;
  // + 1 KB to align the base; D = 64 also keeps 32 KB of tail room so that no
  // operand descriptor of the last V stage can address past the allocation.
  static constexpr uint32_t SMEM = USED + 1024 + (D == 64 ? 32768u : 0u);
  // barrier slots
  static constexpr int B_Q = 0, B_KF = 1, B_KE = 1 + NS, B_VF = 1 + 2 * NS, B_VE = 1 + 3 * NS;
  static constexpr int B_SF = 1 + 4 * NS, B_PF = 3 + 4 * NS, B_OF = 5 + 4 * NS, B_DONE = 6 + 4 * NS;
  static constexpr int NBAR = 7 + 4 * NS;
  static_assert(NBAR * 8 <= 512, "barrier area");
};

__device__ int g_attn_status;  // 0 or kStatusTimeout; read and cleared by the host

struct Abort {
  volatile uint32_t* flag;
  long long limit;
};

// Spin on an mbarrier phase, bounded.  Returns false when another role aborted
// (if honour_abort) or when `limit` cycles pass; the latter records a timeout.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const Abort& ab,
                                             bool honour_abort = true) {
  if (sm103::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (sm103::mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (honour_abort && *ab.flag) return false;
      if (clock64() - t0 > ab.limit) {
        atomicCAS(&g_attn_status, 0, kStatusTimeout);
        *ab.flag = 1u;
        return false;
      }
    }
  }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_sm103(const __grid_constant__ FwdParams p) {
  using C = Cfg<D>;
  constexpr int NS = C::NS;
  constexpr int KB = C::KB;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = sm103::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sbase + 512);
  volatile uint32_t* const abort_flag = reinterpret_cast<volatile uint32_t*>(sbase + 516);
  const uint32_t sQ = base + C::OFF_Q, sK = base + C::OFF_K, sV = base + C::OFF_V;
  auto bar = [base](int i) { return base + 8u * uint32_t(i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Tile order.  Causal: heaviest query tiles first (longest-processing-time
  // order across all heads).  Full: the query tiles of one head are adjacent
  // so that its K and V stay hot in L2.
  int qt, bh;
  if (CAUSAL) {
    qt = p.n_tiles - 1 - int(blockIdx.x / uint32_t(p.bh));
    bh = int(blockIdx.x % uint32_t(p.bh));
  } else {
    qt = int(blockIdx.x % uint32_t(p.n_tiles));
    bh = int(blockIdx.x / uint32_t(p.n_tiles));
  }
  const int m0 = qt * BM;
  const int nk = CAUSAL ? qt + 1 : p.n_tiles;  // key tiles this query tile visits

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i)
      sm103::mbar_init(bar(i), (i == C::B_PF || i == C::B_PF + 1) ? uint32_t(BM) : 1u);
    *abort_flag = 0u;
    sm103::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    sm103::tmem_alloc(sm103::smem_u32(tmem_slot), kTmemCols);
    sm103::tmem_relinquish();
  }
  if (warp == kLoadWarp && lane == 0) {
    sm103::tma_prefetch_map(&p.tq);
    sm103::tma_prefetch_map(&p.tk);
    sm103::tma_prefetch_map(&p.tv);
  }
  sm103::tc_fence_before();
  __syncthreads();
  sm103::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag, p.timeout_cycles};

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      sm103::mbar_arrive_expect_tx(bar(C::B_Q), C::TILE);
      for (int kb = 0; kb < KB; ++kb)
        sm103::tma_load_3d(sQ + kb * kSubTile, &p.tq, bar(C::B_Q), kb * 64, m0, bh);
      int kiss = 0, viss = 0;  // K and V tiles issued
      for (int j = 0; j < nk; ++j) {
        const int s = j % NS;
        const uint32_t ph = uint32_t(j / NS) & 1u;
        if (j >= NS && !wait_bounded(bar(C::B_KE + s), ph ^ 1u, ab)) break;
        sm103::mbar_arrive_expect_tx(bar(C::B_KF + s), C::TILE);
        for (int kb = 0; kb < KB; ++kb)
          sm103::tma_load_3d(sK + s * C::TILE + kb * kSubTile, &p.tk, bar(C::B_KF + s), kb * 64, j * BN, bh);
        ++kiss;
        if (j >= NS && !wait_bounded(bar(C::B_VE + s), ph ^ 1u, ab)) break;
        sm103::mbar_arrive_expect_tx(bar(C::B_VF + s), C::TILE);
        for (int kb = 0; kb < KB; ++kb)
          sm103::tma_load_3d(sV + s * C::TILE + kb * kSubTile, &p.tv, bar(C::B_VF + s), kb * 64, j * BN, bh);
        ++viss;
      }
      // Drain: no copy may land in shared memory after this CTA has left.
      wait_bounded(bar(C::B_Q), 0u, ab, false);
      for (int t = kiss > NS ? kiss - NS : 0; t < kiss; ++t)
        wait_bounded(bar(C::B_KF + t % NS), uint32_t(t / NS) & 1u, ab, false);
      for (int t = viss > NS ? viss - NS : 0; t < viss; ++t)
        wait_bounded(bar(C::B_VF + t % NS), uint32_t(t / NS) & 1u, ab, false);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t kIdescS = sm103::idesc_bf16_f32(BM, BN, 0, 0);  // Q, K both K-major
      constexpr uint32_t kIdescO = sm103::idesc_bf16_f32(BM, D, 0, 1);   // P K-major, V MN-major
      auto issue_pv = [&](int jj) -> bool {
        const int s = jj % NS;
        const int b = jj & 1;
        if (!wait_bounded(bar(C::B_PF + b), uint32_t(jj >> 1) & 1u, ab)) return false;
        if (!wait_bounded(bar(C::B_VF + s), uint32_t(jj / NS) & 1u, ab)) return false;
        sm103::tc_fence_after();
        const uint32_t aP = tmem + kTmemS + uint32_t(b) * BN;
        const uint32_t vbase = sV + s * C::TILE;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)  // 16 keys per MMA: 8 TMEM columns of P, 16 rows of V
          sm103::mma_ts(tmem + kTmemO, aP + kk * 8, sm103::sdesc_sw128(vbase + kk * 2048, kSubTile, 1024),
                        kIdescO, (jj > 0 || kk > 0) ? 1u : 0u);
        sm103::mma_commit(bar(C::B_OF));
        sm103::mma_commit(bar(C::B_VE + s));
        return true;
      };
      bool ok = wait_bounded(bar(C::B_Q), 0u, ab);
      for (int j = 0; ok && j < nk; ++j) {
        const int s = j % NS;
        const int b = j & 1;
        if (!(ok = wait_bounded(bar(C::B_KF + s), uint32_t(j / NS) & 1u, ab))) break;
        sm103::tc_fence_after();
        const uint32_t kbase = sK + s * C::TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {  // 16 of the head dim per MMA
          const uint32_t off = uint32_t(kk >> 2) * kSubTile + uint32_t(kk & 3) * 32u;
          sm103::mma_ss(tmem + kTmemS + uint32_t(b) * BN, sm103::sdesc_sw128(sQ + off, 16, 1024),
                        sm103::sdesc_sw128(kbase + off, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
        }
        sm103::mma_commit(bar(C::B_SF + b));
        sm103::mma_commit(bar(C::B_KE + s));
        if (j > 0) ok = issue_pv(j - 1);
      }
      if (ok) issue_pv(nk - 1);
      // Every MMA must be finished before TMEM is freed.
      sm103::mma_commit(bar(C::B_DONE));
      wait_bounded(bar(C::B_DONE), 0u, ab, false);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------- softmax, epilogue
    const int r = threadIdx.x;  // row within the tile = TMEM lane
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    const uint32_t tO = tmem + lane_off + kTmemO;
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY;  // running max of scale*log2(e)*s
    float l_run = 0.f;        // running sum of p (fp32, before the bf16 rounding of P)
    bool ok = true;
    for (int j = 0; j < nk; ++j) {
      const int b = j & 1;
      ok = __all_sync(0xffffffffu, wait_bounded(bar(C::B_SF + b), uint32_t(j >> 1) & 1u, ab));
      if (!ok) break;
      sm103::tc_fence_after();
      const uint32_t tS = tmem + lane_off + kTmemS + uint32_t(b) * BN;
      float s[BN];
#pragma unroll
      for (int q = 0; q < BN / 32; ++q) {
        uint32_t u[32];
        sm103::tmem_ld32(tS + q * 32, u);
#pragma unroll
        for (int e = 0; e < 32; ++e) s[q * 32 + e] = __uint_as_float(u[e]);
      }
      // Masks: the causal diagonal tile (key c visible iff c <= r) and keys past N.
      int lim = BN - 1;
      if (CAUSAL && j == nk - 1) lim = r;
      if (j == p.n_tiles - 1) lim = min(lim, p.N - 1 - j * BN);
      if (lim < BN - 1) {
#pragma unroll
        for (int c = 0; c < BN; ++c) s[c] = c > lim ? -INFINITY : s[c];
      }
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int c = 4; c < BN; c += 4) {
        mx0 = fmaxf(mx0, s[c]);
        mx1 = fmaxf(mx1, s[c + 1]);
        mx2 = fmaxf(mx2, s[c + 2]);
        mx3 = fmaxf(mx3, s[c + 3]);
      }
      const float m_new = fmaxf(m_run, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2);
      const float alpha = sm103::ex2_approx(m_run - m_new);  // 0 on the first tile
      const float neg_m = -m_new;
      float sum0 = 0.f, sum1 = 0.f, sum2 = 0.f, sum3 = 0.f;
#pragma unroll
      for (int q = 0; q < BN / 32; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = sm103::ex2_approx(fmaf(s[q * 32 + 2 * e], sl2, neg_m));
          const float p1 = sm103::ex2_approx(fmaf(s[q * 32 + 2 * e + 1], sl2, neg_m));
          pk[e] = sm103::pack_bf16x2(p0, p1);
          if (e & 1) {
            sum2 += p0;
            sum3 += p1;
          } else {
            sum0 += p0;
            sum1 += p1;
          }
        }
        sm103::tmem_st16(tS + q * 16, pk);  // P over the first 64 columns of this S buffer
      }
      sm103::tmem_st_wait();
      l_run = alpha * l_run + ((sum0 + sum1) + (sum2 + sum3));
      m_run = m_new;
      if (j > 0) {
        // O holds sum over earlier tiles; P_{j-1} V_{j-1} must have landed first.
        ok = __all_sync(0xffffffffu, wait_bounded(bar(C::B_OF), uint32_t(j - 1) & 1u, ab));
        if (!ok) break;
        sm103::tc_fence_after();
        if (__any_sync(0xffffffffu, alpha < 1.f)) {
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t u[32];
            sm103::tmem_ld32(tO + q * 32, u);
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
            sm103::tmem_st32(tO + q * 32, u);
          }
          sm103::tmem_st_wait();
        }
      }
      sm103::tc_fence_before();
      sm103::mbar_arrive(bar(C::B_PF + b));
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_bounded(bar(C::B_OF), uint32_t(nk - 1) & 1u, ab));
    if (ok) {
      sm103::tc_fence_after();
      const float inv_l = 1.f / l_run;
      const int row = m0 + r;
      const bool live = row < p.N;
      __nv_bfloat16* const orow = p.o + (size_t(bh) * size_t(p.N) + size_t(live ? row : 0)) * D;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t u[32];
        sm103::tmem_ld32(tO + q * 32, u);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = sm103::pack_bf16x2(__uint_as_float(u[2 * e]) * inv_l, __uint_as_float(u[2 * e + 1]) * inv_l);
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(orow + q * 32);
          dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          dst[2] = make_uint4(pk[8], pk[9], pk[10], pk[11]);
          dst[3] = make_uint4(pk[12], pk[13], pk[14], pk[15]);
        }
      }
      if (live) p.lse[size_t(bh) * size_t(p.N) + size_t(row)] = (m_run + log2f(l_run)) * 0.6931471805599453f;
    }
  }

  sm103::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    sm103::tc_fence_after();
    sm103::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace attn
