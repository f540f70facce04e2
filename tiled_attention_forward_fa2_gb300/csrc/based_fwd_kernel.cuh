// Based linear-attention forward for sm_103a (GB300).
//
// What it computes (the pages name the kernel -- "GPU의 폭발적인 성능 향상",
// news.hada.io topic 14783, section "ThunderKittens" -- but print no formula;
// the definition is the published Based layer): causal linear attention with
// the second-order Taylor kernel of exp,
//   s_ij = scale q_i . k_j,  a_ij = 1 + s_ij + s_ij^2 / 2  (j <= i),
//   z_i = sum_j a_ij,        y_i = sum_j a_ij v_j / z_i.
// a_ij = phi_Q(q_i) . phi_K(k_j) for the feature maps below, so the sum over
// all earlier chunks collapses into a running state Sigma = sum_j phi_K(k_j) v'_j^T.
//
// Features (160 columns = 80 bf16 pairs, 153 used), the same order for both
// maps (sc = scale; phi_Q | phi_K):
//   pairs 0..7    (sc q_2i, sc q_2i+1)           | (k_2i, k_2i+1)          linear
//   pairs 8..15   sc^2/2 (q_2i^2, q_2i+1^2)      | (k_2i^2, k_2i+1^2)      squares
//   pairs 16..71  sc^2 q_a (q_2m, q_2m+1)        | k_a (k_2m, k_2m+1)      a = 0..15, 2m > a
//   pairs 72..75  sc^2 (q_4t q_4t+1, q_4t+2 q_4t+3) | (k_4t k_4t+1, ...)   the products (a, a+1), a even
//   pair 76       (1, 0)                         | (1, 0)                  constant
//   pairs 77..79  0
// Every product q_a q_b with a < b appears once, so
// phi_Q(q) . phi_K(k) = s + s^2/2 + 1 exactly.  The order makes each pair one
// packed multiply of registers as loaded: phi_K in bf16x2 (the product of two
// bf16 values is exact before its single rounding), phi_Q in fp32x2 then one
// rounding.  Values carry one extra column: v' = [v (64, zero padded), 1,
// 0 x 15], so every product that gives y also gives z (column 64) with the
// same bf16 weights.
//
// One CTA per (batch, head) sequence walks its chunks of 128 tokens.  Per
// chunk c, on the tensor core (tcgen05, fp32 accumulators in TMEM), in issue order:
//   S      = Q_c K_c^T                 (the raw tiles; the A warps apply the scale)
//   Sig^T += V'_c^T phi_K(K_c)         (M = 80 value columns (of 128), N = 160 features, K = 128 tokens)
//   A'     = causal(1 + s + s^2/2) -> bf16, in TMEM over S  (A warps)
//   Y'_b   = A' V'_c                   (intra-chunk part, b = c mod 2; A' read from TMEM)
//   Y'_b  += phi_Q(Q_c) bf16(Sig before chunk c)            (all earlier chunks)
//   y = Y'_b[:, 0:64] / Y'_b[:, 64], z = Y'_b[:, 64].
// S depends only on the loaded tiles and Y' is double-buffered, so the first
// three products of a chunk are queued while phi_Q of the chunk (which must wait
// for the previous chunk's readout to release its tile) is still being written.
// Roles (512 threads):
//   warps 0-3  : feature warps, one thread per chunk row: phi_Q / phi_K rows into
//                128-byte-swizzled shared tiles; epilogue of the previous chunk
//                (y -> bf16 -> TMA store, z -> global).
//   warps 4-7  : A warps: the Taylor weights of the intra-chunk block, causal mask.
//   warps 8-11 : state warps, one thread per value column (TMEM lane): its row
//                of Sig^T (fp32, TMEM) -> bf16 row of the readout's K-major B
//                operand in shared memory (16-byte stores).
//   warp 12    : TMA producer (q, k as two 8-feature boxes each, in the
//                unswizzled K-major layout the S product reads; v 128-byte swizzled).
//   warp 15    : allocates TMEM and issues every MMA (one elected lane); the
//                next chunk's S is issued right after this chunk's A' V', so the
//                A warps work while the readout and the state update run.
// Every barrier wait is bounded (the forward's status word and abort flag).
#pragma once
#include "attn_fwd_kernel.cuh"

namespace based {

constexpr int C = 128;          // tokens per chunk (= TMEM lanes)
constexpr int NF = 160;         // phi features held (153 used)
constexpr int NV = 80;          // columns of v', Y' and Sig: 64 values, the z column, padding
constexpr int kThreads = 512;
constexpr int kLoadWarp = 12, kMmaWarp = 15;  // the MMA warp on the sub-partition with the idle state warp
constexpr uint32_t kTile = 128u * 128u;    // 16 KB: 128 rows of 128 bytes
constexpr int NQK = 4;                     // q/k stages
constexpr int NVS = 2;                     // v stages
// A q or k tile as loaded: two boxes of 8 features, each 128 rows of 16 bytes
// (the unswizzled K-major layout: 8-row core matrices 128 bytes apart, the
// second 8 features 2048 bytes on).
constexpr uint32_t kHalf = 128u * 16u;
constexpr uint32_t kQK = 4u * kHalf;          // q and k tiles of one chunk
constexpr uint32_t kSbfBlock = 80u * 128u;    // one 64-feature block of the bf16 state: 80 rows x 128 B
constexpr uint32_t kTmemCols = 512;
// Register split (setmaxnreg; warps 13 and 14 idle): 4 x 128 threads, sum = 512 x 128.
// The load/MMA warpgroup spills at 72 or fewer (ptxas); the state warps need
// no more than 176.
constexpr uint32_t kRegFeature = 152, kRegA = 104, kRegState = 176, kRegOther = 80;
constexpr uint32_t kRegLaunch = 65536 / kThreads;  // registers per thread at launch (1 CTA per SM)
static_assert(kRegFeature + kRegA + kRegState + kRegOther == 4 * kRegLaunch, "register split");

// Shared memory (offsets from a 1024-byte aligned base).  The ones block must
// follow the three phi_K blocks: it is the fourth 64-feature block the second
// state MMA group reads (features 192..255, whose state rows are never read),
// and the second 64-column block of every v' operand.
constexpr uint32_t OFF_QK = 1024;
constexpr uint32_t OFF_V = OFF_QK + NQK * kQK;
constexpr uint32_t OFF_PHIQ = OFF_V + NVS * kTile;
constexpr uint32_t OFF_PHIK = OFF_PHIQ + 3 * kTile;
constexpr uint32_t OFF_ONES = OFF_PHIK + 3 * kTile;
constexpr uint32_t OFF_SBF = OFF_ONES + kTile;
constexpr uint32_t OFF_STG = OFF_SBF + 3 * kSbfBlock;
constexpr uint32_t USED = OFF_STG + kTile;
constexpr uint32_t SMEM = USED + 1024;
static_assert(OFF_V % 1024 == 0 && OFF_PHIQ % 1024 == 0 && OFF_PHIK % 1024 == 0 && OFF_ONES % 1024 == 0 &&
                  OFF_SBF % 1024 == 0 && OFF_STG % 1024 == 0 && kSbfBlock % 1024 == 0,
              "swizzled tiles need 1024-byte alignment");
static_assert(SMEM <= 232448, "shared memory");

// Barriers
constexpr int B_QKF = 0;              // [NQK] q, k landed (TMA bytes)
constexpr int B_QKE = B_QKF + NQK;    // [NQK] q, k rows read (128 feature threads) and S done (commit)
constexpr int B_VF = B_QKE + NQK;     // [NVS] v landed
constexpr int B_VE = B_VF + NVS;      // [NVS] last MMA on v done (commit)
constexpr int B_PHIK = B_VE + NVS;    // phi_K of the chunk written (128 feature threads)
constexpr int B_PHIQ = B_PHIK + 1;    // phi_Q written (128)
constexpr int B_S = B_PHIQ + 1;       // S in TMEM (commit)
constexpr int B_A = B_S + 1;          // A' in TMEM (128)
constexpr int B_SIG = B_A + 1;        // state update done (commit)
constexpr int B_SIGF = B_SIG + 1;     // state read out of TMEM (128)
constexpr int B_SBF = B_SIGF + 1;     // bf16 state in shared memory (128)
constexpr int B_Y = B_SBF + 1;        // Y' of the chunk complete (commit)
constexpr int B_YF = B_Y + 1;         // [2] Y' buffer read out of TMEM (128)
constexpr int B_DONE = B_YF + 2;
constexpr int NBAR = B_DONE + 1;
static_assert(NBAR * 8 <= 512, "barrier area");
__host__ __device__ constexpr uint32_t bar_count(int b) {
  return (b >= B_QKE && b < B_QKE + NQK) ? 129u
         : (b == B_PHIK || b == B_PHIQ || b == B_A || b == B_SIGF || b == B_SBF || b == B_YF || b == B_YF + 1)
             ? 128u
             : 1u;
}

// TMEM columns
constexpr uint32_t COL_S = 0;     // S (fp32, 128), then A' (bf16 pairs, 64)
constexpr uint32_t COL_Y = 128;   // Y' buffer b at COL_Y + 96 b (80 each)
constexpr uint32_t COL_SIG = 320; // Sig^T (160): lane = value column, column = feature

struct BasedParams {
  CUtensorMap tq, tk;  // {F, N, B*H}, box {8, 128, 1}, no swizzle, zero fill
  CUtensorMap tv, ty;  // {D, N, B*H}, box {64, 128, 1}, 128-byte swizzle
  float* z;            // [B*H, N]
  int N, n_chunks;
  float scale;
  long long timeout_cycles;
};

// Pair p of the feature order above: kind 0 linear, 1 square, 2 a-times-pair,
// 3 adjacent products, 4 constant, 5 zero; a, m as in the table.
struct Pair {
  int kind, a, m;
};
__host__ __device__ constexpr Pair pair_of(int p) {
  if (p < 8) return {0, 0, p};
  if (p < 16) return {1, 0, p - 8};
  if (p < 72) {
    int t = p - 16;
    for (int a = 0; a < 16; ++a) {
      const int m0 = (a + 2) / 2;  // first m with 2m > a
      const int cnt = 8 - m0;
      if (t < cnt) return {2, a, m0 + t};
      t -= cnt;
    }
  }
  if (p < 76) return {3, 0, p - 72};
  if (p == 76) return {4, 0, 0};
  return {5, 0, 0};
}

// phi_K pair p from the row as loaded: w[i] = (k_2i, k_2i+1) as bf16.
template <int p>
__device__ __forceinline__ uint32_t phik_pair(const uint32_t (&w)[8]) {
  constexpr Pair t = pair_of(p);
  if constexpr (t.kind == 0) {
    return w[t.m];
  } else if constexpr (t.kind == 1) {
    return sm103::bf2_mul(w[t.m], w[t.m]);
  } else if constexpr (t.kind == 2) {
    // (k_a, k_a): the low or high half of w[a / 2] in both halves.
    const uint32_t dup = (t.a & 1) ? sm103::prmt<0x3232>(w[t.a / 2], 0u) : sm103::prmt<0x1010>(w[t.a / 2], 0u);
    return sm103::bf2_mul(dup, w[t.m]);
  } else if constexpr (t.kind == 3) {
    // (k_4t, k_4t+2) * (k_4t+1, k_4t+3)
    const uint32_t lo = sm103::prmt<0x5410>(w[2 * t.m], w[2 * t.m + 1]);
    const uint32_t hi = sm103::prmt<0x7632>(w[2 * t.m], w[2 * t.m + 1]);
    return sm103::bf2_mul(lo, hi);
  } else if constexpr (t.kind == 4) {
    return 0x3F80u;  // (1, 0)
  } else {
    return 0u;
  }
}

// phi_Q pair p from xs = sc q and hs = sc q / 2 (fp32), rounded once to bf16.
template <int p>
__device__ __forceinline__ uint32_t phiq_pair(const float (&xs)[16], const float (&hs)[16]) {
  constexpr Pair t = pair_of(p);
  float lo, hi;
  if constexpr (t.kind == 0) {
    return sm103::pack_bf16x2(xs[2 * t.m], xs[2 * t.m + 1]);
  } else if constexpr (t.kind == 1) {
    sm103::f2_unpack(sm103::f2_mul(sm103::f2_pack(xs[2 * t.m], xs[2 * t.m + 1]),
                                   sm103::f2_pack(hs[2 * t.m], hs[2 * t.m + 1])), lo, hi);
    return sm103::pack_bf16x2(lo, hi);
  } else if constexpr (t.kind == 2) {
    sm103::f2_unpack(sm103::f2_mul(sm103::f2_pack(xs[t.a], xs[t.a]), sm103::f2_pack(xs[2 * t.m], xs[2 * t.m + 1])),
                     lo, hi);
    return sm103::pack_bf16x2(lo, hi);
  } else if constexpr (t.kind == 3) {
    sm103::f2_unpack(sm103::f2_mul(sm103::f2_pack(xs[4 * t.m], xs[4 * t.m + 2]),
                                   sm103::f2_pack(xs[4 * t.m + 1], xs[4 * t.m + 3])), lo, hi);
    return sm103::pack_bf16x2(lo, hi);
  } else if constexpr (t.kind == 4) {
    return 0x3F80u;
  } else {
    return 0u;
  }
}

// Write one phi row into a 128-byte-swizzled K-major tile: 16-byte chunk c
// holds pairs 4c .. 4c+3 (features 8c .. 8c+7), at chunk (c mod 8) of the
// 64-feature block c / 8, swizzled by the row.
template <int c, bool KMAP>
struct PhiRow {
  static __device__ __forceinline__ void run(uint32_t tile, int r, const uint32_t (&w)[8], const float (&xs)[16],
                                             const float (&hs)[16]) {
    uint32_t v[4];
    if constexpr (KMAP) {
      v[0] = phik_pair<4 * c>(w), v[1] = phik_pair<4 * c + 1>(w), v[2] = phik_pair<4 * c + 2>(w),
      v[3] = phik_pair<4 * c + 3>(w);
    } else {
      v[0] = phiq_pair<4 * c>(xs, hs), v[1] = phiq_pair<4 * c + 1>(xs, hs), v[2] = phiq_pair<4 * c + 2>(xs, hs),
      v[3] = phiq_pair<4 * c + 3>(xs, hs);
    }
    const uint32_t addr = tile + uint32_t(c / 8) * kTile + uint32_t(r) * 128u + ((uint32_t(c % 8) ^ uint32_t(r & 7)) << 4);
    sm103::st_shared_v4(addr, v[0], v[1], v[2], v[3]);
    PhiRow<c + 1, KMAP>::run(tile, r, w, xs, hs);
  }
};
template <bool KMAP>
struct PhiRow<NF / 8, KMAP> {
  static __device__ __forceinline__ void run(uint32_t, int, const uint32_t (&)[8], const float (&)[16],
                                             const float (&)[16]) {}
};

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t (&w)[4]) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;\n" ::"r"(addr), "r"(v) : "memory");
}

// Row r of a q or k tile as loaded (two 8-feature halves kHalf bytes apart,
// 16 bytes per row): w[i] = features (2i, 2i+1) as packed bf16.
__device__ __forceinline__ void load_row16(uint32_t tile, int r, uint32_t (&w)[8]) {
  uint32_t h[4];
  ld_shared_v4(tile + uint32_t(r) * 16u, h);
  w[0] = h[0], w[1] = h[1], w[2] = h[2], w[3] = h[3];
  ld_shared_v4(tile + kHalf + uint32_t(r) * 16u, h);
  w[4] = h[0], w[5] = h[1], w[6] = h[2], w[7] = h[3];
}

__global__ void __launch_bounds__(kThreads, 1) based_fwd_sm103(const __grid_constant__ BasedParams p) {
  using attn::Abort;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = sm103::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sbase + 512);
  volatile uint32_t* const abort_flag = reinterpret_cast<volatile uint32_t*>(sbase + 516);
  const uint32_t sQK = base + OFF_QK, sV = base + OFF_V, sPQ = base + OFF_PHIQ, sPK = base + OFF_PHIK;
  const uint32_t sOnes = base + OFF_ONES, sSbf = base + OFF_SBF, sStg = base + OFF_STG;
  auto bar = [base](int i) { return base + 8u * uint32_t(i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = int(blockIdx.x);
  const int n = p.n_chunks;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) sm103::mbar_init(bar(i), bar_count(i));
    *abort_flag = 0u;
    sm103::fence_mbar_init();
  }
  // The ones block: K-row t of a v' operand's second 64-column block holds
  // [1, 0, ..., 0] (column 64 of v' = 1); stored in the 128-byte swizzle.
  for (int i = int(threadIdx.x); i < 128 * 8; i += kThreads) {
    const int row = i >> 3, chunk = i & 7;  // logical 16-byte chunk of the row
    sm103::st_shared_v4(sOnes + uint32_t(row) * 128u + ((uint32_t(chunk) ^ uint32_t(row & 7)) << 4),
                        chunk == 0 ? 0x3F80u : 0u, 0u, 0u, 0u);  // bf16 1.0 = 0x3F80, low half first
  }
  sm103::fence_proxy_async_smem();
  if (warp == kMmaWarp) {
    sm103::tmem_alloc(sm103::smem_u32(tmem_slot), kTmemCols);
    sm103::tmem_relinquish();
  }
  if (warp == kLoadWarp && lane == 0) {
    sm103::tma_prefetch_map(&p.tq);
    sm103::tma_prefetch_map(&p.tk);
    sm103::tma_prefetch_map(&p.tv);
    sm103::tma_prefetch_map(&p.ty);
  }
  sm103::tc_fence_before();
  __syncthreads();
  sm103::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag, p.timeout_cycles};

  if (warp >= kLoadWarp) {
    sm103::regs_set<kRegOther, kRegLaunch>();
    if (warp == kLoadWarp) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        bool ok = true;
        int c = 0;
        for (; c < n && ok; ++c) {
          const int s = c % NQK, sv = c % NVS;
          if (c >= NQK && !(ok = attn::wait_bounded(bar(B_QKE + s), uint32_t(c / NQK - 1) & 1u, ab))) break;
          const uint32_t dst = sQK + uint32_t(s) * kQK;
          sm103::mbar_arrive_expect_tx(bar(B_QKF + s), kQK);
          sm103::tma_load_3d(dst, &p.tq, bar(B_QKF + s), 0, c * C, bh);
          sm103::tma_load_3d(dst + kHalf, &p.tq, bar(B_QKF + s), 8, c * C, bh);
          sm103::tma_load_3d(dst + 2u * kHalf, &p.tk, bar(B_QKF + s), 0, c * C, bh);
          sm103::tma_load_3d(dst + 3u * kHalf, &p.tk, bar(B_QKF + s), 8, c * C, bh);
          if (c >= NVS && !(ok = attn::wait_bounded(bar(B_VE + sv), uint32_t(c / NVS - 1) & 1u, ab))) {
            ++c;  // the q/k copies of this chunk are in flight
            break;
          }
          sm103::mbar_arrive_expect_tx(bar(B_VF + sv), kTile);
          sm103::tma_load_3d(sV + uint32_t(sv) * kTile, &p.tv, bar(B_VF + sv), 0, c * C, bh);
        }
        // Drain: no copy may land after the CTA has left.  q/k copies issued: c;
        // v copies issued: c, or c - 1 when the loop stopped between the two.
        const int nqk = c;
        const int nv = (ok || c == 0) ? c : c - 1;
        for (int t = nqk > NQK ? nqk - NQK : 0; t < nqk; ++t)
          attn::drain_wait(bar(B_QKF + t % NQK), uint32_t(t / NQK) & 1u);
        for (int t = nv > NVS ? nv - NVS : 0; t < nv; ++t) attn::drain_wait(bar(B_VF + t % NVS), uint32_t(t / NVS) & 1u);
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // --------------------------------------------------------- MMA issue
      constexpr uint32_t kIdescS = sm103::idesc_bf16_f32(128, 128, 0, 0);    // q, k K-major (unswizzled)
      constexpr uint32_t kIdescSig = sm103::idesc_bf16_f32(128, 160, 1, 1);  // v'^T (MN-major), phi_K MN-major
      constexpr uint32_t kIdescYt = sm103::idesc_bf16_f32(128, NV, 0, 1);    // A' from TMEM, v' MN-major
      constexpr uint32_t kIdescYs = sm103::idesc_bf16_f32(128, NV, 0, 0);    // phi_Q K-major, state K-major
      const uint32_t hi = sm103::kSdescHi;
      constexpr uint32_t kHiRaw = sm103::sdesc_noswz_hi(128);  // 8-row groups 128 bytes apart
      const uint32_t dPQ = sm103::sdesc_sw128_lo(sPQ, 16);
      const uint32_t dPK = sm103::sdesc_sw128_lo(sPK, kTile);  // phi_K as an MN-major operand: 64-feature blocks
      const uint32_t dSbf = sm103::sdesc_sw128_lo(sSbf, 16);
      bool ok = true;
      // S = Q K^T of chunk c from the raw tiles (the two 8-feature halves kHalf apart along K).
      auto issue_s = [&](int c) -> bool {
        const int s = c % NQK;
        if (!attn::warp_wait(bar(B_QKF + s), uint32_t(c / NQK) & 1u, ab)) return false;
        sm103::tc_fence_after();
        const uint32_t qk = sQK + uint32_t(s) * kQK;
        sm103::mma_ss_warp_lo(tmem + COL_S, sm103::sdesc_sw128_lo(qk, kHalf), sm103::sdesc_sw128_lo(qk + 2u * kHalf, kHalf),
                              kIdescS, 0u, kHiRaw);
        sm103::mma_commit_warp(bar(B_S));
        sm103::mma_commit_warp(bar(B_QKE + s));
        return true;
      };
      if (n > 0) ok = issue_s(0);
      for (int c = 0; c < n && ok; ++c) {
        const int sv = c % NVS, yb = c & 1;
        const uint32_t vslot = sV + uint32_t(sv) * kTile;
        // v' = [v | ones]: the second 64-column block sits at the ones block.
        const uint32_t dV = sm103::sdesc_sw128_lo(vslot, sOnes - vslot);
        const uint32_t tY = tmem + COL_Y + uint32_t(yb) * 96u;
        // Sig^T += v'^T phi_K
        if (!(ok = attn::warp_wait(bar(B_PHIK), uint32_t(c) & 1u, ab))) break;
        if (!(ok = attn::warp_wait(bar(B_VF + sv), uint32_t(c / NVS) & 1u, ab))) break;
        if (c > 0 && !(ok = attn::warp_wait(bar(B_SIGF), uint32_t(c - 1) & 1u, ab))) break;
        sm103::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk)  // 16 tokens per MMA: 2048 bytes of rows
          sm103::mma_ss_warp_lo(tmem + COL_SIG, dV + uint32_t(kk) * 128u, dPK + uint32_t(kk) * 128u, kIdescSig,
                                (c > 0 || kk > 0) ? 1u : 0u, hi);
        sm103::mma_commit_warp(bar(B_SIG));
        // Y'_b = A' v'  (buffer b last read by the epilogue of chunk c - 2)
        if (!(ok = attn::warp_wait(bar(B_A), uint32_t(c) & 1u, ab))) break;
        if (c > 1 && !(ok = attn::warp_wait(bar(B_YF + yb), uint32_t(c / 2 - 1) & 1u, ab))) break;
        sm103::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk)
          sm103::mma_ts_warp_lo(tY, tmem + COL_S + uint32_t(kk) * 8u, dV + uint32_t(kk) * 128u, kIdescYt,
                                kk > 0 ? 1u : 0u, hi);
        sm103::mma_commit_warp(bar(B_VE + sv));
        // The next chunk's S (over A' of this chunk, which the product above has read).
        if (c + 1 < n && !(ok = issue_s(c + 1))) break;
        // Y'_b += phi_Q bf16(Sig of the earlier chunks)
        if (c > 0) {
          if (!(ok = attn::warp_wait(bar(B_PHIQ), uint32_t(c) & 1u, ab))) break;
          if (!(ok = attn::warp_wait(bar(B_SBF), uint32_t(c - 1) & 1u, ab))) break;
          sm103::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < NF / 16; ++kk) {
            const uint32_t oa = (uint32_t(kk >> 2) * kTile + uint32_t(kk & 3) * 32u) >> 4;
            const uint32_t ob = (uint32_t(kk >> 2) * kSbfBlock + uint32_t(kk & 3) * 32u) >> 4;
            sm103::mma_ss_warp_lo(tY, dPQ + oa, dSbf + ob, kIdescYs, 1u, hi);
          }
        }
        sm103::mma_commit_warp(bar(B_Y));
      }
      sm103::mma_commit_warp(bar(B_DONE));
      attn::drain_wait(bar(B_DONE), 0u);
      __syncwarp();
    }
  } else if (warp < 4) {
    // --------------------------------------------- feature warps + epilogue
    sm103::regs_set<kRegFeature, kRegLaunch>();
    const int r = int(threadIdx.x) & 127;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const float sc = p.scale;
    bool ok = true;
    uint32_t wq[8], wk[8];
    // The rows of chunk c (packed bf16) once landed; frees the stage for the
    // next copy together with the S product's commit.
    auto load_rows = [&](int c) -> bool {
      const int s = c % NQK;
      if (!attn::warp_wait(bar(B_QKF + s), uint32_t(c / NQK) & 1u, ab)) return false;
      load_row16(sQK + uint32_t(s) * kQK, r, wq);
      load_row16(sQK + uint32_t(s) * kQK + 2u * kHalf, r, wk);
      sm103::mbar_arrive(bar(B_QKE + s));
      return true;
    };
    auto write_phik = [&]() {
      float unused[16];
      PhiRow<0, true>::run(sPK, r, wk, unused, unused);
      sm103::fence_proxy_async_smem();
      sm103::mbar_arrive(bar(B_PHIK));
    };
    auto write_phiq = [&]() {
      float xs[16], hs[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        xs[2 * i] = sc * sm103::bf16lo_to_f32(wq[i]);
        xs[2 * i + 1] = sc * sm103::bf16hi_to_f32(wq[i]);
        hs[2 * i] = 0.5f * xs[2 * i];
        hs[2 * i + 1] = 0.5f * xs[2 * i + 1];
      }
      PhiRow<0, false>::run(sPQ, r, wq, xs, hs);
      sm103::fence_proxy_async_smem();
      sm103::mbar_arrive(bar(B_PHIQ));
    };
    if (n > 0 && (ok = load_rows(0))) write_phik();
    for (int c = 0; c <= n; ++c) {
      // phi_Q(c), once the readout of chunk c - 1 has read phi_Q(c - 1).
      if (c < n && ok) {
        if (c > 0) ok = attn::warp_wait(bar(B_Y), uint32_t(c - 1) & 1u, ab);
        if (ok) write_phiq();
      }
      if (c > 0) {
        // Epilogue of chunk c - 1 (its Y' is complete: B_Y phase c - 1).
        uint32_t yv[80];
        if (ok && c == n) ok = attn::warp_wait(bar(B_Y), uint32_t(c - 1) & 1u, ab);
        if (ok) {
          sm103::tc_fence_after();
          const uint32_t tY = tmem + lane_off + COL_Y + uint32_t((c - 1) & 1) * 96u;
          uint32_t (&y0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&yv[0]);
          uint32_t (&y1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&yv[32]);
          uint32_t (&y2)[16] = *reinterpret_cast<uint32_t(*)[16]>(&yv[64]);
          sm103::tmem_ld32(tY, y0);
          sm103::tmem_ld32(tY + 32u, y1);
          sm103::tmem_ld16(tY + 64u, y2);
          sm103::tc_fence_before();
          sm103::mbar_arrive(bar(B_YF + ((c - 1) & 1)));
        }
        if (r == 0) sm103::bulk_wait_read0();  // the previous store has read the staging tile
        ok = sm103::named_bar_and(1, 128, ok);
        if (!ok) break;
        const float zr = __uint_as_float(yv[64]);
        const float zinv = 1.f / zr;
        const uint64_t zinv2 = sm103::f2_pack(zinv, zinv);
        auto norm = [&](int e) {  // values e, e + 1 times 1/z, as bf16
          float lo, hi;
          sm103::f2_unpack(sm103::f2_mul(sm103::f2_pack(__uint_as_float(yv[e]), __uint_as_float(yv[e + 1])), zinv2),
                           lo, hi);
          return sm103::pack_bf16x2(lo, hi);
        };
#pragma unroll
        for (int q = 0; q < 8; ++q)  // 16-byte chunk q of row r: values 8q .. 8q+7
          sm103::st_shared_v4(sStg + uint32_t(r) * 128u + ((uint32_t(q) ^ uint32_t(r & 7)) << 4), norm(8 * q),
                              norm(8 * q + 2), norm(8 * q + 4), norm(8 * q + 6));
        sm103::fence_proxy_async_smem();
        sm103::named_bar_sync(1, 128);
        if (r == 0) {
          sm103::tma_store_3d(&p.ty, sStg, 0, (c - 1) * C, bh);
          sm103::bulk_commit();
        }
        const int row = (c - 1) * C + r;
        if (row < p.N) p.z[size_t(bh) * size_t(p.N) + size_t(row)] = zr;
      }
      // The next chunk's rows, and phi_K(c + 1) once the state update of chunk c
      // has read phi_K(c).
      if (c + 1 < n && ok) {
        ok = load_rows(c + 1);
        if (ok) ok = attn::warp_wait(bar(B_SIG), uint32_t(c) & 1u, ab);
        if (ok) write_phik();
      }
      // A warp that gave up keeps iterating without work until the next
      // reduction barrier above, where all four warps agree and leave together.
    }
    if (r == 0) sm103::bulk_wait_read0();
  } else if (warp < 8) {
    // ------------------------------------------------------------- A warps
    sm103::regs_set<kRegA, kRegLaunch>();
    const int r = int(threadIdx.x) & 127;
    const uint32_t tS = tmem + (uint32_t((warp & 3) * 32) << 16) + COL_S;
    const float sc = p.scale;
    const uint64_t sc2 = sm103::f2_pack(sc, sc), half2 = sm103::f2_pack(0.5f, 0.5f), one2 = sm103::f2_pack(1.f, 1.f);
    const int g = warp & 3;  // rows 32 g .. 32 g + 31
    for (int c = 0; c < n; ++c) {
      if (!attn::warp_wait(bar(B_S), uint32_t(c) & 1u, ab)) break;
      sm103::tc_fence_after();
      // Quarter q reads S columns 32q..32q+31 and writes A' columns 16q..16q+15
      // (bf16 pairs), which hold S values already read.  The causal mask is
      // warp-uniform off the diagonal quarter: q < g all visible, q > g none.
      // One quarter body (kept rolled: four roles share each SM sub-partition's
      // instruction cache).
#pragma unroll 1
      for (int q = 0; q <= g; ++q) {
        uint32_t sv[32], pk[16];
        sm103::tmem_ld32(tS + uint32_t(q) * 32u, sv);
        const int lim = r - q * 32;  // columns 32q + j with j <= lim are visible
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          // a = 1 + s (1 + s / 2), s = scale * S, two at a time
          const uint64_t s2 = sm103::f2_mul(sm103::f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), sc2);
          float a0, a1;
          sm103::f2_unpack(sm103::f2_fma(s2, sm103::f2_fma(s2, half2, one2), one2), a0, a1);
          pk[e] = sm103::pack_bf16x2(2 * e <= lim ? a0 : 0.f, 2 * e + 1 <= lim ? a1 : 0.f);
        }
        sm103::tmem_st16(tS + uint32_t(q) * 16u, pk);
      }
      {
        uint32_t zero[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) zero[e] = 0u;
#pragma unroll 1
        for (int q = g + 1; q < 4; ++q) sm103::tmem_st16(tS + uint32_t(q) * 16u, zero);
      }
      sm103::tmem_st_wait();
      sm103::tc_fence_before();
      sm103::mbar_arrive(bar(B_A));
    }
  } else {
    // --------------------------------------------------------- state warps
    sm103::regs_set<kRegState, kRegLaunch>();
    // Thread = value column d (TMEM lane) of Sig^T; columns 0..79 are the
    // readout's B rows (64 values, the z column, zero padding).
    const int d = (warp & 3) * 32 + lane;
    const uint32_t tSig = tmem + (uint32_t((warp & 3) * 32) << 16) + COL_SIG;
    const bool active = (warp & 3) < 3;  // lanes 96..127 hold no value column
    for (int c = 0; c < n; ++c) {
      if (!attn::warp_wait(bar(B_SIG), uint32_t(c) & 1u, ab)) break;
      sm103::tc_fence_after();
      uint32_t pk[80];  // features (2i, 2i+1) of row d, bf16
      if (active) {
#pragma unroll
        for (int g = 0; g < 5; ++g) {
          uint32_t a[32];
          sm103::tmem_ld32(tSig + uint32_t(g) * 32u, a);
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[16 * g + e] = sm103::pack_bf16x2(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
        }
      }
      sm103::tc_fence_before();
      sm103::mbar_arrive(bar(B_SIGF));
      // The readout of chunk c (B_Y) has read the bf16 state of chunk c - 1.
      if (!attn::warp_wait(bar(B_Y), uint32_t(c) & 1u, ab)) break;
      if (active && d < NV) {
        // Row d of the K-major B operand: 16-byte chunk q (features 8q..8q+7) at
        // chunk (q mod 8) of 64-feature block q / 8, swizzled by the row.
#pragma unroll
        for (int q = 0; q < NF / 8; ++q)
          sm103::st_shared_v4(sSbf + uint32_t(q / 8) * kSbfBlock + uint32_t(d) * 128u +
                                  ((uint32_t(q % 8) ^ uint32_t(d & 7)) << 4),
                              pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
      sm103::fence_proxy_async_smem();
      sm103::mbar_arrive(bar(B_SBF));
    }
  }

  sm103::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    sm103::tc_fence_after();
    sm103::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace based
