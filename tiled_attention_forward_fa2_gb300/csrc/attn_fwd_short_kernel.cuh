// Short-unit forward for D <= 64 on sm_103a: two CTAs per SM.
//
// The main forward kernel (attn_fwd_kernel.cuh) owns a whole SM and pairs two
// query tiles per unit; on short rows (a few key tiles per unit) the pair's
// shorter tile waits for the longer one, and every unit boundary leaves the
// tensor core and the softmax warps idle while the next unit's first scores
// are computed (a clock64 timeline of causal b16h32n512d64 showed ~2300 cycles
// per boundary and 68 % of the steady-state step rate).  Here each CTA runs one
// chain of single-tile units with half of the SM (256 threads, 256 TMEM
// columns, ~100 KB of shared memory), and two such CTAs share every SM: while
// one waits at a unit boundary or on a load, the other computes.  Shared
// memory holds two Q buffers, which also stage O, and a four-slot K/V ring
// (two key steps of loads in flight).
//
// Roles (256 threads):
//   warps 0-3 : softmax over the tile's 128 rows (thread = row = TMEM lane),
//               then the unit's epilogue, each warp on its own 32 rows:
//               O / l -> bf16 -> the unit's Q buffer (read for the last time
//               by the unit's last S) -> one TMA store per warp; LSE;
//   warp 4    : TMA producer (Q into one of two buffers, K/V through a ring);
//   warp 5    : TMEM allocation and warp-uniform MMA issue;
//   warps 6-7 : idle (they complete the second warpgroup for setmaxnreg).
// TMEM: S at columns 0..127, O at 128..191, P (bf16 pairs) at 192..255.
// Per unit and key step j: S_j = Q K_j^T -> softmax -> P_j -> O += P_j V_j.
// P has columns of its own, so S_{j+1} is issued as soon as the softmax warps
// have loaded S_j into registers (B_SR), and runs while they compute P_j: a
// key step costs the softmax alone, not the softmax plus P V plus the next S.
// The next unit's S_0 goes out the same way behind the last step's load.  The
// softmax waits for P_{j-1} V_{j-1} (B_PVD) before it writes P_j or rescales
// O.  The softmax warps read O for the epilogue before they hand over the
// next unit's first P, which is what the next unit's first P V (writing O
// afresh) waits for.  Every wait is bounded (wait_bounded).
#pragma once
#include "attn_fwd_kernel.cuh"

namespace attn {

constexpr int kShortThreads = 256;
constexpr int kShortLoadWarp = 4, kShortMmaWarp = 5;
// setmaxnreg: launched at 128 registers a thread (two CTAs of 256 threads fill
// the 65536-register file); the softmax warpgroup takes 168, the other 88.
constexpr uint32_t kShortRegLaunch = 128, kShortRegSoftmax = 168, kShortRegOther = 88;
static_assert(kShortRegSoftmax + kShortRegOther == 2 * kShortRegLaunch, "register split");

struct CfgShort {
  static constexpr int D = 64;
  static constexpr uint32_t TILE = kSubTile;  // 128 rows x 64 bf16
  static constexpr int NQB = 2;               // Q buffers: the next unit's Q loads during this one
  // K/V ring slots: with three the ring ran about one key step ahead and the
  // loads' latency showed at every step (causal b16h32n512d64: 47.8 us with a
  // staging tile for O and three slots).
  static constexpr int NSLOT = 4;
  static constexpr uint32_t OFF_Q = 1024;     // barriers, TMEM slot and abort word below
  static constexpr uint32_t OFF_KV = OFF_Q + NQB * TILE;
  static constexpr uint32_t USED = OFF_KV + NSLOT * TILE;
  static constexpr uint32_t SMEM = USED + 1024;  // + slack to align the base to 1 KB
  // 228 KB of shared memory per SM, 1 KB of it reserved per CTA.
  static_assert(2 * (SMEM + 1024) <= 228u * 1024u, "two CTAs per SM");
  static constexpr int B_Q = 0;                       // [NQB] Q landed (TMA bytes)
  static constexpr int B_OS = NQB;                    // [NQB] the buffer's O stores have read it (4 warps)
  static constexpr int B_FULL = 2 * NQB;              // [NSLOT] ring slot landed
  static constexpr int B_EMPTY = 2 * NQB + NSLOT;     // [NSLOT] ring slot read (MMA commit)
  static constexpr int B_SF = 2 * NQB + 2 * NSLOT;    // S_j ready (MMA commit)
  static constexpr int B_PF = B_SF + 1;               // P_j in TMEM, O rescaled (128 arrivals)
  static constexpr int B_OF = B_PF + 1;               // the unit's last P V done (MMA commit)
  static constexpr int B_SR = B_OF + 1;               // S_j loaded by the softmax warps (128 arrivals)
  static constexpr int B_PVD = B_SR + 1;              // P_j V_j done (MMA commit)
  static constexpr int B_DONE = B_PVD + 1;
  static constexpr int NBAR = B_DONE + 1;
  static_assert(NBAR * 8 <= 512, "barrier area");
  static constexpr uint32_t COL_S = 0, COL_O = 128, COL_P = 192, kCols = 256;
};

template <bool CAUSAL>
__global__ void __launch_bounds__(kShortThreads, 2) attn_fwd_short_sm103(const __grid_constant__ FwdParams p) {
  using C = CfgShort;
  constexpr int NSLOT = C::NSLOT, NQB = C::NQB;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = sm103::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sbase + 512);
  volatile uint32_t* const abort_flag = reinterpret_cast<volatile uint32_t*>(sbase + 516);
  const uint32_t sQ = base + C::OFF_Q, sKV = base + C::OFF_KV;
  auto bar = [base](int i) { return base + 8u * uint32_t(i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Units of this CTA in snake order over the grid, as in the main kernel
  // (units numbered heaviest first when causal).
  const int w0 = int(blockIdx.x), dw = int(gridDim.x);
  auto work = [w0, dw](int k) { return k * dw + ((k & 1) ? dw - 1 - w0 : w0); };
  auto more = [&](int k) { return work(k) < p.n_work; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i)
      sm103::mbar_init(bar(i), (i == C::B_PF || i == C::B_SR) ? uint32_t(BM)
                               : (i >= C::B_OS && i < C::B_OS + NQB) ? 4u : 1u);
    *abort_flag = 0u;
    sm103::fence_mbar_init();
  }
  if (warp == kShortMmaWarp) {
    sm103::tmem_alloc(sm103::smem_u32(tmem_slot), C::kCols);
    sm103::tmem_relinquish();
  }
  if (warp == kShortLoadWarp && lane == 0) {
    sm103::tma_prefetch_map(&p.tq);
    sm103::tma_prefetch_map(&p.tk);
    sm103::tma_prefetch_map(&p.tv);
    sm103::tma_prefetch_map(&p.to32);
  }
  sm103::tc_fence_before();
  __syncthreads();
  sm103::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag, p.timeout_cycles};

  if (warp >= 4) {
    sm103::regs_set<kShortRegOther, kShortRegLaunch>();
    if (warp == kShortLoadWarp) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        int c = 0, nq = 0;  // K/V loads and Q loads issued
        bool ok = true;
        for (int k = 0; ok && more(k); ++k) {
          const Unit u = unit_of<CAUSAL>(p, work(k));
          const int qi = nq % NQB;
          // The buffer is free once the O stores of the unit NQB units back have read it.
          if (nq >= NQB && !(ok = wait_bounded(bar(C::B_OS + qi), uint32_t(nq / NQB - 1) & 1u, ab))) break;
          sm103::mbar_arrive_expect_tx(bar(C::B_Q + qi), C::TILE);
          sm103::tma_load_3d(sQ + uint32_t(qi) * C::TILE, &p.tq, bar(C::B_Q + qi), 0, u.t0 * BM, u.bh);
          ++nq;
          for (int j = 0; ok && j < u.nk0; ++j) {
            for (int kv = 0; kv < 2; ++kv, ++c) {
              const int s = c % NSLOT;
              if (c >= NSLOT && !(ok = wait_bounded(bar(C::B_EMPTY + s), uint32_t(c / NSLOT - 1) & 1u, ab))) break;
              sm103::mbar_arrive_expect_tx(bar(C::B_FULL + s), C::TILE);
              sm103::tma_load_3d(sKV + uint32_t(s) * C::TILE, kv == 0 ? &p.tk : &p.tv, bar(C::B_FULL + s), 0, j * BN,
                                 u.bh);
            }
          }
        }
        // No copy may land after the CTA has left: wait for the loads not yet consumed.
        for (int t = nq > NQB ? nq - NQB : 0; t < nq; ++t) drain_wait(bar(C::B_Q + t % NQB), uint32_t(t / NQB) & 1u);
        for (int t = c > NSLOT ? c - NSLOT : 0; t < c; ++t) drain_wait(bar(C::B_FULL + t % NSLOT), uint32_t(t / NSLOT) & 1u);
      }
      __syncwarp();
    } else if (warp == kShortMmaWarp) {
      // ----------------------------------------------------------- MMA issue
      constexpr uint32_t kIdescS = sm103::idesc_bf16_f32(BM, BN, 0, 0);  // Q, K both K-major
      constexpr uint32_t kIdescO = sm103::idesc_bf16_f32(BM, C::D, 0, 1);  // P from TMEM, V MN-major
      const uint32_t hi = sm103::kSdescHi;
      const uint32_t desc_q = sm103::sdesc_sw128_lo(sQ, 16);
      const uint32_t desc_k = sm103::sdesc_sw128_lo(sKV, 16);
      const uint32_t desc_v = sm103::sdesc_sw128_lo(sKV, kSubTile);
      auto slot_off = [](int c) { return uint32_t(c % NSLOT) * (C::TILE >> 4); };
      auto wait_full = [&](int c) { return warp_wait(bar(C::B_FULL + c % NSLOT), uint32_t(c / NSLOT) & 1u, ab); };
      auto release = [&](int c) { sm103::mma_commit_warp(bar(C::B_EMPTY + c % NSLOT)); };
      const uint32_t dS = tmem + C::COL_S, dO = tmem + C::COL_O, dP = tmem + C::COL_P;
      int cb = 0;   // ring index of the current unit's K_0
      int ns = 0;   // key steps so far (B_SF, B_SR, B_PF, B_PVD phases)
      int nu = 0;   // units so far (Q buffer, B_Q phase, B_OF)
      bool ok = true;
      for (int k = 0; ok && more(k); ++k) {
        const int nk = unit_of<CAUSAL>(p, work(k)).nk0;
        const int qi = nu % NQB;
        // S_j = Q K_j^T, once the softmax warps have loaded S of the step
        // before (global step g - 1) out of TMEM.
        auto issue_s = [&](int j) -> bool {
          const int g = ns + j;
          if (g > 0 && !warp_wait(bar(C::B_SR), uint32_t(g - 1) & 1u, ab)) return false;
          sm103::tc_fence_after();
          const uint32_t dk = desc_k + slot_off(cb + 2 * j), dq = desc_q + uint32_t(qi) * (C::TILE >> 4);
#pragma unroll
          for (int kk = 0; kk < C::D / 16; ++kk)
            sm103::mma_ss_warp_lo(dS, dq + uint32_t(kk) * 2u, dk + uint32_t(kk) * 2u, kIdescS, kk > 0 ? 1u : 0u, hi);
          sm103::mma_commit_warp(bar(C::B_SF));
          release(cb + 2 * j);  // K_j is done with once S_j is
          return true;
        };
        if (!(ok = warp_wait(bar(C::B_Q + qi), uint32_t(nu / NQB) & 1u, ab) && wait_full(cb))) break;
        sm103::tc_fence_after();
        if (!(ok = issue_s(0))) break;
        for (int j = 0; ok && j < nk; ++j) {
          if (j + 1 < nk && !(ok = wait_full(cb + 2 * j + 2) && issue_s(j + 1))) break;
          if (!(ok = wait_full(cb + 2 * j + 1))) break;
          if (!(ok = warp_wait(bar(C::B_PF), uint32_t(ns + j) & 1u, ab))) break;
          sm103::tc_fence_after();
          const uint32_t dv = desc_v + slot_off(cb + 2 * j + 1);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)  // 16 keys per MMA: 8 TMEM columns of P, 16 rows of V
            sm103::mma_ts_warp_lo(dO, dP + uint32_t(kk) * 8u, dv + uint32_t(kk) * (2048u >> 4), kIdescO,
                                  (j > 0 || kk > 0) ? 1u : 0u, hi);
          sm103::mma_commit_warp(bar(C::B_PVD));
          release(cb + 2 * j + 1);
        }
        if (!ok) break;
        sm103::mma_commit_warp(bar(C::B_OF));
        cb += 2 * nk;
        ns += nk;
        ++nu;
      }
      // Every MMA must be finished before TMEM is freed.
      sm103::mma_commit_warp(bar(C::B_DONE));
      drain_wait(bar(C::B_DONE), 0u);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------- softmax and epilogue
    sm103::regs_set<kShortRegSoftmax, kShortRegLaunch>();
    const int r = threadIdx.x;  // row of the tile = TMEM lane
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::COL_S, tO = tmem + lane_off + C::COL_O, tP = tmem + lane_off + C::COL_P;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = sm103::f2_pack(sl2, sl2);
    int ns = 0, nu = 0;  // key steps and units so far (B_SF, B_OF phases)
    bool ok = true;
    for (int k = 0; ok && more(k); ++k) {
      int nk, t0, bh;
      {
        const Unit u = unit_of<CAUSAL>(p, work(k));
        nk = u.nk0;
        t0 = u.t0;
        bh = u.bh;
      }
      const int diag = t0 * BM + r + p.kv_off;  // causal: last visible key of this row
      float m_ref = 0.f, l_run = 0.f;
      for (int j = 0; ok && j < nk; ++j) {
        if (!(ok = warp_wait(bar(C::B_SF), uint32_t(ns + j) & 1u, ab))) break;
        sm103::tc_fence_after();
        float s[BN];
        {
          uint32_t uu[BN];
          sm103::tmem_ld128(tS, uu);
#pragma unroll
          for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(uu[c]);
        }
        // S_j is in registers: its columns go back to the MMA warp for S_{j+1}.
        sm103::tc_fence_before();
        sm103::mbar_arrive(bar(C::B_SR));
        // Masks: keys past N, and keys after the query row when causal.
        int lim = min(BN - 1, p.Nk - 1 - j * BN);
        if (CAUSAL) lim = min(lim, diag - j * BN);
        const int wlim = __reduce_max_sync(0xffffffffu, lim);
        float mrow = -INFINITY;
        if constexpr (CAUSAL) {
          // Per 32-column chunk, decided for the whole warp: chunks every row
          // of the warp sees need no mask, chunks no row sees take no part
          // (their exponentials are skipped below too), and only the chunk the
          // warp's limits fall in is masked row by row (the diagonal tile of a
          // short causal row: 43.7 -> 41.8 us on b16h32n512d64).  Full rows keep
          // one tree over the row (the chunked form measured 1.4 % slower there).
          const int wmin = __reduce_min_sync(0xffffffffu, lim);
          if (wmin < BN - 1) {
#pragma unroll
            for (int q = 0; q < BN / 32; ++q) {
              if (q * 32 + 31 <= wmin || q * 32 > wlim) continue;
#pragma unroll
              for (int e = 0; e < 32; ++e) s[q * 32 + e] = q * 32 + e > lim ? -INFINITY : s[q * 32 + e];
            }
          }
#pragma unroll
          for (int q = 0; q < BN / 32; ++q) {
            if (q * 32 > wlim) continue;
            const float* c = s + q * 32;
            float a0 = sm103::max3(c[0], c[1], c[2]), a1 = sm103::max3(c[3], c[4], c[5]);
            float a2 = sm103::max3(c[6], c[7], c[8]), a3 = sm103::max3(c[9], c[10], c[11]);
#pragma unroll
            for (int e = 12; e < 28; e += 8) {
              a0 = sm103::max3(a0, c[e], c[e + 1]);
              a1 = sm103::max3(a1, c[e + 2], c[e + 3]);
              a2 = sm103::max3(a2, c[e + 4], c[e + 5]);
              a3 = sm103::max3(a3, c[e + 6], c[e + 7]);
            }
            a0 = sm103::max3(a0, c[28], c[29]);
            a1 = sm103::max3(a1, c[30], c[31]);
            mrow = sm103::max3(mrow, fmaxf(a0, a1), fmaxf(a2, a3));
          }
        } else {
          if (lim < BN - 1) {
#pragma unroll
            for (int c = 0; c < BN; ++c) s[c] = c > lim ? -INFINITY : s[c];
          }
          float mx0 = sm103::max3(s[0], s[1], s[2]);
          float mx1 = sm103::max3(s[3], s[4], s[5]);
          float mx2 = sm103::max3(s[6], s[7], s[8]);
          float mx3 = sm103::max3(s[9], s[10], s[11]);
#pragma unroll
          for (int c = 12; c + 8 <= BN - 4; c += 8) {
            mx0 = sm103::max3(mx0, s[c], s[c + 1]);
            mx1 = sm103::max3(mx1, s[c + 2], s[c + 3]);
            mx2 = sm103::max3(mx2, s[c + 4], s[c + 5]);
            mx3 = sm103::max3(mx3, s[c + 6], s[c + 7]);
          }
          mx0 = sm103::max3(mx0, s[BN - 4], s[BN - 3]);
          mx1 = sm103::max3(mx1, s[BN - 2], s[BN - 1]);
          mrow = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
        }
        const float cand = mrow * sl2;
        // Lazy rescale as in the main kernel: the reference max moves only when
        // the row's max grows by more than 2^kRescaleLog2.
        float alpha = 1.f;
        if (j == 0) {
          m_ref = cand;
        } else if (cand > m_ref + kRescaleLog2) {
          alpha = sm103::ex2_approx(m_ref - cand);
          m_ref = cand;
        }
        const uint64_t negm = sm103::f2_pack(-m_ref, -m_ref);
        uint64_t acc0 = 0, acc1 = 0;
        // 32-column chunks masked for every row of the warp (the diagonal tile's
        // upper right, keys past N) need no exponentials: P is zero there.  The
        // exponential unit is what a key step waits on, and the warp of the
        // other CTA on this sub-partition gets the cycles.
        uint32_t pk[BN / 32][16];
#pragma unroll
        for (int q = 0; q < BN / 32; ++q) {
          if (q * 32 > wlim) {
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[q][e] = 0u;
            continue;
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint64_t t = sm103::f2_fma(sm103::f2_pack(s[q * 32 + 2 * e], s[q * 32 + 2 * e + 1]), sl2x2, negm);
            float t_lo, t_hi;
            sm103::f2_unpack(t, t_lo, t_hi);
            const float p0 = sm103::ex2_approx(t_lo);
            const float p1 = sm103::ex2_approx(t_hi);
            pk[q][e] = sm103::pack_bf16x2(p0, p1);
            if (e & 1)
              acc1 = sm103::f2_add(acc1, sm103::f2_pack(p0, p1));
            else
              acc0 = sm103::f2_add(acc0, sm103::f2_pack(p0, p1));
          }
        }
        // P_{j-1} V_{j-1} has read P and written O (at j = 0 the epilogue
        // already waited for the previous unit's last P V): only the stores of
        // P_j and the rescale of O wait for it, the exponentials above do not.
        if (j > 0 && !(ok = warp_wait(bar(C::B_PVD), uint32_t(ns + j - 1) & 1u, ab))) break;
        sm103::tc_fence_after();
#pragma unroll
        for (int q = 0; q < BN / 32; ++q) sm103::tmem_st16(tP + q * 16, pk[q]);
        float a0, a1, a2, a3;
        sm103::f2_unpack(acc0, a0, a1);
        sm103::f2_unpack(acc1, a2, a3);
        const float rowsum = (a0 + a1) + (a2 + a3);
        l_run = j == 0 ? rowsum : fmaf(alpha, l_run, rowsum);
        // O *= alpha when a row of the warp moved its reference max (the P V
        // that last wrote O is done: B_PVD above).
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int q = 0; q < C::D / 32; ++q) {
            uint32_t v[32];
            sm103::tmem_ld32(tO + q * 32, v);
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            sm103::tmem_st32(tO + q * 32, v);
          }
        }
        sm103::tmem_st_wait();
        sm103::tc_fence_before();
        sm103::mbar_arrive(bar(C::B_PF));
        if (j == 0 && nu > 0 && lane == 0) {
          // The previous unit's O store from this warp has read its staging rows
          // by now: that Q buffer is free for the loader once all four warps say so.
          sm103::bulk_wait_read0();
          sm103::mbar_arrive(bar(C::B_OS + (nu - 1) % NQB));
        }
      }
      // Epilogue: O is final once the unit's last P V is done.  Each warp
      // works on its own 32 rows; nothing is shared between the warps.
      if (!ok || !(ok = warp_wait(bar(C::B_OF), uint32_t(nu) & 1u, ab))) break;
      sm103::tc_fence_after();
      const int row = t0 * BM + r;
      if (row < p.Nq) p.lse[size_t(bh) * size_t(p.Nq) + size_t(row)] = (m_ref + log2f(l_run)) * 0.6931471805599453f;
      const float inv_l = 1.f / l_run;
      // Rows 32 w .. 32 w + 31 of the unit's Q buffer, in the 128-byte-swizzled
      // layout of a 32-row box (row r' at 128 r', chunk c at ((c ^ (r' & 7)) * 16)).
      const uint32_t stg = sQ + uint32_t(nu % NQB) * C::TILE + uint32_t(warp) * 4096u;
#pragma unroll
      for (int q = 0; q < C::D / 32; ++q) {
        uint32_t v[32];
        sm103::tmem_ld32(tO + q * 32, v);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = sm103::pack_bf16x2(__uint_as_float(v[2 * e]) * inv_l, __uint_as_float(v[2 * e + 1]) * inv_l);
        const uint32_t rowbase = stg + uint32_t(lane) * 128u;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const uint32_t chunk = uint32_t(q * 4 + c4);
          sm103::st_shared_v4(rowbase + ((chunk ^ uint32_t(lane & 7)) << 4), pk[4 * c4], pk[4 * c4 + 1],
                              pk[4 * c4 + 2], pk[4 * c4 + 3]);
        }
      }
      sm103::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        // Rows past Nq are clipped by the map; a box starting past them is not issued.
        if (t0 * BM + warp * 32 < p.Nq) sm103::tma_store_3d(&p.to32, stg, 0, t0 * BM + warp * 32, bh);
        sm103::bulk_commit();
      }
      ns += nk;
      ++nu;
    }
    if (lane == 0) sm103::bulk_wait_read0();  // the stores have read shared memory
  }

  sm103::tc_fence_before();
  __syncthreads();
  if (warp == kShortMmaWarp) {
    sm103::tc_fence_after();
    sm103::tmem_dealloc(tmem, C::kCols);
  }
}

}  // namespace attn
