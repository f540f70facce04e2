// Attention backward for sm_103a (GB300): dQ, dK, dV of sum(dO * O) for the
// forward in attn_fwd_kernel.cuh.
//
// The pages ("GPUの爆発的な性能向上", ja.news.hada.io topic 14783, closing
// discussion and section "アドレス生成とTMA") call the backward an order of
// magnitude harder than the forward and print no formula; this is the chain
// rule through the softmax with the forward's saved LSE:
//   p_ij  = exp(scale s_ij - LSE_i),  dp_ij = dO_i . v_j,  D_i = dO_i . O_i,
//   ds_ij = p_ij (dp_ij - D_i),  dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
// Two kernels, launched in this order on one stream; neither needs scratch
// memory (D is an output):
//   attn_bwd_dq_sm103  : one CTA per 128-query tile.  D_i from O and dO, then
//       per key tile S = Q K^T (into one of two TMEM buffers, alternating) and
//       dP = dO V^T into TMEM, dS (bf16) over S, dQ += dS K with dS read from
//       TMEM; dQ stored with TMA.  The elementwise warps take dP into
//       registers first and release its columns, so the next key tile's S and
//       dP are computed while they work on this one's dS.
//   attn_bwd_dkdv_sm103: per 128-key tile, transposed: per half of a query
//       tile (64 queries) S^T = K Q^T and dP^T = V dO^T into one of two TMEM
//       buffers, P^T and dS^T (bf16) over them, then dV += P^T dO and
//       dK += dS^T Q; the next half's S^T and dP^T are computed while the
//       elementwise warps work on this one.  The per-query LSE and D reach
//       every thread through shared memory; dK, dV stored with TMA.  One CTA
//       per SM walks the key tiles (D <= 128): the next tile's K and V load,
//       and its first S^T and dP^T run, while this tile's dK and dV are stored.
// Warp roles as in the forward: warps 0-3 elementwise (thread = TMEM lane =
// row), warp 4 TMA producer, warp 5 TMEM allocation and warp-uniform MMA issue.
// Every wait is bounded (see wait_bounded in attn_fwd_kernel.cuh).
#pragma once
#include "attn_fwd_kernel.cuh"

namespace attn {

// 64 consecutive columns of this thread's lane as two x32 loads and one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr), "r"(taddr + 32u)
      : "memory");
}

constexpr int kBwdThreads = 192;
constexpr int kBwdLoadWarp = 4, kBwdMmaWarp = 5;

struct BwdParams {
  CUtensorMap tq, tdo, tk, tv;  // Q, dO {D, Nq, B*H}; K, V {D, Nk, B*H}; box {64, 128, 1}
  CUtensorMap tdq, tdk, tdv;    // stores: dQ {D, Nq, B*H}; dK, dV {D, Nk, B*H}
  const __nv_bfloat16* o;       // [B*H, Nq, D] forward output
  const __nv_bfloat16* dout;    // [B*H, Nq, D]
  const float* lse;             // [B*H, Nq] natural log
  float* delta;                 // [B*H, Nq] D_i: written by the dQ kernel, read by the dK/dV kernel
  int Nq, Nk, kv_off, bh, n_qtiles, n_ktiles;
  int lpt;                      // causal dQ order: heads per longest-first band (0: a head's tiles adjacent)
  int d;                        // true head dim (<= the kernel's D; the rest is zero padding)
  int ld;                       // row stride (elements) of every [.., N, D] tensor: a multiple of 8, >= d
  float scale;                  // softmax scale
  float scale_log2;             // scale * log2(e)
  long long timeout_cycles;
};

// ------------------------------------------------------------------ dQ kernel
template <int D>
struct CfgDq {
  static constexpr int KB = D / 64;
  // Keys per step: 128, or 64 at D = 256, where S, dP and dQ (256 columns)
  // must share TMEM's 512 columns and the K, V tiles shared memory with Q, dO.
  static constexpr int BNK = D == 256 ? 64 : 128;
  static constexpr uint32_t TILE = KB * kSubTile;               // Q, dO: 128 rows
  static constexpr uint32_t KVSUB = uint32_t(BNK) * 128u;       // one 64-column box of a K or V tile
  static constexpr uint32_t TILE_KV = KB * KVSUB;
  // Separate rings for K and V, sized to how long each tile is needed: K_j
  // until dQ_j (the end of step j), V_j only until dP_j.  Three K slots and two
  // V slots give every load a whole step of lead (one four-slot ring left the
  // MMA warp waiting ~1760 cycles a step for K/V); at D = 256 two and one fit.
  static constexpr int NK = D == 64 ? 5 : (D == 128 ? 3 : 2), NV = D == 64 ? 3 : (D == 128 ? 2 : 1);
  static constexpr int NSLOT = NK + NV;            // K slots, then V slots
  static constexpr uint32_t OFF_Q = 1024, OFF_DO = OFF_Q + TILE, OFF_KV = OFF_DO + TILE;
  static constexpr uint32_t SMEM = OFF_KV + NSLOT * TILE_KV + 1024;
  static_assert(SMEM <= 232448, "shared memory");
  // B_SF: S_j and dP_j in TMEM (MMA commit); B_DPR: dP_j in the elementwise
  // warps' registers (128 arrivals); B_DSF[j & 1]: dS_j in TMEM (128 arrivals).
  // Two dS barriers: S_{j+1} is issued before the MMA warp waits for dS_j, so
  // on a single barrier dS_{j+1} could complete a phase the MMA warp had not
  // yet seen; dS_{j+2} needs S_{j+2}, which is only issued after that wait.
  static constexpr int B_Q = 0, B_FULL = 1, B_EMPTY = 1 + NSLOT, B_SF = 1 + 2 * NSLOT, B_DSF = B_SF + 1,
                       B_DPR = B_DSF + 2, B_QDONE = B_DPR + 1, B_DONE = B_QDONE + 1, NBAR = B_DONE + 1;
  // S_j at COL_S + BNK (j & 1), dS_j (bf16) over its first BNK / 2 columns.
  static constexpr uint32_t COL_S = 0, COL_DP = 2 * BNK, COL_DQ = D == 256 ? 256 : 384;
  static_assert(COL_DP + BNK <= COL_DQ && COL_DQ + D <= kTmemCols, "TMEM columns");
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1) attn_bwd_dq_sm103(const __grid_constant__ BwdParams p) {
  using C = CfgDq<D>;
  constexpr int KB = C::KB, NK = C::NK, NV = C::NV, BNK = C::BNK;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = sm103::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sbase + 512);
  volatile uint32_t* const abort_flag = reinterpret_cast<volatile uint32_t*>(sbase + 516);
  const uint32_t sQ = base + C::OFF_Q, sDO = base + C::OFF_DO, sKV = base + C::OFF_KV;
  auto bar = [base](int i) { return base + 8u * uint32_t(i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Causal with bands (p.lpt > 0): heaviest query tiles first within bands of
  // p.lpt heads.  Otherwise (full, or causal tiles of about equal key ranges
  // whose K and V exceed half of L2) the tiles of one head are adjacent, so
  // the CTAs running at one time read its K and V from HBM once.
  int qt, bh;
  if (CAUSAL && p.lpt) {
    const int span = p.lpt * p.n_qtiles;
    const int band = int(blockIdx.x) / span, idx = int(blockIdx.x) - band * span;
    const int g = min(p.lpt, p.bh - band * p.lpt);
    qt = p.n_qtiles - 1 - idx / g;
    bh = band * p.lpt + idx % g;
  } else {
    qt = int(blockIdx.x % uint32_t(p.n_qtiles));
    bh = int(blockIdx.x / uint32_t(p.n_qtiles));
  }
  const int m0 = qt * BM;
  const int n_kt = (p.Nk + BNK - 1) / BNK;
  const int nk = CAUSAL ? min(n_kt, (min(m0 + BM - 1, p.Nq - 1) + p.kv_off) / BNK + 1) : n_kt;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i)
      sm103::mbar_init(bar(i), (i == C::B_DSF || i == C::B_DSF + 1 || i == C::B_DPR) ? uint32_t(BM) : 1u);
    *abort_flag = 0u;
    sm103::fence_mbar_init();
  }
  if (warp == kBwdMmaWarp) {
    sm103::tmem_alloc(sm103::smem_u32(tmem_slot), kTmemCols);
    sm103::tmem_relinquish();
  }
  sm103::tc_fence_before();
  __syncthreads();
  sm103::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag, p.timeout_cycles};

  if (warp == kBwdLoadWarp) {
    if (lane == 0) {
      sm103::mbar_arrive_expect_tx(bar(C::B_Q), 2u * C::TILE);
      for (int kb = 0; kb < KB; ++kb) {
        sm103::tma_load_3d(sQ + kb * kSubTile, &p.tq, bar(C::B_Q), kb * 64, m0, bh);
        sm103::tma_load_3d(sDO + kb * kSubTile, &p.tdo, bar(C::B_Q), kb * 64, m0, bh);
      }
      int ck = 0, cv = 0;  // K and V loads issued
      bool ok = true;
      auto load = [&](int j, bool is_k) -> bool {
        const int n = is_k ? NK : NV, s = (is_k ? 0 : NK) + j % n;
        if (j >= n && !wait_bounded(bar(C::B_EMPTY + s), uint32_t(j / n - 1) & 1u, ab)) return false;
        sm103::mbar_arrive_expect_tx(bar(C::B_FULL + s), C::TILE_KV);
        for (int kb = 0; kb < KB; ++kb)
          sm103::tma_load_3d(sKV + s * C::TILE_KV + kb * C::KVSUB, is_k ? &p.tk : &p.tv, bar(C::B_FULL + s), kb * 64,
                             j * BNK, bh);
        return true;
      };
      for (int j = 0; ok && j < nk; ++j) {
        if (!(ok = load(j, true))) break;
        ++ck;
        if (!(ok = load(j, false))) break;
        ++cv;
      }
      drain_wait(bar(C::B_Q), 0u);
      for (int t = ck > NK ? ck - NK : 0; t < ck; ++t) drain_wait(bar(C::B_FULL + t % NK), uint32_t(t / NK) & 1u);
      for (int t = cv > NV ? cv - NV : 0; t < cv; ++t) drain_wait(bar(C::B_FULL + NK + t % NV), uint32_t(t / NV) & 1u);
    }
    __syncwarp();
  } else if (warp == kBwdMmaWarp) {
    constexpr uint32_t kIdescS = sm103::idesc_bf16_f32(BM, BNK, 0, 0);  // both operands K-major
    constexpr uint32_t kIdescQ = sm103::idesc_bf16_f32(BM, D, 0, 1);    // dS from TMEM, K MN-major
    const uint64_t dq_k = sm103::sdesc_sw128(sQ, 16, 1024), ddo_k = sm103::sdesc_sw128(sDO, 16, 1024);
    const uint64_t dkv_k = sm103::sdesc_sw128(sKV, 16, 1024), dkv_mn = sm103::sdesc_sw128(sKV, C::KVSUB, 1024);
    // Ring slot of K_j (kv = 0) or V_j (kv = 1), its fill phase, and release.
    auto slot = [](int j, int kv) { return kv == 0 ? j % NK : NK + j % NV; };
    auto slot_off = [&](int j, int kv) { return uint64_t(uint32_t(slot(j, kv)) * (C::TILE_KV >> 4)); };
    // 16 columns kk of D: in a 128-row tile (Q, dO) and in a K or V tile.
    auto off_q = [](int kk) { return uint64_t((uint32_t(kk >> 2) * kSubTile + uint32_t(kk & 3) * 32u) >> 4); };
    auto off_kv = [](int kk) { return uint64_t((uint32_t(kk >> 2) * C::KVSUB + uint32_t(kk & 3) * 32u) >> 4); };
    auto wait_full = [&](int j, int kv) {
      return warp_wait(bar(C::B_FULL + slot(j, kv)), uint32_t(j / (kv == 0 ? NK : NV)) & 1u, ab);
    };
    auto release = [&](int j, int kv) { sm103::mma_commit_warp(bar(C::B_EMPTY + slot(j, kv))); };
    auto issue_s = [&](int j) {  // S = Q K_j^T into buffer j & 1
      const uint64_t dk = dkv_k + slot_off(j, 0);
      const uint32_t dS = tmem + C::COL_S + uint32_t(j & 1) * BNK;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) sm103::mma_ss_warp(dS, dq_k + off_q(kk), dk + off_kv(kk), kIdescS, kk > 0 ? 1u : 0u);
    };
    auto issue_dp = [&](int j) {  // dP = dO V_j^T; S_j and dP_j ready together
      const uint64_t dv = dkv_k + slot_off(j, 1);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        sm103::mma_ss_warp(tmem + C::COL_DP, ddo_k + off_q(kk), dv + off_kv(kk), kIdescS, kk > 0 ? 1u : 0u);
      sm103::mma_commit_warp(bar(C::B_SF));
      release(j, 1);  // V_j is done with
    };
    bool ok = warp_wait(bar(C::B_Q), 0u, ab) && wait_full(0, 0) && wait_full(0, 1);
    if (ok) {
      sm103::tc_fence_after();
      issue_s(0);
      issue_dp(0);
    }
    for (int j = 0; ok && j < nk; ++j) {
      if (j + 1 < nk) {
        // S_{j+1} goes to the other buffer as soon as K_{j+1} is in (its dS_{j-1}
        // was read by the dQ MMA issued before, and the elementwise warps had
        // finished with it), so it runs while they work on step j; dP_{j+1} once
        // dP_j has left TMEM.
        if (!(ok = wait_full(j + 1, 0))) break;
        sm103::tc_fence_after();
        issue_s(j + 1);
        if (!(ok = wait_full(j + 1, 1))) break;
        if (!(ok = warp_wait(bar(C::B_DPR), uint32_t(j) & 1u, ab))) break;
        sm103::tc_fence_after();
        issue_dp(j + 1);
      }
      if (!(ok = warp_wait(bar(C::B_DSF + (j & 1)), uint32_t(j >> 1) & 1u, ab))) break;
      sm103::tc_fence_after();
      const uint64_t dkmn = dkv_mn + slot_off(j, 0);
      const uint32_t aS = tmem + C::COL_S + uint32_t(j & 1) * BNK;
#pragma unroll
      for (int kk = 0; kk < BNK / 16; ++kk)  // dQ += dS K_j: 16 keys per MMA
        sm103::mma_ts_warp(tmem + C::COL_DQ, aS + kk * 8, dkmn + uint64_t(kk * (2048 >> 4)), kIdescQ,
                           (j > 0 || kk > 0) ? 1u : 0u);
      release(j, 0);  // K_j is done with
    }
    sm103::mma_commit_warp(bar(C::B_QDONE));
    sm103::mma_commit_warp(bar(C::B_DONE));
    drain_wait(bar(C::B_DONE), 0u);
    __syncwarp();
  } else {
    // ------------------------------------------------------- elementwise
    const int r = threadIdx.x;
    const int row = m0 + r;
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    // D_i = dO_i . O_i and the row's LSE in base 2 (rows past Nq: P = 0).
    float dlt = 0.f, lse2 = INFINITY;
    if (row < p.Nq) {
      // Rows are p.ld elements apart (a multiple of 8, >= d); a partial last
      // group of 8 is read in full (it lies within the row's padding) and
      // masked to the first d elements.
      const uint4* po = reinterpret_cast<const uint4*>(p.o + (size_t(bh) * p.Nq + row) * size_t(p.ld));
      const uint4* pd = reinterpret_cast<const uint4*>(p.dout + (size_t(bh) * p.Nq + row) * size_t(p.ld));
      float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
      for (int x = 0; x < p.d / 8; ++x) {
        const uint4 uo = po[x], ud = pd[x];
        const uint32_t wo[4] = {uo.x, uo.y, uo.z, uo.w}, wd[4] = {ud.x, ud.y, ud.z, ud.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          a0 = fmaf(sm103::bf16lo_to_f32(wo[e]), sm103::bf16lo_to_f32(wd[e]), a0);
          a1 = fmaf(sm103::bf16hi_to_f32(wo[e]), sm103::bf16hi_to_f32(wd[e]), a1);
        }
      }
      if (p.d & 7) {
        const int x = p.d / 8, rem = p.d & 7;
        const uint4 uo = po[x], ud = pd[x];
        const uint32_t wo[4] = {uo.x, uo.y, uo.z, uo.w}, wd[4] = {ud.x, ud.y, ud.z, ud.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (2 * e < rem) a0 = fmaf(sm103::bf16lo_to_f32(wo[e]), sm103::bf16lo_to_f32(wd[e]), a0);
          if (2 * e + 1 < rem) a1 = fmaf(sm103::bf16hi_to_f32(wo[e]), sm103::bf16hi_to_f32(wd[e]), a1);
        }
      }
      dlt = a0 + a1;
      lse2 = p.lse[size_t(bh) * p.Nq + row] * 1.4426950408889634f;
      p.delta[size_t(bh) * p.Nq + row] = dlt;
    }
    const uint64_t sl2x2 = sm103::f2_pack(sl2, sl2), nl2 = sm103::f2_pack(-lse2, -lse2);
    bool ok = true;
    for (int j = 0; j < nk; ++j) {
      if (!(ok = warp_wait(bar(C::B_SF), uint32_t(j) & 1u, ab))) break;
      sm103::tc_fence_after();
      int lim = min(BNK - 1, p.Nk - 1 - j * BNK);
      if (CAUSAL) lim = min(lim, row + p.kv_off - j * BNK);
      // dP_j - D into registers, then its TMEM columns go back to the MMA warp.
      float dpd[BNK];
      {
        uint32_t ud[BNK];
        if constexpr (BNK == 128)
          sm103::tmem_ld128(tmem + lane_off + C::COL_DP, ud);
        else
          tmem_ld64(tmem + lane_off + C::COL_DP, ud);
#pragma unroll
        for (int c = 0; c < BNK; ++c) dpd[c] = __uint_as_float(ud[c]) - dlt;
      }
      sm103::tc_fence_before();
      sm103::mbar_arrive(bar(C::B_DPR));
      const uint32_t tS = tmem + lane_off + C::COL_S + uint32_t(j & 1) * BNK;
#pragma unroll
      for (int q = 0; q < BNK / 32; ++q) {
        uint32_t us[32];
        sm103::tmem_ld32(tS + q * 32, us);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint64_t t = sm103::f2_fma(sm103::f2_pack(__uint_as_float(us[2 * e]), __uint_as_float(us[2 * e + 1])), sl2x2, nl2);
          float t0, t1;
          sm103::f2_unpack(t, t0, t1);
          const int c = q * 32 + 2 * e;
          const float p0 = c > lim ? 0.f : sm103::ex2_approx(t0);
          const float p1 = c + 1 > lim ? 0.f : sm103::ex2_approx(t1);
          pk[e] = sm103::pack_bf16x2(p0 * dpd[c], p1 * dpd[c + 1]);
        }
        sm103::tmem_st16(tS + q * 16, pk);  // dS over the first BNK / 2 columns of S_j
      }
      sm103::tmem_st_wait();
      sm103::tc_fence_before();
      sm103::mbar_arrive(bar(C::B_DSF + (j & 1)));
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_bounded(bar(C::B_QDONE), 0u, ab));
    if (ok) {
      sm103::tc_fence_after();
      // dQ * scale -> bf16 into the idle Q tile (128-byte swizzle layout), then TMA.
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t v[32];
        sm103::tmem_ld32(tmem + lane_off + C::COL_DQ + q * 32, v);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = sm103::pack_bf16x2(__uint_as_float(v[2 * e]) * p.scale, __uint_as_float(v[2 * e + 1]) * p.scale);
        const uint32_t rowbase = sQ + uint32_t(q >> 1) * kSubTile + uint32_t(r) * 128u;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const uint32_t chunk = uint32_t((q & 1) * 4 + c4);
          sm103::st_shared_v4(rowbase + ((chunk ^ uint32_t(r & 7)) << 4), pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2],
                              pk[4 * c4 + 3]);
        }
      }
      sm103::fence_proxy_async_smem();
    }
    ok = sm103::named_bar_and(1, BM, ok);
    if (ok && r == 0) {
      for (int kb = 0; kb < KB; ++kb) sm103::tma_store_3d(&p.tdq, sQ + kb * kSubTile, kb * 64, m0, bh);
      sm103::bulk_commit();
      sm103::bulk_wait_read0();
    }
  }
  sm103::tc_fence_before();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    sm103::tc_fence_after();
    sm103::tmem_dealloc(tmem, kTmemCols);
  }
}

// --------------------------------------------------------------- dK/dV kernel
template <int D>
struct CfgDkv {
  static constexpr int KB = D / 64;
  // At D = 256 dK and dV (256 fp32 columns each) do not fit in TMEM together:
  // each key tile is shared by two CTAs, each accumulating one 128-column half
  // of dK and dV (both compute the whole S^T and dP^T); and with whole K and V
  // tiles of 64 KB in shared memory, a stage holds 32 queries.
  static constexpr int DACC = D == 256 ? 128 : D;          // dK, dV columns per CTA
  static constexpr int NHALF = D / DACC;                   // CTAs per key tile
  static constexpr int SQ = D == 256 ? 32 : 128;           // queries per stage
  static constexpr int HQ = D == 256 ? 32 : 64;            // queries per sub-step
  static constexpr int NSUB = SQ / HQ;                     // sub-steps per stage
  static constexpr uint32_t TILE = KB * kSubTile;          // K, V: 128 rows
  static constexpr uint32_t QSUB = uint32_t(SQ) * 128u;    // one 64-column box of a stage's Q or dO
  static constexpr uint32_t STILE = KB * QSUB;
  static constexpr int NSTAGE = 2;                         // (Q_i, dO_i, LSE, D) stages
  static constexpr uint32_t OFF_VEC = 1024;                // [NSTAGE][2][SQ] fp32: LSE*log2e, D
  static constexpr uint32_t OFF_K = 4096, OFF_V = OFF_K + TILE, OFF_ST = OFF_V + TILE;  // stage s: Q, dO
  static constexpr uint32_t SMEM = OFF_ST + NSTAGE * 2 * STILE + 1024;
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(OFF_VEC + NSTAGE * 2 * SQ * 4 <= OFF_K, "vector area");
  // Sub-steps h (HQ queries): S^T and dP^T in buffer h & 1 (B_SF[h & 1], MMA
  // commit), P^T and dS^T written over them (B_PF[h & 1], 128 arrivals).
  // B_KV: a unit's K and V landed (TMA bytes); B_KVE: its last S^T and dP^T
  // (the products that read K and V) done (MMA commit); B_ACC: its last
  // products done (MMA commit); B_EPI: the epilogue has read dK, dV out of
  // TMEM (128 arrivals); B_STG: a unit's dK, dV stores have read their
  // staging (thread 0).
  static constexpr int B_KV = 0, B_SFULL = 1, B_SEMPTY = 1 + NSTAGE, B_SF = 1 + 2 * NSTAGE, B_PF = B_SF + 2,
                       B_ACC = B_PF + 2, B_EPI = B_ACC + 1, B_STG = B_EPI + 1, B_KVE = B_STG + 1,
                       B_DONE = B_KVE + 1, NBAR = B_DONE + 1;
  // One CTA per SM walking key tiles (D <= 128, where a stage slot holds a
  // unit's dK and dV for their stores), or one CTA per key tile (D = 256).
  static constexpr bool PERSIST = 2u * STILE >= 2u * uint32_t(BM) * uint32_t(DACC) * 2u;
  // Buffer b: S^T at BUF b, dP^T at BUF b + HQ (HQ columns each; P^T, dS^T
  // bf16 over their first HQ / 2).
  static constexpr uint32_t COL_S = 0, COL_DP = HQ, BUF = 2 * HQ, COL_DV = 256, COL_DK = 256 + DACC;
  static_assert(2 * BUF <= COL_DV && COL_DK + DACC <= kTmemCols, "TMEM columns");
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1) attn_bwd_dkdv_sm103(const __grid_constant__ BwdParams p) {
  using C = CfgDkv<D>;
  constexpr int KB = C::KB, NSTAGE = C::NSTAGE, SQ = C::SQ, HQ = C::HQ, NSUB = C::NSUB, DACC = C::DACC;
  constexpr bool PERSIST = C::PERSIST;
  constexpr int kRounds = PERSIST ? 0x7fffffff : 1;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = sm103::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sbase + 512);
  volatile uint32_t* const abort_flag = reinterpret_cast<volatile uint32_t*>(sbase + 516);
  float* const vec = reinterpret_cast<float*>(sbase + C::OFF_VEC);  // [stage][0: lse2, 1: D][SQ]
  const uint32_t sK = base + C::OFF_K, sV = base + C::OFF_V, sST = base + C::OFF_ST;
  auto bar = [base](int i) { return base + 8u * uint32_t(i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Units: one key tile of one (b, h) (and, at D = 256, one column half of dK
  // and dV).  Causal: key-tile major, the key tiles seen by the most queries
  // (the first ones) first; else (b, h) major.  The CTAs of one key tile's
  // column halves are adjacent.  PERSIST: CTA c takes units k G + c (even
  // rounds k) and k G + G - 1 - c (odd rounds), G = grid size, as the forward.
  const int n_units = p.n_ktiles * p.bh * C::NHALF;
  const int w0 = int(blockIdx.x), dw = int(gridDim.x);
  auto work = [w0, dw](int k) { return k * dw + ((k & 1) ? dw - 1 - w0 : w0); };
  auto more = [&](int k) { return work(k) < n_units; };
  struct UnitDkv {
    int half, bh, n0, it0, niter;
  };
  auto unit_at = [&](int w) {
    UnitDkv u;
    u.half = C::NHALF > 1 ? w % C::NHALF : 0;
    const int tile = w / C::NHALF;
    const int kt = CAUSAL ? tile / p.bh : tile % p.n_ktiles;
    u.bh = CAUSAL ? tile % p.bh : tile / p.n_ktiles;
    u.n0 = kt * BN;
    // Query blocks (SQ queries, one stage each) with a query that sees one of
    // these keys (query i sees key n iff n <= i + kv_off): at least one, as
    // causal problems have Nq <= Nk.
    u.it0 = CAUSAL ? max(0, u.n0 - p.kv_off) / SQ : 0;
    u.niter = max(0, (p.Nq + SQ - 1) / SQ - u.it0);
    return u;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      // the producer warp's 32 lanes (vectors written) + lane 0's expect-tx arrival
      if (i >= C::B_SFULL && i < C::B_SFULL + NSTAGE) cnt = 33;
      if (i == C::B_PF || i == C::B_PF + 1 || i == C::B_EPI) cnt = BM;
      sm103::mbar_init(bar(i), cnt);
    }
    *abort_flag = 0u;
    sm103::fence_mbar_init();
  }
  if (warp == kBwdMmaWarp) {
    sm103::tmem_alloc(sm103::smem_u32(tmem_slot), kTmemCols);
    sm103::tmem_relinquish();
  }
  sm103::tc_fence_before();
  __syncthreads();
  sm103::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag, p.timeout_cycles};

  // Phase bookkeeping: every role walks the same units and counts stages (gs:
  // B_SFULL, B_SEMPTY, the stage slot gs % NSTAGE), sub-steps (gh: the S^T /
  // dP^T buffer gh & 1, B_SF, B_PF) and units (nu: B_KV, B_ACC, B_EPI, B_STG)
  // across them.  With PERSIST a unit's dK, dV are staged in the slot of its
  // last stage (free once its MMAs are done), so the next unit's K and V load
  // while they are stored; without it (D = 256) they are staged in the K and V
  // tiles.
  if (warp == kBwdLoadWarp) {
    // -------------------------------------------------------------- producer
    static_assert(NSTAGE == 2, "staging bookkeeping below is for two stage slots");
    int gs = 0;
    int nkv = 0;                // K, V loads issued (one per unit)
    int stg0 = -1, stg1 = -1;   // unit whose dK, dV are staged in slot 0 / 1 (-1: none)
    bool ok = true;
    int nu = 0;
    for (int k = 0; k < kRounds && ok && more(k); ++k, ++nu) {
      const UnitDkv u = unit_at(work(k));
      // K and V: the previous unit's S^T and dP^T must be done with the tiles.
      if (nu > 0 && !(ok = warp_wait(bar(C::B_KVE), uint32_t(nu - 1) & 1u, ab))) break;
      if (lane == 0) {
        sm103::mbar_arrive_expect_tx(bar(C::B_KV), 2u * C::TILE);
        for (int kb = 0; kb < KB; ++kb) {
          sm103::tma_load_3d(sK + kb * kSubTile, &p.tk, bar(C::B_KV), kb * 64, u.n0, u.bh);
          sm103::tma_load_3d(sV + kb * kSubTile, &p.tv, bar(C::B_KV), kb * 64, u.n0, u.bh);
        }
      }
      ++nkv;
      for (int it = 0; ok && it < u.niter; ++it, ++gs) {
        const int st = gs % NSTAGE;
        const int i0 = (u.it0 + it) * SQ;
        // Per-query LSE (base 2) and D for this block (queries past Nq get P = 0),
        // read before the stage is free so the loads overlap the wait; the tile
        // copies go out first once it is free.
        constexpr int NV4 = SQ / 32;  // values per lane
        float lse4[NV4], d4[NV4];
#pragma unroll
        for (int x = 0; x < NV4; ++x) {
          const int i = i0 + lane * NV4 + x;
          const bool live = i < p.Nq;
          lse4[x] = live ? p.lse[size_t(u.bh) * p.Nq + i] * 1.4426950408889634f : INFINITY;
          d4[x] = live ? p.delta[size_t(u.bh) * p.Nq + i] : 0.f;
        }
        if (gs >= NSTAGE && !(ok = warp_wait(bar(C::B_SEMPTY + st), uint32_t(gs / NSTAGE - 1) & 1u, ab))) break;
        // A slot that holds a unit's staged dK, dV is refilled once its stores have read it.
        const int stg = st == 0 ? stg0 : stg1;
        if (PERSIST && stg >= 0) {
          if (!(ok = warp_wait(bar(C::B_STG), uint32_t(stg) & 1u, ab))) break;
          if (st == 0) stg0 = -1; else stg1 = -1;
        }
        if (lane == 0) {
          sm103::mbar_arrive_expect_tx(bar(C::B_SFULL + st), 2u * C::STILE);
          const uint32_t sq = sST + uint32_t(st) * 2u * C::STILE, sdo = sq + C::STILE;
          for (int kb = 0; kb < KB; ++kb) {
            sm103::tma_load_3d(sq + kb * C::QSUB, &p.tq, bar(C::B_SFULL + st), kb * 64, i0, u.bh);
            sm103::tma_load_3d(sdo + kb * C::QSUB, &p.tdo, bar(C::B_SFULL + st), kb * 64, i0, u.bh);
          }
        }
#pragma unroll
        for (int x = 0; x < NV4; ++x) {
          vec[(st * 2 + 0) * SQ + lane * NV4 + x] = lse4[x];
          vec[(st * 2 + 1) * SQ + lane * NV4 + x] = d4[x];
        }
        sm103::mbar_arrive(bar(C::B_SFULL + st));  // releases this lane's vector stores
      }
      if (PERSIST && ok) {  // the unit's last stage will hold its dK, dV
        if ((gs - 1) % NSTAGE == 0) stg0 = nu; else stg1 = nu;
      }
    }
    // No copy may land after the CTA has left.  Loads before the last NSTAGE
    // stages, and K, V before the last unit's, were waited on by their users.
    if (lane == 0) {
      if (nkv > 0) drain_wait(bar(C::B_KV), uint32_t(nkv - 1) & 1u);
      for (int t = gs > NSTAGE ? gs - NSTAGE : 0; t < gs; ++t)
        drain_wait(bar(C::B_SFULL + t % NSTAGE), uint32_t(t / NSTAGE) & 1u);
    }
    __syncwarp();
  } else if (warp == kBwdMmaWarp) {
    // ------------------------------------------------------------- MMA issue
    constexpr uint32_t kIdescS = sm103::idesc_bf16_f32(BM, HQ, 0, 0);    // S^T, dP^T: both K-major
    constexpr uint32_t kIdescA = sm103::idesc_bf16_f32(BM, DACC, 0, 1);  // P^T / dS^T from TMEM, B MN-major
    const uint64_t dk_k = sm103::sdesc_sw128(sK, 16, 1024), dv_k = sm103::sdesc_sw128(sV, 16, 1024);
    const uint64_t dst_k = sm103::sdesc_sw128(sST, 16, 1024), dst_mn = sm103::sdesc_sw128(sST, C::QSUB, 1024);
    constexpr uint64_t kSub = uint64_t((HQ * 128u) >> 4);  // HQ rows of a stage tile
    // 16 columns kk of D: in a K or V tile and in a stage's Q or dO.
    auto off_kv = [](int kk) { return uint64_t((uint32_t(kk >> 2) * kSubTile + uint32_t(kk & 3) * 32u) >> 4); };
    auto off_st = [](int kk) { return uint64_t((uint32_t(kk >> 2) * C::QSUB + uint32_t(kk & 3) * 32u) >> 4); };
    int gs = 0, gh = 0;
    bool ok = true;
    int nu = 0;
    for (int k = 0; k < kRounds && ok && more(k); ++k, ++nu) {
      const UnitDkv u = unit_at(work(k));
      // This unit's columns of dO and Q (the B operands of dV and dK).
      const uint64_t half_off = uint64_t((uint32_t(u.half) * uint32_t(DACC / 64) * C::QSUB) >> 4);
      // S^T and dP^T of the unit's sub-step h into buffer (gh + h) & 1.
      auto issue_s = [&](int h) {
        const int st = (gs + h / NSUB) % NSTAGE;
        const uint64_t soff = uint64_t(uint32_t(st) * 2u * (C::STILE >> 4)) + uint64_t(h % NSUB) * kSub;
        const uint64_t q_k = dst_k + soff, do_k = dst_k + soff + (C::STILE >> 4);
        const uint32_t buf = tmem + uint32_t((gh + h) & 1) * C::BUF;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)  // S^T = K Q^T
          sm103::mma_ss_warp(buf + C::COL_S, dk_k + off_kv(kk), q_k + off_st(kk), kIdescS, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)  // dP^T = V dO^T
          sm103::mma_ss_warp(buf + C::COL_DP, dv_k + off_kv(kk), do_k + off_st(kk), kIdescS, kk > 0 ? 1u : 0u);
        sm103::mma_commit_warp(bar(C::B_SF + ((gh + h) & 1)));
      };
      const int nh = NSUB * u.niter;
      if (!(ok = warp_wait(bar(C::B_KV), uint32_t(nu) & 1u, ab) &&
                 warp_wait(bar(C::B_SFULL + gs % NSTAGE), uint32_t(gs / NSTAGE) & 1u, ab)))
        break;
      sm103::tc_fence_after();
      issue_s(0);
      if (PERSIST && nh == 1) sm103::mma_commit_warp(bar(C::B_KVE));  // K and V no longer read after these
      for (int h = 0; ok && h < nh; ++h) {
        const int st = (gs + h / NSUB) % NSTAGE;
        if (h + 1 < nh) {
          // The other buffer's P^T, dS^T (sub-step h - 1) were read by MMAs issued before.
          if ((h + 1) % NSUB == 0) {
            const int g1 = gs + (h + 1) / NSUB;
            if (!(ok = warp_wait(bar(C::B_SFULL + g1 % NSTAGE), uint32_t(g1 / NSTAGE) & 1u, ab))) break;
            sm103::tc_fence_after();
          }
          issue_s(h + 1);
          if (PERSIST && h + 1 == nh - 1) sm103::mma_commit_warp(bar(C::B_KVE));
        }
        if (!(ok = warp_wait(bar(C::B_PF + ((gh + h) & 1)), uint32_t((gh + h) >> 1) & 1u, ab))) break;
        // The first products of a unit overwrite dV and dK: the previous unit's
        // epilogue must have read them.
        if (h == 0 && nu > 0 && !(ok = warp_wait(bar(C::B_EPI), uint32_t(nu - 1) & 1u, ab))) break;
        sm103::tc_fence_after();
        const uint64_t soff = uint64_t(uint32_t(st) * 2u * (C::STILE >> 4)) + uint64_t(h % NSUB) * kSub + half_off;
        const uint64_t q_mn = dst_mn + soff, do_mn = dst_mn + soff + (C::STILE >> 4);
        const uint32_t buf = tmem + uint32_t((gh + h) & 1) * C::BUF;
#pragma unroll
        for (int kk = 0; kk < HQ / 16; ++kk) {  // dV += P^T dO, dK += dS^T Q: 16 queries per MMA
          const uint64_t off = uint64_t(kk * (2048 >> 4));
          sm103::mma_ts_warp(tmem + C::COL_DV, buf + C::COL_S + kk * 8, do_mn + off, kIdescA,
                             (h > 0 || kk > 0) ? 1u : 0u);
          sm103::mma_ts_warp(tmem + C::COL_DK, buf + C::COL_DP + kk * 8, q_mn + off, kIdescA,
                             (h > 0 || kk > 0) ? 1u : 0u);
        }
        if (h % NSUB == NSUB - 1) sm103::mma_commit_warp(bar(C::B_SEMPTY + st));  // the stage is done with
      }
      if (!ok) break;
      sm103::mma_commit_warp(bar(C::B_ACC));
      gs += u.niter;
      gh += nh;
    }
    sm103::mma_commit_warp(bar(C::B_DONE));
    drain_wait(bar(C::B_DONE), 0u);
    __syncwarp();
  } else {
    // ----------------------------------------------------------- elementwise
    const int r = threadIdx.x;
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    const uint64_t sl2x2 = sm103::f2_pack(p.scale_log2, p.scale_log2);
    int gs = 0, gh = 0;
    bool ok = true;
    int nu = 0;
    // The four warps meet at one reduction barrier per unit, whatever happened
    // to their waits, and leave the loop together.
    for (int k = 0; k < kRounds && more(k); ++k, ++nu) {
      const UnitDkv u = unit_at(work(k));
      const int n = u.n0 + r;  // this thread's key
      const bool key_live = n < p.Nk;
      const int nh = NSUB * u.niter;
      for (int h = 0; ok && h < nh; ++h) {
        const int g = gs + h / NSUB, st = g % NSTAGE, hf = (gh + h) & 1, sub = h % NSUB;
        if (!(ok = warp_wait(bar(C::B_SF + hf), uint32_t((gh + h) >> 1) & 1u, ab))) break;
        if (PERSIST && h == 0 && nu > 0 && r == 0) {
          // The previous unit's dK, dV stores (issued at its end) have read their staging slot.
          sm103::bulk_wait_read0();
          sm103::mbar_arrive(bar(C::B_STG));
        }
        // The stage's LSE and D vectors were written by the producer lanes: wait on
        // their barrier directly (already complete) to acquire those stores.
        if (!(ok = warp_wait(bar(C::B_SFULL + st), uint32_t(g / NSTAGE) & 1u, ab))) break;
        sm103::tc_fence_after();
        const int i0 = (u.it0 + g - gs) * SQ + sub * HQ;
        // query column c sees this key iff n <= i0 + c + kv_off, i.e. c >= n - kv_off - i0
        const int cmin = key_live ? (CAUSAL ? n - p.kv_off - i0 : 0) : HQ;
        const float2* lv = reinterpret_cast<const float2*>(vec + (st * 2 + 0) * SQ + sub * HQ);
        const float2* dv = reinterpret_cast<const float2*>(vec + (st * 2 + 1) * SQ + sub * HQ);
        const uint32_t tS = tmem + lane_off + uint32_t(hf) * C::BUF + C::COL_S, tDP = tS + (C::COL_DP - C::COL_S);
        // S^T and dP^T are adjacent: one load of 2 HQ columns, one wait.
        static_assert(C::COL_DP == C::COL_S + HQ, "S^T, dP^T adjacent");
        uint32_t uu[2 * HQ];
        if constexpr (HQ == 64)
          sm103::tmem_ld128(tS, uu);
        else
          tmem_ld64(tS, uu);
#pragma unroll
        for (int q = 0; q < HQ / 32; ++q) {
          uint32_t pp[16], pd[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c = q * 32 + 2 * e;
            const float2 l2 = lv[c / 2], d2 = dv[c / 2];
            const uint64_t t = sm103::f2_fma(sm103::f2_pack(__uint_as_float(uu[c]), __uint_as_float(uu[c + 1])),
                                             sl2x2, sm103::f2_pack(-l2.x, -l2.y));
            float t0, t1;
            sm103::f2_unpack(t, t0, t1);
            const float p0 = c < cmin ? 0.f : sm103::ex2_approx(t0);
            const float p1 = c + 1 < cmin ? 0.f : sm103::ex2_approx(t1);
            pp[e] = sm103::pack_bf16x2(p0, p1);
            pd[e] = sm103::pack_bf16x2(p0 * (__uint_as_float(uu[HQ + c]) - d2.x),
                                       p1 * (__uint_as_float(uu[HQ + c + 1]) - d2.y));
          }
          sm103::tmem_st16(tS + q * 16, pp);   // P^T over S^T (its first 32 columns)
          sm103::tmem_st16(tDP + q * 16, pd);  // dS^T over dP^T
        }
        sm103::tmem_st_wait();
        sm103::tc_fence_before();
        sm103::mbar_arrive(bar(C::B_PF + hf));
      }
      if (ok) ok = warp_wait(bar(C::B_ACC), uint32_t(nu) & 1u, ab);
      // Staging: the slot of the unit's last stage (PERSIST; its MMAs are done),
      // else the K and V tiles.  dV into the Q half or the V tile, dK * scale
      // into the dO half or the K tile (128-byte-swizzle layout).
      const uint32_t slot = sST + uint32_t((gs + u.niter - 1) % NSTAGE) * 2u * C::STILE;
      const uint32_t stg_v = PERSIST ? slot : sV, stg_k = PERSIST ? slot + C::STILE : sK;
      if (ok) {
        sm103::tc_fence_after();
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const uint32_t col0 = w == 0 ? C::COL_DV : C::COL_DK;
          const uint32_t stage = w == 0 ? stg_v : stg_k;
          const float mul = w == 0 ? 1.f : p.scale;
#pragma unroll
          for (int q = 0; q < DACC / 32; ++q) {
            uint32_t v[32];
            sm103::tmem_ld32(tmem + lane_off + col0 + q * 32, v);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = sm103::pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
            const uint32_t rowbase = stage + uint32_t(q >> 1) * kSubTile + uint32_t(r) * 128u;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const uint32_t chunk = uint32_t((q & 1) * 4 + c4);
              sm103::st_shared_v4(rowbase + ((chunk ^ uint32_t(r & 7)) << 4), pk[4 * c4], pk[4 * c4 + 1],
                                  pk[4 * c4 + 2], pk[4 * c4 + 3]);
            }
          }
        }
        // dK, dV are in registers and shared memory: the next unit may overwrite them in TMEM.
        sm103::tc_fence_before();
        sm103::mbar_arrive(bar(C::B_EPI));
        sm103::fence_proxy_async_smem();
      }
      ok = sm103::named_bar_and(1, BM, ok);
      if (!ok) break;
      if (r == 0) {
        for (int kb = 0; kb < DACC / 64; ++kb) {
          sm103::tma_store_3d(&p.tdv, stg_v + kb * kSubTile, u.half * DACC + kb * 64, u.n0, u.bh);
          sm103::tma_store_3d(&p.tdk, stg_k + kb * kSubTile, u.half * DACC + kb * 64, u.n0, u.bh);
        }
        sm103::bulk_commit();
      }
      gs += u.niter;
      gh += nh;
    }
    if (r == 0) sm103::bulk_wait_read0();  // the stores have read shared memory
  }
  sm103::tc_fence_before();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    sm103::tc_fence_after();
    sm103::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace attn
