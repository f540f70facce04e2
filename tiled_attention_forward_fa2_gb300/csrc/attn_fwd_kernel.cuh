// Fused attention forward for sm_103a (GB300).
//
// What it computes ("[GPU] Deep Learning for HPC", bkkhyunn.github.io, section
// "Flash Attention"): S = Q K^T, a row softmax, O = softmax(S) V, tiled so the
// score matrix only ever lives on chip.  The running-max / running-sum form of
// the softmax is the one the FlashAttention-2 forward returns `Lse` for
// (null-ptr.tistory.com "development", the Triton `_fwd_kernel` post); the
// safe-softmax step (subtract the row max before exp) follows the softmax post
// on the same site ("Original softmax").
//
// Hardware mapping.  The pages' H100 design (wgmma into registers, TMA,
// swizzled shared memory; "GPUの爆発的な性能向上", ja.news.hada.io topic 14783,
// sections "WGMMA", "Shared memoryとbank conflict", "アドレス生成とTMA",
// "Occupancyが隠してくれるコスト") is prior art.  The work is cut into units of
// T = 1 or 2 query tiles of 128 rows of one (batch, head) (T = 1 at D = 256);
// a unit streams that head's K and V tiles once for its tiles.  With PERSIST
// the grid has one CTA per SM, each taking its units in snake order, and every
// role runs through the same sequence, so one unit's epilogue and the next
// unit's loads overlap the tensor-core work instead of a CTA launch; without
// it (long key ranges, D = 256) each CTA runs one unit.
//   warp 12      : TMA producer.  Q tiles of each unit (into a buffer of the
//                  tile once the last S MMA of the unit that used it before has
//                  finished; two buffers per tile at D = 64; at D = 256 into
//                  the K/V ring's slot 0 as the unit's first load); K_j, V_j
//                  into a ring of 128-byte-swizzled shared-memory slots
//                  (full/empty mbarriers).
//   warp 13      : allocates the 512 TMEM columns; one thread issues tcgen05.mma:
//                  S_i = Q_i K_j^T into TMEM buffer i, and O_i += P_i V_j with P_i
//                  read back from TMEM (bf16, written over S_i).  The order
//                  PV_0(j), S_0(j+1), PV_1(j), S_1(j+1) keeps the tensor core on
//                  one tile while the other tile's softmax runs (ping-pong).  At
//                  D = 256 it first copies Q into TMEM (tcgen05.cp) and reads it
//                  from there, which frees Q's slot for K and V.
//   warpgroup i  : (i = 0, 1; warps 4i..4i+3) softmax of query tile i, one
//                  thread per row (= TMEM lane).  Masks, running max in base 2,
//                  p = 2^(s*scale*log2e - m) with packed fp32x2 math, P -> TMEM,
//                  running sum.  The reference max m only moves when a row's max
//                  grows by more than 2^8; then the same warp rescales its rows
//                  of O_i in TMEM before handing P over (the last P V on O_i has
//                  finished by then), so no other role takes part in a key step.
//                  Causal with one unit per CTA: P goes over in two halves.
//                  1/l goes to shared memory; LSE to global.
//   warpgroup 2  : (warps 8..11) epilogue: O_i / l -> bf16 -> swizzled staging
//                  tile -> TMA store.
// Every barrier wait is bounded: on expiry the kernel records a timeout in a
// device status word, the other roles see a shared abort flag, in-flight TMA
// copies and MMAs are drained, TMEM is freed and the CTA returns.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace sm103 {
// 128 rows x 256 bits of a shared-memory operand (descriptor as for an MMA
// operand) into TMEM, 8 columns from `taddr`, in the layout an MMA reads A
// from TMEM; one elected lane issues it.  Ordered with this thread's later
// tcgen05.mma, and tracked by its tcgen05.commit.
__device__ __forceinline__ void tmem_cp_128x256b_warp(uint32_t taddr, uint64_t sdesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\t"
      "@e tcgen05.cp.cta_group::1.128x256b [%0], %1;\n}\n" ::"r"(taddr),
      "l"(sdesc)
      : "memory");
}
}  // namespace sm103

namespace attn {

constexpr int BM = 128;                     // query rows per tile (= TMEM lanes)
constexpr int BN = 128;                     // keys per tile
constexpr int kThreads = 512;               // 4 warpgroups
constexpr int kCorrWarp0 = 8;               // warps 8..11: epilogue
constexpr int kLoadWarp = 12;
constexpr int kMmaWarp = 13;                // warps 14, 15 idle (complete the warpgroup)
constexpr uint32_t kSubTile = 128u * 128u;  // 128 rows x 64 bf16 (one 128-B swizzle span)
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;        // move the reference max only when it grows by > 2^8
constexpr int kStatusTimeout = 4;           // value of ATTN_ERR_TIMEOUT
// Register split (setmaxnreg): 2 x 128 softmax threads at 168, 128 epilogue
// threads at 96, 128 load/MMA/idle threads at 80 = 65536 = 512 threads x 128
// (measured best; 176 / 80 / 80 is as fast on long rows and slower on the
// bench shape).
constexpr uint32_t kRegSoftmax = 168, kRegCorr = 96, kRegOther = 80;
static_assert(2 * 128 * kRegSoftmax + 128 * kRegCorr + 128 * kRegOther == kThreads * 128, "register split");

struct FwdParams {
  CUtensorMap tq, tk, tv, to;  // 3-D maps {D, Nq or Nk, B*H}, box {64, 128, 1}, 128-B swizzle, zero fill
  float* lse;                  // [B*H, Nq]
  int Nq, Nk;                  // query and key lengths
  int kv_off;                  // Nk - Nq: causal key j is visible to query i iff j <= i + kv_off
  int bh;                      // B*H
  int n_qtiles, n_ktiles;      // ceil(Nq / 128), ceil(Nk / 128)
  int tiles_per_cta;           // T = 1 or 2 query tiles per unit
  int n_units;                 // ceil(n_qtiles / T): units per (batch, head)
  int n_work;                  // n_units * B*H: units of the whole problem
  int lpt;                     // causal: heads per band, heaviest units first within each band (0: a head's units adjacent)
  float scale_log2;            // scale * log2(e)
  long long timeout_cycles;
  CUtensorMap to32;            // O with 32-row boxes (the short-unit kernel's per-warp stores)
#ifdef ATTN_TEST_HOOKS
  int withhold_kv;             // test build only: nonzero -> no K/V loads are issued, so the pipeline waits run out
#endif
};

template <int D>
struct Cfg {
  static_assert(D == 64 || D == 128 || D == 256, "head dim");
  static constexpr int KB = D / 64;                      // 64-column sub-tiles per tile
  static constexpr uint32_t TILE = KB * kSubTile;        // bytes of one 128 x D bf16 tile
  // Query tiles per unit at most: at D = 256 one (S 128 + O 256 TMEM columns;
  // a second tile would need 768).
  static constexpr int MAXT = D == 256 ? 1 : 2;
  // Q buffers per query tile: at D = 64 two, so a unit's Q loads while the unit
  // before still reads the other (short units would otherwise wait for it).
  static constexpr int NQB = D == 64 ? 2 : 1;
  // At D = 256 Q is read from TMEM (QT): it lands in ring slot 0 as the
  // unit's first load, the MMA warp copies it into TMEM columns 128..255
  // (free beside S and O there) and releases the slot, so the ring has three
  // 64 KB slots where a separate Q buffer left room for two (K_{j+1} then
  // loads while step j runs instead of after S_j).
  static constexpr bool QT = D == 256;
  // K/V ring slots (one tile each).
  static constexpr int NSLOT = D == 256 ? 3 : (D == 128 ? 4 : 9);
  // At D = 256 the epilogue stages O in ring slot 0 (idle once the unit's
  // products are done), so that kernel runs one unit per CTA.
  static constexpr bool STAGE_IN_Q = D == 256;
  static constexpr uint32_t OFF_INVL = 1024;             // [2][128] fp32: 1/l of each row of tile i
  static constexpr uint32_t OFF_Q = 2048;                // Q buffer i * NQB + b of tile i
  static constexpr uint32_t OFF_STG = STAGE_IN_Q ? OFF_Q : OFF_Q + MAXT * NQB * TILE;  // O staging tile
  static constexpr uint32_t OFF_KV = QT ? OFF_Q : OFF_Q + MAXT * NQB * TILE + (STAGE_IN_Q ? 0u : TILE);
  static constexpr uint32_t USED = OFF_KV + NSLOT * TILE;
  static constexpr uint32_t COL_Q = 128;   // QT: Q (bf16 pairs) in TMEM
  static constexpr uint32_t SMEM = USED + 1024;          // + slack to align the base to 1 KB
  static_assert(SMEM <= 232448, "shared memory");
  // barrier slots ([2]: one per query tile of the unit)
  static constexpr int B_Q = 0;                  // [2 NQB] Q buffer landed (TMA bytes)
  static constexpr int B_QE = 2 * NQB;           // [2 NQB] last S MMA on the buffer finished (MMA commit)
  static constexpr int B_FULL = 4 * NQB, B_EMPTY = 4 * NQB + NSLOT;
  static constexpr int B_SF = 4 * NQB + 2 * NSLOT;  // [2] scores of tile i ready (MMA commit)
  static constexpr int B_PF = B_SF + 2;          // [2] P of tile i in TMEM, O_i rescaled (128 softmax threads)
  static constexpr int B_OF = B_PF + 2;          // [2] O_i += P_i V_j finished (MMA commit)
  static constexpr int B_FIN = B_OF + 2;         // [2] final 1/l in shared memory (128 softmax threads)
  static constexpr int B_OE = B_FIN + 2;         // [2] epilogue has read O_i and 1/l (128 epilogue threads)
  static constexpr int B_DONE = B_OE + 2;
  static constexpr int B_PH = B_DONE + 1;        // [2] (split P) first half of P_i in TMEM, O_i rescaled (128 softmax threads)
  static constexpr int NBAR = B_PH + 2;
  static_assert(NBAR * 8 <= 512, "barrier area");
  // TMEM columns
  static constexpr uint32_t COL_S = 0;     // S_i at COL_S + 128 i (P_i over its first 64 columns)
  static constexpr uint32_t COL_O = 256;   // O_i at COL_O + D i
  __host__ __device__ static constexpr bool count128(int b) {  // barriers completed by 128 thread arrivals
    return (b >= B_PF && b < B_PF + 2) || (b >= B_FIN && b < B_OE + 2) || (b >= B_PH && b < B_PH + 2);
  }
};

// The unit a CTA works on: query tiles t0 (and t0 + 1), key tiles nk0 (nk1)
// visited by them; nk1 = 0 when the unit has one tile.  Causal with units of
// very different lengths (p.lpt): heaviest units first (longest-processing-time
// order) within bands of heads.  Otherwise the units of one head are adjacent,
// so CTAs working at the same time share its K and V in L2.
struct Unit {
  int t0, bh, nk0, nk1;
  __device__ __forceinline__ int nk() const { return max(nk0, nk1); }
};

// Key split (SPLITK): a unit is one query tile whose key tiles are shared out
// between the two softmax warpgroups -- even key tiles to tile slot 0, odd ones
// to slot 1 -- each keeping its own running max, sum and O; the epilogue merges
// the two.  The unit's serial chain of key steps is halved, which is what
// bounds problems with fewer query tiles than SMs.  nk0 / nk1 count the key
// steps of each slot; slot i's step j is key tile 2 j + i.
template <bool SPLITK>
__device__ __forceinline__ int key_tile(int i, int j) {
  return SPLITK ? 2 * j + i : j;
}

template <bool CAUSAL, bool SPLITK = false>
__device__ __forceinline__ Unit unit_of(const FwdParams& p, int w) {
  Unit u;
  int unit;
  if (CAUSAL && p.lpt) {
    // Longest first within bands of p.lpt heads (the last band may be
    // smaller): the CTAs running at one time then read the K and V of only
    // about a band of heads, which stays resident in L2.
    const int span = p.lpt * p.n_units;
    const int band = w / span, idx = w - band * span;
    const int g = min(p.lpt, p.bh - band * p.lpt);
    unit = p.n_units - 1 - idx / g;
    u.bh = band * p.lpt + idx % g;
  } else {
    unit = w % p.n_units;
    u.bh = w / p.n_units;
  }
  u.t0 = unit * p.tiles_per_cta;
  // Causal: key tiles up to the one of the tile's last query row (past Nq: row Nq-1).
  auto tiles = [&](int t) {
    if (!CAUSAL) return p.n_ktiles;
    const int last_row = min(t * BM + BM - 1, p.Nq - 1);
    return min(p.n_ktiles, (last_row + p.kv_off) / BN + 1);
  };
  if constexpr (SPLITK) {
    const int nk = tiles(u.t0);
    u.nk0 = (nk + 1) / 2;
    u.nk1 = nk / 2;
  } else {
    u.nk0 = tiles(u.t0);
    u.nk1 = (p.tiles_per_cta == 2 && u.t0 + 1 < p.n_qtiles) ? tiles(u.t0 + 1) : 0;
  }
  return u;
}

// Key tiles a unit streams (each as K then V).
template <bool SPLITK>
__device__ __forceinline__ int unit_key_tiles(const Unit& u) {
  return SPLITK ? u.nk0 + u.nk1 : u.nk();
}

__device__ int g_attn_status;  // 0 or kStatusTimeout; taken and cleared by status_take

// attn_last_status's read of the status word: one atomic exchange (read and
// clear), its result left in a slot of its own for the host to copy.
constexpr int kStatusSlots = 64;
__device__ int g_status_taken[kStatusSlots];
__global__ void status_take(int slot) { g_status_taken[slot] = atomicExch(&g_attn_status, 0); }

struct Abort {
  volatile uint32_t* flag;
  long long limit;
};

// Wait for an mbarrier phase, bounded.  Each try suspends the thread until the
// phase completes or about a millisecond passes; between tries the wait gives
// up when another role aborted (if honour_abort) or when `limit` cycles have
// passed, the latter recording a timeout.
constexpr uint32_t kSuspendNs = 1000000;
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const Abort& ab,
                                             bool honour_abort = true) {
  if (sm103::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (sm103::mbar_try_wait_sleep(bar, parity, kSuspendNs)) return true;
    if (honour_abort && *ab.flag) return false;
    if (clock64() - t0 > ab.limit) {
      atomicCAS(&g_attn_status, 0, kStatusTimeout);
      *ab.flag = 1u;
      return false;
    }
  }
}

// Wait on work that completes by itself (copies in flight, MMAs before TMEM is
// freed): ignores the abort flag and allows about a second of SM cycles.
constexpr long long kDrainCycles = 1LL << 31;
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  if (sm103::mbar_try_wait(bar, parity)) return;
  const long long t0 = clock64();
  while (!sm103::mbar_try_wait_sleep(bar, parity, kSuspendNs)) {
    if (clock64() - t0 > kDrainCycles) {
      atomicCAS(&g_attn_status, 0, kStatusTimeout);
      return;
    }
  }
}

// Warp-uniform version: every lane waits, the warp proceeds only if all saw it.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Abort& ab) {
  return __all_sync(0xffffffffu, wait_bounded(bar, parity, ab));
}

template <int D, bool CAUSAL, bool PERSIST, bool SPLITK = false>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_sm103(const __grid_constant__ FwdParams p) {
  using C = Cfg<D>;
  static_assert(!(PERSIST && C::STAGE_IN_Q), "O staged in the Q buffer: one unit per CTA");
  static_assert(!SPLITK || (D == 64 && PERSIST), "key split: D = 64 persistent kernel only");
  constexpr int KB = C::KB;
  constexpr int NSLOT = C::NSLOT;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = sm103::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sbase + 512);
  volatile uint32_t* const abort_flag = reinterpret_cast<volatile uint32_t*>(sbase + 516);
  float* const invl = reinterpret_cast<float*>(sbase + C::OFF_INVL);  // [2][128]
  const uint32_t sQ = base + C::OFF_Q;      // Q buffer qi = i * NQB + b at sQ + qi * TILE
  const uint32_t sStg = base + C::OFF_STG;  // O staging tile
  const uint32_t sKV = base + C::OFF_KV;    // slot s at sKV + s * TILE
  // Key split: both slots read tile slot 0's Q buffers; slot 1's hold the two
  // partial (max, sum) rows of every query row, [slot][max | sum][128].
  float* const ml = reinterpret_cast<float*>(sbase + C::OFF_Q + C::NQB * C::TILE);
  auto bar = [base](int i) { return base + 8u * uint32_t(i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Units of this CTA: round k takes unit k G + c for even k and k G + (G - 1 - c)
  // for odd k (G = gridDim.x, c = blockIdx.x).  Units are numbered heaviest
  // first when causal, so the snake order pairs heavy and light rounds and the
  // CTAs' totals stay level.
  // Without PERSIST the grid has one CTA per unit and every loop over units
  // below runs once; the compiler then lays the MMA warp's key loop out as a
  // single loop, which keeps its issue rate (about 6 % more throughput on long
  // key ranges than the same loop nested in a unit loop).
  const int w0 = int(blockIdx.x), dw = int(gridDim.x);
  auto work = [w0, dw](int k) { return k * dw + ((k & 1) ? dw - 1 - w0 : w0); };
  // Rounds of units per CTA; the bound is written as k < kRounds (not k == 0):
  // the compiler only collapses the loops for the former.
  constexpr int kRounds = PERSIST ? 0x7fffffff : 1;
  auto more = [&](int k) { return work(k) < p.n_work; };
  // Split P: the softmax hands P over in two halves (B_PH after keys 0..63,
  // then B_PF), so the first four P V MMAs of a step run while it finishes the
  // rest.  Measured on the causal one-unit grid only: +5 % there (causal
  // N = 16384), -0.6 to -0.8 % on full rows, -1.8 % on the persistent grid.
  constexpr bool kSplitP = CAUSAL && !PERSIST;
  (void)ml;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) sm103::mbar_init(bar(i), C::count128(i) ? uint32_t(BM) : 1u);
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
    sm103::tma_prefetch_map(&p.to);
  }
  sm103::tc_fence_before();
  __syncthreads();
  sm103::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag, p.timeout_cycles};

  // Phase bookkeeping.  Every role walks the same units; per query tile i it
  // counts the units that used tile i (phases of B_Q, B_QE, B_FIN, B_OE) and
  // their key steps (B_SF, B_PF, B_OF).
  if (warp >= kLoadWarp) {
    sm103::regs_decrease<kRegOther>();
    if (warp == kLoadWarp) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        int c = 0;            // K/V loads issued; K_j of a unit is load cb + 2j, V_j load cb + 2j + 1
        int nq0 = 0, nq1 = 0;  // Q loads issued for tile 0 / 1 (the n-th into buffer n % NQB)
        bool ok = true;
        for (int k = 0; k < kRounds && ok && more(k); ++k) {
          const Unit u = unit_of<CAUSAL, SPLITK>(p, work(k));
          // A buffer is free once the last S MMA of the unit that used it before
          // (NQB loads ago) has finished.
          auto load_q = [&](int i, int nq) -> bool {
            const int qi = i * C::NQB + nq % C::NQB;
            if (nq >= C::NQB && !wait_bounded(bar(C::B_QE + qi), uint32_t(nq / C::NQB - 1) & 1u, ab)) return false;
            sm103::mbar_arrive_expect_tx(bar(C::B_Q + qi), C::TILE);
            for (int kb = 0; kb < KB; ++kb)
              sm103::tma_load_3d(sQ + qi * C::TILE + kb * kSubTile, &p.tq, bar(C::B_Q + qi), kb * 64,
                                 (u.t0 + i) * BM, u.bh);
            return true;
          };
          if constexpr (C::QT) {
            // Q into ring slot 0 as the unit's load 0 (one unit per CTA at D = 256).
            sm103::mbar_arrive_expect_tx(bar(C::B_FULL), C::TILE);
            for (int kb = 0; kb < KB; ++kb)
              sm103::tma_load_3d(sKV + kb * kSubTile, &p.tq, bar(C::B_FULL), kb * 64, u.t0 * BM, u.bh);
            ++c;
          } else {
            if (!(ok = load_q(0, nq0))) break;
            ++nq0;
          }
          if (!SPLITK && u.nk1 > 0) {
            if (!(ok = load_q(1, nq1))) break;
            ++nq1;
          }
          const int nk = unit_key_tiles<SPLITK>(u);
#ifdef ATTN_TEST_HOOKS
          const bool withhold = p.withhold_kv != 0;
#else
          constexpr bool withhold = false;
#endif
          for (int j = 0; ok && !withhold && j < nk; ++j) {
            for (int kv = 0; kv < 2; ++kv, ++c) {
              const int s = c % NSLOT;
              if (c >= NSLOT && !(ok = wait_bounded(bar(C::B_EMPTY + s), uint32_t(c / NSLOT - 1) & 1u, ab))) break;
              sm103::mbar_arrive_expect_tx(bar(C::B_FULL + s), C::TILE);
              const CUtensorMap* map = kv == 0 ? &p.tk : &p.tv;
              for (int kb = 0; kb < KB; ++kb)
                sm103::tma_load_3d(sKV + s * C::TILE + kb * kSubTile, map, bar(C::B_FULL + s), kb * 64, j * BN, u.bh);
            }
          }
        }
        // Drain: no copy may land in shared memory after this CTA has left.
        // Earlier Q loads and ring loads before the last NSLOT were consumed
        // (waited on) before their buffers were reused.
        for (int t = nq0 > C::NQB ? nq0 - C::NQB : 0; t < nq0; ++t)
          drain_wait(bar(C::B_Q + t % C::NQB), uint32_t(t / C::NQB) & 1u);
        for (int t = nq1 > C::NQB ? nq1 - C::NQB : 0; t < nq1; ++t)
          drain_wait(bar(C::B_Q + C::NQB + t % C::NQB), uint32_t(t / C::NQB) & 1u);
        for (int t = c > NSLOT ? c - NSLOT : 0; t < c; ++t) drain_wait(bar(C::B_FULL + t % NSLOT), uint32_t(t / NSLOT) & 1u);
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // ----------------------------------------------------------- MMA issue
      // The whole warp runs this loop with warp-uniform values; one elected
      // lane issues each tcgen05.mma and tcgen05.commit.
      constexpr uint32_t kIdescS = sm103::idesc_bf16_f32(BM, BN, 0, 0);  // Q, K both K-major
      // S's MMAs fully unrolled up to D = 128; at D = 256 four at a time (fewer
      // hoisted descriptor offsets: this warp runs at 88 registers).
      constexpr int kUnrollS = D / 16 <= 8 ? D / 16 : 4;
      constexpr uint32_t kIdescO = sm103::idesc_bf16_f32(BM, D, 0, 1);   // P K-major, V MN-major
      // Descriptors (low words) are built once; moving an operand by `off` bytes
      // adds off >> 4 to the start-address field (no carry: shared addresses stay
      // below 256 KB).
      const uint32_t hi = sm103::kSdescHi;
      const uint32_t desc_q = sm103::sdesc_sw128_lo(sQ, 16);         // K-major Q tiles
      const uint32_t desc_k = sm103::sdesc_sw128_lo(sKV, 16);        // K-major K slots
      const uint32_t desc_v = sm103::sdesc_sw128_lo(sKV, kSubTile);  // MN-major V slots
      auto slot_off = [](int c) { return uint32_t(c % NSLOT) * (C::TILE >> 4); };
      auto wait_full = [&](int c) { return warp_wait(bar(C::B_FULL + c % NSLOT), uint32_t(c / NSLOT) & 1u, ab); };
      auto release = [&](int c) { sm103::mma_commit_warp(bar(C::B_EMPTY + c % NSLOT)); };
      // nu0/nu1: units tile 0/1 had (B_Q / B_QE buffer and phase, B_OE); ph bits
      // 2/3 = parity of their key steps (B_PF).
      uint32_t cb = 0;  // ring index of the current unit's K_0
      uint32_t ph = 0;
      int nu0 = 0, nu1 = 0;
      bool ok = true;
      for (int k = 0; k < kRounds && ok && more(k); ++k) {
        int nk0, nk1;
        {
          const Unit u = unit_of<CAUSAL, SPLITK>(p, work(k));
          nk0 = u.nk0;
          nk1 = u.nk1;
        }
        const int nk = max(nk0, nk1);
        auto issue_s = [&](int i, int j) {
          const int qi = SPLITK ? nu0 % C::NQB : i * C::NQB + (i == 0 ? nu0 : nu1) % C::NQB;
          const uint32_t dk = desc_k + slot_off(int(cb) + 2 * key_tile<SPLITK>(i, j));
          const uint32_t dq = desc_q + uint32_t(qi) * (C::TILE >> 4);
          const uint32_t dS = tmem + C::COL_S + uint32_t(i) * BN;
#pragma unroll(kUnrollS)
          for (int kk = 0; kk < D / 16; ++kk) {  // 16 of the head dim per MMA
            const uint32_t off = (uint32_t(kk >> 2) * kSubTile + uint32_t(kk & 3) * 32u) >> 4;
            if constexpr (C::QT)
              sm103::mma_ts_warp_lo(dS, tmem + C::COL_Q + uint32_t(kk) * 8u, dk + off, kIdescS, kk > 0 ? 1u : 0u, hi);
            else
              sm103::mma_ss_warp_lo(dS, dq + off, dk + off, kIdescS, kk > 0 ? 1u : 0u, hi);
          }
          sm103::mma_commit_warp(bar(C::B_SF + i));
          if constexpr (C::QT) return;  // Q is in TMEM: no Q buffer to free
          // Q buffer no longer read: after the unit's last S MMA on it.  With the
          // key split that is slot 0's last S when the unit has an odd number of
          // key tiles (nk0 = nk1 + 1), else slot 1's -- exactly one commit per unit.
          const bool last_s = SPLITK ? (i == 0 ? (j == nk0 - 1 && nk1 < nk0) : (j == nk1 - 1 && nk1 == nk0))
                                     : j == (i == 0 ? nk0 : nk1) - 1;
          if (last_s) sm103::mma_commit_warp(bar(C::B_QE + qi));
        };
        auto issue_pv = [&](int i, int j) -> bool {
          if (!warp_wait(bar((kSplitP ? C::B_PH : C::B_PF) + i), ((ph >> (2 + i)) ^ uint32_t(j)) & 1u, ab)) return false;
          if (j == 0 && (i == 0 ? nu0 : nu1) > 0) {
            // The first P V of a unit overwrites O_i: the previous unit's epilogue must have read it.
            if (!warp_wait(bar(C::B_OE + i), uint32_t((i == 0 ? nu0 : nu1) - 1) & 1u, ab)) return false;
          }
          sm103::tc_fence_after();
          const uint32_t dv = desc_v + slot_off(int(cb) + 2 * key_tile<SPLITK>(i, j) + 1);
          const uint32_t aP = tmem + C::COL_S + uint32_t(i) * BN;
          const uint32_t dO = tmem + C::COL_O + uint32_t(i) * D;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {  // 16 keys per MMA: 8 TMEM columns of P, 16 rows of V
            if (kSplitP && kk == BN / 32) {
              if (!warp_wait(bar(C::B_PF + i), ((ph >> (2 + i)) ^ uint32_t(j)) & 1u, ab)) return false;
              sm103::tc_fence_after();
            }
            sm103::mma_ts_warp_lo(dO, aP + kk * 8, dv + uint32_t(kk * (2048 >> 4)), kIdescO, (j > 0 || kk > 0) ? 1u : 0u, hi);
          }
          sm103::mma_commit_warp(bar(C::B_OF + i));
          return true;
        };
        if constexpr (C::QT) {
          // Q (ring load 0) into TMEM, 16 columns of the head dim per copy,
          // then slot 0 goes back to the ring (the commit follows the copies).
          if (!(ok = wait_full(0))) break;
          sm103::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t dq = sm103::sdesc_sw128(sKV + uint32_t(kk >> 2) * kSubTile + uint32_t(kk & 3) * 32u, 16, 1024);
            sm103::tmem_cp_128x256b_warp(tmem + C::COL_Q + uint32_t(kk) * 8u, dq);
          }
          release(0);
          cb = 1;  // K_j is load 1 + 2 j, V_j load 2 + 2 j
        } else {
          ok = warp_wait(bar(C::B_Q + nu0 % C::NQB), uint32_t(nu0 / C::NQB) & 1u, ab);
          if (!ok) break;
        }
        if (!(ok = wait_full(int(cb)))) break;
        sm103::tc_fence_after();
        issue_s(0, 0);
        if (nk1 > 0) {
          if constexpr (SPLITK) {
            if (!(ok = wait_full(int(cb) + 2))) break;  // K of key tile 1
          } else {
            if (!(ok = warp_wait(bar(C::B_Q + C::NQB + nu1 % C::NQB), uint32_t(nu1 / C::NQB) & 1u, ab))) break;
          }
          sm103::tc_fence_after();
          issue_s(1, 0);
        }
        release(int(cb));
        if (SPLITK && nk1 > 0) release(int(cb) + 2);
        if constexpr (SPLITK) {
          // Step j: P V of key tiles 2j (slot 0) and 2j + 1 (slot 1), then S of
          // key tiles 2j + 2 and 2j + 3 for the next step.
          // Each product waits only for its own tile: a P V for its V, an S
          // for its K (waiting for the next K tiles before this step's P V held
          // the P V back by a load latency whenever those K tiles were still in
          // flight, as on short units whose ring slots refill late).
          for (int j = 0; ok && j < nk; ++j) {
            const bool has1 = j < nk1, next0 = j + 1 < nk0, next1 = j + 1 < nk1;
            if (!(ok = wait_full(int(cb) + 2 * (2 * j) + 1))) break;
            sm103::tc_fence_after();
            if (!(ok = issue_pv(0, j))) break;
            if (next0) {
              if (!(ok = wait_full(int(cb) + 2 * (2 * j + 2)))) break;
              sm103::tc_fence_after();
              issue_s(0, j + 1);
            }
            if (has1) {
              if (!(ok = wait_full(int(cb) + 2 * (2 * j + 1) + 1))) break;
              sm103::tc_fence_after();
              if (!(ok = issue_pv(1, j))) break;
              if (next1) {
                if (!(ok = wait_full(int(cb) + 2 * (2 * j + 3)))) break;
                sm103::tc_fence_after();
                issue_s(1, j + 1);
              }
            }
            release(int(cb) + 2 * (2 * j) + 1);
            if (has1) release(int(cb) + 2 * (2 * j + 1) + 1);
            if (next0) release(int(cb) + 2 * (2 * j + 2));
            if (next1) release(int(cb) + 2 * (2 * j + 3));
          }
          cb += 2u * uint32_t(nk0 + nk1);
        } else {
        for (int j = 0; ok && j < nk; ++j) {
          const bool next = j + 1 < nk;
          if constexpr (D > 128) {
            // One tile per unit (D = 256): its P V waits only for V_j, the next
            // S for K_{j+1}.  Waiting for K_{j+1} first held each P V back by a
            // load latency, the ring being two 64 KB slots (B2 H16 N4096 585 ->
            // 499 us).  The D <= 128 instances keep K_{j+1} and V_j up front:
            // there the split order (as a runtime branch) measured 1-5 % slower.
            if (!(ok = wait_full(int(cb) + 2 * j + 1))) break;
            sm103::tc_fence_after();
            if (!(ok = issue_pv(0, j))) break;
            if (next) {
              if (!(ok = wait_full(int(cb) + 2 * j + 2))) break;
              sm103::tc_fence_after();
              issue_s(0, j + 1);
            }
          } else {
          if (next && !(ok = wait_full(int(cb) + 2 * j + 2))) break;
          if (!(ok = wait_full(int(cb) + 2 * j + 1))) break;
          sm103::tc_fence_after();
          if (j < nk0) {
            if (!(ok = issue_pv(0, j))) break;
            if (j + 1 < nk0) issue_s(0, j + 1);
          }
          if (j < nk1) {
            if (!(ok = issue_pv(1, j))) break;
            if (j + 1 < nk1) issue_s(1, j + 1);
          }
          }
          release(int(cb) + 2 * j + 1);
          if (next) release(int(cb) + 2 * j + 2);
        }
        cb += 2u * uint32_t(nk);
        }
        // Tile i: units +1, steps + nk_i.
        ph ^= uint32_t(nk0 & 1) << 2;
        ++nu0;
        if (nk1 > 0) {
          ph ^= uint32_t(nk1 & 1) << 3;
          ++nu1;
        }
      }
      // Every MMA must be finished before TMEM is freed.
      sm103::mma_commit_warp(bar(C::B_DONE));
      drain_wait(bar(C::B_DONE), 0u);
      __syncwarp();
    }
  } else if (warp < kCorrWarp0) {
    // ------------------------------------------------------------- softmax
    sm103::regs_increase<kRegSoftmax>();
    const int i = warp >> 2;            // query tile of this warpgroup
    const int r = threadIdx.x & 127;    // row within the tile = TMEM lane
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::COL_S + uint32_t(i) * BN;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = sm103::f2_pack(sl2, sl2);
    // Phase word (kept small: this role runs at the register limit): bit 0 =
    // parity of this tile's earlier key steps (B_SF), bit 1 = parity of its
    // earlier units (B_OE), bit 2 = an earlier unit exists.
    uint32_t ph = 0;
    bool ok = true;
    for (int k = 0; k < kRounds && ok && more(k); ++k) {
      int nki, diag;  // key steps; causal: last visible key of this row (row + Nk - Nq)
      {
        const Unit u = unit_of<CAUSAL, SPLITK>(p, work(k));
        nki = i == 0 ? u.nk0 : u.nk1;
        diag = (u.t0 + (SPLITK ? 0 : i)) * BM + r + p.kv_off;
      }
      if (nki == 0) continue;
      float m_ref = 0.f;  // reference max (base 2) the exponents are taken against
      float l_run = 0.f;  // running sum of p (fp32, before the bf16 rounding of P)
      for (int j = 0; j < nki; ++j) {
        if (!(ok = warp_wait(bar(C::B_SF + i), (ph ^ uint32_t(j)) & 1u, ab))) break;
        sm103::tc_fence_after();
        float s[BN];
        {
          uint32_t uu[BN];
          sm103::tmem_ld128(tS, uu);
#pragma unroll
          for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(uu[c]);
        }
        // Masks: keys past N, and keys after the query row when causal.
        const int kt = key_tile<SPLITK>(i, j);
        int lim = min(BN - 1, p.Nk - 1 - kt * BN);
        if (CAUSAL) lim = min(lim, diag - kt * BN);
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
        const float cand = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
        float alpha = 1.f;
        if (j == 0) {
          m_ref = cand;
        } else {
          if (cand > m_ref + kRescaleLog2) {
            alpha = sm103::ex2_approx(m_ref - cand);
            m_ref = cand;
          }
        }
        const uint64_t negm = sm103::f2_pack(-m_ref, -m_ref);
        uint64_t acc0 = 0, acc1 = 0;  // packed fp32 partial sums (+0.0f, +0.0f)
#pragma unroll
        for (int q = 0; q < BN / 32; ++q) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint64_t t = sm103::f2_fma(sm103::f2_pack(s[q * 32 + 2 * e], s[q * 32 + 2 * e + 1]), sl2x2, negm);
            float t_lo, t_hi;
            sm103::f2_unpack(t, t_lo, t_hi);
            const float p0 = sm103::ex2_approx(t_lo);
            const float p1 = sm103::ex2_approx(t_hi);
            pk[e] = sm103::pack_bf16x2(p0, p1);
            if (e & 1)
              acc1 = sm103::f2_add(acc1, sm103::f2_pack(p0, p1));
            else
              acc0 = sm103::f2_add(acc0, sm103::f2_pack(p0, p1));
          }
          sm103::tmem_st16(tS + q * 16, pk);  // P over the first 64 columns of S_i
          if (kSplitP && q == BN / 64 - 1) {
            // O_i *= alpha (rare; the P V that last wrote O_i was issued before
            // this step's S MMAs, so it has finished), then the first half of P
            // goes to the MMA warp.
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
              const uint32_t tO = tmem + lane_off + C::COL_O + uint32_t(i) * D;
#pragma unroll 1
              for (int q2 = 0; q2 < D / 32; ++q2) {
                uint32_t v[32];
                sm103::tmem_ld32(tO + q2 * 32, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                sm103::tmem_st32(tO + q2 * 32, v);
              }
            }
            sm103::tmem_st_wait();
            sm103::tc_fence_before();
            sm103::mbar_arrive(bar(C::B_PH + i));
          }
        }
        float a0, a1, a2, a3;
        sm103::f2_unpack(acc0, a0, a1);
        sm103::f2_unpack(acc1, a2, a3);
        const float rowsum = (a0 + a1) + (a2 + a3);
        l_run = j == 0 ? rowsum : fmaf(alpha, l_run, rowsum);
        // O_i *= alpha when a row of the warp moved its reference max (rare after
        // the first steps).  The P V that last wrote O_i was issued before this
        // step's S MMAs, so it has finished; the next one waits for B_PF below.
        if (!kSplitP && __any_sync(0xffffffffu, alpha != 1.f)) {
          const uint32_t tO = tmem + lane_off + C::COL_O + uint32_t(i) * D;
#pragma unroll 1
          for (int q = 0; q < D / 32; ++q) {
            uint32_t v[32];
            sm103::tmem_ld32(tO + q * 32, v);
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            sm103::tmem_st32(tO + q * 32, v);
          }
        }
        sm103::tmem_st_wait();
        sm103::tc_fence_before();
        sm103::mbar_arrive(bar(C::B_PF + i));
      }
      if (!ok) break;
      // 1/l for the epilogue, once it has read the previous unit's value; LSE from here.
      if ((ph & 4u) && !(ok = warp_wait(bar(C::B_OE + i), ((ph >> 1) & 1u) ^ 1u, ab))) break;
      if constexpr (SPLITK) {
        // The partial max and sum; the epilogue merges the two slots and writes LSE.
        ml[(2 * i) * BM + r] = m_ref;
        ml[(2 * i + 1) * BM + r] = l_run;
        sm103::mbar_arrive(bar(C::B_FIN + i));
        ph = ((ph ^ uint32_t(nki)) & 1u) | ((ph ^ 2u) & 2u) | 4u;
        continue;
      }
      invl[i * BM + r] = 1.f / l_run;
      sm103::mbar_arrive(bar(C::B_FIN + i));
      {
        const Unit u = unit_of<CAUSAL>(p, work(k));
        const int row = (u.t0 + i) * BM + r;
        if (row < p.Nq) p.lse[size_t(u.bh) * size_t(p.Nq) + size_t(row)] = (m_ref + log2f(l_run)) * 0.6931471805599453f;
      }
      ph = ((ph ^ uint32_t(nki)) & 1u) | ((ph ^ 2u) & 2u) | 4u;
    }
  } else {
    // -------------------------------------------------------------- epilogue
    sm103::regs_decrease<kRegCorr>();
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    int nu0 = 0, nu1 = 0, ns0 = 0, ns1 = 0;  // units and key steps of tile 0 / 1 so far (B_FIN, B_OE; B_OF)
    bool ok = true;
    for (int k = 0; k < kRounds && more(k); ++k) {
      const Unit u = unit_of<CAUSAL, SPLITK>(p, work(k));
      if constexpr (SPLITK) {
        // One query tile per unit: merge the two slots' partial results.
        //   m = max(m0, m1), c_i = 2^(m_i - m) / (2^(m0 - m) l0 + 2^(m1 - m) l1),
        //   O = c0 O0 + c1 O1, LSE = ln 2 (m + log2 l).
        const bool two = u.nk1 > 0;
        if (ok) ok = warp_wait(bar(C::B_FIN), uint32_t(nu0) & 1u, ab);
        if (ok) ok = warp_wait(bar(C::B_OF), uint32_t(ns0 + u.nk0 - 1) & 1u, ab);
        if (ok && two) ok = warp_wait(bar(C::B_FIN + 1), uint32_t(nu1) & 1u, ab);
        if (ok && two) ok = warp_wait(bar(C::B_OF + 1), uint32_t(ns1 + u.nk1 - 1) & 1u, ab);
        if (r == 0) sm103::bulk_wait_read0();
        ok = sm103::named_bar_and(1, 128, ok);
        if (!ok) break;
        sm103::tc_fence_after();
        const float m0 = ml[r], l0 = ml[BM + r];
        const float m1 = two ? ml[2 * BM + r] : -INFINITY, l1 = two ? ml[3 * BM + r] : 0.f;
        const float m = fmaxf(m0, m1);
        const float a0 = sm103::ex2_approx(m0 - m), a1 = two ? sm103::ex2_approx(m1 - m) : 0.f;
        const float l = a0 * l0 + a1 * l1;
        const float inv = 1.f / l;
        const float c0 = a0 * inv, c1 = a1 * inv;
        const uint32_t tO0 = tmem + lane_off + C::COL_O, tO1 = tO0 + uint32_t(D);
#pragma unroll
        for (int q = 0; q < D / 16; ++q) {  // 16 columns = two 16-byte chunks of the staging row
          uint32_t v0[16], v1[16];
          sm103::tmem_ld16(tO0 + q * 16, v0);
          if (two) sm103::tmem_ld16(tO1 + q * 16, v1);
          if (q == D / 16 - 1) {
            sm103::tc_fence_before();
            sm103::mbar_arrive(bar(C::B_OE));
            if (two) sm103::mbar_arrive(bar(C::B_OE + 1));
          }
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float lo = __uint_as_float(v0[2 * e]) * c0, hi = __uint_as_float(v0[2 * e + 1]) * c0;
            if (two) {
              lo = fmaf(__uint_as_float(v1[2 * e]), c1, lo);
              hi = fmaf(__uint_as_float(v1[2 * e + 1]), c1, hi);
            }
            pk[e] = sm103::pack_bf16x2(lo, hi);
          }
          const uint32_t rowbase = sStg + uint32_t(r) * 128u;
          sm103::st_shared_v4(rowbase + ((uint32_t(2 * q) ^ uint32_t(r & 7)) << 4), pk[0], pk[1], pk[2], pk[3]);
          sm103::st_shared_v4(rowbase + ((uint32_t(2 * q + 1) ^ uint32_t(r & 7)) << 4), pk[4], pk[5], pk[6], pk[7]);
        }
        sm103::fence_proxy_async_smem();
        sm103::named_bar_sync(1, 128);
        if (r == 0) {
          sm103::tma_store_3d(&p.to, sStg, 0, u.t0 * BM, u.bh);
          sm103::bulk_commit();
        }
        const int row = u.t0 * BM + r;
        if (row < p.Nq) p.lse[size_t(u.bh) * size_t(p.Nq) + size_t(row)] = (m + log2f(l)) * 0.6931471805599453f;
        ++nu0;
        ns0 += u.nk0;
        if (two) {
          ++nu1;
          ns1 += u.nk1;
        }
      } else {
      // The four warps agree (reduction barrier) before touching the
      // shared staging tile, so a warp that gave up on a wait cannot leave the
      // others stuck at the named barrier below.  Tile 0 is in every unit, so the
      // warps meet at least once per unit.
#pragma unroll 1
      for (int i = 0; i < 2; ++i) {
        const int nki = i == 0 ? u.nk0 : u.nk1;
        if (nki == 0) continue;
        const uint32_t tO = tmem + lane_off + C::COL_O + uint32_t(i) * D;
        if (ok) ok = warp_wait(bar(C::B_FIN + i), uint32_t(i == 0 ? nu0 : nu1) & 1u, ab);
        if (ok) ok = warp_wait(bar(C::B_OF + i), uint32_t((i == 0 ? ns0 : ns1) + nki - 1) & 1u, ab);
        if (r == 0) sm103::bulk_wait_read0();  // the previous store has read the staging tile
        ok = sm103::named_bar_and(1, 128, ok);
        if (!ok) break;
        sm103::tc_fence_after();
        const float inv_l = invl[i * BM + r];
        // O_i / l -> bf16 into the staging tile, laid out as TMA's 128-byte
        // swizzle expects: row r at 128 r, 16-byte chunk c at ((c ^ (r & 7)) * 16).
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t v[32];
          sm103::tmem_ld32(tO + q * 32, v);
          if (q == D / 32 - 1) {
            // O_i and 1/l are in registers: the next unit may overwrite both.
            sm103::tc_fence_before();
            sm103::mbar_arrive(bar(C::B_OE + i));
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = sm103::pack_bf16x2(__uint_as_float(v[2 * e]) * inv_l, __uint_as_float(v[2 * e + 1]) * inv_l);
          const uint32_t rowbase = sStg + uint32_t(q >> 1) * kSubTile + uint32_t(r) * 128u;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const uint32_t chunk = uint32_t((q & 1) * 4 + c4);
            sm103::st_shared_v4(rowbase + ((chunk ^ uint32_t(r & 7)) << 4), pk[4 * c4], pk[4 * c4 + 1],
                                pk[4 * c4 + 2], pk[4 * c4 + 3]);
          }
        }
        sm103::fence_proxy_async_smem();
        sm103::named_bar_sync(1, 128);
        if (r == 0) {
          for (int kb = 0; kb < KB; ++kb) sm103::tma_store_3d(&p.to, sStg + kb * kSubTile, kb * 64, (u.t0 + i) * BM, u.bh);
          sm103::bulk_commit();
        }
      }
      if (!ok) break;
      ++nu0;
      ns0 += u.nk0;
      if (u.nk1 > 0) {
        ++nu1;
        ns1 += u.nk1;
      }
      }
    }
    if (r == 0) sm103::bulk_wait_read0();  // the stores have read shared memory
  }

  sm103::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    sm103::tc_fence_after();
    sm103::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace attn
