// Fused decode-GEMM on the 5th-generation tensor cores, for 16 < M <= 256
// activation rows per launch: the trellis is decoded by producer warps
// straight into the tensor-core operand buffers in shared memory, so no
// reconstructed weight is ever written to HBM.
//
// This is the reconstruct-free "dequant fused into the GEMM" kernel that
// vLLM PR #316, "[EXL3] dispatch prefill-shaped GEMMs to reconstruct+hgemm"
// (follow-up comment, the ceiling arithmetic) names as the limit beyond the
// unfused reconstruct+hgemm sequence, rebuilt for sm_103a. It serves the
// decode-shaped side of the runtime dispatch above 16 rows: each weight is
// decoded once per 256 rows instead of once per 16.
//
//   y[m0:m0+M, :] = had_r_128( x'[m0:m0+M] . W ) * sv      (x' already rotated)
//
// Work: stream-K over (128-column n-block, 64-row k step) units, one CTA per
// SM. The decoded W^T block is the M = 128 operand of the tensor-core MMA and
// x' the N operand, N = the rows rounded up to 32, so a few activation rows
// cost a narrow MMA instead of a 128-row padded one. Per k step:
//   * warp 0 (one lane): one TMA load of x' (N x 64, 128-byte swizzle);
//   * warps 2..17 (decoders): four groups of four; group j decodes the four
//     16-row slabs of k steps j, j+4, ...; each warp
//     streams its slab's 8 trellis tiles through a private bulk-copy ring,
//     decodes lane (g, q) = tile g, rows 4q..4q+3, and stores W^T into the
//     A operand: K-major, 128-byte swizzle (the layout the tensor core reads
//     at full rate). Column n = 16g + c goes to operand row 16g + (c ^ g), so
//     the eight lanes storing column step c hit eight different swizzle rows
//     and the warp's 8-byte stores spread over all banks; the address is one
//     XOR of a per-lane constant with a compile-time one;
//   * warp 1 (one lane): tcgen05.mma M=128 N=npad K=16 into a double-buffered
//     TMEM accumulator (TMEM lane = output column, TMEM column = row);
//   * warps 18..21 (epilogue): when a CTA's part of an n-block is done they
//     stream TMEM (one output column per thread, the row permutation undone,
//     32 rows per load) into an
//     fp32 partial slot with coalesced row stores; the decode finalize kernel
//     sums each n-block's slots in slot order and applies had_r_128, sv and
//     the -inf mask.
//
// Roofline: the integer decode (K*N weights once) and the tensor work
// (2*M*K*N) overlap; HBM traffic is the trellis (K*N*BITS/8) plus x'.
#include <cuda.h>
#include <math.h>

#include "exl3_common.cuh"
#include "exl3_internal.h"
#include "exl3_tcgen05.cuh"

namespace exl3 {

namespace {

constexpr int F_BN = 128, F_BK = 64;
constexpr int F_DEC_WARPS = 16, F_EPI_WARPS = 4;
constexpr int F_GROUPS = F_DEC_WARPS / 4;    // k steps decoded concurrently (4 slabs each)
constexpr int F_THREADS = (2 + F_DEC_WARPS + F_EPI_WARPS) * 32;
constexpr int F_MAX_SA = 8;                  // x' stages at most
constexpr int F_B_STAGE = F_BN * F_BK * 2;   // one 128 x 64 fp16 W^T tile (128-byte swizzle)
constexpr int F_A_TILE = 128 * F_BK * 2;     // 128 rows x 64 fp16 of x' (128-byte swizzle)

// MTILES = ceil(npad / 128) sizes the x' region; npad is a runtime value and
// the region holds kARegion / (npad * 128 B) stages (2 .. 8).
template <int BITS, int MTILES>
struct FusedCfg {
  static constexpr int kSeg = 256 * BITS;
  // Trellis bytes each decoder warp keeps in flight (at least two slabs):
  // 16 warps x 2 KB per SM covers the HBM latency at the rate the decoders
  // consume; at 4 bits three slabs measured 0.1-0.9 us faster at 32..256
  // rows (4 KB: slower below 128 rows).
  static constexpr int kRingBytes = BITS == 4 ? 3072 : 2048;
  static constexpr int kRD = kRingBytes / kSeg < 2 ? 2 : kRingBytes / kSeg;
  static constexpr int kBudget = 227 * 1024 - 2048 - 2048;
  static constexpr int kRest = kBudget - F_DEC_WARPS * kRD * kSeg;
  // x' region: three stages at the widest npad of this variant when at least
  // five W^T stages still fit (the MMA issuer batches ready k steps only
  // with three or more x' stages), else two.
  static constexpr int kA3 = 3 * MTILES * F_A_TILE, kA2 = 2 * MTILES * F_A_TILE;
  static constexpr int kARegion = (kRest - kA3) / F_B_STAGE >= F_GROUPS + 1 ? kA3 : kA2;
  // W^T stages: the decoder groups run in rounds of F_GROUPS k steps; with
  // 2 * F_GROUPS stages a group only needs the stage the MMA was handed a
  // whole round earlier. Take as many as shared memory holds, up to that.
  static constexpr int kSBFit = (kRest - kARegion) / F_B_STAGE;
  static constexpr int kSB = kSBFit > 2 * F_GROUPS ? 2 * F_GROUPS : kSBFit;
  static constexpr int kOffB = kARegion;
  static constexpr int kOffD = kOffB + kSB * F_B_STAGE;
  static constexpr int kOffBar = kOffD + F_DEC_WARPS * kRD * kSeg;
  static constexpr int kNumBars = 2 * F_MAX_SA + 2 * kSB + 4 + 1 + F_DEC_WARPS * kRD;
  static constexpr int kSmem = 2048 + kOffBar + kNumBars * 8 + 16;
  static_assert(kSB > F_GROUPS, "W^T stages: one more than the k steps decoded at once, at least");
  static_assert(kNumBars * 8 + 16 <= 2048, "barrier area");
  static_assert(kOffB % 2048 == 0, "W^T stages must stay 2048-byte aligned");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

struct FusedParams {
  const uint8_t *trellis;
  const __half *sv;
  void *y;
  float *partials;
  int *status;
  int64_t tiles_n, n_gemm, n_valid, TS, P;
  int rows, y_f32, KS, smax;
  int npad;       // MMA N: rows rounded up to 32, <= 128 * MTILES
  int tmem_cols;  // power of two >= 2 * npad
  int nsa;        // x' stages of npad * 128 bytes in the x' region
  uint32_t m16;   // 16, opaque to the compiler (a multiply by it stays on the FMA pipe)
};

__device__ __forceinline__ int64_t unit_owner(int64_t z, int64_t P, int64_t TS) { return ((z + 1) * P - 1) / TS; }

__device__ __forceinline__ void wait_prior_grid_f() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// One lane of the (fully active) warp, the same lane every time.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Whole-warp bounded wait: every lane waits, and the warp agrees on the result.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int *status) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status)) != 0;
}
__device__ __forceinline__ void allow_next_grid_f() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <int BITS, int MTILES>
__global__ void __launch_bounds__(F_THREADS, 1)
    fused_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const FusedParams p) {
  using Cfg = FusedCfg<BITS, MTILES>;
  constexpr int F_SA = F_MAX_SA, F_SB = Cfg::kSB, F_RD = Cfg::kRD;
  const int nsa = p.nsa;
  const uint32_t a_stage = (uint32_t)p.npad * (F_BK * 2);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 2047) & ~(uintptr_t)2047);
  const uint32_t smem_s = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
  auto a_full = [&](int s) { return smem_u32(&bars[s]); };
  auto a_empty = [&](int s) { return smem_u32(&bars[F_SA + s]); };
  auto b_full = [&](int s) { return smem_u32(&bars[2 * F_SA + s]); };
  auto b_empty = [&](int s) { return smem_u32(&bars[2 * F_SA + F_SB + s]); };
  auto acc_full = [&](int a) { return smem_u32(&bars[2 * F_SA + 2 * F_SB + a]); };
  auto acc_empty = [&](int a) { return smem_u32(&bars[2 * F_SA + 2 * F_SB + 2 + a]); };
  const uint32_t done_bar = smem_u32(&bars[2 * F_SA + 2 * F_SB + 4]);
  auto dec_full = [&](int w, int s) { return smem_u32(&bars[2 * F_SA + 2 * F_SB + 5 + w * F_RD + s]); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Cfg::kNumBars);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t c = blockIdx.x;
  const int64_t zs = c * p.TS / p.P, ze = (c + 1) * p.TS / p.P;
  const int len = (int)(ze - zs);
  const int KS = p.KS;
  // The layout inside the CTA's shared memory, the x' stages inside their
  // region, the MMA width and the TMEM allocation (CTA-uniform: checked
  // before any barrier or TMEM is set up).
  if (!EXL3_SMEM(smem_s, Cfg::kOffBar + Cfg::kNumBars * 8 + 4) || !EXL3_RANGE(nsa, 1, F_SA + 1) ||
      !EXL3_SPAN(0, nsa * a_stage, Cfg::kARegion) || !EXL3_RANGE(p.npad, 32, 128 * MTILES + 1) ||
      !EXL3_ALIGNED(p.npad, 32) || !EXL3_SPAN(0, 2 * p.npad, p.tmem_cols) || !EXL3_RANGE(p.tmem_cols, 32, 513))
    return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nsa; ++s) {
      mbar_init(a_full(s), 1);
      mbar_init(a_empty(s), 1);
    }
    for (int s = 0; s < F_SB; ++s) {
      mbar_init(b_full(s), 4);
      mbar_init(b_empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full(a), 1);
      mbar_init(acc_empty(a), F_EPI_WARPS);
    }
    mbar_init(done_bar, 1);
    for (int w = 0; w < F_DEC_WARPS; ++w)
      for (int s = 0; s < F_RD; ++s) mbar_init(dec_full(w, s), 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(p.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  allow_next_grid_f();

  if (warp == 0) {
    // ---------------- x' producer (whole warp; one elected lane issues) ----------------
    wait_prior_grid_f();  // x' comes from the rotation kernel
    const bool leader = elect_one();
    int ks = (int)(zs % KS), as = 0, issued = 0;
    uint32_t aph = 0;
    for (int kk = 0; kk < len; ++kk) {
      if (!warp_wait(a_empty(as), aph ^ 1u, p.status)) break;
      if (leader) {
        mbar_arrive_expect_tx(a_full(as), a_stage);
        // box: fp16 columns [64 ks, +64) (128 bytes: the 16-byte rule), rows
        // [0, npad); the stage 1024-byte aligned for the 128-byte swizzle
        if (EXL3_RANGE(ks, 0, KS) && EXL3_RANGE(as, 0, nsa) && EXL3_ALIGNED(smem_s + as * a_stage, 1024))
          tma_load_2d(smem_s + as * a_stage, &tmA, a_full(as), ks * F_BK, 0);
      }
      __syncwarp();
      ++issued;
      if (++ks == KS) ks = 0;
      if (++as == nsa) {
        as = 0;
        aph ^= 1u;
      }
    }
    // Before leaving (also after a timeout), wait for the loads that may still
    // be in flight, in issue order: load u was issued only after load u - nsa
    // had been consumed, so at most the last nsa can be outstanding.
    if (leader)
      for (int u = issued > nsa ? issued - nsa : 0; u < issued; ++u)
        mbar_wait_short(a_full(u % nsa), (uint32_t)(u / nsa) & 1u);
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer (whole warp; one elected lane issues) ----------------
    // With 3 or more x' stages, each round the warp tests, without blocking,
    // whether the next `look` k steps' W^T stages (lanes 0..3) and x' stages
    // (lanes 8..11) are full and issues every consecutive ready k step in
    // one batch: a satisfied
    // barrier costs one test per batch, not a wait per k step. The lookahead
    // stays below both ring sizes, so each tested stage's previous use is
    // already consumed and its next use cannot complete before this warp
    // frees it: the parity tests cannot alias. Only when the current k step
    // is not ready does the warp block (bounded) on it. A batch ends where
    // an n-block ends, so each accumulator hand-off stays per segment.
    const bool leader = elect_one();
    const uint32_t idesc = f16_idesc(F_BN, p.npad);
    int ks = (int)(zs % KS), seg = 0, as = 0, bs = 0;
    uint32_t aph = 0, bph = 0;
    if (nsa < 3) {
      // Two x' stages (wide x' tiles): the next step's x' cannot land before
      // this warp frees a stage, so batches cannot form; one k step at a time.
      for (int kk = 0; kk < len; ++kk) {
        const bool first = (kk == 0) || (ks == 0);
        const bool last = (kk == len - 1) || (ks == KS - 1);
        const int ab = seg & 1;
        if (first) {
          if (!warp_wait(acc_empty(ab), ((uint32_t)(seg >> 1) & 1u) ^ 1u, p.status)) break;
          tc_fence_after();
        }
        if (!warp_wait(a_full(as), aph, p.status)) break;
        if (!warp_wait(b_full(bs), bph, p.status)) break;
        tc_fence_after();
        const uint64_t wdesc = sw128_desc(smem_s + Cfg::kOffB + bs * F_B_STAGE);
        const uint64_t xdesc = sw128_desc(smem_s + as * a_stage);
        const uint32_t d = tmem_base + (uint32_t)(ab * p.npad);
        if (leader) {
          // operand stages and the accumulator's npad TMEM columns
          const bool ok = EXL3_RANGE(as, 0, nsa) && EXL3_RANGE(bs, 0, F_SB) &&
                          EXL3_SPAN(ab * p.npad, p.npad, p.tmem_cols);
#pragma unroll
          for (int k16 = 0; k16 < F_BK / 16; ++k16)
            if (ok)
              tc_mma(d, wdesc + (uint64_t)(2 * k16), xdesc + (uint64_t)(2 * k16), idesc,
                     (!first || k16 > 0) ? 1u : 0u);
          tc_commit(a_empty(as));
          tc_commit(b_empty(bs));
          if (last) tc_commit(acc_full(ab));
        }
        __syncwarp();
        if (last) ++seg;
        if (++ks == KS) ks = 0;
        if (++as == nsa) {
          as = 0;
          aph ^= 1u;
        }
        if (++bs == F_SB) {
          bs = 0;
          bph ^= 1u;
        }
      }
    } else {
      const int look = nsa < 4 ? nsa : 4;  // F_SB > 4 always
      for (int kk = 0; kk < len;) {
        const int ab = seg & 1;
        if (kk == 0 || ks == 0) {
          if (!warp_wait(acc_empty(ab), ((uint32_t)(seg >> 1) & 1u) ^ 1u, p.status)) break;
          tc_fence_after();
        }
        bool rdy = false;
        {
          const int j = lane & 7;
          if (lane < 16 && j < look && kk + j < len) {
            if (lane < 8) {
              int s = bs + j;
              uint32_t ph = bph;
              if (s >= F_SB) {
                s -= F_SB;
                ph ^= 1u;
              }
              rdy = mbar_test_wait(b_full(s), ph);
            } else {
              int s = as + j;
              uint32_t ph = aph;
              if (s >= nsa) {
                s -= nsa;
                ph ^= 1u;
              }
              rdy = mbar_test_wait(a_full(s), ph);
            }
          }
        }
        const uint32_t bal = __ballot_sync(0xffffffffu, rdy);
        __syncwarp();  // the lanes' acquires are ordered before the issuing lane's MMAs
        const uint32_t both = bal & (bal >> 8) & 0xFFu;
        int n = __ffs(~both) - 1;  // leading run of ready k steps
        if (n > KS - ks) n = KS - ks;
        if (n == 0) {
          if (!warp_wait(a_full(as), aph, p.status)) break;
          if (!warp_wait(b_full(bs), bph, p.status)) break;
          n = 1;
        }
        tc_fence_after();
        if (leader) {
          int a = as, b = bs, k2 = ks;
          const uint32_t d = tmem_base + (uint32_t)(ab * p.npad);
          for (int t = 0; t < n; ++t) {
            const bool first = (kk + t == 0) || (k2 == 0);
            const bool last = (kk + t == len - 1) || (k2 == KS - 1);
            const uint64_t wdesc = sw128_desc(smem_s + Cfg::kOffB + b * F_B_STAGE);
            const uint64_t xdesc = sw128_desc(smem_s + a * a_stage);
            const bool ok = EXL3_RANGE(a, 0, nsa) && EXL3_RANGE(b, 0, F_SB) &&
                            EXL3_SPAN(ab * p.npad, p.npad, p.tmem_cols);
#pragma unroll
            for (int k16 = 0; k16 < F_BK / 16; ++k16)
              if (ok)
                tc_mma(d, wdesc + (uint64_t)(2 * k16), xdesc + (uint64_t)(2 * k16), idesc,
                       (!first || k16 > 0) ? 1u : 0u);
            tc_commit(a_empty(a));
            tc_commit(b_empty(b));
            if (last) tc_commit(acc_full(ab));
            if (++a == nsa) a = 0;
            if (++b == F_SB) b = 0;
            if (++k2 == KS) k2 = 0;
          }
        }
        __syncwarp();
        const int kl = kk + n - 1, ksl = ks + n - 1;  // the batch's last k step (ksl < KS)
        if (kl == len - 1 || ksl == KS - 1) ++seg;
        kk += n;
        ks = ksl + 1 == KS ? 0 : ksl + 1;
        as += n;
        if (as >= nsa) {
          as -= nsa;
          aph ^= 1u;
        }
        bs += n;
        if (bs >= F_SB) {
          bs -= F_SB;
          bph ^= 1u;
        }
      }
    }
    if (leader) {
      tc_commit(done_bar);
      mbar_wait_short(done_bar, 0);
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 2 + F_DEC_WARPS) {
    // ---------------- decoders ----------------
    const int dw = warp - 2;
    const int par = dw >> 2, slab_i = dw & 3;  // k steps par, par + F_GROUPS, ...; slab slab_i of each
    const int g = lane >> 2, q = lane & 3;
    const int nmine = len > par ? (len - par + F_GROUPS - 1) / F_GROUPS : 0;
    const uint32_t ring_s = smem_s + Cfg::kOffD + dw * F_RD * Cfg::kSeg;
    // Swizzled W^T address of (column 16g + c, rows 4q..4q+3 of slab slab_i)
    // = (stage + lane_off) ^ (c << 7 | (c & 7) << 4), stage 2048-byte aligned:
    // operand row t = c ^ g of
    // 8-row atom 2g + (t >> 3), 16-byte chunk (2 slab_i + (q >> 1)) ^ (t & 7).
    const uint32_t lane_off = (uint32_t)g * 2048u | (uint32_t)g << 7 |
                              (((uint32_t)(2 * slab_i + (q >> 1)) ^ (uint32_t)g) & 7u) << 4 | (uint32_t)(q & 1) << 3;
    int64_t issued = 0;
    // Cursor of the next slab to fetch (n-block, k step); fetches go in order.
    int64_t inb = (zs + par) / KS;
    int iks = (int)((zs + par) % KS);
    auto issue = [&](int j) {
      const int64_t nb = inb, tk = (int64_t)iks * 4 + slab_i;
      iks += F_GROUPS;
      while (iks >= KS) {
        iks -= KS;
        ++inb;
      }
      const int s = j % F_RD;
      mbar_arrive_expect_tx(dec_full(dw, s), Cfg::kSeg);
      // the slab's 8 tiles: tile row tk of the 4 KS, tiles [8 nb, +8) of tiles_n
      if (EXL3_RANGE(tk, 0, 4 * (int64_t)KS) && EXL3_RANGE(nb, 0, p.n_gemm / 128) &&
          EXL3_SPAN(nb * 8, 8, p.tiles_n) && EXL3_ALIGNED((tk * p.tiles_n + nb * 8) * (32 * BITS), 16))
        bulk_g2s(ring_s + s * Cfg::kSeg, p.trellis + (tk * p.tiles_n + nb * 8) * (32 * BITS), Cfg::kSeg,
                 dec_full(dw, s));
      ++issued;
    };
    if (lane == 0)
      for (int j = 0; j < F_RD - 1 && j < nmine; ++j) issue(j);
    int bs = par % F_SB;  // B stage of k step par + F_GROUPS * j, and its phase
    uint32_t bph = 0;
    // On a timeout the warp stops, but first waits (bounded) for the copies
    // it still has in flight into its ring, in issue order.
    auto drain_from = [&](int64_t u0) {
      if (lane == 0)
        for (int64_t u = u0; u < issued; ++u) mbar_wait_short(dec_full(dw, (int)(u % F_RD)), (uint32_t)(u / F_RD) & 1u);
    };
    for (int j = 0; j < nmine; ++j) {
      if (lane == 0 && j + F_RD - 1 < nmine) issue(j + F_RD - 1);
      const int s = j % F_RD;
      if (!mbar_wait(dec_full(dw, s), (uint32_t)(j / F_RD) & 1u, p.status)) {
        drain_from(j);
        break;
      }
      uint32_t own[2 * BITS];
      if (EXL3_SPAN(s * Cfg::kSeg + lane * 8 * BITS, 8 * BITS, F_RD * Cfg::kSeg)) {
        load_own_words_shared<BITS>(ring_s + s * Cfg::kSeg + lane * 8 * BITS, own);
      } else {
#pragma unroll
        for (int i = 0; i < 2 * BITS; ++i) own[i] = 0;
      }
      const uint32_t prev = prefix_from_neighbour<BITS>(own, lane);
      uint32_t st[4][16];
      if constexpr (BITS == 4) {
#pragma unroll
        for (int r = 0; r < 4; ++r) row4_states(own[2 * r], own[2 * r + 1], r == 0 ? prev : own[2 * r - 1], p.m16, st[r]);
      } else {
        RowWindows<BITS> rw;
        rw.build(own, prev);
        static_for<4>([&](auto R) {
          // plain extraction: the window views' multiplies measured mixed here (the
          // decoders load the FMA pipe too), -4 % to +4.5 % over bits 1..8
          static_for<16>([&](auto C) { st[R.value][C.value] = rw.template state<R.value, C.value>(); });
        });
      }
      if (!mbar_wait(b_empty(bs), bph ^ 1u, p.status)) {
        drain_from(j + 1);
        break;
      }
      const uint32_t bt = smem_s + Cfg::kOffB + bs * F_B_STAGE + lane_off;  // low 11 bits: lane_off's
      static_for<16>([&](auto C) {
        constexpr int cc = C.value;
        constexpr uint32_t cx = (uint32_t)cc << 7 | (uint32_t)(cc & 7) << 4;
        const uint32_t lo = decode_pair_sel<false>(st[0][cc], st[1][cc]);
        const uint32_t hi = decode_pair_sel<false>(st[2][cc], st[3][cc]);
        if (EXL3_RANGE(bs, 0, F_SB) && EXL3_SPAN((bt ^ cx) - (smem_s + Cfg::kOffB + bs * F_B_STAGE), 8, F_B_STAGE))
          st_shared_v2(bt ^ cx, lo, hi);
      });
      fence_proxy_async_shared();  // make the generic stores visible to the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(b_full(bs));
      bs += F_GROUPS;
      if (bs >= F_SB) {
        bs -= F_SB;
        bph ^= 1u;
      }
    }
  } else if (warp >= 2 + F_DEC_WARPS) {
    // ---------------- epilogue ----------------
    wait_prior_grid_f();  // the previous kernel may still read the partial slots
    const int lg = warp & 3;
    int seg = 0;
    int64_t nb = zs / KS;
    // Segment ends (local k step indexes): the last k step of each n-block
    // the range touches, or the range's last k step.
    for (int e = (int)(KS - 1 - zs % KS);; e += KS, ++nb) {
      const int ab = seg & 1;
      if (!mbar_wait(acc_full(ab), (uint32_t)(seg >> 1) & 1u, p.status)) break;
      tc_fence_after();
      // Every CTA stores its part of the n-block as an fp32 partial slot; the
      // finalize kernel sums the slots and applies the output rotation.
      const int64_t pf = unit_owner(nb * KS, p.P, p.TS);
      const int i = lg * 32 + lane;  // operand row = TMEM lane
      float *slot = p.partials + (nb * p.smax + (c - pf)) * (int64_t)(MTILES * 128 * 128) + 16 * (i >> 4) +
                    ((i & 15) ^ (i >> 4));
      const uint32_t taddr = tmem_base + ((uint32_t)(lg * 32) << 16) + (uint32_t)(ab * p.npad);
      // slot c - pf of the n-block's smax, rows < 128 * MTILES of the slot
      const bool slot_ok = EXL3_RANGE(nb, 0, p.n_gemm / 128) && EXL3_RANGE(c - pf, 0, p.smax) &&
                           EXL3_RANGE(p.rows, 1, 128 * MTILES + 1);
#pragma unroll 1
      for (int m0 = 0; m0 < p.rows; m0 += 32) {
        float t[32];
        // 32 TMEM columns inside this accumulator (warp-uniform)
        if (EXL3_SPAN(ab * p.npad + m0, 32, p.tmem_cols) && EXL3_SPAN(m0, 32, p.npad)) {
          tmem_ld32(taddr + m0, t);
        } else {
#pragma unroll
          for (int r = 0; r < 32; ++r) t[r] = 0.f;
        }
        if (slot_ok && m0 + 32 <= p.rows) {
#pragma unroll
          for (int r = 0; r < 32; ++r) slot[(int64_t)(m0 + r) * 128] = t[r];
        } else if (slot_ok) {
#pragma unroll
          for (int r = 0; r < 32; ++r)
            if (m0 + r < p.rows) slot[(int64_t)(m0 + r) * 128] = t[r];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(ab));
      ++seg;
      if (e >= len - 1) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(p.tmem_cols)
                 : "memory");
  }
}

template <int BITS, int MTILES>
cudaError_t init_one() {
  return cudaFuncSetAttribute(fused_gemm_kernel<BITS, MTILES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              FusedCfg<BITS, MTILES>::kSmem);
}

template <int BITS>
cudaError_t init_bits() {
  cudaError_t e = init_one<BITS, 1>();
  if (e != cudaSuccess) return e;
  return init_one<BITS, 2>();
}

template <int BITS, int MTILES>
cudaError_t launch_bits(const CUtensorMap &tmA, const FusedParams &fp, int64_t grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(F_THREADS);
  cfg.dynamicSmemBytes = FusedCfg<BITS, MTILES>::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_gemm_kernel<BITS, MTILES>, tmA, fp);
}

template <int MTILES>
cudaError_t launch_mt(int bits, const CUtensorMap &tmA, const FusedParams &fp, int64_t grid, cudaStream_t st) {
  switch (bits) {
    case 1: return launch_bits<1, MTILES>(tmA, fp, grid, st);
    case 2: return launch_bits<2, MTILES>(tmA, fp, grid, st);
    case 3: return launch_bits<3, MTILES>(tmA, fp, grid, st);
    case 4: return launch_bits<4, MTILES>(tmA, fp, grid, st);
    case 5: return launch_bits<5, MTILES>(tmA, fp, grid, st);
    case 6: return launch_bits<6, MTILES>(tmA, fp, grid, st);
    case 7: return launch_bits<7, MTILES>(tmA, fp, grid, st);
    case 8: return launch_bits<8, MTILES>(tmA, fp, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

int64_t owner_h(int64_t z, int64_t P, int64_t TS) { return ((z + 1) * P - 1) / TS; }

template <int MTILES>
int a_region_mt(int bits) {
  switch (bits) {
    case 1: return FusedCfg<1, MTILES>::kARegion;
    case 2: return FusedCfg<2, MTILES>::kARegion;
    case 3: return FusedCfg<3, MTILES>::kARegion;
    case 4: return FusedCfg<4, MTILES>::kARegion;
    case 5: return FusedCfg<5, MTILES>::kARegion;
    case 6: return FusedCfg<6, MTILES>::kARegion;
    case 7: return FusedCfg<7, MTILES>::kARegion;
    default: return FusedCfg<8, MTILES>::kARegion;
  }
}

int a_region_bytes(int bits, int mtiles) { return mtiles == 1 ? a_region_mt<1>(bits) : a_region_mt<2>(bits); }

}  // namespace

FusedPlan fused_plan(int64_t n_blocks, int64_t K, int num_sms) {
  FusedPlan f;
  const int64_t KS = K / F_BK;
  f.TS = n_blocks * KS;
  f.P = f.TS < num_sms ? f.TS : num_sms;
  f.smax = 1;
  for (int64_t nb = 0; nb < n_blocks; ++nb) {
    const int64_t cnt = owner_h((nb + 1) * KS - 1, f.P, f.TS) - owner_h(nb * KS, f.P, f.TS) + 1;
    if (cnt > f.smax) f.smax = cnt;
  }
  return f;
}

size_t fused_partials_bytes(const FusedPlan &f, int64_t n_blocks) {
  return (size_t)n_blocks * f.smax * 256 * 128 * 4;
}

cudaError_t init_fused_kernels(int *status) {
  cudaError_t e = EXL3_BIND_BOUNDS_WORD(status);
  if (e != cudaSuccess) return e;
  if ((e = init_bits<1>()) != cudaSuccess) return e;
  if ((e = init_bits<2>()) != cudaSuccess) return e;
  if ((e = init_bits<3>()) != cudaSuccess) return e;
  if ((e = init_bits<4>()) != cudaSuccess) return e;
  if ((e = init_bits<5>()) != cudaSuccess) return e;
  if ((e = init_bits<6>()) != cudaSuccess) return e;
  if ((e = init_bits<7>()) != cudaSuccess) return e;
  return init_bits<8>();
}

cudaError_t launch_fused_gemm(const FusedLaunch &L, cudaStream_t st) {
  if (L.rows < 1 || L.rows > kFusedMaxRows) return cudaErrorInvalidValue;
  const int npad = (L.rows + 31) & ~31;
  const int MTILES = npad <= 128 ? 1 : 2;
  int tmem_cols = 32;
  while (tmem_cols < 2 * npad) tmem_cols *= 2;
  alignas(64) CUtensorMap tmA;
  if (!encode_tensor_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, L.xr, (uint64_t)L.K, (uint64_t)L.xr_rows,
                            (uint64_t)L.K * 2, F_BK, (uint32_t)npad, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  FusedParams fp;
  fp.trellis = reinterpret_cast<const uint8_t *>(L.trellis);
  fp.sv = static_cast<const __half *>(L.sv);
  fp.y = L.y;
  fp.partials = L.partials;
  fp.status = L.status;
  fp.tiles_n = L.n_stored / 16;
  fp.n_gemm = L.n_gemm;
  fp.n_valid = L.n_valid;
  fp.TS = L.plan.TS;
  fp.P = L.plan.P;
  fp.rows = L.rows;
  fp.y_f32 = L.y_f32;
  fp.KS = (int)(L.K / F_BK);
  fp.smax = (int)L.plan.smax;
  fp.npad = npad;
  fp.tmem_cols = tmem_cols;
  fp.m16 = 16u;
  fp.nsa = a_region_bytes(L.bits, MTILES) / (npad * F_BK * 2);
  if (fp.nsa > F_MAX_SA) fp.nsa = F_MAX_SA;
  cudaError_t e = MTILES == 1 ? launch_mt<1>(L.bits, tmA, fp, fp.P, st) : launch_mt<2>(L.bits, tmA, fp, fp.P, st);
  if (e != cudaSuccess) return e;
  return launch_decode_finalize(L.partials, fp.smax, (int64_t)MTILES * 128 * 128, L.sv, L.y, L.y_f32, L.n_gemm,
                                L.n_valid, L.rows, fp.P, fp.TS, fp.KS, /*all_blocks=*/1, st);
}

#if EXL3_DEBUG_BOUNDS
cudaError_t bounds_probe_fused(cudaStream_t st) { return launch_bounds_probe(st); }
#endif

}  // namespace exl3
