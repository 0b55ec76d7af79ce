// Fused prefill-shaped layer on CTA pairs: the trellis is decoded by producer
// warps straight into the tensor-core operand buffers, so no reconstructed
// weight is written to HBM, and each decoded weight serves 512 activation
// rows.
//
//     y[:, :] = had_r_128( x' . W ) * sv          (x' already rotated)
//
// This is the "dequant fused into the GEMM" kernel that vLLM PR #316,
// "[EXL3] dispatch prefill-shaped GEMMs to reconstruct+hgemm" (section "The
// remaining gap is structural" and the follow-up comment's ceiling
// arithmetic) names as the step beyond the reconstruct + hgemm sequence,
// built for sm_103a.
//
// Work: a cluster of two CTAs (two SMs) owns a tile of 512 rows x 256 output
// columns and runs its whole K. Per 64-deep k step:
//   * warp 0 (one lane) of each CTA: TMA loads of this CTA's 128 rows of each
//     of the tile's two 256-row sub-blocks of x' (128-byte swizzle); both
//     CTAs' bytes complete on the even CTA's stage barrier;
//   * warps 2..13 of each CTA (decoders): this CTA's 128-column n-block of
//     W^T, decoded into the N operand (K-major, 128-byte swizzle), four warps
//     per k step, each a 16-row slab whose trellis words every lane loads
//     from global memory one slab ahead, into registers (no shared-memory
//     ring: that room goes to a fourth x' stage); the operand-row
//     permutation of the decode-shaped fused kernel: column 16g + c at
//     operand row 16g + (c ^ g);
//   * warp 1 of the even CTA (one lane): two tcgen05.mma.cta_group::2 chains
//     (M = 256 rows, N = 256 columns, K = 16): sub-block j into TMEM columns
//     256 j .. 256 j + 255 of both CTAs (TMEM lane = row, column = output
//     column in operand order);
//   * warps 14..21 of each CTA (epilogue, two per TMEM lane group, one per
//     128-column half): after the tile's last k step, per row and
//     128-column block, had_r_128 as a 32-point transform of each
//     32-column chunk (written back to TMEM in output order) followed by a
//     4-point transform across the chunks, then sv, the -inf mask and the
//     store. The stages run in the order h = 1, 2, ..., 64 with the same
//     additions as the whole-row form.
// The accumulator takes all 512 TMEM columns, so the next tile's MMAs wait
// for the epilogue; the decoders and the x' producer run ahead meanwhile.
//
// Roofline: per SM and k step, 128 x 256 x 2 MACs (about 1050 cycles of
// tensor work) and 128 x 64 weights decoded (8 a cycle keep up); HBM: the
// trellis read once per 512 rows, x' once per 256 output columns. Measured,
// a k step takes about 1.5x its tensor work with the decoders well ahead;
// the shared-memory traffic (about 112 KB per SM per k step of TMA writes,
// decoder writes and operand reads) is the likely bound.
#include <cuda.h>
#include <math.h>

#include "exl3_common.cuh"
#include "exl3_internal.h"
#include "exl3_tcgen05.cuh"

namespace exl3 {

namespace {

constexpr int FP_BK = 64;
// 12 decoder warps keep ahead of the MMA (they wait for free W^T stages most
// of the time); 8 epilogue warps (two per TMEM lane group, one per 128-column
// half) share the single-buffered accumulator's drain.
constexpr int FP_DEC_WARPS = 12, FP_EPI_WARPS = 8;
constexpr int FP_GROUPS = FP_DEC_WARPS / 4;  // k steps decoded concurrently (4 slabs each)
constexpr int FP_THREADS = (2 + FP_DEC_WARPS + FP_EPI_WARPS) * 32;
constexpr int FP_SUB = 128 * FP_BK * 2;      // 128 rows x 64 fp16 (an x' sub-block half or a W^T n-block)
constexpr int FP_TMEM_COLS = 512;
constexpr uint32_t kIdescFP = f16_idesc(256, 256);

template <int BITS>
struct FPCfg {
  static constexpr int kRest = 227 * 1024 - 2048 - 1024;
  // x' stages (two 16 KB halves each): four, leaving room for five W^T
  // stages (the least the four decoder groups need).
  static constexpr int kSA = (kRest - (FP_GROUPS + 1) * FP_SUB) / (2 * FP_SUB) > 4
                                 ? 4 : (kRest - (FP_GROUPS + 1) * FP_SUB) / (2 * FP_SUB);
  // W^T stages: with 2 * FP_GROUPS a decoder group only needs the stage the
  // MMA was handed a whole round earlier; as many as fit, up to that.
  static constexpr int kSBFit = (kRest - kSA * 2 * FP_SUB) / FP_SUB;
  static constexpr int kSB = kSBFit > 2 * FP_GROUPS ? 2 * FP_GROUPS : kSBFit;
  static constexpr int kOffB = kSA * 2 * FP_SUB;
  static constexpr int kOffBar = kOffB + kSB * FP_SUB;
  static constexpr int kNumBars = 2 * kSA + 2 * kSB + 3;
  // barriers and the TMEM slot, then the current tile's 256 sv values
  static constexpr int kOffSv = kOffBar + 512;
  static constexpr int kSmem = 2048 + kOffSv + 512;
  static_assert(kSB > FP_GROUPS, "W^T stages: one more than the k steps decoded at once, at least");
  static_assert(kNumBars * 8 + 16 <= 512, "barrier area");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

struct FPParams {
  const uint8_t *trellis;
  const __half *sv;
  void *y;
  int *status;
  int64_t tiles_n;  // trellis tiles per 16-row k tile (n_stored / 16)
  int64_t n_gemm, n_valid;
  int M, KS, y_f32;
  int ntb;          // 512-row blocks
  int ncp;          // 256-column blocks
  int last_row0;    // first row of the last 128-row block of x'
  uint32_t m16;     // 16, opaque to the compiler
};

// One 128-column block of one output row from TMEM columns taddr .. +127
// (the decoders' operand order), then * sv (the block's 128 values at shared
// address sv_s), mask, store.
__device__ __forceinline__ void fp_epilogue_block(uint32_t taddr, const FPParams &p, int64_t row, int64_t col0,
                                                  uint32_t sv_s) {
  // 32-point transforms (stages h = 1 .. 16) of the four 32-column chunks,
  // in output-column order, written back to TMEM.
  static_for<4>([&](auto A) {
    constexpr int a = A.value;
    float r[32], u[32];
    tmem_ld32(taddr + 32 * a, r);
    static_for<32>([&](auto I) {
      constexpr int i = I.value, h = i >> 4, c = i & 15, g = 2 * a + h;
      u[i] = r[16 * h + (c ^ g)];  // operand row 16g + (c ^ g) holds column 16g + c
    });
#pragma unroll
    for (int s = 1; s < 32; s <<= 1)
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (!(i & s)) {
          const float x0 = u[i], x1 = u[i + s];
          u[i] = x0 + x1;
          u[i + s] = x0 - x1;
        }
    tmem_st32(taddr + 32 * a, u);
  });
  tmem_wait_st();
  const bool store = row < p.M;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    float w[32];  // w[8a + i]: column 32a + 8s + i
    tmem_ld4x8(taddr + 8 * s, 32, w);
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // stages h = 32 (chunks a, a ^ 1) and 64 (a, a ^ 2)
      const float c0 = w[i] + w[8 + i], c1 = w[i] - w[8 + i];
      const float c2 = w[16 + i] + w[24 + i], c3 = w[16 + i] - w[24 + i];
      w[i] = c0 + c2;
      w[16 + i] = c0 - c2;
      w[8 + i] = c1 + c3;
      w[24 + i] = c1 - c3;
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int64_t col = col0 + 32 * a + 8 * s;
      // sv and y columns [col, col + 8) inside the GEMM width
      const bool cols_ok = EXL3_SPAN(col, 8, p.n_gemm);
      uint4 raw;
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(raw.x), "=r"(raw.y), "=r"(raw.z), "=r"(raw.w)
                   : "r"(sv_s + (uint32_t)(2 * (32 * a + 8 * s))));
      const __half *hv = reinterpret_cast<const __half *>(&raw);
      float o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        o[i] = (col + i < p.n_valid) ? w[8 * a + i] * (__half2float(hv[i]) * kInvSqrt128) : -INFINITY;
      if (!store || !cols_ok) continue;
      if (p.y_f32) {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.y) + row * p.n_gemm + col);
        dst[0] = make_float4(o[0], o[1], o[2], o[3]);
        dst[1] = make_float4(o[4], o[5], o[6], o[7]);
      } else {
        uint32_t hw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __half2 h2 = __floats2half2_rn(o[2 * e], o[2 * e + 1]);
          hw[e] = *reinterpret_cast<uint32_t *>(&h2);
        }
        *reinterpret_cast<uint4 *>(static_cast<__half *>(p.y) + row * p.n_gemm + col) =
            make_uint4(hw[0], hw[1], hw[2], hw[3]);
      }
    }
  }
}

// 704 threads, one CTA per SM: 22 warps over four 16 K-register sub-partitions
// (six warps on two of them) allow 80 registers a thread.
template <int BITS>
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(80)
    fused_prefill_kernel(const __grid_constant__ CUtensorMap tmA, const FPParams p) {
  using Cfg = FPCfg<BITS>;
  constexpr int SA = Cfg::kSA, SB = Cfg::kSB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 2047) & ~(uintptr_t)2047);
  const uint32_t smem_s = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
  auto a_full = [&](int s) { return smem_u32(&bars[s]); };
  auto a_empty = [&](int s) { return smem_u32(&bars[SA + s]); };
  auto b_full = [&](int s) { return smem_u32(&bars[2 * SA + s]); };
  auto b_empty = [&](int s) { return smem_u32(&bars[2 * SA + SB + s]); };
  const uint32_t acc_full = smem_u32(&bars[2 * SA + 2 * SB]);
  const uint32_t acc_empty = smem_u32(&bars[2 * SA + 2 * SB + 1]);
  const uint32_t done_bar = smem_u32(&bars[2 * SA + 2 * SB + 2]);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Cfg::kNumBars);
  auto a_s = [&](int s, int j) { return smem_s + (uint32_t)(s * 2 * FP_SUB + j * FP_SUB); };
  auto b_s = [&](int s) { return smem_s + (uint32_t)(Cfg::kOffB + s * FP_SUB); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
  const int KS = p.KS;
  const int ntiles = p.ntb * p.ncp;
  const int my_tiles = pair < ntiles ? (ntiles - 1 - pair) / npairs + 1 : 0;
  const int64_t len = (int64_t)my_tiles * KS;  // this pair's (tile, k step) units, in order
  // Tile i of this pair: 512-row block tb, 256-column block cp.
  auto tile_tb = [&](int i) { return (pair + i * npairs) / p.ncp; };
  auto tile_cp = [&](int i) { return (pair + i * npairs) % p.ncp; };
  // The layout inside the CTA's shared memory (the same in both CTAs, so
  // both leave here or neither).
  if (!EXL3_SMEM(smem_s, Cfg::kOffBar + Cfg::kNumBars * 8 + 4)) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      mbar_init(a_full(s), 1);
      mbar_init(a_empty(s), 1);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(b_full(s), 8);  // four decoder warps of each CTA
      mbar_init(b_empty(s), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * FP_EPI_WARPS);
    mbar_init(done_bar, 1);
    fence_barrier_init();
  }
  if (warp == 1) {  // one warp of each CTA of the pair allocates together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(FP_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();  // both CTAs' barriers initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- x' producer (both CTAs, one lane) ----------------
    if (lane == 0) {
      int as = 0, i = 0, ks = 0;
      uint32_t aph = 0;
      int64_t issued = 0;
      for (int64_t z = 0; z < len; ++z) {
        const int tb = tile_tb(i);
        const int nsub = tb * 512 + 256 < p.M ? 2 : 1;
        if (!mbar_wait(a_empty(as), aph ^ 1u, p.status)) break;
        if (rank == 0) mbar_arrive_expect_tx(a_full(as), (uint32_t)(2 * nsub * FP_SUB));
        const uint32_t fb = map_to_rank(a_full(as), 0);
        for (int j = 0; j < nsub; ++j) {
          // this CTA's 128 rows of sub-block j; past the last rotated row
          // block, the last one again (those rows are never stored)
          const int r0 = min(tb * 512 + 256 * j + 128 * (int)rank, p.last_row0);
          if (EXL3_RANGE(ks, 0, KS) && EXL3_RANGE(r0, 0, p.last_row0 + 1) && EXL3_ALIGNED(ks * FP_BK * 2, 16))
            tma_load_2d_pair(a_s(as, j), &tmA, fb, ks * FP_BK, r0);
        }
        ++issued;
        if (++as == SA) {
          as = 0;
          aph ^= 1u;
        }
        if (++ks == KS) {
          ks = 0;
          ++i;
        }
      }
      // Rank 0's stage barriers count both CTAs' bytes: once each stage's last
      // use has completed there, no copy of either CTA is in flight (the final
      // cluster barrier keeps the odd CTA until then).
      if (rank == 0)
        for (int64_t u = issued > SA ? issued - SA : 0; u < issued; ++u)
          mbar_wait_cluster(a_full((int)(u % SA)), (uint32_t)(u / SA) & 1u, nullptr, 200000000ull);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (even CTA, one lane) ----------------
    if (lane == 0 && rank == 0) {
      int as = 0, bs = 0, i = 0, ks = 0;
      uint32_t aph = 0, bph = 0;
      for (int64_t z = 0; z < len; ++z) {
        const int nsub = tile_tb(i) * 512 + 256 < p.M ? 2 : 1;
        if (ks == 0) {
          if (!mbar_wait_cluster(acc_empty, ((uint32_t)i & 1u) ^ 1u, p.status, kWaitLimitNs)) break;
          tc_fence_after();
        }
        if (!mbar_wait_cluster(a_full(as), aph, p.status, kWaitLimitNs)) break;
        if (!mbar_wait_cluster(b_full(bs), bph, p.status, kWaitLimitNs)) break;
        tc_fence_after();
        const uint64_t bd = sw128_desc(b_s(bs));
        for (int j = 0; j < nsub; ++j) {
          const uint64_t ad = sw128_desc(a_s(as, j));
#pragma unroll
          for (int k16 = 0; k16 < FP_BK / 16; ++k16)
            if (EXL3_RANGE(j, 0, 2))  // 256 TMEM columns of the 512 allocated
              tc_mma_pair(tmem_base + (uint32_t)(256 * j), ad + (uint64_t)(2 * k16), bd + (uint64_t)(2 * k16),
                          kIdescFP, (ks | k16) != 0);
        }
        tc_commit_pair(a_empty(as), 3);
        tc_commit_pair(b_empty(bs), 3);
        if (ks == KS - 1) tc_commit_pair(acc_full, 3);
        if (++as == SA) {
          as = 0;
          aph ^= 1u;
        }
        if (++bs == SB) {
          bs = 0;
          bph ^= 1u;
        }
        if (++ks == KS) {
          ks = 0;
          ++i;
        }
      }
      // Every issued MMA (they write both CTAs' TMEM) finishes before the
      // final cluster barrier, after which both CTAs release their TMEM.
      tc_commit_pair(done_bar, 1);
      mbar_wait_cluster(done_bar, 0, nullptr, 200000000ull);
    }
  } else if (warp < 2 + FP_DEC_WARPS) {
    // ---------------- decoders (both CTAs) ----------------
    const int dw = warp - 2;
    const int par = dw >> 2, slab_i = dw & 3;  // units par, par + FP_GROUPS, ...; slab slab_i of each
    const int g = lane >> 2, q = lane & 3;
    const int64_t nmine = len > par ? (len - par + FP_GROUPS - 1) / FP_GROUPS : 0;
    // Swizzled W^T address of (column 16g + c, rows 4q..4q+3 of slab slab_i)
    // = (stage + lane_off) ^ (c << 7 | (c & 7) << 4), stage 2048-byte aligned:
    // operand row t = c ^ g of 8-row atom 2g + (t >> 3), 16-byte chunk
    // (2 slab_i + (q >> 1)) ^ (t & 7).
    const uint32_t lane_off = (uint32_t)g * 2048u | (uint32_t)g << 7 |
                              (((uint32_t)(2 * slab_i + (q >> 1)) ^ (uint32_t)g) & 7u) << 4 | (uint32_t)(q & 1) << 3;
    const int64_t nblk = p.n_gemm / 128;
    // Cursor of the next slab to load (tile i, k step ks); loads go in order.
    int fi = (int)(par / KS), fks = (int)(par % KS);
    // The lane's 8 * BITS bytes of the next slab, loaded into `w`.
    auto load_next = [&](uint32_t (&w)[2 * BITS]) {
      // this CTA's n-block of the tile (the last real one for a 128-wide last
      // column block: decoded, never stored)
      int64_t nb = 2 * (int64_t)tile_cp(fi) + rank;
      if (nb >= nblk) nb = nblk - 1;
      const int64_t tk = (int64_t)fks * 4 + slab_i;
      fks += FP_GROUPS;
      while (fks >= KS) {
        fks -= KS;
        ++fi;
      }
      // the slab's 8 tiles: tile row tk of the 4 KS, tiles [8 nb, +8) of tiles_n
      if (EXL3_RANGE(tk, 0, 4 * (int64_t)KS) && EXL3_SPAN(nb * 8, 8, p.tiles_n)) {
        load_own_words<BITS, false>(p.trellis + (tk * p.tiles_n + nb * 8) * (32 * BITS) + lane * 8 * BITS, w);
      } else {
#pragma unroll
        for (int k = 0; k < 2 * BITS; ++k) w[k] = 0;
      }
    };
    uint32_t nxt[2 * BITS];
    if (nmine > 0) load_next(nxt);
    int bs = par % SB;  // W^T stage of unit par + FP_GROUPS * j, and its phase
    uint32_t bph = 0;
    const uint32_t bf_leader0 = map_to_rank(b_full(0), 0);
    for (int64_t jj = 0; jj < nmine; ++jj) {
      uint32_t own[2 * BITS];
#pragma unroll
      for (int k = 0; k < 2 * BITS; ++k) own[k] = nxt[k];
      if (jj + 1 < nmine) load_next(nxt);
      const uint32_t prev = prefix_from_neighbour<BITS>(own, lane);
      uint32_t st[4][16];
      if constexpr (BITS == 4) {
#pragma unroll
        for (int r = 0; r < 4; ++r) row4_states(own[2 * r], own[2 * r + 1], r == 0 ? prev : own[2 * r - 1], p.m16, st[r]);
      } else {
        RowWindows<BITS> rw;
        rw.build(own, prev);
        static_for<4>([&](auto R) {
          static_for<16>([&](auto C) { st[R.value][C.value] = rw.template state<R.value, C.value>(); });
        });
      }
      if (!mbar_wait(b_empty(bs), bph ^ 1u, p.status)) break;
      const uint32_t bt = b_s(bs) + lane_off;  // low 11 bits: lane_off's
      static_for<16>([&](auto C) {
        constexpr int cc = C.value;
        constexpr uint32_t cx = (uint32_t)cc << 7 | (uint32_t)(cc & 7) << 4;
        const uint32_t lo = decode_pair_sel<false>(st[0][cc], st[1][cc]);
        const uint32_t hi = decode_pair_sel<false>(st[2][cc], st[3][cc]);
        if (EXL3_RANGE(bs, 0, SB) && EXL3_SPAN((bt ^ cx) - b_s(bs), 8, FP_SUB)) st_shared_v2(bt ^ cx, lo, hi);
      });
      // The generic stores (to this CTA's shared memory), visible to the
      // tensor core; then the stage's arrival on the even CTA's barrier:
      // local there, remote (release at cluster scope) from the odd CTA.
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(b_full(bs)); else mbar_arrive_cluster(bf_leader0 + 8u * (uint32_t)bs);
      }
      bs += FP_GROUPS;
      if (bs >= SB) {
        bs -= SB;
        bph ^= 1u;
      }
    }
  } else {
    // ---------------- epilogue (both CTAs) ----------------
    const int lg = warp & 3;  // TMEM lane group this warp may access
    const int ew = warp - 2 - FP_DEC_WARPS;  // 0 .. 7
    const int h = ew >> 2;                   // the 128-column half this warp rotates
    const uint32_t ae = map_to_rank(acc_empty, 0);
    const uint32_t sv_s = smem_s + Cfg::kOffSv;
    const int et = ew * 32 + lane;  // 0 .. 255
    for (int i = 0; i < my_tiles; ++i) {
      const int tb = tile_tb(i), cp = tile_cp(i);
      const int nsub = tb * 512 + 256 < p.M ? 2 : 1;
      // The tile's sv column 256 cp + et goes to shared memory once every
      // epilogue thread has its accumulator (and is done with the previous
      // tile's sv). The named barrier also makes the decision to stop after
      // a timed-out wait the same in all eight warps.
      const int64_t col = (int64_t)cp * 256 + et;
      const uint32_t v = col < p.n_gemm ? (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(p.sv + col)) : 0u;
      const uint32_t ok = mbar_wait(acc_full, (uint32_t)i & 1u, p.status) ? 1u : 0u;
      uint32_t all_ok;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\t"
          "setp.ne.u32 q, %1, 0;\n\t"
          "barrier.red.and.pred p, 1, %2, q;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(all_ok)
          : "r"(ok), "n"(FP_EPI_WARPS * 32)
          : "memory");
      if (!all_ok) break;
      asm volatile("st.shared.u16 [%0], %1;" ::"r"(sv_s + 2u * (uint32_t)et), "h"((unsigned short)v) : "memory");
      asm volatile("bar.sync 1, %0;" ::"n"(FP_EPI_WARPS * 32) : "memory");
      tc_fence_after();
      const int64_t col0 = (int64_t)cp * 256 + 128 * h;
      for (int j = 0; j < nsub; ++j) {
        const int64_t row = (int64_t)tb * 512 + 256 * j + 128 * (int)rank + lg * 32 + lane;
        if (col0 < p.n_gemm)
          fp_epilogue_block(tmem_base + ((uint32_t)(lg * 32) << 16) + (uint32_t)(256 * j + 128 * h), p, row, col0,
                            sv_s + 256u * (uint32_t)h);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(ae);
    }
  }

  tc_fence_before();
  __syncwarp();
  cluster_sync_all();  // no remote arrival or copy of either CTA is pending
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(FP_TMEM_COLS)
                 : "memory");
  }
}

template <int BITS>
cudaError_t init_one() {
  return cudaFuncSetAttribute(fused_prefill_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              FPCfg<BITS>::kSmem);
}

template <int BITS>
cudaError_t launch_bits(const CUtensorMap &tmA, const FPParams &fp, int grid, cudaStream_t st) {
  fused_prefill_kernel<BITS><<<grid, FP_THREADS, FPCfg<BITS>::kSmem, st>>>(tmA, fp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t init_fused_prefill_kernels(int *status) {
  cudaError_t e = EXL3_BIND_BOUNDS_WORD(status);
  if (e != cudaSuccess) return e;
  if ((e = init_one<1>()) != cudaSuccess) return e;
  if ((e = init_one<2>()) != cudaSuccess) return e;
  if ((e = init_one<3>()) != cudaSuccess) return e;
  if ((e = init_one<4>()) != cudaSuccess) return e;
  if ((e = init_one<5>()) != cudaSuccess) return e;
  if ((e = init_one<6>()) != cudaSuccess) return e;
  if ((e = init_one<7>()) != cudaSuccess) return e;
  return init_one<8>();
}

cudaError_t launch_fused_prefill(const FusedPrefillLaunch &L, cudaStream_t st) {
  if (L.M == 0) return cudaSuccess;
  if (L.M < 0 || L.xr_rows < ceil_div(L.M, 128) * 128 || L.K % FP_BK || L.n_gemm % 128 || L.num_sms < 2)
    return cudaErrorInvalidValue;
  alignas(64) CUtensorMap tmA;
  if (!encode_tensor_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, L.xr, (uint64_t)L.K, (uint64_t)L.xr_rows,
                            (uint64_t)L.K * 2, FP_BK, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  FPParams fp;
  fp.trellis = reinterpret_cast<const uint8_t *>(L.trellis);
  fp.sv = static_cast<const __half *>(L.sv);
  fp.y = L.y;
  fp.status = L.status;
  fp.tiles_n = L.n_stored / 16;
  fp.n_gemm = L.n_gemm;
  fp.n_valid = L.n_valid;
  fp.M = (int)L.M;
  fp.KS = (int)(L.K / FP_BK);
  fp.y_f32 = L.y_f32;
  fp.ntb = (int)ceil_div(L.M, 512);
  fp.ncp = (int)ceil_div(L.n_gemm, 256);
  fp.last_row0 = (int)((ceil_div(L.M, 128) - 1) * 128);
  fp.m16 = 16u;
  const int64_t ntiles = (int64_t)fp.ntb * fp.ncp;
  const int64_t pairs = ntiles < L.num_sms / 2 ? ntiles : L.num_sms / 2;
  const int grid = (int)(2 * pairs);
  switch (L.bits) {
    case 1: return launch_bits<1>(tmA, fp, grid, st);
    case 2: return launch_bits<2>(tmA, fp, grid, st);
    case 3: return launch_bits<3>(tmA, fp, grid, st);
    case 4: return launch_bits<4>(tmA, fp, grid, st);
    case 5: return launch_bits<5>(tmA, fp, grid, st);
    case 6: return launch_bits<6>(tmA, fp, grid, st);
    case 7: return launch_bits<7>(tmA, fp, grid, st);
    case 8: return launch_bits<8>(tmA, fp, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

#if EXL3_DEBUG_BOUNDS
cudaError_t bounds_probe_fused_prefill(cudaStream_t st) { return launch_bounds_probe(st); }
#endif

}  // namespace exl3
