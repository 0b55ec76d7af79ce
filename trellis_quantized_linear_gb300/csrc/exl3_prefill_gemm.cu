// Prefill-shaped dense GEMM on the 5th-generation tensor cores (tcgen05),
// with the output rotation fused into its epilogue:
//
//     y[:, c0:c0+nc] = had_r_128( x' . W[:, c0:c0+nc] ) * sv[c0:c0+nc]
//
// This is the "hgemm" stage of the unfused prefill sequence of vLLM PR #316,
// "[EXL3] dispatch prefill-shaped GEMMs to reconstruct+hgemm" (sections
// "Kernel measurements" and "Change"), rebuilt for sm_103a, plus the final
// had_r_128 of that sequence.
//
// A = x' (rotated activations, rows x K fp16, K-major) and B = W^T (the
// reconstructed chunk, nc x K fp16, K-major) are staged by TMA with 128-byte
// swizzle; tcgen05.mma accumulates in fp32 in TMEM, double-buffered (2 x 256
// columns) so the epilogue of tile i overlaps the main loop of tile i+1.
// Persistent grids, one CTA per SM. Two forms:
//   * prefill_pair_kernel (from two 128-row tiles up): clusters of two CTAs
//     share a 256 x 256 tile through tcgen05.mma.cta_group::2 (M=256, N=256),
//     each CTA staging its 128 x' rows and half of the tile's W^T rows in a
//     6-stage ring (32 KB per SM per 64-deep k block);
//   * prefill_gemm_kernel (one 128-row tile, small problems, and the
//     stream-K split of a short last wave): one CTA per 128 x 256 tile,
//     tcgen05.mma M=128, N=256, a 4-stage ring (48 KB per k block).
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM allocator
// and MMA issuer (the even CTA's, for a pair), warps 2..5 = epilogue (warp w
// reads TMEM lanes 32*(w%4) .. 32*(w%4)+31, i.e. one output row per thread).
//
// Roofline: tensor-bound, 2*M*K*nc flops per launch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "exl3_common.cuh"
#include "exl3_internal.h"
#include "exl3_tcgen05.cuh"

namespace exl3 {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int RING_BYTES = STAGES * (A_BYTES + B_BYTES);
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 512;
constexpr int SMEM_BYTES = 1024 + RING_BYTES + 256;

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B fp16
// (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

struct PrefillParams {
  const __half *sv;
  void *y;
  int *status;
  int64_t ldy, n_valid_local;
  int M, nc, K, y_f32, tiles_m, tiles_n;
  int rotate;  // 0: the weight already carries both rotations and sv
  // Schedule: each CTA first takes full_waves whole tiles (tile c + i * G),
  // then its contiguous range of the tail's (tile, k block) units, U units
  // cut evenly over the first Gsk CTAs (stream-K). A tail tile shared by
  // several CTAs is accumulated in fp32 partial slots (128 x 256, in CTA
  // order) that prefill_tail_finalize_kernel reduces.
  int G, full_waves, dp_tiles, Gsk, smax;
  int pair_cols;  // CTA-pair launch: tile columns 0 .. pair_cols-1, every tile row
  int64_t U;
  float *partials;
};

// One unit of a CTA's work: output tile, k-block range, and whether the
// result is a partial (slot `slot` of that tail tile) or the final tile.
struct Work {
  int tile, kb0, kb1, slot;
  bool partial;
};

__device__ __forceinline__ int64_t sk_owner(int64_t z, int64_t Gsk, int64_t U) { return ((z + 1) * Gsk - 1) / U; }

// The CTA's work list, walked identically by the producer, MMA and epilogue.
struct WorkIter {
  int i;
  int64_t u, u_end;
  __device__ __forceinline__ void init(const PrefillParams &p) {
    i = 0;
    const int64_t c = blockIdx.x;
    if (c < p.Gsk) {
      u = c * p.U / p.Gsk;
      u_end = (c + 1) * p.U / p.Gsk;
    } else {
      u = u_end = 0;
    }
  }
  __device__ __forceinline__ bool next(const PrefillParams &p, int kblocks, Work &w) {
    if (i < p.full_waves && (int)blockIdx.x + i * p.G < p.dp_tiles) {
      w.tile = (int)blockIdx.x + i * p.G;
      w.kb0 = 0;
      w.kb1 = kblocks;
      w.partial = false;
      w.slot = 0;
      ++i;
      return true;
    }
    if (u >= u_end) return false;
    const int64_t t = u / kblocks;
    w.kb0 = (int)(u % kblocks);
    const int64_t left = u_end - u;
    w.kb1 = (int)((kblocks - w.kb0) < left ? kblocks : w.kb0 + left);
    const int64_t first = sk_owner(t * kblocks, p.Gsk, p.U), last = sk_owner((t + 1) * kblocks - 1, p.Gsk, p.U);
    w.tile = p.dp_tiles + (int)t;
    w.partial = last > first;
    w.slot = (int)((int64_t)blockIdx.x - first);
    u += w.kb1 - w.kb0;
    return true;
  }
};

// In-register orthonormal had_r_128 of one row block, then * sv, mask, store
// (rotation and sv skipped for a pre-rotated weight).
__device__ __forceinline__ void epilogue_block(float (&v)[128], const PrefillParams &p, int64_t row, int col0) {
  const bool cols_ok = EXL3_SPAN(col0, 128, p.nc);  // sv and y columns of this chunk
  if (p.rotate) {
#pragma unroll
    for (int h = 1; h < 128; h <<= 1) {
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        if (!(i & h)) {
          float a = v[i], b = v[i + h];
          v[i] = a + b;
          v[i + h] = a - b;
        }
      }
    }
    const uint4 *svp = reinterpret_cast<const uint4 *>(p.sv + col0);
#pragma unroll
    for (int a = 0; a < 16; ++a) {
      const uint4 raw = cols_ok ? __ldg(svp + a) : uint4{};
      const __half *h = reinterpret_cast<const __half *>(&raw);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c = 8 * a + e;
        v[c] = (col0 + c < p.n_valid_local) ? v[c] * (__half2float(h[e]) * kInvSqrt128) : -INFINITY;
      }
    }
  }
  if (row >= p.M || !cols_ok) return;
  if (p.y_f32) {
    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.y) + row * p.ldy + col0);
#pragma unroll
    for (int a = 0; a < 32; ++a) dst[a] = make_float4(v[4 * a], v[4 * a + 1], v[4 * a + 2], v[4 * a + 3]);
  } else {
    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__half *>(p.y) + row * p.ldy + col0);
#pragma unroll
    for (int a = 0; a < 16; ++a) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __half2 h2 = __floats2half2_rn(v[8 * a + 2 * e], v[8 * a + 2 * e + 1]);
        w[e] = *reinterpret_cast<uint32_t *>(&h2);
      }
      dst[a] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// SK = false: whole tiles 0 .. dp_tiles-1 in data-parallel waves (tile
// c + i * gridDim.x). SK = true: only the stream-K tail (see PrefillParams).
template <bool SK>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + RING_BYTES);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
  const uint32_t smem_s = smem_u32(smem);
  auto a_s = [&](int s) { return smem_s + (uint32_t)(s * A_BYTES); };
  auto b_s = [&](int s) { return smem_s + (uint32_t)(STAGES * A_BYTES + s * B_BYTES); };
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[STAGES + s]); };
  auto tfull_bar = [&](int a) { return smem_u32(&bars[2 * STAGES + a]); };
  auto tempty_bar = [&](int a) { return smem_u32(&bars[2 * STAGES + 2 + a]); };
  const uint32_t done_bar = smem_u32(&bars[2 * STAGES + 4]);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kblocks = p.K / BK;
  const int ntiles = p.dp_tiles;  // whole tiles of a data-parallel launch
  // ring, barriers and TMEM slot inside the CTA's shared memory (CTA-uniform,
  // before any barrier or TMEM is set up)
  if (!EXL3_SMEM(smem_s, RING_BYTES + (2 * STAGES + 5) * 8 + 4)) return;
  // A tile (tm, tn, kb): TMA boxes at fp16 column 64 kb (128 bytes: the
  // 16-byte rule), A rows 128 tm of the rotated rows, B rows 256 tn of the
  // chunk; both inside the problem.
  auto tile_ok = [&](int tm, int tn, int kb) {
    return EXL3_RANGE(tm, 0, p.tiles_m) && EXL3_RANGE(tn, 0, p.tiles_n) && EXL3_RANGE(kb, 0, kblocks) &&
           EXL3_ALIGNED(kb * BK * 2, 16);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);
    }
    mbar_init(done_bar, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // A split tail's launch may start on SMs this launch leaves (no shared data).
  if constexpr (!SK) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    if constexpr (!SK) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        const int tm = tile % p.tiles_m, tn = tile / p.tiles_m;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), A_BYTES + B_BYTES);
          if (tile_ok(tm, tn, kb)) {
            tma_load_2d(a_s(stage), &tmA, full_bar(stage), kb * BK, tm * BM);
            tma_load_2d(b_s(stage), &tmB, full_bar(stage), kb * BK, tn * BN);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < STAGES; ++s) {
        const int64_t uses = issued / STAGES + (s < issued % STAGES ? 1 : 0);
        if (uses > 0) mbar_wait_short(full_bar(s), (uint32_t)((uses - 1) & 1));
      }
    } else {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      WorkIter it;
      it.init(p);
      Work w;
      while (ok && it.next(p, kblocks, w)) {
        const int tm = w.tile % p.tiles_m, tn = w.tile / p.tiles_m;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), A_BYTES + B_BYTES);
          if (tile_ok(tm, tn, kb)) {
            tma_load_2d(a_s(stage), &tmA, full_bar(stage), kb * BK, tm * BM);
            tma_load_2d(b_s(stage), &tmB, full_bar(stage), kb * BK, tn * BN);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < STAGES; ++s) {
        const int64_t uses = issued / STAGES + (s < issued % STAGES ? 1 : 0);
        if (uses > 0) mbar_wait_short(full_bar(s), (uint32_t)((uses - 1) & 1));
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    if constexpr (!SK) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int local = 0;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(tempty_bar(acc), (use & 1u) ^ 1u, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sw128_desc(a_s(stage));
          const uint64_t bd = sw128_desc(b_s(stage));
  #pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // +32 bytes per 16-element K step inside the 128-byte swizzle atom
            if (EXL3_RANGE(acc, 0, 2))  // 256 columns of the 512 allocated
              tc_mma(d_tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), kIdesc, (kb | kk) != 0);
          }
          tc_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(tfull_bar(acc));
      }
      // All issued MMAs must finish before TMEM is released.
      tc_commit(done_bar);
      mbar_wait_short(done_bar, 0);
    } else {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int local = 0;
      WorkIter it;
      it.init(p);
      Work w;
      for (; ok && it.next(p, kblocks, w); ++local) {
        const int acc = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(tempty_bar(acc), (use & 1u) ^ 1u, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sw128_desc(a_s(stage));
          const uint64_t bd = sw128_desc(b_s(stage));
  #pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // +32 bytes per 16-element K step inside the 128-byte swizzle atom
            if (EXL3_RANGE(acc, 0, 2))
              tc_mma(d_tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), kIdesc, (kb != w.kb0 || kk != 0));
          }
          tc_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(tfull_bar(acc));
      }
      // All issued MMAs must finish before TMEM is released.
      tc_commit(done_bar);
      mbar_wait_short(done_bar, 0);
    }
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    if constexpr (!SK) {
      const int lg = warp & 3;  // TMEM lane group this warp may access
      const int row_in_tile = lg * 32 + lane;
      int local = 0;
      for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++local) {
        const int tm = tile % p.tiles_m, tn = tile / p.tiles_m;
        const int acc = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(tfull_bar(acc), use & 1u, p.status)) break;
        tc_fence_after();
        const int64_t row = (int64_t)tm * BM + row_in_tile;
        const uint32_t tbase = tmem_base + ((uint32_t)(lg * 32) << 16) + (uint32_t)(acc * BN);
        const int c0 = tn * BN;
        const bool second = c0 + 128 < p.nc;
        float v[128];
  #pragma unroll
        for (int j = 0; j < 4; ++j) {
          float t[32];
          tmem_ld32(tbase + 32 * j, t);
  #pragma unroll
          for (int i = 0; i < 32; ++i) v[32 * j + i] = t[i];
        }
        if (!second) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(acc));
        }
        epilogue_block(v, p, row, c0);
        if (second) {
  #pragma unroll
          for (int j = 0; j < 4; ++j) {
            float t[32];
            tmem_ld32(tbase + 128 + 32 * j, t);
  #pragma unroll
            for (int i = 0; i < 32; ++i) v[32 * j + i] = t[i];
          }
            tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(acc));
          epilogue_block(v, p, row, c0 + 128);
        }
      }
    } else {
      const int lg = warp & 3;  // TMEM lane group this warp may access
      const int row_in_tile = lg * 32 + lane;
      int local = 0;
      WorkIter it;
      it.init(p);
      Work w;
      for (; it.next(p, kblocks, w); ++local) {
        const int tm = w.tile % p.tiles_m, tn = w.tile / p.tiles_m;
        const int acc = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(tfull_bar(acc), use & 1u, p.status)) break;
        tc_fence_after();
        const int64_t row = (int64_t)tm * BM + row_in_tile;
        const uint32_t tbase = tmem_base + ((uint32_t)(lg * 32) << 16) + (uint32_t)(acc * BN);
        const int c0 = tn * BN;
        const bool second = c0 + 128 < p.nc;
        if (w.partial) {
          // This CTA's share of a tail tile: fp32 partial sums, row-major 128 x 256.
          float *slot = p.partials + ((int64_t)(w.tile - p.dp_tiles) * p.smax + w.slot) * (BM * BN) +
                        (int64_t)row_in_tile * BN;
          // slot w.slot of the tail tile's smax (the host sized the buffer for
          // every tail tile's smax slots)
          const bool slot_ok = EXL3_RANGE(w.tile - p.dp_tiles, 0, (int64_t)p.tiles_m * p.tiles_n - p.dp_tiles) &&
                               EXL3_RANGE(w.slot, 0, p.smax);
          const int ncols = second ? BN : 128;
          for (int j = 0; j < ncols; j += 32) {
            float t[32];
            tmem_ld32(tbase + j, t);
            if (row < p.M && slot_ok) {
              float4 *dst = reinterpret_cast<float4 *>(slot + j);
  #pragma unroll
              for (int a = 0; a < 8; ++a) dst[a] = make_float4(t[4 * a], t[4 * a + 1], t[4 * a + 2], t[4 * a + 3]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(acc));
          continue;
        }
        float v[128];
  #pragma unroll
        for (int j = 0; j < 4; ++j) {
          float t[32];
          tmem_ld32(tbase + 32 * j, t);
  #pragma unroll
          for (int i = 0; i < 32; ++i) v[32 * j + i] = t[i];
        }
        if (!second) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(acc));
        }
        epilogue_block(v, p, row, c0);
        if (second) {
  #pragma unroll
          for (int j = 0; j < 4; ++j) {
            float t[32];
            tmem_ld32(tbase + 128 + 32 * j, t);
  #pragma unroll
            for (int i = 0; i < 32; ++i) v[32 * j + i] = t[i];
          }
            tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(acc));
          epilogue_block(v, p, row, c0 + 128);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
  // Launched as a programmatic dependent of the whole-tile launch: finish
  // only after it, so that work queued behind this launch sees both done.
  if constexpr (SK) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// CTA-pair form of the whole-tile launch. A cluster of two CTAs (two SMs)
// computes one 256 x 256 output tile with tcgen05.mma.cta_group::2 (M = 256,
// N = 256, K = 16): the even CTA (rank 0) stages x' rows 0-127 of the tile and
// W^T rows (output columns) 0-127, the odd CTA rows 128-255 of each, and the
// even CTA's thread issues the MMA for both. Each SM thus stages 32 KB per
// 64-deep k block (16 KB of A, 16 KB of B) instead of the 48 KB of a
// one-SM 128 x 256 tile, for the same tensor work per SM. Each CTA's TMEM
// holds its 128 rows x 256 columns (double-buffered, 512 columns), and its
// four epilogue warps run the same fused had_r_128 / sv / mask epilogue.
//
// Barriers (same offsets in both CTAs):
//   full[s]   rank 0's counts both CTAs' TMA bytes of stage s (the odd CTA's
//             loads complete on it through its cluster address);
//   empty[s]  each CTA's, completed by the pair MMA's commit (multicast);
//   tfull[a]  each CTA's, accumulator a ready (commit, multicast);
//   tempty[a] rank 0's, 8 arrivals: the four epilogue warps of both CTAs;
//   done      rank 0's, every pair MMA finished.
constexpr int P_STAGES = 6;
constexpr int PA_BYTES = 128 * BK * 2;  // 16 KB: this CTA's 128 rows of x'
constexpr int PB_BYTES = 128 * BK * 2;  // 16 KB: this CTA's 128 rows of W^T
constexpr int P_RING_BYTES = P_STAGES * (PA_BYTES + PB_BYTES);
constexpr int P_NBARS = 2 * P_STAGES + 5;
constexpr int P_SMEM_BYTES = 1024 + P_RING_BYTES + 256;
static_assert(P_NBARS * 8 + 4 <= 256, "pair barrier area");
constexpr uint32_t kIdescPair = f16_idesc(256, 256);

// Pair tile t: rows 256 (t % tiles_mp) .., columns 256 (t / tiles_mp) ..,
// for the first pair_cols tile columns.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + P_RING_BYTES);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + P_NBARS);
  const uint32_t smem_s = smem_u32(smem);
  auto a_s = [&](int s) { return smem_s + (uint32_t)(s * PA_BYTES); };
  auto b_s = [&](int s) { return smem_s + (uint32_t)(P_STAGES * PA_BYTES + s * PB_BYTES); };
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[P_STAGES + s]); };
  auto tfull_bar = [&](int a) { return smem_u32(&bars[2 * P_STAGES + a]); };
  auto tempty_bar = [&](int a) { return smem_u32(&bars[2 * P_STAGES + 2 + a]); };
  const uint32_t done_bar = smem_u32(&bars[2 * P_STAGES + 4]);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
  const int kblocks = p.K / BK;
  const int tiles_mp = (p.tiles_m + 1) >> 1;
  const int ptiles = tiles_mp * p.pair_cols;
  // Ring, barriers and TMEM slot inside the CTA's shared memory. The same
  // in both CTAs (same kernel, same size), so both leave here or neither.
  if (!EXL3_SMEM(smem_s, P_RING_BYTES + P_NBARS * 8 + 4)) return;
  // This CTA's boxes of pair tile (tmp, tn) at k block kb: fp16 column 64 kb
  // (128 bytes: the 16-byte rule); 128 x' rows inside the rotated rows, W^T
  // rows 256 tn + 128 rank inside the chunk.
  auto box_ok = [&](int tmp, int tn, int kb) {
    return EXL3_RANGE(tmp, 0, tiles_mp) && EXL3_RANGE(tn, 0, p.pair_cols) && EXL3_RANGE(kb, 0, kblocks) &&
           EXL3_ALIGNED(kb * BK * 2, 16);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 8);
    }
    mbar_init(done_bar, 1);
    fence_barrier_init();
  }
  if (warp == 1) {  // one warp of each CTA of the pair allocates together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();  // both CTAs' barriers initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int t = pair; t < ptiles && ok; t += npairs) {
      const int tmp = t % tiles_mp, tn = t / tiles_mp;
      // With an odd number of 128-row tiles the last pair's odd CTA re-reads
      // the last real row tile (its rows are past M and never stored).
      const int arow = min(tmp * 256 + (int)rank * 128, (p.tiles_m - 1) * 128);
      const int brow = tn * 256 + (int)rank * 128;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_cluster(empty_bar(stage), phase ^ 1u, p.status, kWaitLimitNs)) {
          ok = false;
          break;
        }
        if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * (PA_BYTES + PB_BYTES));
        if (box_ok(tmp, tn, kb)) {
          const uint32_t fb = map_to_rank(full_bar(stage), 0);
          tma_load_2d_pair(a_s(stage), &tmA, fb, kb * BK, arow);
          tma_load_2d_pair(b_s(stage), &tmB, fb, kb * BK, brow);
        }
        ++issued;
        if (++stage == P_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // Rank 0's full barriers count both CTAs' bytes: once each stage's last
    // use has completed there, no copy of either CTA is in flight (the final
    // cluster barrier keeps the odd CTA until then).
    if (rank == 0)
      for (int s = 0; s < P_STAGES; ++s) {
        const int64_t uses = issued / P_STAGES + (s < issued % P_STAGES ? 1 : 0);
        if (uses > 0) mbar_wait_cluster(full_bar(s), (uint32_t)((uses - 1) & 1), nullptr, 200000000ull);
      }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------- MMA issuer (even CTA) ----------------
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int local = 0;
    for (int t = pair; t < ptiles && ok; t += npairs, ++local) {
      const int acc = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      if (!mbar_wait_cluster(tempty_bar(acc), (use & 1u) ^ 1u, p.status, kWaitLimitNs)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_cluster(full_bar(stage), phase, p.status, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = sw128_desc(a_s(stage));
        const uint64_t bd = sw128_desc(b_s(stage));
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          // +32 bytes per 16-element K step inside the 128-byte swizzle atom
          if (EXL3_RANGE(acc, 0, 2))  // 256 columns of the 512 allocated
            tc_mma_pair(d_tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), kIdescPair, (kb | kk) != 0);
        }
        tc_commit_pair(empty_bar(stage), 3);
        if (++stage == P_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit_pair(tfull_bar(acc), 3);
    }
    // All issued MMAs (which write both CTAs' TMEM) finish before the final
    // cluster barrier, after which both CTAs release their TMEM.
    tc_commit_pair(done_bar, 1);
    mbar_wait_cluster(done_bar, 0, nullptr, 200000000ull);
  } else if (warp >= 2) {
    // ---------------- epilogue (both CTAs) ----------------
    const int lg = warp & 3;  // TMEM lane group this warp may access
    const int row_in_tile = (int)rank * 128 + lg * 32 + lane;
    int local = 0;
    for (int t = pair; t < ptiles; t += npairs, ++local) {
      const int tmp = t % tiles_mp, tn = t / tiles_mp;
      const int acc = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      if (!mbar_wait_cluster(tfull_bar(acc), use & 1u, p.status, kWaitLimitNs)) break;
      tc_fence_after();
      const int64_t row = (int64_t)tmp * 256 + row_in_tile;
      const uint32_t tbase = tmem_base + ((uint32_t)(lg * 32) << 16) + (uint32_t)(acc * BN);
      const uint32_t te = map_to_rank(tempty_bar(acc), 0);
      const int c0 = tn * BN;
      const bool second = c0 + 128 < p.nc;
      float v[128];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float tt[32];
        tmem_ld32(tbase + 32 * j, tt);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[32 * j + i] = tt[i];
      }
      if (!second) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(te);
      }
      epilogue_block(v, p, row, c0);
      if (second) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float tt[32];
          tmem_ld32(tbase + 128 + 32 * j, tt);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[32 * j + i] = tt[i];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(te);
        epilogue_block(v, p, row, c0 + 128);
      }
    }
  }

  tc_fence_before();
  __syncwarp();
  cluster_sync_all();  // no remote arrival or copy of either CTA is pending
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}

// Reduces the partial slots of every tail tile shared by several CTAs, in
// CTA order, then applies the epilogue (had_r_128 per 128-column block, sv,
// mask) and stores y. One warp per (tail tile, row); lane l holds the eight
// columns 128*(l/16) + 8*(l%16) .. +7 of the tile's 256.
__global__ void __launch_bounds__(256) prefill_tail_finalize_kernel(const PrefillParams p, int kblocks) {
  const int lane = threadIdx.x & 31;
  const int64_t wi = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t t = wi >> 7;
  const int r = (int)(wi & 127);
  const int64_t tail = (int64_t)p.tiles_m * p.tiles_n - p.dp_tiles;
  if (t >= tail) return;
  const int64_t first = sk_owner(t * kblocks, p.Gsk, p.U), last = sk_owner((t + 1) * kblocks - 1, p.Gsk, p.U);
  if (last == first) return;  // finished by its single CTA
  const int tile = p.dp_tiles + (int)t;
  const int tm = tile % p.tiles_m, tn = tile / p.tiles_m;
  const int64_t row = (int64_t)tm * BM + r;
  if (row >= p.M) return;
  const int c0 = tn * BN, half = lane >> 4, l16 = lane & 15;
  const bool second = c0 + 128 < p.nc;
  const float *src = p.partials + t * p.smax * (int64_t)(BM * BN) + (int64_t)r * BN + 128 * half + 8 * l16;
  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const int cnt = (int)(last - first + 1);
  const bool slots_ok = EXL3_RANGE(cnt, 1, p.smax + 1);  // cnt of the tile's smax slots
  for (int s = 0; s < (slots_ok ? cnt : 0); ++s) {  // slot (CTA) order
    if (half == 0 || second) {
      const float4 a = __ldcg(reinterpret_cast<const float4 *>(src + (int64_t)s * (BM * BN)));
      const float4 b = __ldcg(reinterpret_cast<const float4 *>(src + (int64_t)s * (BM * BN)) + 1);
      v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w;
      v[4] += b.x; v[5] += b.y; v[6] += b.z; v[7] += b.w;
    }
  }
  const int col0 = c0 + 128 * half + 8 * l16;
  if (p.rotate) {
#pragma unroll
    for (int h = 1; h < 8; h <<= 1)
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (!(i & h)) {
          const float a = v[i], b = v[i + h];
          v[i] = a + b;
          v[i + h] = a - b;
        }
#pragma unroll
    for (int s = 1; s < 16; s <<= 1) {
      const float sgn = (l16 & s) ? -1.f : 1.f;  // o + v or o - v, one rounding either way
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float o = __shfl_xor_sync(0xffffffffu, v[i], s);
        v[i] = fmaf(v[i], sgn, o);
      }
    }
    if (half == 1 && !second) return;
    if (!EXL3_SPAN(col0, 8, p.nc)) return;
    const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(p.sv + col0));
    const __half *h = reinterpret_cast<const __half *>(&raw);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      v[i] = (col0 + i < p.n_valid_local) ? v[i] * (__half2float(h[i]) * kInvSqrt128) : -INFINITY;
  } else if (half == 1 && !second) {
    return;
  }
  if (!EXL3_SPAN(col0, 8, p.nc)) return;
  if (p.y_f32) {
    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.y) + row * p.ldy + col0);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    uint32_t wv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __half2 h2 = __floats2half2_rn(v[2 * e], v[2 * e + 1]);
      wv[e] = *reinterpret_cast<uint32_t *>(&h2);
    }
    *reinterpret_cast<uint4 *>(static_cast<__half *>(p.y) + row * p.ldy + col0) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool make_map(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

bool encode_tensor_map_2d(CUtensorMap *m, CUtensorMapDataType type, const void *ptr, uint64_t dim0, uint64_t dim1,
                          uint64_t stride_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle) {
  if (!g_encode) return false;
  cuuint64_t dims[2] = {(cuuint64_t)dim0, (cuuint64_t)dim1};
  cuuint64_t strides[1] = {(cuuint64_t)stride_bytes};
  cuuint32_t box[2] = {box0, box1};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, type, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t init_prefill_kernels(int *status) {
  const cudaError_t eb = EXL3_BIND_BOUNDS_WORD(status);
  if (eb != cudaSuccess) return eb;
  if (!g_encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  cudaError_t e = cudaFuncSetAttribute(prefill_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(prefill_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(prefill_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes a;
  return cudaFuncGetAttributes(&a, prefill_tail_finalize_kernel);
}

size_t prefill_tail_partials_bytes(int num_sms) { return (size_t)3 * num_sms * BM * BN * 4; }

cudaError_t launch_prefill_gemm(const PrefillLaunch &L, cudaStream_t st) {
  if (L.M == 0 || L.nc == 0) return cudaSuccess;
  alignas(64) CUtensorMap ma, mb;
  if (!make_map(&ma, L.xr, L.xr_rows, L.K, BM)) return cudaErrorInvalidValue;
  if (!make_map(&mb, L.wt, L.chunk_rows, L.K, BN)) return cudaErrorInvalidValue;
  PrefillParams p;
  p.sv = static_cast<const __half *>(L.sv);
  p.y = L.y;
  p.status = L.status;
  p.ldy = L.ldy;
  p.n_valid_local = L.n_valid_local;
  p.rotate = L.rotate;
  p.M = (int)L.M;
  p.nc = (int)L.nc;
  p.K = (int)L.K;
  p.y_f32 = L.y_f32;
  p.tiles_m = (int)ceil_div(L.M, BM);
  p.tiles_n = (int)ceil_div(L.nc, BN);
  const int ntiles = p.tiles_m * p.tiles_n;
  const int kblocks = p.K / BK;
  // Data-parallel waves of whole tiles, then the remaining tiles' k blocks
  // spread evenly over the CTAs (at least 4 k blocks each); see PrefillParams.
  p.G = L.num_sms;
  p.full_waves = ntiles / p.G;
  p.dp_tiles = p.full_waves * p.G;
  const int64_t tail = ntiles - p.dp_tiles;
  p.U = tail * kblocks;
  p.Gsk = 0;
  p.smax = 1;
  p.partials = L.partials;
  // Splitting the tail pays off when it fills at most half a wave and either
  // the whole problem is small (the split multiplies the CTAs at work) or K
  // is long (each saved round is expensive). Otherwise the split tiles'
  // fp32 partials and the lost lockstep of CTAs that share weight columns
  // (re-read from HBM when the chunk exceeds L2) cost more than the idle
  // SMs of the last wave (measured on the 4-bit MLP geometries).
  const bool split_tail = p.U > 0 && 2 * tail <= p.G && (2 * ntiles <= p.G || kblocks >= 128);
  p.pair_cols = 0;
  const int G2 = L.num_sms / 2;
  if (p.tiles_m >= 2 && G2 >= 1) {
    // CTA pairs over 256 x 256 tiles: the same rule in pair units. A split
    // tail keeps whole tile columns in the pair launch (those the full pair
    // waves cover) and spreads the remaining columns' 128-row tiles over
    // all CTAs as below; a problem whose full pair waves cover no whole
    // column keeps the one-SM schedule.
    const int tiles_mp = (p.tiles_m + 1) / 2;
    const int64_t P = (int64_t)tiles_mp * p.tiles_n, tailp = P % G2;
    const bool split = tailp > 0 && 2 * tailp <= G2 && (2 * P <= G2 || kblocks >= 128);
    p.pair_cols = split ? (int)((P / G2) * G2 / tiles_mp) : p.tiles_n;
  }
  if (p.pair_cols > 0) {
    p.full_waves = 0;
    p.dp_tiles = p.pair_cols * p.tiles_m;
    p.U = (int64_t)(ntiles - p.dp_tiles) * kblocks;
  } else if (p.U > 0 && !split_tail) {
    p.full_waves += 1;
    p.dp_tiles = ntiles;
    p.U = 0;
  }
  const int64_t tail_tiles = ntiles - p.dp_tiles;
  if (p.U > 0) {
    int64_t gsk = p.U / 4;
    if (gsk < 1) gsk = 1;
    if (gsk > p.G) gsk = p.G;
    int64_t smax = 1;
    for (int64_t t = 0; t < tail_tiles; ++t) {
      const int64_t c = (((t + 1) * kblocks) * gsk - 1) / p.U - (((t * kblocks + 1) * gsk - 1) / p.U) + 1;
      if (c > smax) smax = c;
    }
    if (L.partials != nullptr && (size_t)(tail_tiles * smax) * BM * BN * 4 <= L.partials_bytes) {
      p.Gsk = (int)gsk;
      p.smax = (int)smax;
    } else if (p.pair_cols > 0) {  // no room for partial slots: every column in pair tiles
      p.pair_cols = p.tiles_n;
      p.dp_tiles = ntiles;
      p.U = 0;
    } else {  // no room for partial slots: the tail runs as one more wave of whole tiles
      p.full_waves += 1;
      p.dp_tiles = ntiles;
      p.U = 0;
    }
  }
  // Whole tiles first (data-parallel waves), then, when the tail is split, a
  // second launch that spreads the tail's k blocks over Gsk CTAs.
  if (p.pair_cols > 0) {
    alignas(64) CUtensorMap mbp;  // W^T boxes of 128 rows: each CTA stages half of a tile's columns
    if (!make_map(&mbp, L.wt, L.chunk_rows, L.K, 128)) return cudaErrorInvalidValue;
    const int64_t ptiles = (int64_t)((p.tiles_m + 1) / 2) * p.pair_cols;
    const int pairs = (int)(ptiles < G2 ? ptiles : G2);
    prefill_pair_kernel<<<2 * pairs, NUM_THREADS, P_SMEM_BYTES, st>>>(ma, mbp, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  } else if (p.dp_tiles > 0) {
    prefill_gemm_kernel<false><<<p.dp_tiles < p.G ? p.dp_tiles : p.G, NUM_THREADS, SMEM_BYTES, st>>>(ma, mb, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (p.Gsk == 0) return cudaSuccess;
  PrefillParams q = p;
  q.full_waves = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.Gsk);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.dp_tiles > 0 ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_gemm_kernel<true>, ma, mb, q);
  if (e != cudaSuccess) return e;
  const int64_t warps = tail_tiles * BM;
  prefill_tail_finalize_kernel<<<(unsigned)ceil_div(warps, 8), 256, 0, st>>>(q, kblocks);
  return cudaGetLastError();
}

#if EXL3_DEBUG_BOUNDS
cudaError_t bounds_probe_prefill(cudaStream_t st) { return launch_bounds_probe(st); }
#endif

}  // namespace exl3
