// Decode-shaped trellis linear: the fused decode-inside-GEMM path for up to
// 16 activation rows per launch.
//
// The decode-shaped kernel of vLLM PR #316, "[EXL3] dispatch prefill-shaped
// GEMMs to reconstruct+hgemm" (sections "Problem" and "Change": below the M
// threshold the op keeps a kernel that decodes the trellis inside the GEMM),
// rebuilt for sm_103a. Each weight is decoded exactly once per launch.
//
// Up to three kernels per launch:
//   1. rotate_frag_kernel: x' = RNE_fp16(had_r_128(x * su)) for the (<= 16)
//      rows, written in mma fragment order (per 16-row k slab, lane (g, q)
//      finds x'[g][4q..4q+3] and x'[g+8][4q..4q+3] as 8 or 16 contiguous
//      bytes).
//   2. decode_gemm_kernel: stream-K over all (n-block, k-slab) work. A slab
//      is 16 k-rows x 128 output columns = 8 horizontally adjacent trellis
//      tiles, 256*BITS contiguous bytes. The P = SMs x warps-per-CTA warps
//      each own a contiguous range of slabs in n-block-major order, so every
//      warp on every SM has the same amount of work. Each warp feeds itself:
//      lane 0 streams its slabs (weights plus the slab's x' fragments) into a
//      private ring in shared memory with cp.async.bulk, one mbarrier per
//      stage.
//      Lane (g, q) decodes tile g, rows 4q..4q+3 straight into m16n8k16 A
//      fragments (A = W^T: mma row r <-> output column 16*(r%8) + j +
//      8*(r/8) for mma j), B = x'^T (8 tokens per mma). Each A register
//      holds one weight in both halves and the matching B register {x', 0}:
//      mma k index 2q <-> tile row 4q and 2q+8 <-> row 4q+1 in the first
//      mma of a column group, rows 4q+2 and 4q+3 in the second (odd k
//      indices multiply zeros). This spends twice the mmas (tensor pipe
//      ~20 % busy) to save the two instructions per weight pair that would
//      pack two decoded weights into one register. After 16 mmas per slab
//      and token group, lane (g, q) holds output columns 16g .. 16g+15 of
//      tokens 2q, 2q+1 (+8).
//      When a warp finishes its part of an n-block it either owns the whole
//      n-block (then it applies had_r_128 over the 128 columns, sv and the
//      -inf mask and writes y), or it stores an fp32 partial in its slot.
//   3. decode_finalize_kernel (only when some n-block is shared): one warp
//      per (n-block, row) sums the slots in slot order (deterministic),
//      applies had_r_128, sv and the mask and writes y.
//
// Roofline: HBM-bound on the trellis bytes (K*N*BITS/8 per launch) unless
// the per-weight integer decode (a half-rate ALU pipe) binds first.
#include <cuda.h>
#include <math.h>

#include "exl3_common.cuh"
#include "exl3_internal.h"

// Tuning knobs (compile-time): warps per CTA for <= 8 rows.
#ifndef EXL3_DECODE_WARPS_M8
#define EXL3_DECODE_WARPS_M8 12
#endif
// ... and for 9..16 rows.
#ifndef EXL3_DECODE_WARPS_M16
#define EXL3_DECODE_WARPS_M16 12
#endif
// Packing of two decoded fp16 weights into one mma register, per variant
// (0: byte permute on the integer pipe; 1: multiply-add on the fp16 pipe).
#ifndef EXL3_DECODE_PACK_FMA_M8
#define EXL3_DECODE_PACK_FMA_M8 1
#endif
#ifndef EXL3_DECODE_PACK_FMA_M16
#define EXL3_DECODE_PACK_FMA_M16 1
#endif
// A operand form, per variant (1: each weight duplicated in both halves of
// its register against zero-interleaved x', two mmas per slab and column
// group; 0: two weights packed per register, one mma).
#ifndef EXL3_DECODE_DUP_M8
#define EXL3_DECODE_DUP_M8 1
#endif
#ifndef EXL3_DECODE_DUP_M16
#define EXL3_DECODE_DUP_M16 0
#endif
// Where the end of this warp's part of an n-block is tested, per variant
// (1: once per chunk, after its last slab; 0: after every slab).
#ifndef EXL3_DECODE_BLOCK_PER_CHUNK_M8
#define EXL3_DECODE_BLOCK_PER_CHUNK_M8 1
#endif
#ifndef EXL3_DECODE_BLOCK_PER_CHUNK_M16
#define EXL3_DECODE_BLOCK_PER_CHUNK_M16 0
#endif
// Nibble-shifted window copy made on the FMA pipe for BITS = 4 (see
// Windows; 1: on). Also taking the offset-0 and offset-4 states from the
// high word of a multiply (IMAD.HI) measured 18 % slower at 1 row.
#ifndef EXL3_DECODE_FMA_EXTRACT_M8
#define EXL3_DECODE_FMA_EXTRACT_M8 1
#endif
#ifndef EXL3_DECODE_FMA_EXTRACT_M16
#define EXL3_DECODE_FMA_EXTRACT_M16 0
#endif
// Slabs per inner-loop iteration, per variant (for <= 8 rows two measured
// 1-1.5 % faster than one and 3 % faster than four; for 9..16 rows two
// spills and is 2 % slower than one).
#ifndef EXL3_DECODE_UNROLL_M8
#define EXL3_DECODE_UNROLL_M8 2
#endif
#ifndef EXL3_DECODE_UNROLL_M16
#define EXL3_DECODE_UNROLL_M16 1
#endif
#ifndef EXL3_DECODE_STAGES_M8
#define EXL3_DECODE_STAGES_M8 2
#endif
// Proxy fence after reading a ring stage (1) or none (0): the stage's words
// are consumed by register-dependent decode work before the warp reaches the
// reissue point, so the reuse is ordered without it.
#ifndef EXL3_DECODE_PROXY_FENCE
#define EXL3_DECODE_PROXY_FENCE 0
#endif
// Programmatic dependent launch between the rotation, decode and finalize
// kernels (1: on).
#ifndef EXL3_DECODE_PDL
#define EXL3_DECODE_PDL 1
#endif
// Most rows for which the slot reduction runs one warp per CTA.
#ifndef EXL3_DECODE_FIN_1W_ROWS
#define EXL3_DECODE_FIN_1W_ROWS 2
#endif
// The input rotation, too, as a programmatic dependent of whatever precedes
// it in the stream (1: on).
#ifndef EXL3_DECODE_ROTATE_PDL
#define EXL3_DECODE_ROTATE_PDL 1
#endif

namespace exl3 {

namespace {

#ifndef EXL3_DECODE_CHUNK
#define EXL3_DECODE_CHUNK 4  // slabs per copy for BITS <= 4 (half that above)
#endif

template <int BITS, int MT>
struct DecodeCfg {
  static constexpr int kWarps = MT == 1 ? EXL3_DECODE_WARPS_M8 : EXL3_DECODE_WARPS_M16;  // warps per CTA
  static constexpr int kSeg = 256 * BITS;                    // trellis bytes per slab
  static constexpr int kChunk = BITS <= 4 ? EXL3_DECODE_CHUNK : (EXL3_DECODE_CHUNK + 1) / 2;  // slabs per copy
  static constexpr int kStages = MT == 1 ? EXL3_DECODE_STAGES_M8 : 3;  // ring stages (chunks) per warp
  static constexpr int kXB = 32 * 4 * MT * 2;                // x' fragment bytes per slab
  static constexpr int kStage = kChunk * kSeg;
  static constexpr int kWarpRing = kStages * kStage;
  static constexpr int kSmem = kWarps * kWarpRing + kWarps * kStages * 8;
};

struct DecodeParams {
  const uint8_t *trellis;
  const uint8_t *xf;  // rotated x in fragment order, K/16 slabs of 256*MT bytes
  const __half *sv;
  void *y;
  float *partials;
  int *status;
  int64_t tiles_n, n_gemm, n_valid, TS, P;
  int rows, y_f32, KT, smax;
  uint32_t m16;  // 16, opaque to the compiler (see Windows)
};

__device__ __forceinline__ void tma_load_2d_u64(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Output rotation, sv, mask and store for the lane's values
// v[mt][t][c] = token 8*mt + 2q + t, column nb*128 + 16g + c.
template <int MT>
__device__ __forceinline__ void finish_block(float (&v)[MT][2][16], const DecodeParams &p, int64_t nb, int lane) {
  const int g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int t = 0; t < 2; ++t) {
#pragma unroll
      for (int h = 1; h < 16; h <<= 1)
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (!(i & h)) {
            const float a = v[mt][t][i], b = v[mt][t][i + h];
            v[mt][t][i] = a + b;
            v[mt][t][i + h] = a - b;
          }
#pragma unroll
      for (int s = 1; s < 8; s <<= 1)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float o = __shfl_xor_sync(0xffffffffu, v[mt][t][i], s * 4);
          v[mt][t][i] = (g & s) ? (o - v[mt][t][i]) : (v[mt][t][i] + o);
        }
    }
  const int64_t col0 = nb * 128 + 16 * g;
  float scale[16];
  {
    const uint4 *svp = reinterpret_cast<const uint4 *>(p.sv + col0);
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const uint4 raw = __ldg(svp + a);
      const __half *h = reinterpret_cast<const __half *>(&raw);
#pragma unroll
      for (int e = 0; e < 8; ++e) scale[8 * a + e] = __half2float(h[e]) * kInvSqrt128;
    }
  }
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int m = 8 * mt + 2 * q + t;
      float o[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) o[c] = (col0 + c < p.n_valid) ? v[mt][t][c] * scale[c] : -INFINITY;
      if (m < p.rows) {
        if (p.y_f32) {
          float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.y) + (int64_t)m * p.n_gemm + col0);
#pragma unroll
          for (int a = 0; a < 4; ++a) dst[a] = make_float4(o[4 * a], o[4 * a + 1], o[4 * a + 2], o[4 * a + 3]);
        } else {
          uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__half *>(p.y) + (int64_t)m * p.n_gemm + col0);
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __half2 h2 = __floats2half2_rn(o[8 * a + 2 * e], o[8 * a + 2 * e + 1]);
              w[e] = *reinterpret_cast<uint32_t *>(&h2);
            }
            dst[a] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
}

__device__ __forceinline__ int64_t slab_owner(int64_t z, int64_t P, int64_t TS) { return ((z + 1) * P - 1) / TS; }

// The lane's four sv values of n-block nb (columns nb*128 + 4*lane ..).
// sv is a weight, not an output of the GEMM: a kernel that waits for the
// GEMM loads it before the wait, off the critical path (after a long decode
// it has usually left L2).
__device__ __forceinline__ uint2 load_sv4(const __half *__restrict__ sv, int64_t nb, int lane) {
  return __ldg(reinterpret_cast<const uint2 *>(sv + nb * 128 + 4 * lane));
}

// Output rotation (had_r_128 over the 128 columns spread as 4 per lane), sv
// (the lane's four values from load_sv4), mask and store of one row of
// n-block nb.
__device__ __forceinline__ void finalize_row(float (&v)[4], uint2 sraw, void *y, int y_f32, int64_t n_gemm,
                                             int64_t n_valid, int64_t nb, int m, int lane) {
  {
    float a = v[0], b = v[1];
    v[0] = a + b;
    v[1] = a - b;
    a = v[2];
    b = v[3];
    v[2] = a + b;
    v[3] = a - b;
    a = v[0];
    b = v[2];
    v[0] = a + b;
    v[2] = a - b;
    a = v[1];
    b = v[3];
    v[1] = a + b;
    v[3] = a - b;
  }
#pragma unroll
  for (int s = 1; s < 32; s <<= 1)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], s);
      v[i] = (lane & s) ? (o - v[i]) : (v[i] + o);
    }
  const int64_t col = nb * 128 + 4 * lane;
  const __half *sh = reinterpret_cast<const __half *>(&sraw);
  float o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = (col + i < n_valid) ? v[i] * (__half2float(sh[i]) * kInvSqrt128) : -INFINITY;
  if (y_f32) {
    *reinterpret_cast<float4 *>(static_cast<float *>(y) + (int64_t)m * n_gemm + col) = make_float4(o[0], o[1], o[2], o[3]);
  } else {
    __half2 h0 = __floats2half2_rn(o[0], o[1]), h1 = __floats2half2_rn(o[2], o[3]);
    *reinterpret_cast<uint2 *>(static_cast<__half *>(y) + (int64_t)m * n_gemm + col) =
        make_uint2(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1));
  }
}

// Sum of the `cnt` partial slots at base, base + slot_elems, ... in slot
// order (deterministic), four columns per lane; 16 loads per lane in flight.
// The slots were written by other SMs: loads bypass L1.
__device__ __forceinline__ void sum_slots(const float *base, int cnt, int64_t slot_elems, float (&v)[4]) {
  v[0] = v[1] = v[2] = v[3] = 0.f;
  for (int s0 = 0; s0 < cnt; s0 += 16) {
    float4 f[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)  // all loads of the chunk in flight at once
      f[i] = (s0 + i < cnt) ? __ldcg(reinterpret_cast<const float4 *>(base + (s0 + i) * slot_elems))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 16; ++i) {  // summed in slot order
      v[0] += f[i].x;
      v[1] += f[i].y;
      v[2] += f[i].z;
      v[3] += f[i].w;
    }
  }
}

// Waits until the preceding kernel in the stream has completed and its
// memory is visible (no-op when launched without programmatic dependency).
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream (if launched with programmatic
// dependency) start its prologue now.
__device__ __forceinline__ void allow_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <int BITS, int MT>
__global__ void __launch_bounds__(DecodeCfg<BITS, MT>::kWarps * 32, 1)
    decode_gemm_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeParams p) {
  using Cfg = DecodeCfg<BITS, MT>;
  constexpr int R = Cfg::kStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int64_t pw = (int64_t)blockIdx.x * Cfg::kWarps + warp;
  if (pw >= p.P) return;
  const int64_t z0 = pw * p.TS / p.P, z1 = (pw + 1) * p.TS / p.P;

  uint8_t *ring = smem + warp * Cfg::kWarpRing;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kWarps * Cfg::kWarpRing) + warp * R;
  const uint32_t ring_s = smem_u32(ring);
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < R; ++s) mbar_init(smem_u32(&bars[s]), 1);
    fence_barrier_init();
  }
  __syncwarp();

  // Issue cursor (lane 0 only): the next chunk to stream in. A chunk is up
  // to kChunk consecutive k slabs of one n-block, fetched by one 2-D TMA copy
  // (box: one slab row of 8 tiles x kChunk tile rows; rows past K read as 0).
  constexpr int CHK = Cfg::kChunk;
  const int KT = p.KT;
  int i_nb = (int)(z0 / KT), i_tk = (int)(z0 % KT), i_st = 0;
  int64_t zi = z0;
  int64_t issued = 0;
  auto issue_next = [&]() {
    const int64_t left = z1 - zi;
    const int len = (int)((KT - i_tk) < CHK ? ((int64_t)(KT - i_tk) < left ? (KT - i_tk) : left)
                                            : (CHK < left ? CHK : left));
    const uint32_t bar = smem_u32(&bars[i_st]);
    mbar_arrive_expect_tx(bar, Cfg::kStage);
    tma_load_2d_u64(ring_s + i_st * Cfg::kStage, &tmap, bar, i_nb * (32 * BITS), i_tk);
    zi += len;
    i_tk += len;
    if (i_tk == KT) {
      i_tk = 0;
      ++i_nb;
    }
    if (++i_st == R) i_st = 0;
    ++issued;
  };
  if (lane == 0) {
    for (int c = 0; c < R - 1 && zi < z1; ++c) issue_next();
  }
  allow_next_grid();
  wait_prior_grid();  // x' comes from the rotation kernel

  float acc[MT][8][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[mt][j][0] = acc[mt][j][1] = acc[mt][j][2] = acc[mt][j][3] = 0.f;

  // Consumer cursor.
  int nb = (int)(z0 / KT), tk = (int)(z0 % KT), s = 0;
  uint32_t phase = 0;
  int64_t consumed = 0;
  // x' fragments of the current slab, loaded one slab ahead.
  uint32_t bx[2 * MT], bx_next[2 * MT];
  auto load_x = [&](int k_slab, uint32_t (&dst)[2 * MT]) {
    if constexpr (MT == 1) {
      const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p.xf + (int64_t)k_slab * Cfg::kXB) + lane);
      dst[0] = v.x;
      dst[1] = v.y;
    } else {
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.xf + (int64_t)k_slab * Cfg::kXB) + lane);
      dst[0] = v.x;
      dst[1] = v.y;
      dst[2] = v.z;
      dst[3] = v.w;
    }
  };
  // This warp's part of n-block cnb is complete: finish it or store the
  // partial, then clear the accumulators.
  auto block_end = [&](const int64_t cnb) {
    float v[MT][2][16];
    const bool whole = (z0 <= cnb * p.KT) && (z1 >= (cnb + 1) * p.KT);
    if (whole) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int tt = 0; tt < 2; ++tt)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            v[mt][tt][c] = acc[mt][c][tt];
            v[mt][tt][c + 8] = acc[mt][c][2 + tt];
          }
      finish_block<MT>(v, p, cnb, lane);
    } else {
      // Store this warp's contribution in its slot; decode_finalize_kernel
      // sums the n-block's slots in slot order.
      const int64_t pf = slab_owner(cnb * p.KT, p.P, p.TS);
      const int64_t slot_elems = (int64_t)8 * MT * 128;
      float *part = p.partials + (cnb * p.smax + (pw - pf)) * slot_elems;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
          const int m = 8 * mt + 2 * q + tt;
          if (m < p.rows) {
            float4 *dst = reinterpret_cast<float4 *>(part + m * 128 + 16 * g);
            dst[0] = make_float4(acc[mt][0][tt], acc[mt][1][tt], acc[mt][2][tt], acc[mt][3][tt]);
            dst[1] = make_float4(acc[mt][4][tt], acc[mt][5][tt], acc[mt][6][tt], acc[mt][7][tt]);
            dst[2] = make_float4(acc[mt][0][2 + tt], acc[mt][1][2 + tt], acc[mt][2][2 + tt], acc[mt][3][2 + tt]);
            dst[3] = make_float4(acc[mt][4][2 + tt], acc[mt][5][2 + tt], acc[mt][6][2 + tt], acc[mt][7][2 + tt]);
          }
        }
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[mt][j][0] = acc[mt][j][1] = acc[mt][j][2] = acc[mt][j][3] = 0.f;
  };
  constexpr bool kPerChunk = MT == 1 ? EXL3_DECODE_BLOCK_PER_CHUNK_M8 : EXL3_DECODE_BLOCK_PER_CHUNK_M16;
  int xk = tk;  // k slab of bx_next
  load_x(xk, bx_next);
  int64_t z = z0;
  while (z < z1) {
    if (lane == 0 && zi < z1) issue_next();
    // warp-uniform outcome: a lane that gave up takes the whole warp out
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars[s]), phase, p.status))) {
      if (lane == 0) {  // let this warp's copies in flight land before it retires
        int ws = s;
        uint32_t wp = phase;
        for (int64_t u = consumed; u < issued; ++u) {
          mbar_wait_short(smem_u32(&bars[ws]), wp);
          if (++ws == R) {
            ws = 0;
            wp ^= 1u;
          }
        }
      }
      return;
    }
    const uint8_t *stage = ring + s * Cfg::kStage;
    const int64_t left = z1 - z;
    const int len = (int)((KT - tk) < CHK ? ((int64_t)(KT - tk) < left ? (KT - tk) : left)
                                          : (CHK < left ? CHK : left));
    // A chunk lies inside one n-block, so only its last slab can end this
    // warp's part of an n-block (kPerChunk tests it once per chunk).
    constexpr int kUnroll = MT == 1 ? EXL3_DECODE_UNROLL_M8 : EXL3_DECODE_UNROLL_M16;
#pragma unroll(kUnroll)
    for (int i = 0; i < len; ++i) {
      uint32_t own[2 * BITS];
      load_own_words<BITS, true>(stage + i * Cfg::kSeg + lane * 8 * BITS, own);
#pragma unroll
      for (int r = 0; r < 2 * MT; ++r) bx[r] = bx_next[r];
      // x' of the next k slab (none past the end of this warp's range)
      if constexpr (kPerChunk) {
        xk = xk + 1 == KT ? 0 : xk + 1;
      } else {
        xk = tk + 1 == KT ? 0 : tk + 1;  // tk: this slab
      }
      if (z + i + 1 < z1) load_x(xk, bx_next);
      const uint32_t prev = prefix_from_neighbour<BITS>(own, lane);
      constexpr bool kFx = MT == 1 ? EXL3_DECODE_FMA_EXTRACT_M8 : EXL3_DECODE_FMA_EXTRACT_M16;
      Windows<BITS, kFx> win;
      win.build(own, prev, p.m16);
      constexpr bool kDup = MT == 1 ? EXL3_DECODE_DUP_M8 : EXL3_DECODE_DUP_M16;
      if constexpr (kDup) {
        // B registers {x'[k], 0} for slab rows 4q .. 4q+3 of each token group.
        uint32_t bz[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          bz[mt][0] = bx[2 * mt] & 0xFFFFu;
          bz[mt][1] = bx[2 * mt] >> 16;
          bz[mt][2] = bx[2 * mt + 1] & 0xFFFFu;
          bz[mt][3] = bx[2 * mt + 1] >> 16;
        }
        static_for<8>([&](auto J) {
          constexpr int j = J.value;
          // rows 4q, 4q+1 of the lane's tile (mma k 2q and 2q+8), then 4q+2, 4q+3
          const uint32_t a0 = decode_dup(win.template state<0, j>());
          const uint32_t a1 = decode_dup(win.template state<0, j + 8>());
          const uint32_t a2 = decode_dup(win.template state<1, j>());
          const uint32_t a3 = decode_dup(win.template state<1, j + 8>());
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) mma16816(acc[mt][j], a0, a1, a2, a3, bz[mt][0], bz[mt][1]);
          const uint32_t c0 = decode_dup(win.template state<2, j>());
          const uint32_t c1 = decode_dup(win.template state<2, j + 8>());
          const uint32_t c2 = decode_dup(win.template state<3, j>());
          const uint32_t c3 = decode_dup(win.template state<3, j + 8>());
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) mma16816(acc[mt][j], c0, c1, c2, c3, bz[mt][2], bz[mt][3]);
        });
      } else {
        static_for<8>([&](auto J) {
          constexpr int j = J.value;
          constexpr bool kPF = MT == 1 ? EXL3_DECODE_PACK_FMA_M8 : EXL3_DECODE_PACK_FMA_M16;
          const uint32_t a0 = decode_pair_sel<kPF>(win.template state<0, j>(), win.template state<1, j>());
          const uint32_t a1 = decode_pair_sel<kPF>(win.template state<0, j + 8>(), win.template state<1, j + 8>());
          const uint32_t a2 = decode_pair_sel<kPF>(win.template state<2, j>(), win.template state<3, j>());
          const uint32_t a3 = decode_pair_sel<kPF>(win.template state<2, j + 8>(), win.template state<3, j + 8>());
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) mma16816(acc[mt][j], a0, a1, a2, a3, bx[2 * mt], bx[2 * mt + 1]);
        });
      }
      if constexpr (!kPerChunk) {
        const bool done = (tk == KT - 1) || (z + i == z1 - 1);
        const int cur_nb = nb;
        if (++tk == KT) {
          tk = 0;
          ++nb;
        }
        if (done) block_end(cur_nb);
      }
    }  // slabs of this chunk
    if constexpr (kPerChunk) {
      tk += len;
      if (tk == KT || z + len == z1) {
        block_end(nb);
        if (tk == KT) {
          tk = 0;
          ++nb;
        }
      }
    }
    __syncwarp();  // every lane has consumed this stage before lane 0 refills it
#if EXL3_DECODE_PROXY_FENCE
    fence_proxy_async_shared();
#endif
    if (++s == R) {
      s = 0;
      phase ^= 1u;
    }
    z += len;
    ++consumed;
  }
}


// Sums the partial slots of every n-block shared by several warps, in slot
// order, then applies had_r_128 over the block's 128 columns, sv and the
// -inf mask, and writes y. One warp per (n-block, row); lane l owns columns
// 4l .. 4l+3. N-blocks owned by a single warp were finished by that warp.
// The decode GEMM splits an n-block over up to ~20 slots: 16 loads per lane
// are kept in flight at once.
__global__ void __launch_bounds__(256) decode_finalize_kernel(const float *__restrict__ partials, int64_t smax,
                                                              int64_t slot_elems, const __half *__restrict__ sv,
                                                              void *y, int y_f32, int64_t n_gemm, int64_t n_valid,
                                                              int rows, int64_t P, int64_t TS, int KT, int all_blocks) {
  // The next op's input rotation may launch now; it waits for this grid
  // before it touches memory.
  if (EXL3_DECODE_ROTATE_PDL) allow_next_grid();
  const int lane = threadIdx.x & 31;
  const int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nb = w / rows;
  const int m = (int)(w % rows);
  if (nb >= n_gemm / 128) return;
  const int64_t pf = slab_owner(nb * KT, P, TS);
  const int cnt = (int)(slab_owner((nb + 1) * KT - 1, P, TS) - pf + 1);
  if (cnt == 1 && !all_blocks) return;  // finished by its single owner
  const uint2 s4 = load_sv4(sv, nb, lane);
  wait_prior_grid();  // partial slots come from the decode kernel
  const float *base = partials + nb * smax * slot_elems + m * 128 + 4 * lane;
  float v[4];
  sum_slots(base, cnt, slot_elems, v);
  finalize_row(v, s4, y, y_f32, n_gemm, n_valid, nb, m, lane);
}

// The same reduction for the fused tensor-core GEMM (up to 256 rows, 2-3
// slots per n-block): one warp per (n-block, RPW rows) with the loads of all
// its rows for 4 slots at a time in flight together. RPW grows with the rows
// so that the grid keeps a few thousand warps.
template <int RPW>
__global__ void __launch_bounds__(256) fused_finalize_kernel(const float *__restrict__ partials, int64_t smax,
                                                             int64_t slot_elems, const __half *__restrict__ sv,
                                                             void *y, int y_f32, int64_t n_gemm, int64_t n_valid,
                                                             int rows, int64_t P, int64_t TS, int KT) {
  constexpr int SC = 4;
  const int lane = threadIdx.x & 31;
  if (EXL3_DECODE_ROTATE_PDL) allow_next_grid();  // as in decode_finalize_kernel
  const unsigned groups = (unsigned)((rows + RPW - 1) / RPW);
  const unsigned w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nb = w / groups;
  const int m0 = (int)(w % groups) * RPW;
  if (nb >= n_gemm / 128) return;
  const int64_t pf = slab_owner(nb * KT, P, TS);
  const int cnt = (int)(slab_owner((nb + 1) * KT - 1, P, TS) - pf + 1);
  const uint2 s4 = load_sv4(sv, nb, lane);
  wait_prior_grid();  // partial slots come from the GEMM kernel
  const float *base = partials + nb * smax * slot_elems + (int64_t)m0 * 128 + 4 * lane;
  const int nr = rows - m0 < RPW ? rows - m0 : RPW;
  float v[RPW][4];
#pragma unroll
  for (int r = 0; r < RPW; ++r) v[r][0] = v[r][1] = v[r][2] = v[r][3] = 0.f;
  for (int s0 = 0; s0 < cnt; s0 += SC) {
    float4 f[SC][RPW];
#pragma unroll
    for (int s = 0; s < SC; ++s)
#pragma unroll
      for (int r = 0; r < RPW; ++r)
        // unconditional (clamped) so that all of them are issued together
        f[s][r] = __ldcg(reinterpret_cast<const float4 *>(base + (s0 + s < cnt ? s0 + s : cnt - 1) * slot_elems +
                                                          (r < nr ? r : nr - 1) * 128));
#pragma unroll
    for (int s = 0; s < SC; ++s)  // summed in slot order
      if (s0 + s < cnt)
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
          v[r][0] += f[s][r].x;
          v[r][1] += f[s][r].y;
          v[r][2] += f[s][r].z;
          v[r][3] += f[s][r].w;
        }
  }
#pragma unroll
  for (int r = 0; r < RPW; ++r)
    if (r < nr) finalize_row(v[r], s4, y, y_f32, n_gemm, n_valid, nb, m0 + r, lane);
}

// x' = RNE_fp16(had_r_128(x * su)) for up to 8*MT rows, in fragment order:
// for k slab tk, lane (g, q) owns 4*MT halves at xf[(tk*32 + 4g + q)*4*MT],
// {x'[g][16tk+4q .. +3], x'[g+8][16tk+4q .. +3]}. Rows >= `rows` are zero.
// One half-warp per (row, 128-block): lane l16 holds elements 8*l16 .. +7,
// butterfly stages h = 1, 2, 4 in-lane and 8 .. 64 across lanes.
template <int MT>
__global__ void __launch_bounds__(256) rotate_frag_kernel(const __half *__restrict__ x, const __half *__restrict__ su,
                                                          int rows, int64_t K, __half *__restrict__ xf) {
  constexpr int CH = 4 * MT;
  allow_next_grid();
  // When launched as a programmatic dependent of the previous kernel in the
  // stream (only its launch latency is hidden): x may be that kernel's
  // output, and the previous decode GEMM may still read xf.
  wait_prior_grid();
  const int lane = threadIdx.x & 31, l16 = lane & 15;
  const int64_t KB = K / 128;
  const int64_t jobs = 8 * MT * KB;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t jp = warp; jp * 2 < jobs; jp += nwarps) {
    const int64_t job = jp * 2 + (lane >> 4);
    const bool valid = job < jobs;
    const int m = valid ? (int)(job / KB) : 0;
    const int64_t kb = valid ? job % KB : 0;
    float v[8];
    if (valid && m < rows) {
      const int64_t k = kb * 128 + 8 * l16;
      const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(x + (int64_t)m * K + k));
      const uint4 sraw = __ldg(reinterpret_cast<const uint4 *>(su + k));
      const __half *h = reinterpret_cast<const __half *>(&raw);
      const __half *sh = reinterpret_cast<const __half *>(&sraw);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = __half2float(h[i]) * __half2float(sh[i]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
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
    for (int s = 1; s < 16; s <<= 1)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float o = __shfl_xor_sync(0xffffffffu, v[i], s);
        v[i] = (l16 & s) ? (o - v[i]) : (v[i] + o);
      }
    if (valid) {
      __half2 hv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) hv[e] = __floats2half2_rn(v[2 * e] * kInvSqrt128, v[2 * e + 1] * kInvSqrt128);
      const int64_t tk = kb * 8 + (l16 >> 1);
      const int qq = 2 * (l16 & 1);
      const int gg = m & 7;
      const int off = (m >> 3) * 4;
      __half *d0 = xf + (tk * 32 + gg * 4 + qq) * CH + off;
      __half *d1 = xf + (tk * 32 + gg * 4 + qq + 1) * CH + off;
      *reinterpret_cast<uint2 *>(d0) =
          make_uint2(*reinterpret_cast<uint32_t *>(&hv[0]), *reinterpret_cast<uint32_t *>(&hv[1]));
      *reinterpret_cast<uint2 *>(d1) =
          make_uint2(*reinterpret_cast<uint32_t *>(&hv[2]), *reinterpret_cast<uint32_t *>(&hv[3]));
    }
  }
}

template <int BITS, int MT>
cudaError_t init_one() {
  cudaError_t e = cudaFuncSetAttribute(decode_gemm_kernel<BITS, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       DecodeCfg<BITS, MT>::kSmem);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes a;
  e = cudaFuncGetAttributes(&a, decode_finalize_kernel);
  if (e != cudaSuccess) return e;
  for (auto *k : {fused_finalize_kernel<1>, fused_finalize_kernel<2>}) {
    e = cudaFuncGetAttributes(&a, k);
    if (e != cudaSuccess) return e;
  }
  return cudaFuncGetAttributes(&a, rotate_frag_kernel<MT>);
}

template <int BITS>
cudaError_t init_bits() {
  cudaError_t e = init_one<BITS, 1>();
  if (e != cudaSuccess) return e;
  return init_one<BITS, 2>();
}

// Launches `kernel` after the previous work in `st`; with EXL3_DECODE_PDL its
// prologue may overlap the tail of the previous kernel (programmatic
// dependency), and the kernel itself waits before reading that kernel's
// output.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, unsigned block, size_t smem, cudaStream_t st,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = EXL3_DECODE_PDL ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int BITS, int MT>
cudaError_t launch_bits(const DecodeParams &dp, int64_t grid, cudaStream_t st) {
  // The trellis as rows of 16-row tile strips (8-byte elements): one row is
  // every tile of one k slab; the box is one n-block's slab x kChunk rows.
  alignas(64) CUtensorMap tmap;
  const uint64_t row_elems = (uint64_t)dp.tiles_n * 4 * BITS;
  if (!encode_tensor_map_2d(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, dp.trellis, row_elems, (uint64_t)dp.KT,
                            row_elems * 8, 32 * BITS, DecodeCfg<BITS, MT>::kChunk, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  return launch_dependent(decode_gemm_kernel<BITS, MT>, (unsigned)grid, DecodeCfg<BITS, MT>::kWarps * 32,
                          DecodeCfg<BITS, MT>::kSmem, st, tmap, dp);
}

template <int MT>
cudaError_t launch_mt(int bits, const DecodeParams &dp, int64_t grid, cudaStream_t st) {
  switch (bits) {
    case 1: return launch_bits<1, MT>(dp, grid, st);
    case 7: return launch_bits<7, MT>(dp, grid, st);
    case 2: return launch_bits<2, MT>(dp, grid, st);
    case 3: return launch_bits<3, MT>(dp, grid, st);
    case 4: return launch_bits<4, MT>(dp, grid, st);
    case 5: return launch_bits<5, MT>(dp, grid, st);
    case 6: return launch_bits<6, MT>(dp, grid, st);
    case 8: return launch_bits<8, MT>(dp, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

int64_t owner_host(int64_t z, int64_t P, int64_t TS) { return ((z + 1) * P - 1) / TS; }

}  // namespace

DecodePlan decode_plan(int64_t n_blocks, int64_t k_blocks, int num_sms) {
  DecodePlan plan;
  const int64_t KT = k_blocks * 8;
  const int64_t TS = n_blocks * KT;
  for (int mt = 1; mt <= 2; ++mt) {
    const int warps = mt == 1 ? DecodeCfg<4, 1>::kWarps : DecodeCfg<4, 2>::kWarps;
    int64_t P = (int64_t)num_sms * warps;
    if (P > TS) P = TS;
    int64_t smax = 1;
    for (int64_t nb = 0; nb < n_blocks; ++nb) {
      const int64_t c = owner_host((nb + 1) * KT - 1, P, TS) - owner_host(nb * KT, P, TS) + 1;
      if (c > smax) smax = c;
    }
    plan.P[mt - 1] = P;
    plan.grid[mt - 1] = ceil_div(P, warps);
    plan.smax[mt - 1] = smax;
  }
  return plan;
}

size_t decode_partials_bytes(const DecodePlan &plan, int64_t n_blocks) {
  const size_t a = (size_t)n_blocks * plan.smax[0] * 8 * 128 * 4;
  const size_t b = (size_t)n_blocks * plan.smax[1] * 16 * 128 * 4;
  return a > b ? a : b;
}

cudaError_t init_decode_kernels() {
  cudaError_t e;
  if ((e = init_bits<1>()) != cudaSuccess) return e;
  if ((e = init_bits<7>()) != cudaSuccess) return e;
  if ((e = init_bits<2>()) != cudaSuccess) return e;
  if ((e = init_bits<3>()) != cudaSuccess) return e;
  if ((e = init_bits<4>()) != cudaSuccess) return e;
  if ((e = init_bits<5>()) != cudaSuccess) return e;
  if ((e = init_bits<6>()) != cudaSuccess) return e;
  return init_bits<8>();
}

cudaError_t launch_decode_finalize(const float *partials, int64_t smax, int64_t slot_elems, const void *sv, void *y,
                                   int y_f32, int64_t n_gemm, int64_t n_valid, int rows, int64_t P, int64_t TS,
                                   int units_per_block, int all_blocks, cudaStream_t st) {
  if (!all_blocks) {
    const int64_t warps = (n_gemm / 128) * rows;
    // One warp per CTA for few rows spreads the slot loads over more SMs
    // (0.35 us less at 1 row, 0.1 us at 2; 4 rows measured 0.1 us slower).
    const unsigned wpc = rows <= EXL3_DECODE_FIN_1W_ROWS ? 1u : 8u;
    return launch_dependent(decode_finalize_kernel, (unsigned)ceil_div(warps, (int64_t)wpc), 32u * wpc, (size_t)0, st, partials,
                            smax, slot_elems, static_cast<const __half *>(sv), y, y_f32, n_gemm, n_valid, rows, P, TS,
                            units_per_block, all_blocks);
  }
  const int rpw = rows <= 64 ? 1 : 2;  // measured: 4 rows per warp was 4 % slower at 256 rows
  const unsigned grid = (unsigned)ceil_div((n_gemm / 128) * ceil_div(rows, rpw), 8);
  auto *kern = rpw == 1 ? fused_finalize_kernel<1> : fused_finalize_kernel<2>;
  return launch_dependent(kern, grid, 256u, (size_t)0, st, partials, smax, slot_elems,
                          static_cast<const __half *>(sv), y, y_f32, n_gemm, n_valid, rows, P, TS, units_per_block);
}

cudaError_t launch_decode_gemm(const DecodeLaunch &L, cudaStream_t st) {
  const int MT = L.rows <= 8 ? 1 : 2;
  const int64_t K = L.K;
  // 1. rotated activations in fragment order
  {
    const int64_t jobs = 8 * MT * (K / 128);
    int64_t grid = ceil_div(ceil_div(jobs, 2), 8);
    const __half *x = static_cast<const __half *>(L.x), *su = static_cast<const __half *>(L.su);
    __half *xf = static_cast<__half *>(L.xf);
    cudaError_t e;
    if (EXL3_DECODE_ROTATE_PDL && MT == 1)  // (measured 0.5 us slower for 9..16 rows)
      e = launch_dependent(rotate_frag_kernel<1>, (unsigned)grid, 256, 0, st, x, su, L.rows, K, xf);
    else if (MT == 1)
      rotate_frag_kernel<1><<<(unsigned)grid, 256, 0, st>>>(x, su, L.rows, K, xf);
    else
      rotate_frag_kernel<2><<<(unsigned)grid, 256, 0, st>>>(x, su, L.rows, K, xf);
    if (!(EXL3_DECODE_ROTATE_PDL && MT == 1)) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // 2. stream-K decode GEMM
  DecodeParams dp;
  dp.trellis = reinterpret_cast<const uint8_t *>(L.trellis);
  dp.xf = static_cast<const uint8_t *>(L.xf);
  dp.sv = static_cast<const __half *>(L.sv);
  dp.y = L.y;
  dp.partials = L.partials;
  dp.status = L.status;
  dp.tiles_n = L.n_stored / 16;
  dp.n_gemm = L.n_gemm;
  dp.n_valid = L.n_valid;
  dp.KT = (int)(K / 16);
  dp.TS = (L.n_gemm / 128) * dp.KT;
  dp.P = L.plan.P[MT - 1];
  dp.smax = (int)L.plan.smax[MT - 1];
  dp.rows = L.rows;
  dp.m16 = 16u;
  dp.y_f32 = L.y_f32;
  const int64_t grid = L.plan.grid[MT - 1];
  cudaError_t e = MT == 1 ? launch_mt<1>(L.bits, dp, grid, st) : launch_mt<2>(L.bits, dp, grid, st);
  if (e != cudaSuccess || dp.smax == 1) return e;
  // 3. reduce the slots of n-blocks shared by several warps
  return launch_decode_finalize(L.partials, dp.smax, (int64_t)8 * MT * 128, L.sv, L.y, L.y_f32, L.n_gemm, L.n_valid,
                                L.rows, dp.P, dp.TS, dp.KT, /*all_blocks=*/0, st);
}

}  // namespace exl3
