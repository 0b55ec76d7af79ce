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
//      rows, written in mma fragment order: per 16-row k slab, lane (g, q)
//      finds its B registers as 16 contiguous bytes (for <= 8 rows already
//      in the {x', 0} form the duplicated-weight mma takes).
//   2. decode_gemm_kernel: stream-K over all (n-block, k-slab) work. A slab
//      is 16 k-rows x 128 output columns = 8 horizontally adjacent trellis
//      tiles, 256*BITS contiguous bytes. The P = SMs x 12 warps each own a
//      contiguous range of slabs in n-block-major order, so every warp on
//      every SM has the same amount of work. Each warp feeds itself: lane 0
//      streams chunks of up to 4 slabs (one 2-D TMA copy of the trellis plus
//      one bulk copy of the chunk's x' fragments) into a private ring of
//      stages in shared memory, one mbarrier per stage.
//      Lane (g, q) decodes tile g, rows 4q..4q+3 straight into m16n8k16 A
//      fragments (A = W^T: mma row r <-> output column 16*(r%8) + j +
//      8*(r/8) for mma j), B = x'^T (8 tokens per mma). For <= 8 rows each A
//      register holds one weight in both halves and the matching B register
//      {x', 0}: mma k index 2q <-> tile row 4q and 2q+8 <-> row 4q+1 in the
//      first mma of a column group, rows 4q+2 and 4q+3 in the second (odd k
//      indices multiply zeros). This spends twice the mmas (the tensor pipe
//      has room) to save the instructions that would pack two decoded
//      weights into one register. For 9..16 rows the registers hold weight
//      pairs (rows 4q and 4q+1, rows 4q+2 and 4q+3) and one mma per column
//      group and token group. After a slab, lane (g, q) holds output columns
//      16g .. 16g+15 of tokens 2q, 2q+1 (+8).
//      When a warp finishes its part of an n-block it either owns the whole
//      n-block (then it applies had_r_128 over the 128 columns, sv and the
//      -inf mask and writes y), or it stores an fp32 partial in its slot.
//   3. decode_finalize_kernel (only when some n-block is shared): one warp
//      per (n-block, row) sums the slots in slot order (deterministic),
//      applies had_r_128, sv and the mask and writes y.
//
// Roofline: HBM-bound on the trellis bytes (K*N*BITS/8 per launch) unless
// the per-weight integer decode (a half-rate ALU pipe) binds first, which
// it does on GB300: per weight one window extraction, one IMAD (LCG), one
// LOP3 (mask and xor) and one fp16 add, plus an mma per 4 weights.
#include <cuda.h>
#include <math.h>

#include "exl3_common.cuh"
#include "exl3_internal.h"

namespace exl3 {

namespace {

// Warps per CTA (one CTA per SM) for <= 8 rows and for 9..16 rows.
template <int MT>
constexpr int dec_warps() { return MT == 1 ? 12 : 12; }
constexpr int kXFrag = 512;     // x' fragment bytes per 16-row k slab (32 lanes x 16 B)

template <int BITS, int MT>
struct DecodeCfg {
  static constexpr int kWarps = dec_warps<MT>();
  static constexpr int kSeg = 256 * BITS;                    // trellis bytes per slab
  // slabs per copy: 4, or 3 where two stages of 4 would not fit (8 bits)
  static constexpr int kChunk = 2 * kWarps * 4 * (kSeg + kXFrag) <= 226 * 1024 ? 4 : 3;
  static constexpr int kStage = kChunk * (kSeg + kXFrag);    // trellis box, then the chunk's x'
  // ring stages (chunks) per warp (with full chunks run as straight-line
  // slabs, a third stage measured slower for 1..8 rows and for 9..16 rows)
  static constexpr int kStages = 2;
  static constexpr int kWarpRing = kStages * kStage;
  static constexpr int kSmem = kWarps * kWarpRing + kWarps * kStages * 8;
  static_assert(kSmem <= 227 * 1024, "decode ring exceeds shared memory");
};

struct DecodeParams {
  const uint8_t *xf;  // rotated x in fragment order, K/16 slabs of kXFrag bytes
  const __half *sv;
  void *y;
  float *partials;
  int *status;
  int64_t n_gemm, n_valid;
  int TS, P, KT, rows, y_f32, smax;
  uint32_t m16;  // 16, opaque to the compiler (a multiply by it stays on the FMA pipe)
  uint32_t mk[8];  // mk[k] = 2^k, opaque likewise (window views for widths other than 4)
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
      for (int s = 1; s < 8; s <<= 1) {
        // the lane's side of the butterfly: o + v or o - v, one rounding either way
        const float sgn = (g & s) ? -1.f : 1.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float o = __shfl_xor_sync(0xffffffffu, v[mt][t][i], s * 4);
          v[mt][t][i] = fmaf(v[mt][t][i], sgn, o);
        }
      }
    }
  const int64_t col0 = nb * 128 + 16 * g;
  const bool cols_ok = EXL3_SPAN(col0, 16, p.n_gemm);
  float scale[16];
  {
    const uint4 *svp = reinterpret_cast<const uint4 *>(p.sv + col0);
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const uint4 raw = cols_ok ? __ldg(svp + a) : uint4{};
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
      if (m < p.rows && cols_ok) {
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
__device__ __forceinline__ uint2 load_sv4(const __half *__restrict__ sv, int64_t nb, int lane, int64_t n_gemm) {
  return EXL3_SPAN(nb * 128 + 4 * lane, 4, n_gemm) ? __ldg(reinterpret_cast<const uint2 *>(sv + nb * 128 + 4 * lane))
                                                    : uint2{};
}

// Output rotation (had_r_128 over the 128 columns spread as 4 per lane), sv
// (the lane's four values from load_sv4), mask and store of one row of
// n-block nb.
__device__ __forceinline__ void finalize_row(float (&v)[4], uint2 sraw, void *y, int y_f32, int64_t n_gemm,
                                             int64_t n_valid, int64_t nb, int m, int rows, int lane) {
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
  for (int s = 1; s < 32; s <<= 1) {
    const float sgn = (lane & s) ? -1.f : 1.f;  // o + v or o - v, one rounding either way
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], s);
      v[i] = fmaf(v[i], sgn, o);
    }
  }
  const int64_t col = nb * 128 + 4 * lane;
  const __half *sh = reinterpret_cast<const __half *>(&sraw);
  float o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = (col + i < n_valid) ? v[i] * (__half2float(sh[i]) * kInvSqrt128) : -INFINITY;
  if (!EXL3_RANGE(m, 0, rows) || !EXL3_SPAN(col, 4, n_gemm)) return;
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

// The lane's 64 states of one slab: st[r][c] = tile row 4q + r, column c.
template <int BITS>
__device__ __forceinline__ void slab_states(const uint32_t (&own)[2 * BITS], uint32_t prev, uint32_t m16,
                                            const uint32_t (&mk)[8], uint32_t (&st)[4][16]) {
  if constexpr (BITS == 4) {
#pragma unroll
    for (int r = 0; r < 4; ++r) row4_states(own[2 * r], own[2 * r + 1], r == 0 ? prev : own[2 * r - 1], m16, st[r]);
  } else {
    RowWindows<BITS> rw;
    rw.build(own, prev);
    static_for<4>([&](auto R) {
      static_for<16>([&](auto C) { st[R.value][C.value] = rw.template state_fma<R.value, C.value>(mk); });
    });
  }
}

template <int BITS, int MT>
__global__ void __launch_bounds__(DecodeCfg<BITS, MT>::kWarps * 32, 1)
    decode_gemm_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeParams p) {
  using Cfg = DecodeCfg<BITS, MT>;
  constexpr int R = Cfg::kStages, CHK = Cfg::kChunk;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int pw = blockIdx.x * Cfg::kWarps + warp;
  if (pw >= p.P) return;
  const int z0 = (int)((int64_t)pw * p.TS / p.P), z1 = (int)((int64_t)(pw + 1) * p.TS / p.P);
  const int KT = p.KT;
  uint8_t *ring = smem + warp * Cfg::kWarpRing;
  const uint32_t ring_s = smem_u32(ring);
  const uint32_t bar0 = smem_u32(smem + Cfg::kWarps * Cfg::kWarpRing) + warp * R * 8;
  // this warp's ring and barriers inside the CTA's shared memory (warp-uniform)
  if (!EXL3_SMEM(ring_s, Cfg::kWarpRing) || !EXL3_SMEM(bar0, 8 * R)) return;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < R; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_barrier_init();
  }
  __syncwarp();

  // Producer cursor (lane 0 only): the next chunk to stream in. A chunk is
  // up to CHK consecutive k slabs of one n-block: one 2-D TMA copy of the
  // trellis (box: one slab row of 8 tiles x CHK tile rows; rows past K read
  // as zero and are never used) and one bulk copy of the chunk's x'.
  int i_nb = z0 / KT, i_tk = z0 - i_nb * KT, i_z = z0, i_st = 0, issued = 0;
  auto chunk_len = [&](int tk, int z) { return min(min(CHK, KT - tk), z1 - z); };
  auto issue_trellis = [&]() {
    const int len = chunk_len(i_tk, i_z);
    const uint32_t bar = bar0 + 8 * i_st;
    mbar_arrive_expect_tx(bar, CHK * Cfg::kSeg + len * kXFrag);
    // box: 8-byte columns [32*BITS*i_nb, +32*BITS) (an even start: the
    // 16-byte rule), rows [i_tk, +CHK) of KT (rows past KT read zero)
    if (EXL3_RANGE(i_nb, 0, p.n_gemm / 128) && EXL3_RANGE(i_tk, 0, KT) && EXL3_RANGE(len, 1, CHK + 1) &&
        EXL3_ALIGNED(i_nb * (32 * BITS) * 8, 16) && EXL3_RANGE(i_st, 0, R))
      tma_load_2d_u64(ring_s + i_st * Cfg::kStage, &tmap, bar, i_nb * (32 * BITS), i_tk);
    return len;
  };
  auto issue_x = [&](int st, int tk, int len) {
    const uint32_t dst = ring_s + st * Cfg::kStage + CHK * Cfg::kSeg;
    if (EXL3_SPAN((int64_t)tk * kXFrag, len * kXFrag, (int64_t)KT * kXFrag) &&
        EXL3_SPAN(dst - ring_s, len * kXFrag, Cfg::kWarpRing) && EXL3_ALIGNED(dst, 16) &&
        EXL3_ALIGNED(reinterpret_cast<uintptr_t>(p.xf + (size_t)tk * kXFrag), 16))
      bulk_g2s(dst, p.xf + (size_t)tk * kXFrag, len * kXFrag, bar0 + 8 * st);
  };
  auto advance = [&](int len) {
    i_z += len;
    i_tk += len;
    if (i_tk == KT) {
      i_tk = 0;
      ++i_nb;
    }
    if (++i_st == R) i_st = 0;
    ++issued;
  };
  // Fill the ring with trellis before waiting for the rotation kernel (the
  // weights do not depend on it); the x' halves follow after the wait.
  int pro_tk[R], pro_len[R];
  if (lane == 0) {
#pragma unroll
    for (int c = 0; c < R; ++c) {
      pro_len[c] = 0;
      if (i_z < z1) {
        pro_tk[c] = i_tk;
        pro_len[c] = issue_trellis();
        advance(pro_len[c]);
      }
    }
  }
  allow_next_grid();
  wait_prior_grid();  // x' comes from the rotation kernel
  if (lane == 0) {
#pragma unroll
    for (int c = 0; c < R; ++c)
      if (pro_len[c]) issue_x(c, pro_tk[c], pro_len[c]);
  }

  float acc[MT][8][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[mt][j][0] = acc[mt][j][1] = acc[mt][j][2] = acc[mt][j][3] = 0.f;

  // This warp's part of n-block cnb is complete: finish it or store the
  // partial, then clear the accumulators.
  auto block_end = [&](const int cnb) {
    const bool whole = (z0 <= cnb * KT) && (z1 >= (cnb + 1) * KT);
    if (whole) {
      float v[MT][2][16];
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
      // this warp's contribution goes to its slot; decode_finalize_kernel
      // sums the n-block's slots in slot order
      const int64_t pf = slab_owner((int64_t)cnb * KT, p.P, p.TS);
      const int64_t slot_elems = (int64_t)8 * MT * 128;
      // slot pw - pf of the n-block's smax, row m of the slot's 8 * MT
      const bool slot_ok = EXL3_RANGE(cnb, 0, p.n_gemm / 128) && EXL3_RANGE(pw - pf, 0, p.smax) &&
                           EXL3_SPAN(16 * g, 16, 128);
      float *part = p.partials + ((int64_t)cnb * p.smax + (pw - pf)) * slot_elems;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
          const int m = 8 * mt + 2 * q + tt;
          if (m < p.rows && slot_ok && EXL3_RANGE(m, 0, 8 * MT)) {
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

  // One slab: the lane's 64 weights (tile g, rows 4q..4q+3) into 16 (or,
  // for 9..16 rows, 2 x 8) mmas. tr: the slab's trellis in the stage; xb:
  // the lane's 16 bytes of x' fragments for the slab.
  auto slab = [&](const uint8_t *tr, const uint8_t *xb) {
    uint32_t own[2 * BITS];
    if (EXL3_SPAN(smem_u32(tr + lane * 8 * BITS) - ring_s, 8 * BITS, Cfg::kWarpRing)) {
      load_own_words<BITS, true>(tr + lane * 8 * BITS, own);
    } else {
#pragma unroll
      for (int i = 0; i < 2 * BITS; ++i) own[i] = 0;
    }
    const uint4 bxv = EXL3_SPAN(smem_u32(xb + lane * 16) - ring_s, 16, Cfg::kWarpRing)
                          ? *reinterpret_cast<const uint4 *>(xb + lane * 16)
                          : uint4{};
    const uint32_t prev = prefix_from_neighbour<BITS>(own, lane);
    uint32_t st[4][16];
    slab_states<BITS>(own, prev, p.m16, p.mk, st);
    if constexpr (MT == 1) {
      // B registers {x'[row], 0} for tile rows 4q .. 4q+3 of token g
      static_for<8>([&](auto J) {
        constexpr int j = J.value;
        mma16816(acc[0][j], decode_dup(st[0][j]), decode_dup(st[0][j + 8]), decode_dup(st[1][j]),
                 decode_dup(st[1][j + 8]), bxv.x, bxv.y);
        mma16816(acc[0][j], decode_dup(st[2][j]), decode_dup(st[2][j + 8]), decode_dup(st[3][j]),
                 decode_dup(st[3][j + 8]), bxv.z, bxv.w);
      });
    } else {
      // B registers: {x'[4q], x'[4q+1]}, {x'[4q+2], x'[4q+3]} of tokens g and g + 8
      static_for<8>([&](auto J) {
        constexpr int j = J.value;
        // pairs packed by two half-selected fp16 adds and a byte permute (measured
        // 4 % faster at 16 rows than packing with fp16 multiply-adds, which load
        // the half-rate fp16 pipe twice as much)
        const uint32_t a0 = decode_pair_sel<false>(st[0][j], st[1][j]);
        const uint32_t a1 = decode_pair_sel<false>(st[0][j + 8], st[1][j + 8]);
        const uint32_t a2 = decode_pair_sel<false>(st[2][j], st[3][j]);
        const uint32_t a3 = decode_pair_sel<false>(st[2][j + 8], st[3][j + 8]);
        mma16816(acc[0][j], a0, a1, a2, a3, bxv.x, bxv.y);
        mma16816(acc[1][j], a0, a1, a2, a3, bxv.z, bxv.w);
      });
    }
  };

  // Consumer cursor.
  int nb = z0 / KT, tk = z0 - nb * KT, z = z0, s = 0, consumed = 0;
  uint32_t phase = 0;
  while (z < z1) {
    const int len = chunk_len(tk, z);
    // warp-uniform outcome: a lane that gave up takes the whole warp out
    if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * s, phase, p.status))) {
      if (lane == 0) {  // let this warp's copies in flight land before it retires
        int ws = s;
        uint32_t wp = phase;
        for (int u = consumed; u < issued; ++u) {
          mbar_wait_short(bar0 + 8 * ws, wp);
          if (++ws == R) {
            ws = 0;
            wp ^= 1u;
          }
        }
      }
      return;
    }
    const uint8_t *stage = ring + s * Cfg::kStage;
    const uint8_t *xst = stage + CHK * Cfg::kSeg;
    if (len == CHK) {  // a full chunk: straight-line slabs the scheduler can interleave
      static_for<CHK>([&](auto I) { slab(stage + I.value * Cfg::kSeg, xst + I.value * kXFrag); });
    } else {
#pragma unroll 1
      for (int i = 0; i < len; ++i) slab(stage + i * Cfg::kSeg, xst + i * kXFrag);
    }
    // a chunk lies inside one n-block, so only its end can end this warp's part of it
    tk += len;
    z += len;
    if (tk == KT || z == z1) {
      block_end(nb);
      if (tk == KT) {
        tk = 0;
        ++nb;
      }
    }
    // every lane has read this stage (its words are in registers and consumed
    // by register-dependent work) before lane 0 hands it to the next copy
    __syncwarp();
    if (lane == 0 && i_z < z1) {
      const int itk = i_tk, ist = i_st;
      const int ilen = issue_trellis();
      issue_x(ist, itk, ilen);
      advance(ilen);
    }
    if (++s == R) {
      s = 0;
      phase ^= 1u;
    }
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
  allow_next_grid();
  const int lane = threadIdx.x & 31;
  const int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nb = w / rows;
  const int m = (int)(w % rows);
  if (nb >= n_gemm / 128) return;
  const int64_t pf = slab_owner(nb * KT, P, TS);
  const int cnt = (int)(slab_owner((nb + 1) * KT - 1, P, TS) - pf + 1);
  if (cnt == 1 && !all_blocks) return;  // finished by its single owner
  const uint2 s4 = load_sv4(sv, nb, lane, n_gemm);
  wait_prior_grid();  // partial slots come from the decode kernel
  const float *base = partials + nb * smax * slot_elems + m * 128 + 4 * lane;
  // cnt of the n-block's smax slots; the lane's columns of row m in a slot
  const bool ok = EXL3_RANGE(cnt, 1, smax + 1) && EXL3_SPAN(m * 128 + 4 * lane, 4, slot_elems);
  float v[4];
  sum_slots(base, ok ? cnt : 0, slot_elems, v);
  finalize_row(v, s4, y, y_f32, n_gemm, n_valid, nb, m, rows, lane);
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
  allow_next_grid();  // as in decode_finalize_kernel
  const unsigned groups = (unsigned)((rows + RPW - 1) / RPW);
  const unsigned w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nb = w / groups;
  const int m0 = (int)(w % groups) * RPW;
  if (nb >= n_gemm / 128) return;
  const int64_t pf = slab_owner(nb * KT, P, TS);
  const int cnt = (int)(slab_owner((nb + 1) * KT - 1, P, TS) - pf + 1);
  const uint2 s4 = load_sv4(sv, nb, lane, n_gemm);
  wait_prior_grid();  // partial slots come from the GEMM kernel
  const float *base = partials + nb * smax * slot_elems + (int64_t)m0 * 128 + 4 * lane;
  const int nr = rows - m0 < RPW ? rows - m0 : RPW;
  // cnt of the n-block's smax slots; rows m0 .. m0 + nr - 1 of a slot
  const bool ok = EXL3_RANGE(cnt, 1, smax + 1) && EXL3_RANGE(nr, 1, RPW + 1) &&
                  EXL3_SPAN((int64_t)(m0 + nr - 1) * 128 + 4 * lane, 4, slot_elems);
  float v[RPW][4];
#pragma unroll
  for (int r = 0; r < RPW; ++r) v[r][0] = v[r][1] = v[r][2] = v[r][3] = 0.f;
  for (int s0 = 0; s0 < (ok ? cnt : 0); s0 += SC) {
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
    if (r < nr) finalize_row(v[r], s4, y, y_f32, n_gemm, n_valid, nb, m0 + r, rows, lane);
}

// x' = RNE_fp16(had_r_128(x * su)) for up to 8*MT rows, in fragment order:
// for k slab tk, lane (g, q) owns the 16 bytes at xf + (tk*32 + 4g + q)*16.
// MT = 1 (up to 8 rows): the B registers of the duplicated-weight mma,
// {x'[g][16tk+4q+i], 0} for i = 0..3. MT = 2: {x'[g][16tk+4q .. +3],
// x'[g+8][16tk+4q .. +3]}. Rows >= `rows` are zero.
// One half-warp per (row, 128-block): lane l16 holds elements 8*l16 .. +7,
// butterfly stages h = 1, 2, 4 in-lane and 8 .. 64 across lanes.
template <int MT>
__global__ void __launch_bounds__(256) rotate_frag_kernel(const __half *__restrict__ x, const __half *__restrict__ su,
                                                          int rows, int64_t K, uint8_t *__restrict__ xf) {
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
      const bool ok = EXL3_SPAN((int64_t)m * K + k, 8, (int64_t)rows * K) && EXL3_SPAN(k, 8, K);
      const uint4 raw = ok ? __ldg(reinterpret_cast<const uint4 *>(x + (int64_t)m * K + k)) : uint4{};
      const uint4 sraw = ok ? __ldg(reinterpret_cast<const uint4 *>(su + k)) : uint4{};
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
    for (int s = 1; s < 16; s <<= 1) {
      const float sgn = (l16 & s) ? -1.f : 1.f;  // o + v or o - v, one rounding either way
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float o = __shfl_xor_sync(0xffffffffu, v[i], s);
        v[i] = fmaf(v[i], sgn, o);
      }
    }
    if (valid) {
      uint32_t hb[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) hb[i] = __half_as_ushort(__float2half_rn(v[i] * kInvSqrt128));
      // elements 8*l16 .. +7 of block kb: slab kb*8 + l16/2, tile rows
      // 8*(l16&1) .. +7, i.e. lanes q = 2*(l16&1) and q + 1 of group m & 7
      const int64_t tk = kb * 8 + (l16 >> 1);
      const int qq = 2 * (l16 & 1);
      const int64_t xo = (tk * 32 + (m & 7) * 4 + qq) * 16;  // K/16 slabs of 512 bytes
      uint8_t *d0 = xf + xo;
      if constexpr (MT == 1) {
        if (EXL3_SPAN(xo, 32, K * 32)) {
          *reinterpret_cast<uint4 *>(d0) = make_uint4(hb[0], hb[1], hb[2], hb[3]);
          *reinterpret_cast<uint4 *>(d0 + 16) = make_uint4(hb[4], hb[5], hb[6], hb[7]);
        }
      } else {
        const int off = (m >> 3) * 8;
        if (EXL3_RANGE(m, 0, 16) && EXL3_SPAN(xo + off, 24, K * 32)) {
          *reinterpret_cast<uint2 *>(d0 + off) = make_uint2(hb[0] | hb[1] << 16, hb[2] | hb[3] << 16);
          *reinterpret_cast<uint2 *>(d0 + 16 + off) = make_uint2(hb[4] | hb[5] << 16, hb[6] | hb[7] << 16);
        }
      }
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

// Launches `kernel` after the previous work in `st` as a programmatic
// dependent: its prologue may overlap the tail of the previous kernel, and
// the kernel itself waits (griddepcontrol.wait) before reading that
// kernel's output.
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
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int BITS, int MT>
cudaError_t launch_bits(const DecodeParams &dp, const uint16_t *trellis, int64_t tiles_n, int64_t grid,
                        cudaStream_t st) {
  // The trellis as rows of 16-row tile strips (8-byte elements): one row is
  // every tile of one k slab; the box is one n-block's slab x kChunk rows.
  alignas(64) CUtensorMap tmap;
  const uint64_t row_elems = (uint64_t)tiles_n * 4 * BITS;
  if (!encode_tensor_map_2d(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, trellis, row_elems, (uint64_t)dp.KT,
                            row_elems * 8, 32 * BITS, DecodeCfg<BITS, MT>::kChunk, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  return launch_dependent(decode_gemm_kernel<BITS, MT>, (unsigned)grid, DecodeCfg<BITS, MT>::kWarps * 32,
                          DecodeCfg<BITS, MT>::kSmem, st, tmap, dp);
}

template <int MT>
cudaError_t launch_mt(int bits, const DecodeParams &dp, const uint16_t *trellis, int64_t tiles_n, int64_t grid,
                      cudaStream_t st) {
  switch (bits) {
    case 1: return launch_bits<1, MT>(dp, trellis, tiles_n, grid, st);
    case 2: return launch_bits<2, MT>(dp, trellis, tiles_n, grid, st);
    case 3: return launch_bits<3, MT>(dp, trellis, tiles_n, grid, st);
    case 4: return launch_bits<4, MT>(dp, trellis, tiles_n, grid, st);
    case 5: return launch_bits<5, MT>(dp, trellis, tiles_n, grid, st);
    case 6: return launch_bits<6, MT>(dp, trellis, tiles_n, grid, st);
    case 7: return launch_bits<7, MT>(dp, trellis, tiles_n, grid, st);
    case 8: return launch_bits<8, MT>(dp, trellis, tiles_n, grid, st);
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
    const int warps = mt == 1 ? dec_warps<1>() : dec_warps<2>();
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

cudaError_t init_decode_kernels(int *status) {
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

cudaError_t launch_decode_finalize(const float *partials, int64_t smax, int64_t slot_elems, const void *sv, void *y,
                                   int y_f32, int64_t n_gemm, int64_t n_valid, int rows, int64_t P, int64_t TS,
                                   int units_per_block, int all_blocks, cudaStream_t st) {
  if (!all_blocks) {
    const int64_t warps = (n_gemm / 128) * rows;
    // One warp per CTA for 1-4 rows spreads the slot loads over more SMs
    // (0.35 us less at 1 row, 0.1 us at 2, 0.25 us at 4; 8 rows measured
    // 0.1 us slower).
    const unsigned wpc = rows <= 4 ? 1u : 8u;
    return launch_dependent(decode_finalize_kernel, (unsigned)ceil_div(warps, (int64_t)wpc), 32u * wpc, (size_t)0, st,
                            partials, smax, slot_elems, static_cast<const __half *>(sv), y, y_f32, n_gemm, n_valid,
                            rows, P, TS, units_per_block, all_blocks);
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
    const unsigned grid = (unsigned)ceil_div(ceil_div(jobs, 2), 8);
    const __half *x = static_cast<const __half *>(L.x), *su = static_cast<const __half *>(L.su);
    uint8_t *xf = static_cast<uint8_t *>(L.xf);
    cudaError_t e;
    if (MT == 1)  // (a programmatic dependent measured 0.5 us slower for 9..16 rows)
      e = launch_dependent(rotate_frag_kernel<1>, grid, 256, 0, st, x, su, L.rows, K, xf);
    else {
      rotate_frag_kernel<2><<<grid, 256, 0, st>>>(x, su, L.rows, K, xf);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
  }
  // 2. stream-K decode GEMM
  DecodeParams dp;
  dp.xf = static_cast<const uint8_t *>(L.xf);
  dp.sv = static_cast<const __half *>(L.sv);
  dp.y = L.y;
  dp.partials = L.partials;
  dp.status = L.status;
  dp.n_gemm = L.n_gemm;
  dp.n_valid = L.n_valid;
  dp.KT = (int)(K / 16);
  dp.TS = (int)((L.n_gemm / 128) * dp.KT);
  dp.P = (int)L.plan.P[MT - 1];
  dp.smax = (int)L.plan.smax[MT - 1];
  dp.rows = L.rows;
  dp.m16 = 16u;
  for (int k = 0; k < 8; ++k) dp.mk[k] = 1u << k;
  dp.y_f32 = L.y_f32;
  const int64_t grid = L.plan.grid[MT - 1];
  const int64_t tiles_n = L.n_stored / 16;
  cudaError_t e = MT == 1 ? launch_mt<1>(L.bits, dp, L.trellis, tiles_n, grid, st)
                          : launch_mt<2>(L.bits, dp, L.trellis, tiles_n, grid, st);
  if (e != cudaSuccess || dp.smax == 1) return e;
  // 3. reduce the slots of n-blocks shared by several warps
  return launch_decode_finalize(L.partials, dp.smax, (int64_t)8 * MT * 128, L.sv, L.y, L.y_f32, L.n_gemm, L.n_valid,
                                L.rows, dp.P, dp.TS, dp.KT, /*all_blocks=*/0, st);
}

#if EXL3_DEBUG_BOUNDS
cudaError_t bounds_probe_decode(cudaStream_t st) { return launch_bounds_probe(st); }
#endif

}  // namespace exl3
