// Decode-shaped trellis linear: one fused kernel per <= 16 activation rows.
//
// The fused decode-inside-GEMM path of vLLM PR #316, "[EXL3] dispatch
// prefill-shaped GEMMs to reconstruct+hgemm" (sections "Problem" and
// "Change": the op keeps its decode-shaped kernel below the M threshold),
// rebuilt for sm_103a. Each weight is decoded exactly once per launch.
//
// Structure of a CTA (1 producer warp + 8 consumer warps, 1 CTA per SM):
//   * the CTA owns one K split [kb0, kb1) (in 128-row blocks) and the
//     n-blocks gs, gs+Gs, ... (128 output columns each); each consumer warp
//     owns one n-block at a time and walks the whole K split;
//   * prologue: the consumer warps rotate their K slice of x,
//     x' = RNE_fp16(had_r_128(x * su)), into shared memory, already laid out
//     as mma.sync A fragments;
//   * producer: one lane streams each warp's 16 x 128 slab of bitstreams
//     (8 tiles, 256*BITS contiguous bytes) into a shared-memory ring with
//     cp.async.bulk, one mbarrier pair per stage;
//   * consumer lane (g, q) decodes tile g rows 4q..4q+3 straight into
//     m16n8k16 B fragments: the mma's k index 2q, 2q+1, 2q+8, 2q+9 is mapped
//     to tile rows 4q .. 4q+3 (the same permutation is applied to x'), and
//     mma j's column g to tile column 16g + j; after 16 mmas per slab the
//     lane holds output columns 32q .. 32q+31 of rows g and g+8;
//   * epilogue: with one K split the warp finishes the n-block itself; with
//     several, it stores an fp32 partial, and the last warp to arrive on the
//     n-block's counter sums the partials in split order (deterministic),
//     applies had_r_128 over the 128 columns and sv, masks columns >= n_valid
//     to -inf and writes y; it then resets the counter.
//
// Roofline: HBM-bound on the trellis bytes (K*N*BITS/8 per launch); the
// per-weight integer decode is the competing ALU bound.
#include <math.h>

#include "exl3_common.cuh"
#include "exl3_internal.h"

namespace exl3 {

namespace {

constexpr int NC = kDecodeConsumerWarps;

template <int BITS>
struct DecodeCfg {
  static constexpr int kSeg = 256 * BITS;                 // bytes of one 16x128 slab
  static constexpr int kStages = BITS <= 4 ? 8 : 6;
  static constexpr int kRingBytes = kStages * NC * kSeg;
};

struct DecodeParams {
  const __half *x;
  const uint8_t *trellis;
  const __half *su;
  const __half *sv;
  void *y;
  float *partials;
  int *counters;
  int *status;
  int64_t K, tiles_n, n_gemm, n_valid;
  int rows, y_f32, NB, KB, S, Gs;
};

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Output rotation + sv + mask + store of one 128-column block held as
// v[rr][c] = row (g + 8 rr), column 32q + c, by lane (g, q).
__device__ __forceinline__ void finish_block(float (&v)[2][32], const DecodeParams &p, int nb, int lane) {
  const int g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (!(i & h)) {
          float a = v[rr][i], b = v[rr][i + h];
          v[rr][i] = a + b;
          v[rr][i + h] = a - b;
        }
      }
    }
#pragma unroll
    for (int s = 1; s < 4; s <<= 1) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float o = __shfl_xor_sync(0xffffffffu, v[rr][i], s);
        v[rr][i] = (q & s) ? (o - v[rr][i]) : (v[rr][i] + o);
      }
    }
  }
  const int64_t col0 = (int64_t)nb * 128 + 32 * q;
  float scale[32];
  {
    const uint4 *svp = reinterpret_cast<const uint4 *>(p.sv + col0);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      uint4 raw = __ldg(svp + a);
      const __half *h = reinterpret_cast<const __half *>(&raw);
#pragma unroll
      for (int e = 0; e < 8; ++e) scale[8 * a + e] = __half2float(h[e]) * kInvSqrt128;
    }
  }
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int m = g + 8 * rr;
    float o[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      o[c] = (col0 + c < p.n_valid) ? v[rr][c] * scale[c] : -INFINITY;
    }
    if (m < p.rows) {
      if (p.y_f32) {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.y) + (int64_t)m * p.n_gemm + col0);
#pragma unroll
        for (int a = 0; a < 8; ++a) dst[a] = make_float4(o[4 * a], o[4 * a + 1], o[4 * a + 2], o[4 * a + 3]);
      } else {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__half *>(p.y) + (int64_t)m * p.n_gemm + col0);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
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

template <int BITS, int MROWS>
__global__ void __launch_bounds__(32 * (1 + NC), 1) decode_gemm_kernel(const DecodeParams p) {
  using Cfg = DecodeCfg<BITS>;
  constexpr int kSeg = Cfg::kSeg;
  constexpr int kStages = Cfg::kStages;
  constexpr int CH = MROWS == 16 ? 8 : 4;  // fp16 A-fragment values per lane per k16 step
  extern __shared__ __align__(1024) uint8_t smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = blockIdx.x % p.S, gs = blockIdx.x / p.S;
  const int kb0 = (int)((int64_t)ks * p.KB / p.S), kb1 = (int)((int64_t)(ks + 1) * p.KB / p.S);
  const int nkb = kb1 - kb0;
  const int T = nkb * 8;  // 16-row slabs in this K split
  const int count = (p.NB - gs + p.Gs - 1) / p.Gs;
  const int rounds = (count + NC - 1) / NC;
  const int tmax = ((p.KB + p.S - 1) / p.S) * 8;

  __half *xs = reinterpret_cast<__half *>(smem);
  uint8_t *ring = smem + align1024(tmax * 32 * CH * 2);
  uint64_t *bars = reinterpret_cast<uint64_t *>(ring + Cfg::kRingBytes);
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[kStages + s]); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), NC);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      const uint32_t ring_s = smem_u32(ring);
      for (int r = 0; r < rounds && ok; ++r) {
        const int nvalid = min(NC, count - r * NC);
        for (int t = 0; t < T; ++t) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), (uint32_t)(nvalid * kSeg));
          const int64_t tk = (int64_t)kb0 * 8 + t;
          for (int w = 0; w < nvalid; ++w) {
            const int64_t nb = gs + (int64_t)(r * NC + w) * p.Gs;
            const uint8_t *src = p.trellis + (tk * p.tiles_n + nb * 8) * (32 * BITS);
            bulk_g2s(ring_s + (uint32_t)((stage * NC + w) * kSeg), src, kSeg, full_bar(stage));
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every issued copy must land before the CTA may retire.
      for (int s = 0; s < kStages; ++s) {
        const int64_t uses = issued / kStages + (s < issued % kStages ? 1 : 0);
        if (uses > 0) mbar_wait_short(full_bar(s), (uint32_t)((uses - 1) & 1));
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  const int cw = warp - 1;
  const int g = lane >> 2, q = lane & 3;

  // Prologue: x' = RNE_fp16(had_r_128(x * su)) for this K split, stored so
  // that lane (g, q) of k16 step t finds {x'[g][4q..4q+3], x'[g+8][4q..4q+3]}
  // at xs[(t*32 + lane)*CH].
  {
    const int l16 = lane & 15;
    const int jobs = MROWS * nkb;
    for (int jp = cw; jp * 2 < jobs; jp += NC) {
      const int job = jp * 2 + (lane >> 4);
      const bool valid = job < jobs;
      const int m = valid ? job / nkb : 0;
      const int kbl = valid ? job % nkb : 0;
      float v[8];
      if (valid && m < p.rows) {
        const int64_t kofs = (int64_t)(kb0 + kbl) * 128 + 8 * l16;
        uint4 raw = __ldg(reinterpret_cast<const uint4 *>(p.x + (int64_t)m * p.K + kofs));
        uint4 sraw = __ldg(reinterpret_cast<const uint4 *>(p.su + kofs));
        const __half *h = reinterpret_cast<const __half *>(&raw);
        const __half *sh = reinterpret_cast<const __half *>(&sraw);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __half2float(h[i]) * __half2float(sh[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
      }
#pragma unroll
      for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (!(i & h)) {
            float a = v[i], b = v[i + h];
            v[i] = a + b;
            v[i + h] = a - b;
          }
        }
      }
#pragma unroll
      for (int s = 1; s < 16; s <<= 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float o = __shfl_xor_sync(0xffffffffu, v[i], s);
          v[i] = (l16 & s) ? (o - v[i]) : (v[i] + o);
        }
      }
      if (valid) {
        __half2 hv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) hv[e] = __floats2half2_rn(v[2 * e] * kInvSqrt128, v[2 * e + 1] * kInvSqrt128);
        const int t = kbl * 8 + (l16 >> 1);
        const int qq = 2 * (l16 & 1);
        const int gg = m & 7;
        const int off = (m >= 8) ? 4 : 0;
        __half *d0 = xs + (size_t)(t * 32 + gg * 4 + qq) * CH + off;
        __half *d1 = xs + (size_t)(t * 32 + gg * 4 + qq + 1) * CH + off;
        *reinterpret_cast<uint2 *>(d0) = make_uint2(*reinterpret_cast<uint32_t *>(&hv[0]),
                                                    *reinterpret_cast<uint32_t *>(&hv[1]));
        *reinterpret_cast<uint2 *>(d1) = make_uint2(*reinterpret_cast<uint32_t *>(&hv[2]),
                                                    *reinterpret_cast<uint32_t *>(&hv[3]));
      }
    }
  }
  named_bar_sync(1, NC * 32);

  int stage = 0;
  uint32_t phase = 0;
  for (int r = 0; r < rounds; ++r) {
    const int i = r * NC + cw;
    const bool valid = i < count;
    const int nb = gs + i * p.Gs;
    float acc[16][4];
#pragma unroll
    for (int c = 0; c < 16; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;

    for (int t = 0; t < T; ++t) {
      if (!mbar_wait(full_bar(stage), phase, p.status)) return;
      if (valid) {
        uint32_t own[2 * BITS];
        load_own_words<BITS, true>(ring + (stage * NC + cw) * kSeg + lane * 8 * BITS, own);
        const uint32_t prev = prefix_from_neighbour<BITS>(own, lane);
        RowWindows<BITS> rw;
        rw.build(own, prev);
        uint32_t a0, a1, a2, a3;
        if constexpr (MROWS == 16) {
          uint4 av = *reinterpret_cast<const uint4 *>(xs + (size_t)(t * 32 + lane) * CH);
          a0 = av.x; a2 = av.y; a1 = av.z; a3 = av.w;
        } else {
          uint2 av = *reinterpret_cast<const uint2 *>(xs + (size_t)(t * 32 + lane) * CH);
          a0 = av.x; a2 = av.y; a1 = 0u; a3 = 0u;
        }
        static_for<16>([&](auto C) {
          const uint32_t b0 = decode_pair(rw.template state<0, C.value>(), rw.template state<1, C.value>());
          const uint32_t b1 = decode_pair(rw.template state<2, C.value>(), rw.template state<3, C.value>());
          mma16816(acc[C.value], a0, a1, a2, a3, b0, b1);
        });
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(stage));
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!valid) continue;

    float v[2][32];
    if (p.S == 1) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          v[rr][c] = acc[c][2 * rr];
          v[rr][c + 16] = acc[c][2 * rr + 1];
        }
      finish_block(v, p, nb, lane);
      continue;
    }
    // Split K: publish this split's partial, then let the last arrival finish.
    {
      float *part = p.partials + (int64_t)ks * 16 * p.n_gemm + (int64_t)nb * 128 + 32 * q;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int m = g + 8 * rr;
        if (m < p.rows) {
          float4 *dst = reinterpret_cast<float4 *>(part + (int64_t)m * p.n_gemm);
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            dst[a] = make_float4(acc[4 * a][2 * rr], acc[4 * a + 1][2 * rr], acc[4 * a + 2][2 * rr],
                                 acc[4 * a + 3][2 * rr]);
            dst[a + 4] = make_float4(acc[4 * a][2 * rr + 1], acc[4 * a + 1][2 * rr + 1],
                                     acc[4 * a + 2][2 * rr + 1], acc[4 * a + 3][2 * rr + 1]);
          }
        }
      }
    }
    __threadfence();
    __syncwarp();
    int old = 0;
    if (lane == 0) old = atomicAdd(&p.counters[nb], 1);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old != p.S - 1) continue;
    __threadfence();
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
      for (int c = 0; c < 32; ++c) v[rr][c] = 0.f;
    for (int s = 0; s < p.S; ++s) {
      const float *part = p.partials + (int64_t)s * 16 * p.n_gemm + (int64_t)nb * 128 + 32 * q;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int m = g + 8 * rr;
        if (m < p.rows) {
          const float4 *src = reinterpret_cast<const float4 *>(part + (int64_t)m * p.n_gemm);
#pragma unroll
          for (int a = 0; a < 8; ++a) {
            float4 f = __ldcg(src + a);
            v[rr][4 * a] += f.x;
            v[rr][4 * a + 1] += f.y;
            v[rr][4 * a + 2] += f.z;
            v[rr][4 * a + 3] += f.w;
          }
        }
      }
    }
    finish_block(v, p, nb, lane);
    if (lane == 0) atomicExch(&p.counters[nb], 0);
  }
}

template <int BITS, int MROWS>
size_t smem_bytes_for(int tmax) {
  constexpr int CH = MROWS == 16 ? 8 : 4;
  return (size_t)align1024(tmax * 32 * CH * 2) + DecodeCfg<BITS>::kRingBytes +
         2 * DecodeCfg<BITS>::kStages * sizeof(uint64_t);
}

template <int BITS, int MROWS>
cudaError_t init_one() {
  const int tmax = (kDecodeMaxKSplit / 16);
  return cudaFuncSetAttribute(decode_gemm_kernel<BITS, MROWS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_bytes_for<BITS, MROWS>(tmax));
}

template <int BITS>
cudaError_t init_bits() {
  cudaError_t e = init_one<BITS, 8>();
  if (e != cudaSuccess) return e;
  return init_one<BITS, 16>();
}

template <int BITS>
cudaError_t launch_bits(const DecodeParams &dp, int tmax, cudaStream_t st) {
  const unsigned grid = (unsigned)(dp.S * dp.Gs);
  if (dp.rows <= 8) {
    decode_gemm_kernel<BITS, 8><<<grid, 32 * (1 + NC), smem_bytes_for<BITS, 8>(tmax), st>>>(dp);
  } else {
    decode_gemm_kernel<BITS, 16><<<grid, 32 * (1 + NC), smem_bytes_for<BITS, 16>(tmax), st>>>(dp);
  }
  return cudaGetLastError();
}

}  // namespace

DecodePlan decode_plan(int64_t n_blocks, int64_t k_blocks, int num_sms) {
  DecodePlan best;
  int64_t best_cost = -1, best_grid = 0;
  const int64_t s_min = ceil_div(k_blocks, kDecodeMaxKSplit / 128);
  const int64_t s_max = k_blocks < 64 ? k_blocks : 64;
  for (int64_t S = s_min; S <= s_max; ++S) {
    if (S > num_sms) break;
    const int64_t gs_max = n_blocks < num_sms / S ? n_blocks : num_sms / S;
    for (int64_t Gs = 1; Gs <= gs_max; ++Gs) {
      const int64_t rounds = ceil_div(ceil_div(n_blocks, Gs), NC);
      const int64_t cost = rounds * ceil_div(k_blocks, S);
      const int64_t grid = S * Gs;
      if (best_cost < 0 || cost < best_cost || (cost == best_cost && grid > best_grid && S == best.S)) {
        best_cost = cost;
        best_grid = grid;
        best.S = (int)S;
        best.Gs = (int)Gs;
      }
    }
  }
  return best;
}

cudaError_t init_decode_kernels() {
  cudaError_t e;
  if ((e = init_bits<2>()) != cudaSuccess) return e;
  if ((e = init_bits<3>()) != cudaSuccess) return e;
  if ((e = init_bits<4>()) != cudaSuccess) return e;
  if ((e = init_bits<5>()) != cudaSuccess) return e;
  if ((e = init_bits<6>()) != cudaSuccess) return e;
  return init_bits<8>();
}

cudaError_t launch_decode_gemm(const DecodeLaunch &L, cudaStream_t st) {
  DecodeParams dp;
  dp.x = static_cast<const __half *>(L.x);
  dp.trellis = reinterpret_cast<const uint8_t *>(L.trellis);
  dp.su = static_cast<const __half *>(L.su);
  dp.sv = static_cast<const __half *>(L.sv);
  dp.y = L.y;
  dp.partials = L.partials;
  dp.counters = L.counters;
  dp.status = L.status;
  dp.K = L.K;
  dp.tiles_n = L.n_stored / 16;
  dp.n_gemm = L.n_gemm;
  dp.n_valid = L.n_valid;
  dp.rows = L.rows;
  dp.y_f32 = L.y_f32;
  dp.NB = (int)(L.n_gemm / 128);
  dp.KB = (int)(L.K / 128);
  dp.S = L.plan.S;
  dp.Gs = L.plan.Gs;
  const int tmax = (int)ceil_div(dp.KB, dp.S) * 8;
  switch (L.bits) {
    case 2: return launch_bits<2>(dp, tmax, st);
    case 3: return launch_bits<3>(dp, tmax, st);
    case 4: return launch_bits<4>(dp, tmax, st);
    case 5: return launch_bits<5>(dp, tmax, st);
    case 6: return launch_bits<6>(dp, tmax, st);
    case 8: return launch_bits<8>(dp, tmax, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace exl3
