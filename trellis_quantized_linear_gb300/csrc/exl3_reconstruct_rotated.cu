// Weight-side rotation variant of the reconstruct step: a slice of
//
//     W' = diag(su) . had_r_128(K) . W . had_r_128(N) . diag(sv)
//
// so that the prefill-shaped layer becomes y = x . W' with no activation or
// output rotation (the "reconstruct_had_slice" of vLLM PR #316, "[EXL3]
// dispatch prefill-shaped GEMMs to reconstruct+hgemm", section "Kernel
// measurements"). The pages give no arithmetic for it; this library defines
// it per 128 x 128 block of W, in this order, all in fp32 without contraction:
//   fp32(w); fast WHT of every column along k (stages h = 1 .. 64);
//   * fp32(su[k]); fast WHT of every row along n (same stages);
//   * 2^-7 (exact); * fp32(sv[n]); RNE to fp16.
//
// One CTA (8 warps) per block:
//   1. warp s decodes slab s (16 k-rows x 128 columns) with the per-lane
//      layout of the plain reconstruct (lane (g, q) = tile g, rows 4q..4q+3)
//      into an fp32 tile in shared memory: element (r, c) at
//      r*145 + c + 16*(r >= 64) + 16*(c >= 64), which keeps both passes below
//      free of bank conflicts (the two lanes of a pair touch rows or columns
//      64 apart);
//   2. column pass: a lane pair (l, l+16) of warp w owns column 16w + l%16,
//      64 rows each: stages h = 1 .. 32 in registers, h = 64 by one shuffle;
//   3. row pass: the same per row, after the su multiply; then 2^-7, sv, RNE
//      into an fp16 tile, copied out with 16-byte coalesced stores in the
//      requested layout.
//
// Roofline: the HBM bytes are those of the plain reconstruct (K*nc*(BITS/8+2));
// the two 128-point transforms add ~14 fp32 operations per weight.
#include "exl3_common.cuh"
#include "exl3_internal.h"

namespace exl3 {

namespace {

constexpr int RR_T = 145;                    // fp32 tile row stride (floats), = 17 mod 32
constexpr int RR_TN = 128 * RR_T + 16;       // fp32 tile size incl. the half-block skews
constexpr int RR_O = 136;                    // fp16 output tile row stride (halves; 16-byte rows)
constexpr int RR_SMEM = RR_TN * 4 + 128 * RR_O * 2;

__device__ __forceinline__ int rr_ix(int r, int c) { return r * RR_T + c + ((r >> 6) << 4) + ((c >> 6) << 4); }

// In-register unnormalised WHT of 64 values (stages h = 1 .. 32), then the
// h = 64 stage across the lane pair (l, l ^ 16): the lower half keeps a + b,
// the upper half a - b.
__device__ __forceinline__ void wht128_pair(float (&v)[64], int upper) {
#pragma unroll
  for (int h = 1; h < 64; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      if (!(i & h)) {
        const float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const float o = __shfl_xor_sync(0xffffffffu, v[i], 16);
    v[i] = upper ? __fsub_rn(o, v[i]) : __fadd_rn(v[i], o);
  }
}

// LAYOUT 0 (KN): w[k][j], ld = n_cols.  LAYOUT 1 (NK): w[j][k], ld = K.
template <int BITS, int LAYOUT>
__global__ void __launch_bounds__(256, 2) reconstruct_rotated_kernel(const uint8_t *__restrict__ trellis,
                                                                     int64_t tiles_n, int64_t nb0, int64_t nbc,
                                                                     const __half *__restrict__ su,
                                                                     const __half *__restrict__ sv, __half *w,
                                                                     int64_t K, int64_t n_cols) {
  extern __shared__ __align__(16) uint8_t rr_smem[];
  float *T = reinterpret_cast<float *>(rr_smem);
  __half *O = reinterpret_cast<__half *>(rr_smem + RR_TN * 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t kb = blockIdx.x / nbc, nb = blockIdx.x % nbc;  // 128-row block, slice-local 128-column block
  // tiles inside the CTA's shared memory; the block inside K x n_cols and
  // its sv columns inside the stored width (CTA-uniform)
  if (!EXL3_SMEM(smem_u32(rr_smem), RR_SMEM) || !EXL3_SPAN(kb * 128, 128, K) || !EXL3_SPAN(nb * 128, 128, n_cols) ||
      !EXL3_SPAN((nb0 + nb) * 128, 128, tiles_n * 16))
    return;

  // 1. decode slab `warp` of the block
  {
    const int g = lane >> 2, q = lane & 3;
    const int64_t tk = kb * 8 + warp;
    const uint8_t *src = trellis + ((tk * tiles_n + (nb0 + nb) * 8) * (32 * BITS)) + lane * 8 * BITS;
    uint32_t own[2 * BITS];
    if (EXL3_RANGE(warp, 0, 8)) {  // slab kb * 8 + warp of the block's 8
      load_own_words<BITS, false>(src, own);
    } else {
#pragma unroll
      for (int i = 0; i < 2 * BITS; ++i) own[i] = 0;
    }
    const uint32_t prev = prefix_from_neighbour<BITS>(own, lane);
    RowWindows<BITS> rw;
    rw.build(own, prev);
    static_for<4>([&](auto R) {
      float *row = T + rr_ix(16 * warp + 4 * q + R.value, 16 * g);  // 16 columns in one half
      if (!EXL3_SPAN(rr_ix(16 * warp + 4 * q + R.value, 16 * g), 16, RR_TN)) return;
      static_for<8>([&](auto C2) {
        const uint32_t p2 = decode_pair(rw.template state<R.value, 2 * C2.value>(),
                                        rw.template state<R.value, 2 * C2.value + 1>());
        const __half2 h2 = *reinterpret_cast<const __half2 *>(&p2);
        row[2 * C2.value] = __low2float(h2);
        row[2 * C2.value + 1] = __high2float(h2);
      });
    });
  }
  __syncthreads();

  const int upper = lane >> 4;
  const int idx = 16 * warp + (lane & 15);  // column (pass 2) / row (pass 3) of this lane pair
  // 2. column pass along k (the lane's 64 tile entries lie between its first
  // and last, rr_ix being monotonic in each index)
  const bool col_ok = EXL3_RANGE(rr_ix(64 * upper, idx), 0, RR_TN) && EXL3_RANGE(rr_ix(64 * upper + 63, idx), 0, RR_TN);
  const bool row_ok = EXL3_RANGE(rr_ix(idx, 64 * upper), 0, RR_TN) && EXL3_RANGE(rr_ix(idx, 64 * upper + 63), 0, RR_TN);
  {
    float v[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = col_ok ? T[rr_ix(64 * upper + i, idx)] : 0.f;
    wht128_pair(v, upper);
#pragma unroll
    for (int i = 0; i < 64; ++i)
      if (col_ok) T[rr_ix(64 * upper + i, idx)] = v[i];
  }
  __syncthreads();
  // 3. row pass along n, then scale and round
  {
    const float s = __half2float(su[kb * 128 + idx]);
    float v[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = row_ok ? __fmul_rn(T[rr_ix(idx, 64 * upper + i)], s) : 0.f;
    wht128_pair(v, upper);
    const __half *svb = sv + nb0 * 128 + nb * 128 + 64 * upper;
#pragma unroll
    for (int i = 0; i < 64; i += 2) {
      const float a = __fmul_rn(__fmul_rn(v[i], 0.0078125f), __half2float(svb[i]));
      const float b = __fmul_rn(__fmul_rn(v[i + 1], 0.0078125f), __half2float(svb[i + 1]));
      if (LAYOUT == 0) {
        if (EXL3_SPAN(idx * RR_O + 64 * upper + i, 2, 128 * RR_O))
          *reinterpret_cast<__half2 *>(O + idx * RR_O + 64 * upper + i) = __floats2half2_rn(a, b);
      } else if (EXL3_RANGE((64 * upper + i + 1) * RR_O + idx, 0, 128 * RR_O)) {
        O[(64 * upper + i) * RR_O + idx] = __float2half_rn(a);
        O[(64 * upper + i + 1) * RR_O + idx] = __float2half_rn(b);
      }
    }
  }
  __syncthreads();
  // 4. copy out: 128 rows of 256 bytes, 16 bytes per thread per step
  for (int e = threadIdx.x; e < 128 * 16; e += blockDim.x) {
    const int r = e >> 4, c = (e & 15) * 8;
    if (!EXL3_SPAN(r * RR_O + c, 8, 128 * RR_O)) continue;
    const uint4 val = *reinterpret_cast<const uint4 *>(O + r * RR_O + c);
    if (LAYOUT == 0)
      *reinterpret_cast<uint4 *>(w + (kb * 128 + r) * n_cols + nb * 128 + c) = val;
    else
      *reinterpret_cast<uint4 *>(w + (nb * 128 + r) * K + kb * 128 + c) = val;
  }
}

template <int BITS>
cudaError_t init_bits() {
  cudaError_t e = cudaFuncSetAttribute(reconstruct_rotated_kernel<BITS, 0>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, RR_SMEM);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(reconstruct_rotated_kernel<BITS, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              RR_SMEM);
}

template <int BITS>
void launch_bits(const uint8_t *t, int64_t tiles_n, int64_t nb0, int64_t nbc, const __half *su, const __half *sv,
                 __half *w, int64_t K, int64_t n_cols, int layout, unsigned grid, cudaStream_t st) {
  if (layout == 0)
    reconstruct_rotated_kernel<BITS, 0><<<grid, 256, RR_SMEM, st>>>(t, tiles_n, nb0, nbc, su, sv, w, K, n_cols);
  else
    reconstruct_rotated_kernel<BITS, 1><<<grid, 256, RR_SMEM, st>>>(t, tiles_n, nb0, nbc, su, sv, w, K, n_cols);
}

}  // namespace

cudaError_t init_reconstruct_rotated_kernels(int *status) {
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

cudaError_t launch_reconstruct_rotated(const uint16_t *trellis, int bits, int64_t K, int64_t n_stored, int64_t n0,
                                       int64_t n_cols, const void *su, const void *sv, void *w, int layout,
                                       cudaStream_t st) {
  const int64_t nbc = n_cols / 128, blocks = (K / 128) * nbc;
  if (blocks == 0) return cudaSuccess;
  const uint8_t *t = reinterpret_cast<const uint8_t *>(trellis);
  const __half *s_u = static_cast<const __half *>(su), *s_v = static_cast<const __half *>(sv);
  __half *wp = static_cast<__half *>(w);
  const int64_t tiles_n = n_stored / 16, nb0 = n0 / 128;
  const unsigned grid = (unsigned)blocks;
  switch (bits) {
    case 1: launch_bits<1>(t, tiles_n, nb0, nbc, s_u, s_v, wp, K, n_cols, layout, grid, st); break;
    case 2: launch_bits<2>(t, tiles_n, nb0, nbc, s_u, s_v, wp, K, n_cols, layout, grid, st); break;
    case 3: launch_bits<3>(t, tiles_n, nb0, nbc, s_u, s_v, wp, K, n_cols, layout, grid, st); break;
    case 4: launch_bits<4>(t, tiles_n, nb0, nbc, s_u, s_v, wp, K, n_cols, layout, grid, st); break;
    case 5: launch_bits<5>(t, tiles_n, nb0, nbc, s_u, s_v, wp, K, n_cols, layout, grid, st); break;
    case 6: launch_bits<6>(t, tiles_n, nb0, nbc, s_u, s_v, wp, K, n_cols, layout, grid, st); break;
    case 7: launch_bits<7>(t, tiles_n, nb0, nbc, s_u, s_v, wp, K, n_cols, layout, grid, st); break;
    case 8: launch_bits<8>(t, tiles_n, nb0, nbc, s_u, s_v, wp, K, n_cols, layout, grid, st); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

#if EXL3_DEBUG_BOUNDS
cudaError_t bounds_probe_reconstruct_rotated(cudaStream_t st) { return launch_bounds_probe(st); }
#endif

}  // namespace exl3
