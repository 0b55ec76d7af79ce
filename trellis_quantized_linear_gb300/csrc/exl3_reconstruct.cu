// Trellis -> dense fp16 weight slice ("reconstruct" / "reconstruct_slice" of
// vLLM PR #316, "[EXL3] dispatch prefill-shaped GEMMs to reconstruct+hgemm",
// sections "Kernel measurements" and "Change").
//
// Work unit: one slab = 16 k-rows x 128 columns = 8 horizontally adjacent
// tiles, whose 8*32*BITS bitstream bytes are contiguous in the trellis. Lane
// (g, q) = (lane/4, lane%4) owns tile g, rows 4q..4q+3: it loads its own
// 8*BITS bytes at byte offset lane*8*BITS (one fully coalesced warp load),
// takes the word preceding them from its neighbour lane, and decodes its 64
// weights from registers.
//
// Roofline: HBM-bound. Algorithmic bytes per weight = BITS/8 read + 2 written
// (measured 5.7-5.8 TB/s for the gate and down geometries). The decode
// arithmetic keeps the half-rate integer pipe busy as well, so decoded
// pairs are packed on the fp16 pipe (exact: a decoded weight is never -0,
// so adding a signed zero leaves it unchanged): 1-3 % faster than a byte
// permute; the nibble-shifted window copies measured slower here.
#include "exl3_common.cuh"
#include "exl3_internal.h"

namespace exl3 {

// LAYOUT 0 (KN): w[k][j], ld = n_cols.  LAYOUT 1 (NK): w[j][k], ld = K.
// With `overlap` set the kernel was launched as a programmatic dependent of
// the input rotation (which neither reads nor writes its operands): it runs
// alongside it and only waits for it before exiting, so that the GEMM queued
// after this kernel sees both finished.
template <int BITS, int LAYOUT>
__global__ void __launch_bounds__(256) reconstruct_kernel(const uint8_t *__restrict__ trellis,
                                                          int64_t tiles_n, int64_t tk_count,
                                                          int64_t nb0, int64_t nbc, __half *w,
                                                          int64_t K, int64_t n_cols, int overlap) {
  constexpr int kTileBytes = 32 * BITS;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t nslabs = tk_count * nbc;
  for (int64_t s = warp; s < nslabs; s += nwarps) {
    int64_t tk, nb;
    if (LAYOUT == 0) {
      tk = s / nbc;
      nb = s % nbc;
    } else {
      tk = s % tk_count;
      nb = s / tk_count;
    }
    const uint8_t *src = trellis + ((tk * tiles_n + (nb0 + nb) * 8) * kTileBytes) + lane * 8 * BITS;
    uint32_t own[2 * BITS];
    // the slab's 8 tiles: tile row tk of tk_count, tiles [8 (nb0 + nb), +8) of tiles_n
    if (EXL3_RANGE(tk, 0, tk_count) && EXL3_SPAN((nb0 + nb) * 8, 8, tiles_n)) {
      load_own_words<BITS, false>(src, own);
    } else {
#pragma unroll
      for (int i = 0; i < 2 * BITS; ++i) own[i] = 0;
    }
    const uint32_t prev = prefix_from_neighbour<BITS>(own, lane);
    RowWindows<BITS> rw;
    rw.build(own, prev);
    auto pair = [&](uint32_t sa, uint32_t sb) { return decode_pair_sel<true>(sa, sb); };
    const int64_t k0 = tk * 16 + 4 * q;      // first of this lane's 4 rows
    const int64_t j0 = nb * 128 + 16 * g;    // first column of this lane's tile (slice-local)
    if (!EXL3_SPAN(k0, 4, K) || !EXL3_SPAN(j0, 16, n_cols)) continue;  // the lane's 4 x 16 block of w
    if (LAYOUT == 0) {
      static_for<4>([&](auto R) {
        uint32_t p[8];
        static_for<8>([&](auto C2) {
          p[C2.value] = pair(rw.template state<R.value, 2 * C2.value>(), rw.template state<R.value, 2 * C2.value + 1>());
        });
        uint4 *dst = reinterpret_cast<uint4 *>(w + (k0 + R.value) * n_cols + j0);
        dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
        dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
      });
    } else {
      static_for<16>([&](auto C) {
        uint32_t lo = pair(rw.template state<0, C.value>(), rw.template state<1, C.value>());
        uint32_t hi = pair(rw.template state<2, C.value>(), rw.template state<3, C.value>());
        *reinterpret_cast<uint2 *>(w + (j0 + C.value) * K + k0) = make_uint2(lo, hi);
      });
    }
  }
  if (overlap) asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int BITS>
static cudaError_t init_bits() {
  cudaFuncAttributes a;
  cudaError_t e = cudaFuncGetAttributes(&a, reconstruct_kernel<BITS, 0>);
  if (e != cudaSuccess) return e;
  return cudaFuncGetAttributes(&a, reconstruct_kernel<BITS, 1>);
}

cudaError_t init_reconstruct_kernels(int *status) {
  cudaError_t e = EXL3_BIND_BOUNDS_WORD(status);
  if (e != cudaSuccess) return e;
  if ((e = init_bits<1>()) != cudaSuccess) return e;
  if ((e = init_bits<7>()) != cudaSuccess) return e;
  if ((e = init_bits<2>()) != cudaSuccess) return e;
  if ((e = init_bits<3>()) != cudaSuccess) return e;
  if ((e = init_bits<4>()) != cudaSuccess) return e;
  if ((e = init_bits<5>()) != cudaSuccess) return e;
  if ((e = init_bits<6>()) != cudaSuccess) return e;
  return init_bits<8>();
}

template <int BITS, int LAYOUT>
static cudaError_t launch_one(const uint8_t *t, int64_t tiles_n, int64_t tkc, int64_t nb0, int64_t nbc,
                              __half *w, int64_t K, int64_t n_cols, unsigned grid, int overlap, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, reconstruct_kernel<BITS, LAYOUT>, t, tiles_n, tkc, nb0, nbc, w, K, n_cols,
                            overlap);
}

template <int BITS>
static cudaError_t launch_bits(const uint8_t *t, int64_t tiles_n, int64_t tkc, int64_t nb0, int64_t nbc,
                               __half *w, int64_t K, int64_t n_cols, int layout, unsigned grid, int overlap,
                               cudaStream_t st) {
  return layout == 0 ? launch_one<BITS, 0>(t, tiles_n, tkc, nb0, nbc, w, K, n_cols, grid, overlap, st)
                     : launch_one<BITS, 1>(t, tiles_n, tkc, nb0, nbc, w, K, n_cols, grid, overlap, st);
}

cudaError_t launch_reconstruct(const uint16_t *trellis, int bits, int64_t K, int64_t n_stored,
                               int64_t n0, int64_t n_cols, void *w, int layout, int num_sms,
                               cudaStream_t st, int overlap) {
  const int64_t tkc = K / 16, nbc = n_cols / 128;
  const int64_t slabs = tkc * nbc;
  if (slabs == 0) return cudaSuccess;
  int64_t grid = ceil_div(slabs, 8);
  const int64_t cap = (int64_t)num_sms * 8;
  if (grid > cap) grid = cap;
  const uint8_t *t = reinterpret_cast<const uint8_t *>(trellis);
  __half *wp = static_cast<__half *>(w);
  const int64_t tiles_n = n_stored / 16, nb0 = n0 / 128;
  switch (bits) {
    case 1: return launch_bits<1>(t, tiles_n, tkc, nb0, nbc, wp, K, n_cols, layout, (unsigned)grid, overlap, st);
    case 2: return launch_bits<2>(t, tiles_n, tkc, nb0, nbc, wp, K, n_cols, layout, (unsigned)grid, overlap, st);
    case 3: return launch_bits<3>(t, tiles_n, tkc, nb0, nbc, wp, K, n_cols, layout, (unsigned)grid, overlap, st);
    case 4: return launch_bits<4>(t, tiles_n, tkc, nb0, nbc, wp, K, n_cols, layout, (unsigned)grid, overlap, st);
    case 5: return launch_bits<5>(t, tiles_n, tkc, nb0, nbc, wp, K, n_cols, layout, (unsigned)grid, overlap, st);
    case 6: return launch_bits<6>(t, tiles_n, tkc, nb0, nbc, wp, K, n_cols, layout, (unsigned)grid, overlap, st);
    case 7: return launch_bits<7>(t, tiles_n, tkc, nb0, nbc, wp, K, n_cols, layout, (unsigned)grid, overlap, st);
    case 8: return launch_bits<8>(t, tiles_n, tkc, nb0, nbc, wp, K, n_cols, layout, (unsigned)grid, overlap, st);
    default: return cudaErrorInvalidValue;
  }
}

#if EXL3_DEBUG_BOUNDS
cudaError_t bounds_probe_reconstruct(cudaStream_t st) { return launch_bounds_probe(st); }
#endif

}  // namespace exl3
