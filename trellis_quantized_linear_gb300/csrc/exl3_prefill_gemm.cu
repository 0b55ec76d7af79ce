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
// swizzle into a 4-stage ring; one thread issues tcgen05.mma (M=128, N=256,
// K=16, fp32 accumulation in TMEM); the accumulator is double-buffered in
// TMEM (2 x 256 columns) so the epilogue of tile i overlaps the main loop of
// tile i+1. Persistent grid, one CTA per SM.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM allocator
// and MMA issuer, warps 2..5 = epilogue (warp w reads TMEM lanes
// 32*(w%4) .. 32*(w%4)+31, i.e. one output row per thread).
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
};

// In-register orthonormal had_r_128 of one row block, then * sv, mask, store
// (rotation and sv skipped for a pre-rotated weight).
__device__ __forceinline__ void epilogue_block(float (&v)[128], const PrefillParams &p, int64_t row, int col0) {
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
      uint4 raw = __ldg(svp + a);
      const __half *h = reinterpret_cast<const __half *>(&raw);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c = 8 * a + e;
        v[c] = (col0 + c < p.n_valid_local) ? v[c] * (__half2float(h[e]) * kInvSqrt128) : -INFINITY;
      }
    }
  }
  if (row >= p.M) return;
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
  const int ntiles = p.tiles_m * p.tiles_n;
  const int kblocks = p.K / BK;

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

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
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
        tma_load_2d(a_s(stage), &tmA, full_bar(stage), kb * BK, tm * BM);
        tma_load_2d(b_s(stage), &tmB, full_bar(stage), kb * BK, tn * BN);
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
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
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
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
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
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
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

cudaError_t init_prefill_kernels() {
  if (!g_encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return cudaFuncSetAttribute(prefill_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
}

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
  const int grid = ntiles < L.num_sms ? ntiles : L.num_sms;
  prefill_gemm_kernel<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(ma, mb, p);
  return cudaGetLastError();
}

}  // namespace exl3
