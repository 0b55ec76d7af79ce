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
// SM. Per k step:
//   * warp 0 (one lane): TMA loads of x' (M x 64, 128-byte swizzle, one
//     128-row tile per 128 rows);
//   * warps 2..17 (decoders): four groups of four; group j decodes the four
//     16-row slabs of k steps j, j+4, ...; each warp
//     streams its slab's 8 trellis tiles through a private bulk-copy ring,
//     decodes lane (g, q) = tile g, rows 4q..4q+3, and stores W^T into the
//     B operand: K-major, no swizzle, 8x16-byte core matrices with strides
//     chosen so the warp's 8-byte stores hit distinct banks;
//   * warp 1 (one lane): tcgen05.mma M=128 N=128 K=16 per 128-row tile into a
//     double-buffered TMEM accumulator;
//   * warps 18..21 (epilogue): when a CTA's part of an n-block is done they
//     stream TMEM (one row per thread) into an fp32 partial slot; the decode
//     finalize kernel sums each n-block's slots in slot order and applies
//     had_r_128, sv and the -inf mask.
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
constexpr int F_SB = F_GROUPS + 1, F_RD = 2;  // B stages, trellis stages per decoder warp
constexpr int F_LBO = 144;                   // bytes between B core matrices along K
constexpr int F_SBO = 1168;                  // bytes between B 8-row groups along N
constexpr int F_B_STAGE = 16 * F_SBO;        // one 128 x 64 fp16 B tile with padding
constexpr int F_A_TILE = 128 * F_BK * 2;     // one 128 x 64 fp16 x' tile (128-byte swizzle)

template <int BITS, int MTILES>
struct FusedCfg {
  static constexpr int kSA = MTILES == 1 ? 4 : 2;  // x' stages
  static constexpr int kSeg = 256 * BITS;
  static constexpr int kAStage = MTILES * F_A_TILE;
  static constexpr int kOffB = kSA * kAStage;
  static constexpr int kOffD = kOffB + F_SB * F_B_STAGE;
  static constexpr int kOffBar = kOffD + F_DEC_WARPS * F_RD * kSeg;
  static constexpr int kNumBars = 2 * kSA + 2 * F_SB + 4 + 1 + F_DEC_WARPS * F_RD;
  static constexpr int kSmem = 1024 + kOffBar + kNumBars * 8 + 16;
  static constexpr int kTmemCols = MTILES == 1 ? 256 : 512;  // 2 buffers x MTILES x 128 columns
  static_assert(kOffB % 1024 == 0, "x' stages must stay 1024-byte aligned");
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
};

__device__ __forceinline__ int64_t unit_owner(int64_t z, int64_t P, int64_t TS) { return ((z + 1) * P - 1) / TS; }

__device__ __forceinline__ void wait_prior_grid_f() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_next_grid_f() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <int BITS, int MTILES>
__global__ void __launch_bounds__(F_THREADS, 1)
    fused_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const FusedParams p) {
  using Cfg = FusedCfg<BITS, MTILES>;
  constexpr int F_SA = Cfg::kSA;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
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

  if (threadIdx.x == 0) {
    for (int s = 0; s < F_SA; ++s) {
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
                 "r"(Cfg::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  allow_next_grid_f();

  if (warp == 0 && lane == 0) {
    // ---------------- x' producer ----------------
    wait_prior_grid_f();  // x' comes from the rotation kernel
    int64_t issued = 0;
    for (int kk = 0; kk < len; ++kk) {
      const int ks = (int)((zs + kk) % KS);
      const int as = kk % F_SA;
      const uint32_t ua = (uint32_t)(kk / F_SA);
      if (!mbar_wait(a_empty(as), (ua & 1u) ^ 1u, p.status)) break;
      mbar_arrive_expect_tx(a_full(as), Cfg::kAStage);
#pragma unroll
      for (int mt = 0; mt < MTILES; ++mt)
        tma_load_2d(smem_s + as * Cfg::kAStage + mt * F_A_TILE, &tmA, a_full(as), ks * F_BK, mt * 128);
      ++issued;
    }
    for (int s = 0; s < F_SA; ++s) {
      const int64_t uses = issued / F_SA + (s < issued % F_SA ? 1 : 0);
      if (uses > 0) mbar_wait_short(a_full(s), (uint32_t)((uses - 1) & 1));
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = f16_idesc(128, F_BN);
    int seg = 0;
    bool ok = true;
    for (int kk = 0; kk < len && ok; ++kk) {
      const int ks = (int)((zs + kk) % KS);
      const bool first = (kk == 0) || (ks == 0);
      const bool last = (kk == len - 1) || (ks == KS - 1);
      const int ab = seg & 1;
      if (first) {
        if (!mbar_wait(acc_empty(ab), ((uint32_t)(seg >> 1) & 1u) ^ 1u, p.status)) break;
        tc_fence_after();
      }
      const int as = kk % F_SA, bs = kk % F_SB;
      if (!mbar_wait(a_full(as), (uint32_t)(kk / F_SA) & 1u, p.status)) break;
      if (!mbar_wait(b_full(bs), (uint32_t)(kk / F_SB) & 1u, p.status)) break;
      tc_fence_after();
      const uint64_t bdesc = noswizzle_desc(smem_s + Cfg::kOffB + bs * F_B_STAGE, F_LBO, F_SBO);
#pragma unroll
      for (int mt = 0; mt < MTILES; ++mt) {
        const uint32_t d = tmem_base + (uint32_t)((ab * MTILES + mt) * F_BN);
        const uint64_t adesc = sw128_desc(smem_s + as * Cfg::kAStage + mt * F_A_TILE);
#pragma unroll
        for (int k16 = 0; k16 < F_BK / 16; ++k16)
          tc_mma(d, adesc + (uint64_t)(2 * k16), bdesc + (uint64_t)((2 * F_LBO / 16) * k16), idesc,
                 (!first || k16 > 0) ? 1u : 0u);
      }
      tc_commit(a_empty(as));
      tc_commit(b_empty(bs));
      if (last) {
        tc_commit(acc_full(ab));
        ++seg;
      }
    }
    tc_commit(done_bar);
    mbar_wait_short(done_bar, 0);
  } else if (warp >= 2 && warp < 2 + F_DEC_WARPS) {
    // ---------------- decoders ----------------
    const int dw = warp - 2;
    const int par = dw >> 2, slab_i = dw & 3;  // k steps par, par + F_GROUPS, ...; slab slab_i of each
    const int g = lane >> 2, q = lane & 3;
    const int nmine = len > par ? (len - par + F_GROUPS - 1) / F_GROUPS : 0;
    const uint32_t ring_s = smem_s + Cfg::kOffD + dw * F_RD * Cfg::kSeg;
    int64_t issued = 0;
    auto issue = [&](int j) {
      const int64_t z = zs + par + (int64_t)F_GROUPS * j;
      const int64_t nb = z / KS, tk = (z % KS) * 4 + slab_i;
      const int s = j % F_RD;
      mbar_arrive_expect_tx(dec_full(dw, s), Cfg::kSeg);
      bulk_g2s(ring_s + s * Cfg::kSeg, p.trellis + (tk * p.tiles_n + nb * 8) * (32 * BITS), Cfg::kSeg,
               dec_full(dw, s));
      ++issued;
    };
    if (lane == 0)
      for (int j = 0; j < F_RD - 1 && j < nmine; ++j) issue(j);
    for (int j = 0; j < nmine; ++j) {
      if (lane == 0 && j + F_RD - 1 < nmine) issue(j + F_RD - 1);
      const int s = j % F_RD;
      if (!mbar_wait(dec_full(dw, s), (uint32_t)(j / F_RD) & 1u, p.status)) {
        if (lane == 0)
          for (int64_t u = j; u < issued; ++u) mbar_wait_short(dec_full(dw, (int)(u % F_RD)), (uint32_t)(u / F_RD) & 1u);
        break;
      }
      uint32_t own[2 * BITS];
      load_own_words_shared<BITS>(ring_s + s * Cfg::kSeg + lane * 8 * BITS, own);
      const uint32_t prev = prefix_from_neighbour<BITS>(own, lane);
      Windows<BITS> win;
      win.build(own, prev);
      const int kk = par + F_GROUPS * j;
      const int bs = kk % F_SB;
      if (!mbar_wait(b_empty(bs), ((uint32_t)(kk / F_SB) & 1u) ^ 1u, p.status)) break;
      const uint32_t bt = smem_s + Cfg::kOffB + bs * F_B_STAGE + (2 * slab_i + (q >> 1)) * F_LBO + (q & 1) * 8;
      static_for<16>([&](auto C) {
        constexpr int cc = C.value;
        const uint32_t lo = decode_pair_sel<false>(win.template state<0, cc>(), win.template state<1, cc>());
        const uint32_t hi = decode_pair_sel<false>(win.template state<2, cc>(), win.template state<3, cc>());
        const int n = 16 * g + cc;
        st_shared_v2(bt + (n >> 3) * F_SBO + (n & 7) * 16, lo, hi);
      });
      fence_proxy_async_shared();  // make the generic stores visible to the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(b_full(bs));
    }
  } else if (warp >= 2 + F_DEC_WARPS) {
    // ---------------- epilogue ----------------
    wait_prior_grid_f();  // the previous kernel may still read the partial slots
    const int lg = warp & 3;
    int seg = 0;
    for (int kk = 0; kk < len; ++kk) {
      const int64_t z = zs + kk;
      const int ks = (int)(z % KS);
      if (!((kk == len - 1) || (ks == KS - 1))) continue;
      const int64_t nb = z / KS;
      const int ab = seg & 1;
      if (!mbar_wait(acc_full(ab), (uint32_t)(seg >> 1) & 1u, p.status)) break;
      tc_fence_after();
      // Every CTA stores its part of the n-block as an fp32 partial slot; the
      // finalize kernel sums the slots and applies the output rotation.
      const int64_t pf = unit_owner(nb * KS, p.P, p.TS);
      float *slot = p.partials + (nb * p.smax + (c - pf)) * (int64_t)(MTILES * 128 * 128);
#pragma unroll 1
      for (int mt = 0; mt < MTILES; ++mt) {
        const int m = mt * 128 + lg * 32 + lane;
        const uint32_t taddr = tmem_base + ((uint32_t)(lg * 32) << 16) + (uint32_t)((ab * MTILES + mt) * F_BN);
#pragma unroll 1
        for (int j4 = 0; j4 < 4; ++j4) {
          float t[32];
          tmem_ld32(taddr + 32 * j4, t);
          if (m < p.rows) {
            float4 *dst = reinterpret_cast<float4 *>(slot + (int64_t)m * 128 + 32 * j4);
#pragma unroll
            for (int a = 0; a < 8; ++a) dst[a] = make_float4(t[4 * a], t[4 * a + 1], t[4 * a + 2], t[4 * a + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(ab));
      ++seg;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(Cfg::kTmemCols)
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

cudaError_t init_fused_kernels() {
  cudaError_t e;
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
  const int MTILES = L.rows <= 128 ? 1 : 2;
  alignas(64) CUtensorMap tmA;
  if (!encode_tensor_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, L.xr, (uint64_t)L.K, (uint64_t)L.xr_rows,
                            (uint64_t)L.K * 2, F_BK, 128, CU_TENSOR_MAP_SWIZZLE_128B))
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
  cudaError_t e = MTILES == 1 ? launch_mt<1>(L.bits, tmA, fp, fp.P, st) : launch_mt<2>(L.bits, tmA, fp, fp.P, st);
  if (e != cudaSuccess) return e;
  return launch_decode_finalize(L.partials, fp.smax, (int64_t)MTILES * 128 * 128, L.sv, L.y, L.y_f32, L.n_gemm,
                                L.n_valid, L.rows, fp.P, fp.TS, fp.KS, /*all_blocks=*/1, st);
}

}  // namespace exl3
