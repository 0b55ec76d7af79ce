// Input rotation (had_r_128 with an optional pre-scale) and greedy selection
// over masked logits.
//
// had_r_128 stage of the unfused prefill sequence: vLLM PR #316, "[EXL3]
// dispatch prefill-shaped GEMMs to reconstruct+hgemm", section "Kernel
// measurements". Greedy selection over pad-masked logits: pegainfer PR #1046,
// "perf(qwen35): align the logits GEMM width ...", section "Review follow-ups".
#include <float.h>
#include <limits.h>

#include "exl3_common.cuh"
#include "exl3_internal.h"

namespace exl3 {

// One 128-block per half-warp: lane l16 holds elements 8*l16 .. 8*l16+7.
// Butterfly stages h = 1, 2, 4 run inside a lane, h = 8 .. 64 across lanes
// (xor 1, 2, 4, 8), in that order; then one multiply by fp32(1/sqrt(128)).
// Memory-bound: 4 bytes moved per element (2 read, 2 written).
__global__ void __launch_bounds__(256) hadamard128_kernel(const __half *x, __half *y,
                                                          const __half *__restrict__ pre,
                                                          int64_t nblk, int64_t cblk, int64_t cols) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // a dependent kernel may start its prologue
  const int lane = threadIdx.x & 31;
  const int l16 = lane & 15;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t w = warp; w * 2 < nblk; w += nwarps) {
    const int64_t blk = w * 2 + (lane >> 4);
    const bool valid = blk < nblk;
    const int64_t row = valid ? blk / cblk : 0;
    const int64_t cb = valid ? blk % cblk : 0;
    const int64_t off = row * cols + cb * 128 + l16 * 8;
    float v[8];
    if (valid) {
      const uint4 raw = EXL3_SPAN(off, 8, nblk * 128) ? *reinterpret_cast<const uint4 *>(x + off) : uint4{};
      const __half *h = reinterpret_cast<const __half *>(&raw);
      if (pre) {
        const uint4 praw = EXL3_SPAN(cb * 128 + l16 * 8, 8, cols)
                               ? __ldg(reinterpret_cast<const uint4 *>(pre + cb * 128 + l16 * 8))
                               : uint4{};
        const __half *p = reinterpret_cast<const __half *>(&praw);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __half2float(h[i]) * __half2float(p[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __half2float(h[i]);
      }
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
      // the lane's side of the butterfly, p + v or p - v, as one fma with an
      // exact +-1 product: the same single rounding as the add or subtract
      const float sgn = (l16 & s) ? -1.f : 1.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float p = __shfl_xor_sync(0xffffffffu, v[i], s);
        v[i] = fmaf(v[i], sgn, p);
      }
    }
    if (valid) {
      uint4 out;
      __half *o = reinterpret_cast<__half *>(&out);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = __float2half_rn(v[i] * kInvSqrt128);
      if (EXL3_SPAN(off, 8, nblk * 128)) *reinterpret_cast<uint4 *>(y + off) = out;
    }
  }
}

// One CTA per row; first index of the maximum (ties keep the lower index).
__global__ void __launch_bounds__(256) argmax_rows_kernel(const float *__restrict__ logits, int64_t n,
                                                          int32_t *argmax) {
  const float *row = logits + (int64_t)blockIdx.x * n;
  float best = -INFINITY;
  int bidx = INT_MAX;
  for (int64_t c = (int64_t)threadIdx.x * 4; c < n; c += (int64_t)blockDim.x * 4) {
    const float4 v = EXL3_SPAN(c, 4, n) ? __ldg(reinterpret_cast<const float4 *>(row + c))
                                        : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int idx = (int)(c + i);
      if (vv[i] > best || (vv[i] == best && idx < bidx)) {
        best = vv[i];
        bidx = idx;
      }
    }
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) {
    float ob = __shfl_xor_sync(0xffffffffu, best, s);
    int oi = __shfl_xor_sync(0xffffffffu, bidx, s);
    if (ob > best || (ob == best && oi < bidx)) {
      best = ob;
      bidx = oi;
    }
  }
  __shared__ float sb[8];
  __shared__ int si[8];
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0 && EXL3_RANGE(w, 0, 8)) {
    sb[w] = best;
    si[w] = bidx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < (int)(blockDim.x >> 5) && EXL3_RANGE(i, 0, 8); ++i) {
      if (sb[i] > best || (sb[i] == best && si[i] < bidx)) {
        best = sb[i];
        bidx = si[i];
      }
    }
    argmax[blockIdx.x] = (bidx == INT_MAX) ? 0 : bidx;
  }
}

// Self-test of the bounded-wait path: waits on an mbarrier phase that nothing
// completes, gives up after limit_ns and records the timeout in the status
// word. Returns on its own; never traps.
__global__ void wait_timeout_selftest_kernel(int *status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_limit(smem_u32(&bar), 0, status, limit_ns);
  __syncthreads();
  if (threadIdx.x == 0) mbar_arrive(smem_u32(&bar));  // retire the phase before exit
}

cudaError_t launch_wait_timeout_selftest(int *status, unsigned long long limit_ns, cudaStream_t st) {
  wait_timeout_selftest_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

// out = RNE_fp16(silu(gate) * up), computed in fp32, 8 elements per thread.
__global__ void __launch_bounds__(256) silu_mul_kernel(const __half *__restrict__ gate, const __half *__restrict__ up,
                                                       __half *__restrict__ out, int64_t n8) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 g = __ldg(reinterpret_cast<const uint4 *>(gate) + i);
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(up) + i);
    const __half *gh = reinterpret_cast<const __half *>(&g);
    const __half *uh = reinterpret_cast<const __half *>(&u);
    uint4 r;
    __half *rh = reinterpret_cast<__half *>(&r);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float a = __half2float(gh[e]);
      rh[e] = __float2half_rn(a / (1.0f + __expf(-a)) * __half2float(uh[e]));
    }
    reinterpret_cast<uint4 *>(out)[i] = r;
  }
}

cudaError_t launch_silu_mul(const void *gate, const void *up, void *out, int64_t n, int num_sms, cudaStream_t st) {
  const int64_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  int64_t grid = ceil_div(n8, 256);
  if (grid > (int64_t)num_sms * 8) grid = (int64_t)num_sms * 8;
  silu_mul_kernel<<<(unsigned)grid, 256, 0, st>>>(static_cast<const __half *>(gate), static_cast<const __half *>(up),
                                                  static_cast<__half *>(out), n8);
  return cudaGetLastError();
}

cudaError_t init_rotate_kernels(int *status) {
  cudaError_t e = EXL3_BIND_BOUNDS_WORD(status);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes a;
  e = cudaFuncGetAttributes(&a, hadamard128_kernel);
  if (e != cudaSuccess) return e;
  e = cudaFuncGetAttributes(&a, wait_timeout_selftest_kernel);
  if (e != cudaSuccess) return e;
  e = cudaFuncGetAttributes(&a, silu_mul_kernel);
  if (e != cudaSuccess) return e;
  return cudaFuncGetAttributes(&a, argmax_rows_kernel);
}

cudaError_t launch_hadamard128(const void *x, void *y, const void *pre, int64_t rows, int64_t cols,
                               int num_sms, cudaStream_t st) {
  const int64_t cblk = cols / 128;
  const int64_t nblk = rows * cblk;
  if (nblk == 0) return cudaSuccess;
  const int64_t warps = ceil_div(nblk, 2);
  int64_t grid = ceil_div(warps, 8);
  const int64_t cap = (int64_t)num_sms * 16;
  if (grid > cap) grid = cap;
  hadamard128_kernel<<<(unsigned)grid, 256, 0, st>>>(static_cast<const __half *>(x),
                                                     static_cast<__half *>(y),
                                                     static_cast<const __half *>(pre), nblk, cblk, cols);
  return cudaGetLastError();
}

cudaError_t launch_argmax(const float *logits, int64_t M, int64_t n, int32_t *argmax, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  argmax_rows_kernel<<<(unsigned)M, 256, 0, st>>>(logits, n, argmax);
  return cudaGetLastError();
}

#if EXL3_DEBUG_BOUNDS
cudaError_t bounds_probe_rotate(cudaStream_t st) { return launch_bounds_probe(st); }
#endif

}  // namespace exl3
