// Bounds-checked build of the kernels (compiled with -DEXL3_DEBUG_BOUNDS=1
// into libexl3_bounds.so; the normal library is built without it).
//
// It stands in for a memory checker that cannot run here. Before an access
// is made, the checks test it against the extents the launch parameters
// imply:
//   - every global load and store whose index a kernel computes;
//   - every shared-memory address, against the CTA's dynamic
//     shared-memory window;
//   - every TMA coordinate (the 16-byte rule on the innermost coordinate,
//     and the tile inside the tensor);
//   - every bulk-copy span and alignment;
//   - every mbarrier address;
//   - every TMEM column.
//
// When a check fails:
//   - the first failure records EXL3_ERR_OUT_OF_BOUNDS in the device error
//     word and prints its source line and values;
//   - the access is skipped: a load reads zero, and a copy is not issued.
//
// Control flow stays as it was (barriers, shuffles, mbarrier phases), so a
// kernel with a violation still ends. Waiters on a copy that was never
// issued give up through the bounded wait. The error word keeps the first
// error, so such a timeout does not overwrite it.
//
// In the normal build every check is the constant `true`: no code, no
// registers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include "../../include/exl3.h"

#ifndef EXL3_DEBUG_BOUNDS
#define EXL3_DEBUG_BOUNDS 0
#endif

namespace exl3 {

#if EXL3_DEBUG_BOUNDS

// Device address of the error word. Kernels are built without relocatable
// device code, so each translation unit has its own copy; its init function
// sets it (EXL3_BIND_BOUNDS_WORD) when the device is initialized.
static __device__ int *g_bounds_word;

// The dynamic shared-memory window of the CTA (every extern __shared__
// array starts at its base).
extern __shared__ __align__(16) uint8_t exl3_dyn_smem_base[];

__device__ __noinline__ static bool bounds_fail(const char *file, int line, long long v, long long lim) {
  int *w = g_bounds_word;
  if (w && atomicCAS(w, 0, (int)EXL3_ERR_OUT_OF_BOUNDS) == 0)
    printf("exl3 bounds check failed at %s:%d: value %lld, limit %lld (block %d, thread %d)\n", file, line, v, lim,
           (int)blockIdx.x, (int)threadIdx.x);
  return false;
}

// 0 <= off and off + len <= size.
__device__ __forceinline__ static bool check_span(long long off, long long len, long long size, const char *file,
                                                  int line) {
  return (off >= 0 && len >= 0 && off + len <= size) ? true : bounds_fail(file, line, off + len, size);
}

// lo <= v < hi.
__device__ __forceinline__ static bool check_range(long long v, long long lo, long long hi, const char *file,
                                                   int line) {
  return (v >= lo && v < hi) ? true : bounds_fail(file, line, v, v < lo ? lo : hi);
}

__device__ __forceinline__ static bool check_aligned(long long v, long long a, const char *file, int line) {
  return (v % a == 0) ? true : bounds_fail(file, line, v, a);
}

// [saddr, saddr + len) inside the dynamic shared-memory window.
__device__ __forceinline__ static bool check_smem(uint32_t saddr, long long len, const char *file, int line) {
  uint32_t dyn;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(exl3_dyn_smem_base));
  return check_span((long long)saddr - (long long)base, len, (long long)dyn, file, line);
}

#define EXL3_SPAN(off, len, size) \
  ::exl3::check_span((long long)(off), (long long)(len), (long long)(size), __FILE__, __LINE__)
#define EXL3_RANGE(v, lo, hi) ::exl3::check_range((long long)(v), (long long)(lo), (long long)(hi), __FILE__, __LINE__)
#define EXL3_ALIGNED(v, a) ::exl3::check_aligned((long long)(v), (long long)(a), __FILE__, __LINE__)
#define EXL3_SMEM(saddr, len) ::exl3::check_smem((uint32_t)(saddr), (long long)(len), __FILE__, __LINE__)

#define EXL3_BIND_BOUNDS_WORD(w) cudaMemcpyToSymbol(::exl3::g_bounds_word, &(w), sizeof(int *))

// Self-test of the reporting path of one translation unit: submits an index
// equal to its extent to the checks and accesses no memory. Each kernel
// translation unit wraps it (bounds_probe_<unit>), so that a unit whose
// error word was never bound shows up.
__global__ static void bounds_probe_kernel(long long n) { (void)EXL3_RANGE(n, 0, n); }
static inline cudaError_t launch_bounds_probe(cudaStream_t st) {
  bounds_probe_kernel<<<1, 32, 0, st>>>(1);
  return cudaGetLastError();
}

#else

#define EXL3_SPAN(off, len, size) true
#define EXL3_RANGE(v, lo, hi) true
#define EXL3_ALIGNED(v, a) true
#define EXL3_SMEM(saddr, len) true
#define EXL3_BIND_BOUNDS_WORD(w) ((void)(w), cudaSuccess)

#endif

}  // namespace exl3
