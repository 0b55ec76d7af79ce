// Decode-shaped linear layer for callers that cannot allocate device memory.
//
// The rotated activations and the split-K partial sums that exl3_linear
// keeps in the caller's workspace live here in one fixed, file-scope device
// array instead. In host code the array's name is only a host-side stand-in,
// so its device address is looked up once per device (with that device
// current) and passed to the kernels as a plain pointer.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/exl3.h"
#include "exl3_common.cuh"
#include "exl3_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = EXL3_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mutex;

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of the scratch array on the current device (looked up on
// the first call per device).
uint8_t *scratch_on_current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[d]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_ptr[d] = p;
  }
  return static_cast<uint8_t *>(g_scratch_ptr[d]);
}

}  // namespace

extern "C" exl3_status exl3_linear_decode_noalloc(const void *x, int64_t M, int64_t K, const uint16_t *trellis,
                                                  int bits, int64_t n_stored, int64_t n_gemm, const void *su,
                                                  const void *sv, void *y, int y_dtype, void *stream) {
  using namespace exl3;
  if (!linear_rows_ok(M) || !linear_shape_ok(K, n_stored, n_gemm) || (y_dtype != EXL3_F16 && y_dtype != EXL3_F32))
    return EXL3_ERR_INVALID_ARG;
  if (!bits_supported(bits)) return EXL3_ERR_UNSUPPORTED_BITS;
  if (!aligned16(x) || !aligned16(trellis) || !aligned16(su) || !aligned16(sv) || !aligned16(y))
    return EXL3_ERR_ALIGNMENT;
  const DeviceInfo *dev = initialized_device();
  if (!dev) return EXL3_ERR_NOT_INITIALIZED;
  WorkspaceLayout L;
  if (!workspace_layout(kDecodeRows, K, n_gemm, bits, 0, dev->num_sms, &L)) return EXL3_ERR_INVALID_ARG;
  if (L.total > kNoallocScratchBytes) return EXL3_ERR_NOALLOC_TOO_LARGE;
  if (M == 0) return EXL3_OK;
  uint8_t *ws = scratch_on_current_device();
  if (!ws) return EXL3_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t ysz = y_dtype == EXL3_F32 ? 4 : 2;
  for (int64_t m0 = 0; m0 < M; m0 += kDecodeRows) {
    DecodeLaunch d;
    d.x = static_cast<const uint8_t *>(x) + (size_t)(m0 * K) * 2;
    d.rows = (int)((M - m0) < kDecodeRows ? (M - m0) : kDecodeRows);
    d.K = K;
    d.trellis = trellis;
    d.bits = bits;
    d.n_stored = n_stored;
    d.n_gemm = n_gemm;
    d.n_valid = n_gemm;
    d.su = su;
    d.sv = sv;
    d.y = static_cast<uint8_t *>(y) + (size_t)(m0 * n_gemm) * ysz;
    d.y_f32 = y_dtype == EXL3_F32;
    d.xf = ws + L.xf_off;
    d.partials = reinterpret_cast<float *>(ws + L.partials_off);
    d.status = dev->status;
    d.plan = L.plan;
    if (launch_decode_gemm(d, st) != cudaSuccess) return EXL3_ERR_CUDA;
  }
  return EXL3_OK;
}
