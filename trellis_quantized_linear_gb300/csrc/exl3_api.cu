// C ABI of libexl3: argument validation, workspace layout and the runtime
// decode / prefill dispatch. Declarations and argument contracts are in
// include/exl3.h.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/exl3.h"
#include "exl3_common.cuh"
#include "exl3_internal.h"

// Device error word: kernels record in it the first bounded wait they gave
// up (and, in the bounds-checked build, the first failed bounds check).
__device__ int g_exl3_status_word;

namespace exl3 {

namespace {

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_mutex;

const DeviceInfo *current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return nullptr;
  const DeviceInfo *info = &g_devices[d];
  return info->ready ? info : nullptr;
}

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

exl3_status from_cuda(cudaError_t e) { return e == cudaSuccess ? EXL3_OK : EXL3_ERR_CUDA; }

// The fused prefill kernel (decode in producer warps, one 512-row block) is
// used where it was measured faster than reconstruct + GEMM: a single
// 512-row block (it decodes W once, as the reconstruct does, but writes no
// W^T) over enough 256-column blocks to keep most CTA pairs busy. Gate
// geometry (5120 -> 17408, 68 column blocks): 66.8 vs 86.5 us at M = 256,
// 83.0 vs 108.1 us at M = 512; at M = 768 and up, and on the down geometry
// (20 column blocks), reconstruct + GEMM wins.
bool fused_prefill_pays(int64_t M, int64_t n_gemm, int num_sms) {
  const int64_t col_blocks = (n_gemm + 255) / 256;
  return M <= 512 && 10 * col_blocks >= 3 * (int64_t)num_sms;
}

// Shared by exl3_linear and exl3_logits_masked once arguments are validated.
exl3_status run_linear(const DeviceInfo *dev, const WorkspaceLayout &L, const void *x, int64_t M, int64_t K,
                       const uint16_t *trellis, int bits, int64_t n_stored, int64_t n_gemm, int64_t n_valid,
                       const void *su, const void *sv, void *y, int y_dtype, int64_t m_threshold,
                       uint8_t *ws, cudaStream_t st) {
  const bool prefill = m_threshold > 0 && M >= m_threshold;
  const size_t ysz = y_dtype == EXL3_F32 ? 4 : 2;
  if (!prefill && M > kDecodeRows) {
    // Decode-shaped with more than 16 rows: the fused tensor-core kernel,
    // 256 rows per launch, on activations rotated once for all rows.
    cudaError_t e = launch_hadamard128(x, ws + L.xr_off, su, M, K, dev->num_sms, st);
    if (e != cudaSuccess) return EXL3_ERR_CUDA;
    for (int64_t m0 = 0; m0 < M; m0 += kFusedMaxRows) {
      FusedLaunch f;
      f.xr = ws + L.xr_off + (size_t)(m0 * K) * 2;
      f.xr_rows = L.xr_rows - m0;
      f.K = K;
      f.trellis = trellis;
      f.bits = bits;
      f.n_stored = n_stored;
      f.n_gemm = n_gemm;
      f.n_valid = n_valid;
      f.sv = sv;
      f.y = static_cast<uint8_t *>(y) + (size_t)(m0 * n_gemm) * ysz;
      f.y_f32 = y_dtype == EXL3_F32;
      f.partials = reinterpret_cast<float *>(ws + L.partials_off);
      f.status = dev->status;
      f.rows = (int)((M - m0) < kFusedMaxRows ? (M - m0) : kFusedMaxRows);
      f.plan = L.fplan;
      e = launch_fused_gemm(f, st);
      if (e != cudaSuccess) return EXL3_ERR_CUDA;
    }
    return EXL3_OK;
  }
  if (!prefill) {
    for (int64_t m0 = 0; m0 < M; m0 += kDecodeRows) {
      DecodeLaunch d;
      d.x = static_cast<const uint8_t *>(x) + (size_t)(m0 * K) * 2;
      d.rows = (int)((M - m0) < kDecodeRows ? (M - m0) : kDecodeRows);
      d.K = K;
      d.trellis = trellis;
      d.bits = bits;
      d.n_stored = n_stored;
      d.n_gemm = n_gemm;
      d.n_valid = n_valid;
      d.su = su;
      d.sv = sv;
      d.y = static_cast<uint8_t *>(y) + (size_t)(m0 * n_gemm) * ysz;
      d.y_f32 = y_dtype == EXL3_F32;
      d.xf = ws + L.xf_off;
      d.partials = reinterpret_cast<float *>(ws + L.partials_off);
      d.status = dev->status;
      d.plan = L.plan;
      cudaError_t e = launch_decode_gemm(d, st);
      if (e != cudaSuccess) return EXL3_ERR_CUDA;
    }
    return EXL3_OK;
  }
  void *xr = ws + L.xr_off;
  void *wchunk = ws + L.wchunk_off;
  cudaError_t e = launch_hadamard128(x, xr, su, M, K, dev->num_sms, st);
  if (e != cudaSuccess) return EXL3_ERR_CUDA;
  if (fused_prefill_pays(M, n_gemm, dev->num_sms)) {
    FusedPrefillLaunch f;
    f.xr = xr;
    f.xr_rows = L.xr_rows;
    f.M = M;
    f.K = K;
    f.trellis = trellis;
    f.bits = bits;
    f.n_stored = n_stored;
    f.n_gemm = n_gemm;
    f.n_valid = n_valid;
    f.sv = sv;
    f.y = y;
    f.y_f32 = y_dtype == EXL3_F32;
    f.status = dev->status;
    f.num_sms = dev->num_sms;
    return launch_fused_prefill(f, st) == cudaSuccess ? EXL3_OK : EXL3_ERR_CUDA;
  }
  for (int64_t c0 = 0; c0 < n_gemm; c0 += EXL3_RECONSTRUCT_CHUNK_COLS) {
    const int64_t nc = (n_gemm - c0) < EXL3_RECONSTRUCT_CHUNK_COLS ? (n_gemm - c0) : EXL3_RECONSTRUCT_CHUNK_COLS;
    // The first chunk may run alongside the input rotation (independent
    // operands); later chunks follow the GEMM that reads the chunk buffer.
    e = launch_reconstruct(trellis, bits, K, n_stored, c0, nc, wchunk, EXL3_LAYOUT_NK, dev->num_sms, st,
                           c0 == 0 ? 1 : 0);
    if (e != cudaSuccess) return EXL3_ERR_CUDA;
    PrefillLaunch p;
    p.xr = xr;
    p.xr_rows = L.xr_rows;
    p.M = M;
    p.K = K;
    p.wt = wchunk;
    p.chunk_rows = L.chunk_rows;
    p.nc = nc;
    p.sv = static_cast<const uint8_t *>(sv) + (size_t)c0 * 2;
    p.y = static_cast<uint8_t *>(y) + (size_t)c0 * ysz;
    p.ldy = n_gemm;
    p.y_f32 = y_dtype == EXL3_F32;
    p.n_valid_local = n_valid - c0;
    p.status = dev->status;
    p.num_sms = dev->num_sms;
    p.partials = reinterpret_cast<float *>(ws + L.partials_off);
    p.partials_bytes = L.partials_bytes;
    e = launch_prefill_gemm(p, st);
    if (e != cudaSuccess) return EXL3_ERR_CUDA;
  }
  return EXL3_OK;
}

// Validation shared by exl3_linear and exl3_logits_masked. On success fills
// `layout` for this call's M.
exl3_status validate_linear(const void *x, int64_t M, int64_t K, const uint16_t *trellis, int bits,
                            int64_t n_stored, int64_t n_gemm, const void *su, const void *sv, const void *y,
                            int64_t m_threshold, void *workspace, size_t workspace_bytes,
                            const DeviceInfo **dev_out, WorkspaceLayout *layout) {
  if (!linear_rows_ok(M) || m_threshold < 0 || !linear_shape_ok(K, n_stored, n_gemm)) return EXL3_ERR_INVALID_ARG;
  if (!bits_supported(bits)) return EXL3_ERR_UNSUPPORTED_BITS;
  if (!aligned16(x) || !aligned16(trellis) || !aligned16(su) || !aligned16(sv) || !aligned16(y) ||
      !aligned16(workspace))
    return EXL3_ERR_ALIGNMENT;
  const DeviceInfo *dev = current_device();
  if (!dev) return EXL3_ERR_NOT_INITIALIZED;
  if (!workspace_layout(M, K, n_gemm, bits, m_threshold, dev->num_sms, layout)) return EXL3_ERR_INVALID_ARG;
  if (layout->total > workspace_bytes) return EXL3_ERR_WORKSPACE_TOO_SMALL;
  *dev_out = dev;
  return EXL3_OK;
}

}  // namespace

const DeviceInfo *initialized_device() { return current_device(); }

bool bits_supported(int bits) { return bits >= 1 && bits <= 8; }

bool workspace_layout(int64_t M_max, int64_t K, int64_t n_gemm, int bits, int64_t m_threshold, int num_sms,
                      WorkspaceLayout *out) {
  if (M_max < 0 || m_threshold < 0 || num_sms <= 0 || !bits_supported(bits)) return false;
  if (K <= 0 || K % 128 || K > 131072 || n_gemm <= 0 || n_gemm % 128) return false;
  WorkspaceLayout L;
  const int64_t NB = n_gemm / 128, KB = K / 128;
  L.plan = decode_plan(NB, KB, num_sms);
  size_t off = 0;
  L.fplan = fused_plan(NB, K, num_sms);
  L.prefill = m_threshold > 0 && M_max >= m_threshold;
  L.fused = M_max > kDecodeRows && (m_threshold == 0 || m_threshold > kDecodeRows + 1);
  L.partials_off = off;
  {
    size_t pb = decode_partials_bytes(L.plan, NB);
    if (L.fused) {
      const size_t fb = fused_partials_bytes(L.fplan, NB);
      if (fb > pb) pb = fb;
    }
    if (L.prefill) {  // the prefill GEMM's stream-K tail slots share the region
      const size_t tb = prefill_tail_partials_bytes(num_sms);
      if (tb > pb) pb = tb;
    }
    L.partials_bytes = pb;
    off += align_up(pb, 256);
  }
  L.xf_off = off;
  off += align_up((size_t)K * 32, 256);
  if (L.prefill || L.fused) {
    L.xr_rows = ceil_div(M_max, 128) * 128;
    L.xr_off = off;
    off += align_up((size_t)L.xr_rows * (size_t)K * 2, 256);
  }
  if (L.prefill) {
    const int64_t cols = n_gemm < EXL3_RECONSTRUCT_CHUNK_COLS ? n_gemm : EXL3_RECONSTRUCT_CHUNK_COLS;
    L.chunk_rows = ceil_div(cols, 256) * 256;
    L.wchunk_off = off;
    off += align_up((size_t)L.chunk_rows * (size_t)K * 2, 256);
  }
  L.total = off;
  *out = L;
  return true;
}

}  // namespace exl3

using namespace exl3;

extern "C" {

exl3_status exl3_init(int device) {
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess) return EXL3_ERR_CUDA;
  if (device < 0 || device >= n || device >= kMaxDevices) return EXL3_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (cudaSetDevice(device) != cudaSuccess) return EXL3_ERR_CUDA;
  if (g_devices[device].ready) return EXL3_OK;
  DeviceInfo info;
  if (cudaDeviceGetAttribute(&info.num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return EXL3_ERR_CUDA;
  void *status = nullptr;
  if (cudaGetSymbolAddress(&status, g_exl3_status_word) != cudaSuccess) return EXL3_ERR_CUDA;
  info.status = static_cast<int *>(status);
  if (cudaMemset(info.status, 0, sizeof(int)) != cudaSuccess) return EXL3_ERR_CUDA;
  if (init_rotate_kernels(info.status) != cudaSuccess || init_reconstruct_kernels(info.status) != cudaSuccess ||
      init_reconstruct_rotated_kernels(info.status) != cudaSuccess ||
      init_decode_kernels(info.status) != cudaSuccess || init_prefill_kernels(info.status) != cudaSuccess ||
      init_fused_kernels(info.status) != cudaSuccess || init_fused_prefill_kernels(info.status) != cudaSuccess)
    return EXL3_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return EXL3_ERR_CUDA;
  info.ready = true;
  g_devices[device] = info;
  return EXL3_OK;
}

const char *exl3_status_string(int status) {
  switch (status) {
    case EXL3_OK: return "ok";
    case EXL3_ERR_INVALID_ARG: return "invalid argument (shape, size or enum out of range)";
    case EXL3_ERR_ALIGNMENT: return "pointer is NULL or not 16-byte aligned";
    case EXL3_ERR_UNSUPPORTED_BITS: return "unsupported trellis bit width";
    case EXL3_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than the required size";
    case EXL3_ERR_NOT_INITIALIZED: return "exl3_init was not called for the current device";
    case EXL3_ERR_CUDA: return "CUDA runtime error or failed launch";
    case EXL3_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait on the device";
    case EXL3_ERR_NOALLOC_TOO_LARGE: return "problem needs more scratch than the fixed no-alloc buffer holds";
    case EXL3_ERR_OUT_OF_BOUNDS: return "a bounds check of the bounds-checked build failed on the device";
    default: return "unknown status";
  }
}

int exl3_supported_bits(int bits) { return bits_supported(bits) ? 1 : 0; }

int64_t exl3_aligned_logits_width(int64_t n_decodable, int64_t n_stored) {
  if (n_decodable <= 0 || n_stored <= 0 || n_decodable > n_stored) return -1;
  const int64_t aligned = ceil_div(n_decodable, 128) * 128;
  return aligned < n_stored ? aligned : n_stored;
}

int exl3_decode_plan(int64_t K, int64_t n_gemm, int num_sms, int *splits, int *ctas_per_split) {
  if (K <= 0 || K % 128 || K > 131072 || n_gemm <= 0 || n_gemm % 128 || num_sms <= 0 || !splits ||
      !ctas_per_split)
    return -1;
  DecodePlan p = decode_plan(n_gemm / 128, K / 128, num_sms);
  *splits = (int)p.smax[0];
  *ctas_per_split = (int)p.grid[0];
  return 0;
}

int exl3_prefill_path(int64_t M, int64_t n_gemm, int num_sms) {
  if (M < 1 || n_gemm <= 0 || n_gemm % 128 || num_sms < 1) return -1;
  return fused_prefill_pays(M, n_gemm, num_sms) ? 1 : 0;
}

size_t exl3_linear_workspace_bytes_for(int64_t M_max, int64_t K, int64_t n_gemm, int bits, int64_t m_threshold,
                                       int num_sms) {
  WorkspaceLayout L;
  if (!workspace_layout(M_max, K, n_gemm, bits, m_threshold, num_sms, &L)) return 0;
  return L.total;
}

size_t exl3_linear_workspace_bytes(int64_t M_max, int64_t K, int64_t n_gemm, int bits, int64_t m_threshold) {
  int d = -1, sms = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return 0;
  if (d >= 0 && d < kMaxDevices && g_devices[d].ready) {
    sms = g_devices[d].num_sms;
  } else if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) {
    return 0;
  }
  return exl3_linear_workspace_bytes_for(M_max, K, n_gemm, bits, m_threshold, sms);
}

exl3_status exl3_workspace_init(void *workspace, size_t workspace_bytes, void *stream) {
  if (!aligned16(workspace)) return EXL3_ERR_ALIGNMENT;
  if (!current_device()) return EXL3_ERR_NOT_INITIALIZED;
  return from_cuda(cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)));
}

exl3_status exl3_hadamard128(const void *x, void *y, const void *pre_scale, int64_t rows, int64_t cols,
                             void *stream) {
  if (rows < 0 || cols <= 0 || cols % 128) return EXL3_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || (pre_scale && !aligned16(pre_scale))) return EXL3_ERR_ALIGNMENT;
  const DeviceInfo *dev = current_device();
  if (!dev) return EXL3_ERR_NOT_INITIALIZED;
  return from_cuda(launch_hadamard128(x, y, pre_scale, rows, cols, dev->num_sms, static_cast<cudaStream_t>(stream)));
}

exl3_status exl3_reconstruct(const uint16_t *trellis, int bits, int64_t K, int64_t n_stored, int64_t n0,
                             int64_t n_cols, void *w, int layout, void *stream) {
  if (K <= 0 || K % 16 || n_stored <= 0 || n_stored % 128 || n0 < 0 || n0 % 128 || n_cols < 0 || n_cols % 128 ||
      n0 + n_cols > n_stored || (layout != EXL3_LAYOUT_KN && layout != EXL3_LAYOUT_NK))
    return EXL3_ERR_INVALID_ARG;
  if (!bits_supported(bits)) return EXL3_ERR_UNSUPPORTED_BITS;
  if (!aligned16(trellis) || !aligned16(w)) return EXL3_ERR_ALIGNMENT;
  const DeviceInfo *dev = current_device();
  if (!dev) return EXL3_ERR_NOT_INITIALIZED;
  return from_cuda(launch_reconstruct(trellis, bits, K, n_stored, n0, n_cols, w, layout, dev->num_sms,
                                      static_cast<cudaStream_t>(stream)));
}

exl3_status exl3_reconstruct_rotated(const uint16_t *trellis, int bits, int64_t K, int64_t n_stored, int64_t n0,
                                     int64_t n_cols, const void *su, const void *sv, void *w, int layout,
                                     void *stream) {
  if (K <= 0 || K % 128 || K > 131072 || n_stored <= 0 || n_stored % 128 || n_stored > ((int64_t)1 << 24) ||
      n0 < 0 || n0 % 128 || n_cols < 0 || n_cols % 128 || n0 + n_cols > n_stored ||
      (layout != EXL3_LAYOUT_KN && layout != EXL3_LAYOUT_NK))
    return EXL3_ERR_INVALID_ARG;
  if (!bits_supported(bits)) return EXL3_ERR_UNSUPPORTED_BITS;
  if (!aligned16(trellis) || !aligned16(su) || !aligned16(sv) || !aligned16(w)) return EXL3_ERR_ALIGNMENT;
  const DeviceInfo *dev = current_device();
  if (!dev) return EXL3_ERR_NOT_INITIALIZED;
  return from_cuda(launch_reconstruct_rotated(trellis, bits, K, n_stored, n0, n_cols, su, sv, w, layout,
                                              static_cast<cudaStream_t>(stream)));
}

size_t exl3_weight_rotated_workspace_bytes(int64_t K, int64_t n_gemm) {
  if (K <= 0 || K % 128 || K > 131072 || n_gemm <= 0 || n_gemm % 128 || n_gemm > ((int64_t)1 << 24)) return 0;
  const int64_t cols = n_gemm < EXL3_RECONSTRUCT_CHUNK_COLS ? n_gemm : EXL3_RECONSTRUCT_CHUNK_COLS;
  return (size_t)((cols + 255) / 256 * 256) * (size_t)K * 2;
}

exl3_status exl3_linear_weight_rotated(const void *x, int64_t M, int64_t K, const uint16_t *trellis, int bits,
                                       int64_t n_stored, int64_t n_gemm, const void *su, const void *sv, void *y,
                                       int y_dtype, void *workspace, size_t workspace_bytes, void *stream) {
  if (y_dtype != EXL3_F16 && y_dtype != EXL3_F32) return EXL3_ERR_INVALID_ARG;
  if (!linear_rows_ok(M) || !linear_shape_ok(K, n_stored, n_gemm)) return EXL3_ERR_INVALID_ARG;
  if (!bits_supported(bits)) return EXL3_ERR_UNSUPPORTED_BITS;
  if (!aligned16(x) || !aligned16(trellis) || !aligned16(su) || !aligned16(sv) || !aligned16(y) ||
      !aligned16(workspace))
    return EXL3_ERR_ALIGNMENT;
  const DeviceInfo *dev = current_device();
  if (!dev) return EXL3_ERR_NOT_INITIALIZED;
  const size_t need = exl3_weight_rotated_workspace_bytes(K, n_gemm);
  if (need == 0) return EXL3_ERR_INVALID_ARG;
  if (need > workspace_bytes) return EXL3_ERR_WORKSPACE_TOO_SMALL;
  if (M == 0) return EXL3_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t ysz = y_dtype == EXL3_F32 ? 4 : 2;
  const int64_t chunk_rows = (int64_t)(need / ((size_t)K * 2));
  for (int64_t c0 = 0; c0 < n_gemm; c0 += EXL3_RECONSTRUCT_CHUNK_COLS) {
    const int64_t nc = (n_gemm - c0) < EXL3_RECONSTRUCT_CHUNK_COLS ? (n_gemm - c0) : EXL3_RECONSTRUCT_CHUNK_COLS;
    cudaError_t e = launch_reconstruct_rotated(trellis, bits, K, n_stored, c0, nc, su, sv, workspace,
                                               EXL3_LAYOUT_NK, st);
    if (e != cudaSuccess) return EXL3_ERR_CUDA;
    PrefillLaunch p;
    p.xr = x;
    p.xr_rows = M;
    p.M = M;
    p.K = K;
    p.wt = workspace;
    p.chunk_rows = chunk_rows;
    p.nc = nc;
    p.sv = sv;  // unused: the weight carries sv
    p.y = static_cast<uint8_t *>(y) + (size_t)c0 * ysz;
    p.ldy = n_gemm;
    p.y_f32 = y_dtype == EXL3_F32;
    p.n_valid_local = nc;
    p.status = dev->status;
    p.num_sms = dev->num_sms;
    p.rotate = 0;
    e = launch_prefill_gemm(p, st);
    if (e != cudaSuccess) return EXL3_ERR_CUDA;
  }
  return EXL3_OK;
}

exl3_status exl3_linear(const void *x, int64_t M, int64_t K, const uint16_t *trellis, int bits, int64_t n_stored,
                        int64_t n_gemm, const void *su, const void *sv, void *y, int y_dtype, int64_t m_threshold,
                        void *workspace, size_t workspace_bytes, void *stream) {
  if (y_dtype != EXL3_F16 && y_dtype != EXL3_F32) return EXL3_ERR_INVALID_ARG;
  const DeviceInfo *dev = nullptr;
  WorkspaceLayout L;
  exl3_status s = validate_linear(x, M, K, trellis, bits, n_stored, n_gemm, su, sv, y, m_threshold, workspace,
                                  workspace_bytes, &dev, &L);
  if (s != EXL3_OK) return s;
  if (M == 0) return EXL3_OK;
  return run_linear(dev, L, x, M, K, trellis, bits, n_stored, n_gemm, n_gemm, su, sv, y, y_dtype, m_threshold,
                    static_cast<uint8_t *>(workspace), static_cast<cudaStream_t>(stream));
}

exl3_status exl3_logits_masked(const void *x, int64_t M, int64_t K, const uint16_t *trellis, int bits,
                               int64_t n_stored, int64_t n_gemm, int64_t n_decodable, const void *su,
                               const void *sv, float *logits, int32_t *argmax, int64_t m_threshold,
                               void *workspace, size_t workspace_bytes, void *stream) {
  if (n_decodable < 1 || n_decodable > n_gemm) return EXL3_ERR_INVALID_ARG;
  const DeviceInfo *dev = nullptr;
  WorkspaceLayout L;
  exl3_status s = validate_linear(x, M, K, trellis, bits, n_stored, n_gemm, su, sv, logits, m_threshold,
                                  workspace, workspace_bytes, &dev, &L);
  if (s != EXL3_OK) return s;
  if (!aligned16(argmax)) return EXL3_ERR_ALIGNMENT;
  if (M == 0) return EXL3_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  s = run_linear(dev, L, x, M, K, trellis, bits, n_stored, n_gemm, n_decodable, su, sv, logits, EXL3_F32,
                 m_threshold, static_cast<uint8_t *>(workspace), st);
  if (s != EXL3_OK) return s;
  return from_cuda(launch_argmax(logits, M, n_gemm, argmax, st));
}

exl3_status exl3_silu_mul(const void *gate, const void *up, void *out, int64_t n, void *stream) {
  if (n < 0 || n % 8) return EXL3_ERR_INVALID_ARG;
  if (!aligned16(gate) || !aligned16(up) || !aligned16(out)) return EXL3_ERR_ALIGNMENT;
  const DeviceInfo *dev = current_device();
  if (!dev) return EXL3_ERR_NOT_INITIALIZED;
  return from_cuda(launch_silu_mul(gate, up, out, n, dev->num_sms, static_cast<cudaStream_t>(stream)));
}

exl3_status exl3_selftest_wait_timeout(uint32_t limit_us, void *stream) {
  if (limit_us == 0 || limit_us > 2000000u) return EXL3_ERR_INVALID_ARG;
  const DeviceInfo *dev = current_device();
  if (!dev) return EXL3_ERR_NOT_INITIALIZED;
  return from_cuda(launch_wait_timeout_selftest(dev->status, (unsigned long long)limit_us * 1000ull,
                                                static_cast<cudaStream_t>(stream)));
}

int exl3_bounds_checked(void) { return EXL3_DEBUG_BOUNDS ? 1 : 0; }

exl3_status exl3_selftest_bounds(int *units_reported, int *units_total, void *stream) {
  if (!units_reported || !units_total) return EXL3_ERR_INVALID_ARG;
  *units_reported = 0;
  *units_total = 0;
  const DeviceInfo *dev = current_device();
  if (!dev) return EXL3_ERR_NOT_INITIALIZED;
#if EXL3_DEBUG_BOUNDS
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // An error recorded before the self-test is returned (and cleared) first.
  const exl3_status pending = exl3_get_device_status(stream);
  if (pending != EXL3_OK) return pending;
  cudaError_t (*const probes[])(cudaStream_t) = {bounds_probe_rotate,  bounds_probe_decode,
                                                 bounds_probe_fused,   bounds_probe_prefill,
                                                 bounds_probe_reconstruct, bounds_probe_reconstruct_rotated,
                                                 bounds_probe_fused_prefill};
  for (auto *probe : probes) {
    ++*units_total;
    if (probe(st) != cudaSuccess) return EXL3_ERR_CUDA;
    const exl3_status s = exl3_get_device_status(stream);
    if (s == EXL3_ERR_OUT_OF_BOUNDS) ++*units_reported;
    else if (s != EXL3_OK) return s;
  }
#else
  (void)stream;
#endif
  return EXL3_OK;
}

exl3_status exl3_get_device_status(void *stream) {
  const DeviceInfo *dev = current_device();
  if (!dev) return EXL3_ERR_NOT_INITIALIZED;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return EXL3_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return EXL3_ERR_CUDA;
  if (v != 0 && cudaMemset(dev->status, 0, sizeof(int)) != cudaSuccess) return EXL3_ERR_CUDA;
  return v == 0 ? EXL3_OK : static_cast<exl3_status>(v);
}

}  // extern "C"
