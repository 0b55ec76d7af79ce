// Host-side interfaces between the libexl3 translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace exl3 {

constexpr int kDecodeRows = 16;           // activation rows per decode-GEMM launch

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Shape rules every linear-layer entry point enforces before any launch:
// K and n_gemm multiples of 128, n_stored a multiple of 128 and at most 2^24
// columns, n_gemm <= n_stored, K <= 131072.
inline bool linear_shape_ok(int64_t K, int64_t n_stored, int64_t n_gemm) {
  return K > 0 && K % 128 == 0 && K <= 131072 && n_gemm > 0 && n_gemm % 128 == 0 && n_stored % 128 == 0 &&
         n_gemm <= n_stored && n_stored <= ((int64_t)1 << 24);
}
// Activation rows every linear-layer entry point accepts: 0 .. 2^31.
inline bool linear_rows_ok(int64_t M) { return M >= 0 && M <= ((int64_t)1 << 31); }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Stream-K assignment of the decode-shaped GEMM, per token-group variant
// (index 0: <= 8 rows, index 1: <= 16 rows): P warps in total over `grid`
// CTAs, at most smax partial slots per 128-column n-block.
struct DecodePlan {
  int64_t P[2] = {1, 1};
  int64_t grid[2] = {1, 1};
  int64_t smax[2] = {1, 1};
};
DecodePlan decode_plan(int64_t n_blocks, int64_t k_blocks, int num_sms);
size_t decode_partials_bytes(const DecodePlan &plan, int64_t n_blocks);

// Stream-K assignment of the fused tensor-core decode GEMM (16 < rows <= 256
// per launch) over (128-column n-block, 64-row k step) units.
constexpr int kFusedMaxRows = 256;
struct FusedPlan {
  int64_t TS = 0, P = 1, smax = 1;
};
FusedPlan fused_plan(int64_t n_blocks, int64_t K, int num_sms);
size_t fused_partials_bytes(const FusedPlan &f, int64_t n_blocks);

// Workspace layout shared by the size query and the calls.
struct WorkspaceLayout {
  DecodePlan plan;
  FusedPlan fplan;
  bool fused = false;  // a decode-shaped call with more than 16 rows is possible
  size_t partials_off = 0, partials_bytes = 0, xf_off = 0, xr_off = 0, wchunk_off = 0, total = 0;
  int64_t xr_rows = 0;      // rows of the rotated-activation buffer (multiple of 128)
  int64_t chunk_rows = 0;   // rows of the reconstruct chunk (multiple of 256)
  bool prefill = false;
};
bool workspace_layout(int64_t M_max, int64_t K, int64_t n_gemm, int bits, int64_t m_threshold,
                      int num_sms, WorkspaceLayout *out);

struct DecodeLaunch {
  const void *x;          // rows m0.. of x (fp16), ld = K
  int rows;               // 1..16
  int64_t K;
  const uint16_t *trellis;
  int bits;
  int64_t n_stored, n_gemm, n_valid;
  const void *su, *sv;
  void *y;                // rows m0.. of y, ld = n_gemm
  int y_f32;
  void *xf;               // rotated rows in mma fragment order, K * 32 bytes
  float *partials;        // n-blocks x smax slots x (8 or 16) x 128 fp32
  int *status;
  DecodePlan plan;
};

struct PrefillLaunch {
  const void *xr;         // rotated activations, xr_rows x K fp16
  int64_t xr_rows, M, K;
  const void *wt;         // reconstructed chunk, W^T, chunk_rows x K fp16
  int64_t chunk_rows, nc; // rows allocated / columns used (nc % 128 == 0)
  const void *sv;         // sv + c0
  void *y;                // y + c0 (element offset), ld = ldy
  int64_t ldy;
  int y_f32;
  int64_t n_valid_local;  // columns >= this are written as -inf
  int *status;
  int num_sms;
  int rotate = 1;         // 0: plain store of x . W (weight-side rotation variant), no sv
  float *partials = nullptr;  // fp32 slots for tail tiles split across CTAs (stream-K tail)
  size_t partials_bytes = 0;
};
// Size of the stream-K tail's partial slots for any prefill GEMM launch.
size_t prefill_tail_partials_bytes(int num_sms);

struct FusedLaunch {
  const void *xr;          // rotated rows m0.. (fp16), ld = K
  int64_t xr_rows, K;      // rows addressable from xr (>= 1)
  const uint16_t *trellis;
  int bits;
  int64_t n_stored, n_gemm, n_valid;
  const void *sv;
  void *y;                 // rows m0.. of y, ld = n_gemm
  int y_f32;
  float *partials;
  int *status;
  int rows;                // 17 .. 256
  FusedPlan plan;
};

// Fused prefill-shaped layer (decode in producer warps, CTA pairs, 512 x 256
// tiles): y = had_r_128(x' . W) * sv with the -inf mask past n_valid.
struct FusedPrefillLaunch {
  const void *xr;          // rotated rows (fp16), ld = K
  int64_t xr_rows, M, K;   // xr_rows >= M rounded up to 128
  const uint16_t *trellis;
  int bits;
  int64_t n_stored, n_gemm, n_valid;
  const void *sv;
  void *y;                 // M x n_gemm
  int y_f32;
  int *status;
  int num_sms;
};

// Each kernel translation unit's set-up; `status` is the device error word
// (bound into the unit's bounds checks in the bounds-checked build).
cudaError_t init_rotate_kernels(int *status);
cudaError_t init_fused_kernels(int *status);
cudaError_t init_fused_prefill_kernels(int *status);
cudaError_t launch_fused_prefill(const FusedPrefillLaunch &p, cudaStream_t st);
cudaError_t launch_fused_gemm(const FusedLaunch &p, cudaStream_t st);
// Sums the partial slots of shared n-blocks (slot order), output rotation,
// sv, mask, store. Units are k slabs (decode GEMM) or k steps (fused GEMM).
cudaError_t launch_decode_finalize(const float *partials, int64_t smax, int64_t slot_elems, const void *sv, void *y,
                                   int y_f32, int64_t n_gemm, int64_t n_valid, int rows, int64_t P, int64_t TS,
                                   int units_per_block, int all_blocks, cudaStream_t st);
cudaError_t init_reconstruct_kernels(int *status);
cudaError_t init_reconstruct_rotated_kernels(int *status);
cudaError_t launch_reconstruct_rotated(const uint16_t *trellis, int bits, int64_t K, int64_t n_stored, int64_t n0,
                                       int64_t n_cols, const void *su, const void *sv, void *w, int layout,
                                       cudaStream_t st);
cudaError_t init_decode_kernels(int *status);
cudaError_t init_prefill_kernels(int *status);

#if EXL3_DEBUG_BOUNDS
// One probe launch per kernel translation unit (exl3_selftest_bounds).
cudaError_t bounds_probe_rotate(cudaStream_t st);
cudaError_t bounds_probe_decode(cudaStream_t st);
cudaError_t bounds_probe_fused(cudaStream_t st);
cudaError_t bounds_probe_fused_prefill(cudaStream_t st);
cudaError_t bounds_probe_prefill(cudaStream_t st);
cudaError_t bounds_probe_reconstruct(cudaStream_t st);
cudaError_t bounds_probe_reconstruct_rotated(cudaStream_t st);
#endif

cudaError_t launch_hadamard128(const void *x, void *y, const void *pre, int64_t rows, int64_t cols,
                               int num_sms, cudaStream_t st);
// overlap: launched right after the input rotation of the prefill path, which
// it may run alongside (waits for it before exiting).
cudaError_t launch_reconstruct(const uint16_t *trellis, int bits, int64_t K, int64_t n_stored,
                               int64_t n0, int64_t n_cols, void *w, int layout, int num_sms,
                               cudaStream_t st, int overlap = 0);
cudaError_t launch_decode_gemm(const DecodeLaunch &p, cudaStream_t st);
cudaError_t launch_prefill_gemm(const PrefillLaunch &p, cudaStream_t st);
cudaError_t launch_argmax(const float *logits, int64_t M, int64_t n, int32_t *argmax,
                          cudaStream_t st);

bool bits_supported(int bits);

// 2-D TMA descriptor (row-major, dim0 contiguous), OOB reads as zero.
bool encode_tensor_map_2d(CUtensorMap *m, CUtensorMapDataType type, const void *ptr, uint64_t dim0, uint64_t dim1,
                          uint64_t stride_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle);

struct DeviceInfo;
// The current device's cached set-up, or nullptr before exl3_init.
const DeviceInfo *initialized_device();
cudaError_t launch_silu_mul(const void *gate, const void *up, void *out, int64_t n, int num_sms, cudaStream_t st);
cudaError_t launch_wait_timeout_selftest(int *status, unsigned long long limit_ns, cudaStream_t st);

}  // namespace exl3
