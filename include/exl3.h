/*
 * exl3.h — C ABI of libexl3.so, a single-GPU (sm_103a) implementation of the
 * EXL3-style trellis-quantized linear layer
 *
 *     y = had_r_128( had_r_128(x * su) . W ) * sv
 *
 * Sources of the operations (page title, section):
 *   [P1] vLLM PR #316, "[EXL3] dispatch prefill-shaped GEMMs to
 *        reconstruct+hgemm (+113 % prefill, decode unchanged)": sections
 *        "Problem", "Kernel measurements", "Change".
 *   [P2] vLLM PR #314, "[EXL3] allow CUDA-graph decode for dense checkpoints
 *        by priming exl3_gemm autotune": sections "Problem", "Change".
 *   [P3] pegainfer PR #1046, "perf(qwen35): align the logits GEMM width so
 *        the output projection stops landing on an align-1 sm_75 kernel":
 *        sections "Summary", "Review follow-ups", "Testing".
 *
 * Storage format of W (the pages leave it open; this library fixes it):
 *   W is K x n_stored. It is stored as 16x16 tiles ordered row-major over
 *   (k/16, n/16), weights row-major inside a tile. Tile t owns 16*bits
 *   little-endian uint16 words at trellis[t*16*bits ...], a circular stream
 *   of 256*bits bits read MSB-first inside each word. Weight i of a tile
 *   has as its 16-bit state the circular window of stream bits ending at bit
 *   (i+1)*bits-1 (earliest bit = most significant). Its value is
 *       u = state*89226354 + 64248484 (mod 2^32)
 *       u = (u & 0x8FFF8FFF) ^ 0x3B603B60
 *       w = RNE_fp16( fp32(fp16 bits u[15:0]) + fp32(fp16 bits u[31:16]) ).
 *   had_r_128 is the orthonormal 128-point Walsh-Hadamard transform in
 *   natural (Sylvester) order, H[i][j] = (-1)^popcount(i&j) / sqrt(128),
 *   applied to every 128-wide block.
 *
 * General conventions:
 *   - Every data pointer is a caller-owned DEVICE pointer that must be
 *     16-byte aligned. The library never allocates or frees device memory
 *     and never synchronizes a stream except in exl3_get_device_status.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - Matrices are row-major and densely packed unless a leading dimension
 *     is stated.
 *   - Arguments are validated before anything is launched; a rejected call
 *     launches nothing and returns the named status. A failed launch
 *     returns EXL3_ERR_CUDA.
 *   - exl3_init(device) must run once per device, with that device
 *     current, before any other call that touches it and before any CUDA
 *     graph capture: it loads every kernel and sets their attributes, so
 *     no later call loads modules, allocates or queries the device.
 *   - Consecutive kernels of one call overlap their launches through
 *     programmatic dependent launch; each waits for its predecessor before
 *     touching memory it shares with it. The last kernel of a call lets the
 *     next kernel in the stream begin early as well: a caller kernel that
 *     opts into programmatic stream serialization must, as that contract
 *     requires, wait on its grid dependency (cudaGridDependencySynchronize)
 *     before reading this call's outputs. Ordinary launches are unaffected.
 *   - Supported trellis widths: bits in 1..8.
 *   - Shapes: K % 128 == 0, K <= 131072, n_gemm % 128 == 0,
 *     n_gemm <= n_stored, n_stored % 128 == 0, n_stored <= 2^24; others
 *     return EXL3_ERR_INVALID_ARG.
 */
#ifndef EXL3_H_
#define EXL3_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EXL3_OK = 0,
    EXL3_ERR_INVALID_ARG = 1,        /* a shape, size or enum is out of range */
    EXL3_ERR_ALIGNMENT = 2,          /* a pointer is NULL or not 16-byte aligned */
    EXL3_ERR_UNSUPPORTED_BITS = 3,   /* bits is not a supported trellis width */
    EXL3_ERR_WORKSPACE_TOO_SMALL = 4,/* workspace_bytes below the required size */
    EXL3_ERR_NOT_INITIALIZED = 5,    /* exl3_init was not called for the current device */
    EXL3_ERR_CUDA = 6,               /* a CUDA runtime call or a launch failed */
    EXL3_ERR_DEVICE_TIMEOUT = 7,     /* a kernel gave up a bounded wait (see exl3_get_device_status) */
    EXL3_ERR_NOALLOC_TOO_LARGE = 8,  /* the problem needs more scratch than the fixed no-alloc buffer holds */
    EXL3_ERR_OUT_OF_BOUNDS = 9       /* bounds-checked build only: a kernel's index left its buffer */
} exl3_status;

typedef enum { EXL3_F16 = 0, EXL3_F32 = 1 } exl3_dtype;

/* Layout of a reconstructed weight slice. */
typedef enum {
    EXL3_LAYOUT_KN = 0, /* w[k][j] = W[k][n0+j], K rows of n_cols, ld = n_cols */
    EXL3_LAYOUT_NK = 1  /* w[j][k] = W[k][n0+j], n_cols rows of K, ld = K (GEMM operand layout) */
} exl3_layout;

/* Columns reconstructed per prefill chunk; bounds the scratch at
 * 32768*K*2 bytes ([P1] "Change": 336 MB at K = 5120). */
#define EXL3_RECONSTRUCT_CHUNK_COLS 32768

/*
 * exl3_init: one-time set-up for `device` (made current by this call).
 * Loads all kernels, raises their shared-memory limits and caches the SM
 * count. Idempotent. Call before any stream capture ([P2] "Change": every
 * lazy initialisation must happen before capture).
 * Errors: EXL3_ERR_INVALID_ARG (no such device), EXL3_ERR_CUDA.
 */
exl3_status exl3_init(int device);

/* Static English text for a status code (never NULL). */
const char *exl3_status_string(int status);

/* 1 if `bits` is a supported trellis width, else 0. Host only. */
int exl3_supported_bits(int bits);

/*
 * Logits GEMM width for an odd decodable vocabulary: n_decodable rounded up
 * to a multiple of 128, clamped to n_stored ([P3] "Summary": 248077 ->
 * 248192 <= 248320). Returns -1 on invalid input. Host only.
 */
int64_t exl3_aligned_logits_width(int64_t n_decodable, int64_t n_stored);

/*
 * The decode-shaped path's work split for a (K, n_gemm) geometry on a GPU
 * with `num_sms` SMs, for calls of at most 8 rows: the whole (128-column
 * n-block x 16-row k slab) space is cut into equal contiguous ranges, one
 * per warp (stream-K); *splits receives the largest number of warps that
 * share one n-block (its partial-sum slots) and *ctas_per_split the number
 * of CTAs launched. Returns 0, or -1 on invalid input. Host only.
 */
int exl3_decode_plan(int64_t K, int64_t n_gemm, int num_sms, int *splits, int *ctas_per_split);

/*
 * The kernels a prefill-shaped call (m_threshold > 0 and M >= m_threshold)
 * of M rows takes on a layer n_gemm columns wide, on a GPU with `num_sms`
 * SMs: 1 for the fused prefill kernel, whose producer warps decode the
 * trellis straight into the tensor-core operand (the "dequant fused into
 * the GEMM" of [P1] "The remaining gap is structural"), used for
 * M <= 512 on layers with at least 0.3 x num_sms column blocks of 256; 0 for
 * reconstruct (32768-column chunks) followed by the tensor-core GEMM.
 * Both apply the input and output rotations, sv and the logits mask.
 * Returns -1 on invalid input (M < 1, n_gemm not a positive multiple of
 * 128, num_sms < 1). Host only.
 */
int exl3_prefill_path(int64_t M, int64_t n_gemm, int num_sms);

/*
 * Workspace bytes an exl3_linear / exl3_logits_masked call with M <= M_max
 * needs on a GPU with `num_sms` streaming multiprocessors. The workspace is
 * laid out as: split-K partial sums (shared by the decode-shaped kernels
 * and, when a prefill-shaped call is possible, the prefill GEMM's split
 * tail tiles: at most 3 x num_sms fp32 128 x 256 tiles) and rotated
 * activations; then, when a prefill-shaped call is possible (m_threshold > 0
 * and M_max >= m_threshold), the rotated activations (M_max x K fp16) and
 * one reconstruct chunk (min(n_gemm, 32768) x K fp16) ([P1] "Change": one
 * scratch per geometry, reused by every layer of that geometry on one
 * stream). Returns 0 for invalid arguments. Host only.
 */
size_t exl3_linear_workspace_bytes_for(int64_t M_max, int64_t K, int64_t n_gemm, int bits,
                                       int64_t m_threshold, int num_sms);

/* Same, for the current device's SM count (queried, not allocated). */
size_t exl3_linear_workspace_bytes(int64_t M_max, int64_t K, int64_t n_gemm, int bits,
                                   int64_t m_threshold);

/*
 * Clears a workspace (cudaMemsetAsync on `stream`). Optional: no call needs
 * particular initial workspace contents; it only makes a fresh buffer's
 * contents defined.
 */
exl3_status exl3_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/*
 * exl3_hadamard128: y = RNE_fp16( had_r_128(x * pre_scale) ) on every
 * 128-block of each row ([P1] "Kernel measurements": the had_r_128 stage).
 *   x, y:       rows x cols fp16 (may alias for an in-place transform).
 *   pre_scale:  cols fp16, or NULL for none (su of the layer).
 *   cols % 128 == 0, rows >= 0.
 * Arithmetic: fp32, butterfly stages h = 1, 2, 4, ..., 64, then one multiply
 * by fp32(1/sqrt(128)), then round to nearest even.
 */
exl3_status exl3_hadamard128(const void *x, void *y, const void *pre_scale, int64_t rows,
                             int64_t cols, void *stream);

/*
 * exl3_reconstruct: decode columns [n0, n0+n_cols) of W from the trellis
 * ([P1] "Kernel measurements", "Change": reconstruct / reconstruct_slice).
 *   trellis: tiles of the K x n_stored matrix (format above), uint16.
 *   w:       fp16 output in `layout` (exl3_layout).
 *   n0 % 128 == 0, n_cols % 128 == 0, n0 + n_cols <= n_stored.
 * Output is bit-exact with the format definition.
 */
exl3_status exl3_reconstruct(const uint16_t *trellis, int bits, int64_t K, int64_t n_stored,
                             int64_t n0, int64_t n_cols, void *w, int layout, void *stream);

/*
 * Weight-side rotation variant ([P1] "Kernel measurements":
 * reconstruct_had_slice). Moves both rotations and both scales onto the
 * weight, W' = diag(su) . had_r_128(K) . W . had_r_128(N) . diag(sv), so the
 * prefill-shaped layer is the plain product y = x . W'. The pages give no
 * arithmetic for it; this library defines it per 128 x 128 block of W as
 * fp32(w) -> fast WHT of each column along k (fp32, stages h = 1 .. 64)
 * -> * fp32(su[k]) -> fast WHT of each row along n -> * 2^-7 (exact)
 * -> * fp32(sv[n]) -> round to nearest even fp16, and the output is
 * bit-exact with that definition.
 *
 * exl3_reconstruct_rotated: columns [n0, n0+n_cols) of W' into `w`
 *   (fp16, `layout` as exl3_reconstruct); su: K fp16, sv: n_stored fp16.
 *   K % 128 == 0, n0 % 128 == 0, n_cols % 128 == 0, n0 + n_cols <= n_stored.
 *
 * exl3_weight_rotated_workspace_bytes: scratch for
 *   exl3_linear_weight_rotated (one 32768-column W'^T slice), 0 if invalid.
 *
 * exl3_linear_weight_rotated: y = x . W'[:, :n_gemm], reconstructing W' in
 *   32768-column slices into the caller's workspace and running the
 *   tensor-core GEMM without input or output rotation. x: M x K fp16 (not
 *   rotated); y: M x n_gemm (`y_dtype`), ld = n_gemm; fp32 accumulation.
 *   It differs from exl3_linear by where the fp16 roundings fall (W' instead
 *   of x'): max|y - y_linear| / rms(y_linear) stays below 3e-3.
 *   Errors as exl3_linear (EXL3_ERR_WORKSPACE_TOO_SMALL below the size above).
 */
exl3_status exl3_reconstruct_rotated(const uint16_t *trellis, int bits, int64_t K, int64_t n_stored,
                                     int64_t n0, int64_t n_cols, const void *su, const void *sv, void *w,
                                     int layout, void *stream);
size_t exl3_weight_rotated_workspace_bytes(int64_t K, int64_t n_gemm);
exl3_status exl3_linear_weight_rotated(const void *x, int64_t M, int64_t K, const uint16_t *trellis, int bits,
                                       int64_t n_stored, int64_t n_gemm, const void *su, const void *sv, void *y,
                                       int y_dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * exl3_linear: y = had_r_128( RNE_fp16(had_r_128(x * su)) . W[:, :n_gemm] )
 *                  * sv[:n_gemm]
 *   x:     M x K fp16.            su: K fp16.         sv: n_stored fp16.
 *   y:     M x n_gemm, `y_dtype` (EXL3_F32 or EXL3_F16 = RNE of the fp32
 *          result), ld = n_gemm.
 *   m_threshold: path choice made inside this call on its own M ([P1]
 *          "Change": the dispatch must live inside the op, not in a branch
 *          a tracer can freeze). M < m_threshold, or m_threshold == 0,
 *          takes the decode-shaped path, where the trellis is decoded
 *          inside the GEMM and never materialised: for M <= 16 a stream-K
 *          kernel with the decoded weights as the mma.sync operand; for
 *          larger M one tensor-core (tcgen05) kernel per 256 rows whose
 *          producer warps decode straight into the MMA operand buffers.
 *          Otherwise the prefill-shaped path runs had_r_128, then either
 *          (M <= 512 on a layer with at least 0.3 x SMs column blocks of
 *          256) one fused tensor-core kernel whose producer warps decode
 *          straight into the MMA operand, 512 rows per decoded tile, or
 *          reconstruct (32768-column chunks into the workspace) followed by
 *          a tensor-core GEMM; both apply the output rotation, sv and the
 *          mask in their epilogue. On one GB300 the prefill-shaped path is
 *          faster from M = 384 (4-bit 5120 -> 17408) and from M = 768
 *          (4-bit 17408 -> 5120).
 *   workspace: device buffer of at least
 *          exl3_linear_workspace_bytes(M, K, n_gemm, bits, m_threshold)
 *          bytes, cleared once by exl3_workspace_init. Calls that share a
 *          workspace must be ordered (same stream, or synchronised).
 * Accumulation is fp32. M == 0 is a no-op.
 */
exl3_status exl3_linear(const void *x, int64_t M, int64_t K, const uint16_t *trellis, int bits,
                        int64_t n_stored, int64_t n_gemm, const void *su, const void *sv, void *y,
                        int y_dtype, int64_t m_threshold, void *workspace, size_t workspace_bytes,
                        void *stream);

/*
 * exl3_logits_masked: the logits projection with the pad mask and greedy
 * selection fused behind one entry point, so the GEMM cannot be reached
 * without the mask ([P3] "Review follow-ups": output_logits_into owns both).
 *   logits: M x n_gemm fp32 (ld = n_gemm), = exl3_linear's fp32 output with
 *           columns [n_decodable, n_gemm) forced to -inf.
 *   argmax: M int32, the first index of each row's maximum.
 *   1 <= n_decodable <= n_gemm. Other arguments as exl3_linear.
 */
exl3_status exl3_logits_masked(const void *x, int64_t M, int64_t K, const uint16_t *trellis,
                               int bits, int64_t n_stored, int64_t n_gemm, int64_t n_decodable,
                               const void *su, const void *sv, float *logits, int32_t *argmax,
                               int64_t m_threshold, void *workspace, size_t workspace_bytes,
                               void *stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word, which holds the first device-side error since the last read:
 * EXL3_ERR_DEVICE_TIMEOUT if a kernel gave up one of its bounded waits,
 * EXL3_ERR_OUT_OF_BOUNDS if a check of the bounds-checked build failed;
 * EXL3_OK otherwise.
 * The word is one per device, shared by every stream and workspace on it
 * (some entry points that wait on the device have no workspace): with
 * several streams, a timeout is reported to whichever caller reads first.
 */
exl3_status exl3_get_device_status(void *stream);

/*
 * exl3_silu_mul: out = RNE_fp16(silu(gate) * up) elementwise (fp32 math,
 * silu(a) = a / (1 + exp(-a))), n % 8 == 0. The glue between the gate/up
 * and down projections of a dense MLP ([P1] follow-up comment: gate + up +
 * down per layer); not itself part of the trellis layer.
 */
exl3_status exl3_silu_mul(const void *gate, const void *up, void *out, int64_t n, void *stream);

/*
 * Self-test of the failure-detection path: launches one kernel that waits
 * on a barrier nothing will complete, gives up after limit_us microseconds
 * (1 .. 2,000,000) and records EXL3_ERR_DEVICE_TIMEOUT in the device error
 * word, which exl3_get_device_status then returns. The kernel always
 * returns on its own; it neither traps nor faults. The pages have no
 * counterpart; it exercises the bounded waits every pipelined kernel uses.
 */
exl3_status exl3_selftest_wait_timeout(uint32_t limit_us, void *stream);

/*
 * Bounds-checked build. The same sources compiled with EXL3_DEBUG_BOUNDS=1
 * give libexl3_bounds.so, with the same entry points. Before each access,
 * its kernels check against the extents implied by the launch's arguments:
 *   - every computed global index;
 *   - every shared-memory address and mbarrier;
 *   - every TMA coordinate and bulk-copy span;
 *   - every TMEM column.
 * A failed check skips the access (a load reads zero) and records
 * EXL3_ERR_OUT_OF_BOUNDS in the device error word. It also prints the
 * source line once. The check stands in for a memory checker; the pages
 * have no counterpart to it.
 *
 * exl3_bounds_checked: 1 in the bounds-checked library, 0 in libexl3.so.
 * Host only.
 *
 * exl3_selftest_bounds: checks that every kernel translation unit of the
 * bounds-checked build reports to the device error word. It launches one
 * probe kernel per unit, on `stream`. Each probe submits an index equal to
 * its extent to the checks and touches no memory. After each probe the
 * word is read and cleared.
 *   *units_total   receives the number of units probed.
 *   *units_reported receives how many recorded EXL3_ERR_OUT_OF_BOUNDS.
 * In libexl3.so it launches nothing and sets both to 0.
 * An error already pending in the word is returned (and cleared) before
 * any probe runs.
 * Synchronises `stream`.
 * Errors: EXL3_ERR_INVALID_ARG (NULL pointer), EXL3_ERR_NOT_INITIALIZED,
 * EXL3_ERR_CUDA.
 */
int exl3_bounds_checked(void);
exl3_status exl3_selftest_bounds(int *units_reported, int *units_total, void *stream);

/*
 * exl3_linear_decode_noalloc: the decode-shaped linear layer for callers
 * that cannot allocate device memory: a
 * plugin inside a host program that owns every device buffer, or code that
 * must not call cudaMalloc at run time because it synchronises the whole
 * device. The caller passes only inputs and outputs; the split-K partial
 * sums and rotated activations live in a fixed 24 MiB buffer inside the
 * library (a static device array that every GPU which loads libexl3.so
 * keeps until the process exits). The pages have no counterpart to this
 * entry point.
 *   Arguments as exl3_linear, without m_threshold and workspace; the same
 *   shape, row-count, bit-width and alignment rules, with the same status
 *   codes.
 *   Kernels: the rows run in groups of up to 16 through the 16-row
 *   decode-shaped kernel (exactly what exl3_linear runs for M <= 16). For
 *   M > 16 exl3_linear switches to its tensor-core kernel, which needs a
 *   rotated copy of all M rows in the workspace; this entry point instead
 *   repeats the 16-row kernel ceil(M/16) times, so its cost grows about
 *   ceil(M/16)-fold over the M = 16 call (results agree with exl3_linear
 *   within the layer tolerance, not bit for bit).
 *   Limit: exl3_linear_workspace_bytes(16, K, n_gemm, bits, 0) must not
 *   exceed EXL3_NOALLOC_SCRATCH_BYTES (24 MiB; the MLP projections fit, a
 *   248192-wide logits layer does not); larger problems return
 *   EXL3_ERR_NOALLOC_TOO_LARGE and launch nothing.
 *   The first call on a device looks up the buffer's device address, so
 *   make that first call before any stream capture. No call needs the
 *   buffer to start at zero. Every call shares the one buffer
 *   and it keeps the last call's contents, so calls that may overlap on the
 *   GPU (different streams, no ordering) race: order them. It never calls
 *   cudaMalloc, cudaFree or any allocating routine. exl3_init must have run.
 */
#define EXL3_NOALLOC_SCRATCH_BYTES ((size_t)24 << 20)
exl3_status exl3_linear_decode_noalloc(const void *x, int64_t M, int64_t K, const uint16_t *trellis,
                                       int bits, int64_t n_stored, int64_t n_gemm, const void *su,
                                       const void *sv, void *y, int y_dtype, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* EXL3_H_ */
