/*
 * Plain CPU oracle for the EXL3-style trellis-quantized linear layer
 *
 *     y = had_r_128( had_r_128(x * su) . W ) * sv
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg load this file. The library's product path
 * never calls it, and it shares no code, header, table or constant with the
 * CUDA kernels.
 *
 * Sources of the arithmetic:
 *   - The op sequence had_r_128 -> reconstruct -> GEMM -> had_r_128 and the
 *     column slicing of the reconstructed weight: vLLM PR #316 "[EXL3]
 *     dispatch prefill-shaped GEMMs to reconstruct+hgemm", sections
 *     "Kernel measurements" and "Change".
 *   - The odd-width logits with pad columns forced to -inf before greedy
 *     selection: pegainfer PR #1046 "perf(qwen35): align the logits GEMM
 *     width ...", sections "Summary" and "Review follow-ups".
 *   - The pages leave the trellis bit layout, the per-state decode and the
 *     Hadamard ordering open. This library's storage-format specification
 *     fixes them, and this file follows it literally:
 *       * W (K x N) is stored as 16x16 tiles ordered row-major over
 *         (k/16, n/16), weights row-major inside a tile;
 *       * each tile owns a circular stream of 256*bits bits, held as
 *         little-endian uint16 words, read MSB-first inside each word;
 *       * weight i's 16-bit state is the circular window of stream bits
 *         that ends at bit (i+1)*bits-1 (earliest bit = state MSB);
 *       * u = state*89226354 + 64248484 (mod 2^32),
 *         u = (u & 0x8FFF8FFF) ^ 0x3B603B60, value = RNE_fp16(fp32(lo16(u)
 *         as fp16) + fp32(hi16(u) as fp16));
 *       * had_r_128 is the orthonormal 128-point Walsh-Hadamard transform in
 *         natural (Sylvester) order, H[i][j] = (-1)^popcount(i&j)/sqrt(128),
 *         applied to each 128-wide block.
 *
 * Precision choices (readings where the sources are silent):
 *   - the input rotation runs in fp32 with the butterfly stages in the order
 *     h = 1, 2, 4, ..., 64 and one final multiply by fp32(1/sqrt(128)); its
 *     result is rounded to fp16 (the GEMM's A operand is fp16);
 *   - the matmul accumulates in fp64 in ascending k; the output rotation and
 *     the sv scale run in fp64.
 *
 * Compiled with -O2 -ffp-contract=off; OpenMP only splits independent rows
 * and tiles across threads and never changes the order of any sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* fp16 <-> fp32, written out from the IEEE 754 binary16 definition           */
/* ------------------------------------------------------------------------ */

float oracle_half_to_float(uint16_t h)
{
    uint32_t sign = (h >> 15) & 1u;
    uint32_t exp = (h >> 10) & 0x1Fu;
    uint32_t man = h & 0x3FFu;
    float mag;
    if (exp == 0)
        mag = ldexpf((float)man, -24);                 /* subnormal: man * 2^-24 */
    else if (exp == 31)
        mag = man ? NAN : INFINITY;
    else
        mag = ldexpf((float)(man | 0x400u), (int)exp - 25); /* 1.man * 2^(exp-15) */
    return sign ? -mag : mag;
}

/* Round-to-nearest-even conversion of an fp32 value to binary16. */
uint16_t oracle_float_to_half_rne(float f)
{
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t exp = (x >> 23) & 0xFFu;
    uint32_t man = x & 0x7FFFFFu;
    if (exp == 0xFF)
        return (uint16_t)(sign | (man ? 0x7E00u : 0x7C00u));
    if (exp == 0)
        return sign; /* fp32 zero/subnormal: below 2^-126, rounds to signed zero */
    int e = (int)exp - 127;          /* value = sig * 2^(e-23) */
    uint32_t sig = man | 0x800000u;  /* 24 significant bits */
    int drop = (e >= -14) ? 13 : 13 + (-14 - e);
    if (drop > 25)
        return sign;                 /* below half the smallest subnormal */
    uint32_t kept = sig >> drop;
    uint32_t rem = sig & ((1u << drop) - 1u);
    uint32_t halfway = 1u << (drop - 1);
    if (rem > halfway || (rem == halfway && (kept & 1u)))
        kept++;
    if (e >= -14) {
        int E = e + 15;
        if (kept == 0x800u) { kept = 0x400u; E++; }
        if (E >= 31)
            return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | ((uint32_t)E << 10) | (kept & 0x3FFu));
    }
    return (uint16_t)(sign | kept);  /* subnormal (0x400 encodes the smallest normal) */
}

/* ------------------------------------------------------------------------ */
/* Trellis decode                                                             */
/* ------------------------------------------------------------------------ */

/* The raw LCG step u = state*89226354 + 64248484 (mod 2^32). */
uint32_t oracle_lcg_raw(uint32_t state)
{
    return state * 89226354u + 64248484u;
}

/* The masked word: (u & 0x8FFF8FFF) ^ 0x3B603B60. */
uint32_t oracle_lcg_masked(uint32_t state)
{
    return (oracle_lcg_raw(state) & 0x8FFF8FFFu) ^ 0x3B603B60u;
}

/* One 16-bit state to its fp16 weight (returned as binary16 bits). */
uint16_t oracle_decode_state(uint32_t state)
{
    uint32_t u = oracle_lcg_masked(state & 0xFFFFu);
    float lo = oracle_half_to_float((uint16_t)(u & 0xFFFFu));
    float hi = oracle_half_to_float((uint16_t)(u >> 16));
    return oracle_float_to_half_rne(lo + hi);
}

/* Stream bit j of a tile: word j/16, read MSB-first. */
static uint32_t stream_bit(const uint16_t *words, int64_t j)
{
    return (uint32_t)(words[j >> 4] >> (15 - (j & 15))) & 1u;
}

/*
 * Tail-biting walk: preload the 16-bit register with the last (16-bits)
 * stream bits, then for each weight shift in its `bits` bits; the register
 * after weight i's bits is weight i's state.
 */
void oracle_tile_states_walk(const uint16_t *words, int bits, uint16_t *states256)
{
    int64_t L = 256 * (int64_t)bits;
    uint32_t s = 0;
    for (int64_t j = L - (16 - bits); j < L; ++j)
        s = ((s << 1) | stream_bit(words, j)) & 0xFFFFu;
    for (int i = 0; i < 256; ++i) {
        for (int b = 0; b < bits; ++b)
            s = ((s << 1) | stream_bit(words, (int64_t)i * bits + b)) & 0xFFFFu;
        states256[i] = (uint16_t)s;
    }
}

/* Direct circular window: bits e-15 .. e (mod L), e = (i+1)*bits-1, MSB first. */
void oracle_tile_states_window(const uint16_t *words, int bits, uint16_t *states256)
{
    int64_t L = 256 * (int64_t)bits;
    for (int i = 0; i < 256; ++i) {
        int64_t e = (int64_t)(i + 1) * bits - 1;
        uint32_t s = 0;
        for (int t = 0; t < 16; ++t) {
            int64_t j = ((e - 15 + t) % L + L) % L;
            s |= stream_bit(words, j) << (15 - t);
        }
        states256[i] = (uint16_t)s;
    }
}

/* All 256 decoded weights of one tile (walk decoder), binary16 bits. */
void oracle_decode_tile(const uint16_t *words, int bits, uint16_t *w256)
{
    uint16_t st[256];
    oracle_tile_states_walk(words, bits, st);
    for (int i = 0; i < 256; ++i)
        w256[i] = oracle_decode_state(st[i]);
}

/*
 * Reconstruct columns [n0, n0+ncols) of W (K x n_stored) into w (K x ncols,
 * row-major, binary16 bits). n0 and ncols are multiples of 16.
 */
void oracle_reconstruct(const uint16_t *trellis, int bits, int64_t K, int64_t n_stored,
                        int64_t n0, int64_t ncols, uint16_t *w)
{
    int64_t tiles_n = n_stored / 16;
    int64_t wpt = 16 * (int64_t)bits;
    int64_t tk_count = K / 16;
#pragma omp parallel for schedule(static)
    for (int64_t tk = 0; tk < tk_count; ++tk) {
        uint16_t v[256];
        for (int64_t tn = n0 / 16; tn < (n0 + ncols) / 16; ++tn) {
            oracle_decode_tile(trellis + (tk * tiles_n + tn) * wpt, bits, v);
            for (int r = 0; r < 16; ++r)
                for (int c = 0; c < 16; ++c)
                    w[(tk * 16 + r) * ncols + (tn * 16 - n0) + c] = v[r * 16 + c];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Walsh-Hadamard                                                             */
/* ------------------------------------------------------------------------ */

/* Unnormalised in-place fast WHT of 128 floats, stages h = 1, 2, ..., 64. */
static void fwht128_f32(float *v)
{
    for (int h = 1; h < 128; h <<= 1)
        for (int i = 0; i < 128; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                float a = v[j], b = v[j + h];
                v[j] = a + b;
                v[j + h] = a - b;
            }
}

static void fwht128_f64(double *v)
{
    for (int h = 1; h < 128; h <<= 1)
        for (int i = 0; i < 128; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                double a = v[j], b = v[j + h];
                v[j] = a + b;
                v[j + h] = a - b;
            }
}

/* Orthonormal had_r_128 of every 128-block of an fp64 vector (length n). */
void oracle_hadamard128_f64(const double *in, double *out, int64_t n)
{
    double scale = 1.0 / sqrt(128.0);
    for (int64_t b = 0; b < n; b += 128) {
        double v[128];
        for (int i = 0; i < 128; ++i) v[i] = in[b + i];
        fwht128_f64(v);
        for (int i = 0; i < 128; ++i) out[b + i] = v[i] * scale;
    }
}

/* Orthonormal had_r_128 of every 128-block of an fp32 vector (length n). */
void oracle_hadamard128_f32(const float *in, float *out, int64_t n)
{
    float scale = (float)(1.0 / sqrt(128.0));
    for (int64_t b = 0; b < n; b += 128) {
        float v[128];
        for (int i = 0; i < 128; ++i) v[i] = in[b + i];
        fwht128_f32(v);
        for (int i = 0; i < 128; ++i) out[b + i] = v[i] * scale;
    }
}

/*
 * Input rotation x' = RNE_fp16(had_r_128(x * su)) per 128-block of each row,
 * in fp32. su may be NULL (no pre-scale). x, su, out are binary16 bits.
 */
void oracle_input_rotation(const uint16_t *x, const uint16_t *su, int64_t rows, int64_t cols,
                           uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < rows; ++m) {
        float v[128], r[128];
        for (int64_t b = 0; b < cols; b += 128) {
            for (int i = 0; i < 128; ++i) {
                float xv = oracle_half_to_float(x[m * cols + b + i]);
                v[i] = su ? xv * oracle_half_to_float(su[b + i]) : xv;
            }
            oracle_hadamard128_f32(v, r, 128);
            for (int i = 0; i < 128; ++i)
                out[m * cols + b + i] = oracle_float_to_half_rne(r[i]);
        }
    }
}

/*
 * Weight-side rotation variant: columns [n0, n0+ncols) of
 *     W' = diag(su) . had_r_128(K) . W . had_r_128(N) . diag(sv)
 * (the rotations of the linear layer moved onto the weight, so that
 * x . W' = had_r_128(had_r_128(x * su) . W) * sv in exact arithmetic; the
 * "reconstruct_had_slice" of vLLM PR #316, section "Kernel measurements").
 * The pages do not give its arithmetic; this library defines it per
 * 128 x 128 block of W as:
 *   1. t = fp32(w);
 *   2. fast WHT of every column along k, fp32, stages h = 1, 2, ..., 64;
 *   3. t = t * fp32(su[k])                      (fp32 product);
 *   4. fast WHT of every row along n, same stages;
 *   5. t = t * 2^-7                              (exact: the two 1/sqrt(128));
 *   6. t = t * fp32(sv[n])                      (fp32 product);
 *   7. RNE to fp16.
 * layout 0: out is K x ncols (ld ncols); layout 1: ncols x K (ld K).
 */
int oracle_reconstruct_rotated(const uint16_t *trellis, int bits, int64_t K, int64_t n_stored,
                               const uint16_t *su, const uint16_t *sv, int64_t n0, int64_t ncols,
                               int layout, uint16_t *out)
{
    if (K % 128 || n0 % 128 || ncols % 128 || n0 + ncols > n_stored || bits < 1 || bits > 8 ||
        (layout != 0 && layout != 1))
        return -1;
    uint16_t *w = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(K * ncols));
    if (!w) return -2;
    oracle_reconstruct(trellis, bits, K, n_stored, n0, ncols, w);
    int64_t nkb = K / 128, nnb = ncols / 128;
#pragma omp parallel for schedule(static)
    for (int64_t blk = 0; blk < nkb * nnb; ++blk) {
        int64_t kb = blk / nnb, nb = blk % nnb;
        float *t = (float *)malloc(sizeof(float) * 128 * 128);
        float col[128];
        for (int i = 0; i < 128; ++i)
            for (int j = 0; j < 128; ++j)
                t[i * 128 + j] = oracle_half_to_float(w[(kb * 128 + i) * ncols + nb * 128 + j]);
        for (int j = 0; j < 128; ++j) {
            for (int i = 0; i < 128; ++i) col[i] = t[i * 128 + j];
            fwht128_f32(col);
            for (int i = 0; i < 128; ++i) t[i * 128 + j] = col[i];
        }
        for (int i = 0; i < 128; ++i) {
            float s = oracle_half_to_float(su[kb * 128 + i]);
            for (int j = 0; j < 128; ++j) t[i * 128 + j] = t[i * 128 + j] * s;
            fwht128_f32(t + i * 128);
        }
        for (int i = 0; i < 128; ++i)
            for (int j = 0; j < 128; ++j) {
                float v = t[i * 128 + j] * 0.0078125f;
                v = v * oracle_half_to_float(sv[n0 + nb * 128 + j]);
                int64_t k = kb * 128 + i, n = nb * 128 + j;
                out[layout == 0 ? k * ncols + n : n * K + k] = oracle_float_to_half_rne(v);
            }
        free(t);
    }
    free(w);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Linear layer                                                               */
/* ------------------------------------------------------------------------ */

/*
 * y[:, 0:ncols] = output columns [c0, c0+ncols) of
 *     had_r_128( RNE_fp16(had_r_128(x * su)) . W ) * sv
 * for all M rows, in fp64. c0 and ncols are multiples of 128.
 * x: M x K binary16; su: K; sv: n_stored; y: M x ncols doubles.
 */
int oracle_linear(const uint16_t *x, int64_t M, int64_t K, const uint16_t *trellis, int bits,
                  int64_t n_stored, const uint16_t *su, const uint16_t *sv, int64_t c0,
                  int64_t ncols, double *y)
{
    if (K % 128 || c0 % 128 || ncols % 128 || c0 + ncols > n_stored || bits < 1 || bits > 8)
        return -1;
    uint16_t *xr = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(M * K));
    uint16_t *w = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(K * ncols));
    float *h2f = (float *)malloc(sizeof(float) * 65536);
    if (!xr || !w || !h2f) {
        free(xr); free(w); free(h2f);
        return -2;
    }
    for (int i = 0; i < 65536; ++i) h2f[i] = oracle_half_to_float((uint16_t)i);
    oracle_input_rotation(x, su, M, K, xr);
    oracle_reconstruct(trellis, bits, K, n_stored, c0, ncols, w);
    int64_t nblk = ncols / 128;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t mb = 0; mb < M * nblk; ++mb) {
        int64_t m = mb / nblk, b = mb % nblk;
        double acc[128], rot[128];
        for (int j = 0; j < 128; ++j) acc[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double xv = (double)h2f[xr[m * K + k]];
            const uint16_t *wrow = w + k * ncols + b * 128;
            for (int j = 0; j < 128; ++j) acc[j] += xv * (double)h2f[wrow[j]];
        }
        oracle_hadamard128_f64(acc, rot, 128);
        for (int j = 0; j < 128; ++j)
            y[m * ncols + b * 128 + j] = rot[j] * (double)h2f[sv[c0 + b * 128 + j]];
    }
    free(xr); free(w); free(h2f);
    return 0;
}

/*
 * Masked logits and greedy selection over an already computed logits block:
 * columns [n_decodable, n_gemm) are set to -inf, then argmax per row over
 * [0, n_gemm), first index on ties. skip_mask != 0 leaves the pad columns
 * untouched (a planted mistake for the invariant test's mutation check).
 */
void oracle_mask_argmax(double *logits, int64_t M, int64_t n_gemm, int64_t n_decodable,
                        int32_t *argmax, int skip_mask)
{
    for (int64_t m = 0; m < M; ++m) {
        double *row = logits + m * n_gemm;
        if (!skip_mask)
            for (int64_t n = n_decodable; n < n_gemm; ++n) row[n] = -INFINITY;
        int64_t best = 0;
        for (int64_t n = 1; n < n_gemm; ++n)
            if (row[n] > row[best]) best = n;
        argmax[m] = (int32_t)best;
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
