/*
 * CPU oracle for the FP8 scaled linear layer.  TEST INFRASTRUCTURE ONLY: the
 * tests, the smoke check and the benchmark's CPU-baseline leg use it; the
 * product path never links, loads or calls it.
 *
 * Plain, single-threaded C.  Every result is computed from its definition:
 *   - E4M3 ("e4m3fn": 1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
 *     no infinities, 0x7F/0xFF are NaN, largest finite 448) is decoded from
 *     the bit fields and encoded by searching the table of representable
 *     values for the nearest one, ties to the even code, saturating at 448.
 *     The format and its 448 maximum come from the AstrAI page
 *     "astrai/extension/fp8_state.py", module constant E4M3_MAX; the
 *     saturating round-to-nearest-even cast is the plainest reading of
 *     saturating E4M3 quantisation where the pages name no rounding mode.
 *   - scale = amax/448 and scale_inv = 448/amax, each one IEEE fp32 division
 *     (same page, comment above FP8TensorMeta: the GEMM scales its product by
 *     both operands' scales, quantisation multiplies by 1/scale; _update_delayed_scale clamps the
 *     amax to at least 1e-12 and computes scale_inv directly, not as 1/scale).
 *   - GEMMs are summed in fp64 over dequantised values.  Every product of two
 *     e4m3 values is exact in fp64 and every partial sum of up to 2^15 such
 *     products is too (they are multiples of 2^-18 below 2^33), so the sum is
 *     the exact dot product whatever the order.
 *
 * Parity pins live in tests/test_oracle_*.py; every function below is pinned
 * there against a closed form, a library routine, brute force or an invariant.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define E4M3_MAX 448.0

/* ---------------------------------------------------------------- bf16 ---- */

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
float orc_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a double to the nearest bf16 value (8 significant bits, exponent
 * range of binary32), ties to even, and return that value as a double.
 * Overflow past the largest finite bf16 gives +-inf, as IEEE RNE does. */
double orc_round_to_bf16(double x)
{
    if (isnan(x) || isinf(x) || x == 0.0) return x;
    double a = fabs(x);
    int e;
    frexp(a, &e);                   /* a = f * 2^e, f in [0.5, 1) */
    int lead = e - 1;               /* 2^lead <= a < 2^(lead+1) */
    if (lead < -126) lead = -126;   /* below the normal range: fixed quantum */
    double quantum = ldexp(1.0, lead - 7);
    double r = nearbyint(a / quantum) * quantum; /* a/quantum is exact */
    double bf16_max = ldexp(255.0, 120);          /* (2 - 2^-7) * 2^127 */
    if (r > bf16_max) r = INFINITY;
    return x < 0 ? -r : r;
}

/* ---------------------------------------------------------------- e4m3 ---- */

/* Value of an e4m3fn code.  Exponent field 0 holds the subnormals
 * m/8 * 2^-6; otherwise (1 + m/8) * 2^(e-7).  0x7F and 0xFF are NaN. */
double orc_e4m3_decode(uint8_t c)
{
    int sign = c >> 7;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Encode a binary32 value as e4m3fn: round to the nearest representable
 * magnitude (the 127 non-NaN codes 0x00..0x7E, whose values increase with
 * the code), ties to the code with the even last bit, magnitudes at or above
 * 448 (infinity included) saturate to 448, NaN gives 0x7F, and the sign bit is
 * carried over (so -0 gives 0x80). */
uint8_t orc_e4m3_encode(float x)
{
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= E4M3_MAX) return sign | 0x7E;
    /* binary search for the largest code lo with decode(lo) <= a */
    int lo = 0, hi = 0x7E;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (orc_e4m3_decode((uint8_t)mid) <= a) lo = mid; else hi = mid - 1;
    }
    if (lo == 0x7E) return sign | 0x7E;
    double below = orc_e4m3_decode((uint8_t)lo);
    double above = orc_e4m3_decode((uint8_t)(lo + 1));
    int code;
    if (a - below < above - a)
        code = lo;
    else if (a - below > above - a)
        code = lo + 1;
    else
        code = (lo % 2 == 0) ? lo : lo + 1; /* tie: even code */
    return sign | (uint8_t)code;
}

/* ---------------------------------------------------------------- amax ---- */

/* max |x| over a bf16 tensor, compared as fp32.  A NaN anywhere makes the
 * result NaN (the NaN with the largest magnitude bit pattern, sign cleared);
 * the configurations never contain one. */
float orc_amax_bf16(const uint16_t *x, int64_t n)
{
    float best = 0.0f;
    int have_nan = 0;
    uint16_t nan_bits = 0;
    for (int64_t i = 0; i < n; i++) {
        float v = fabsf(orc_bf16_to_f32(x[i]));
        if (isnan(v)) {
            uint16_t b = x[i] & 0x7FFF;
            if (!have_nan || b > nan_bits) nan_bits = b;
            have_nan = 1;
        } else if (v > best) {
            best = v;
        }
    }
    return have_nan ? orc_bf16_to_f32(nan_bits) : best;
}

/* -------------------------------------------------------------- scales ---- */

/* The lag / current-amax rule: a = max(amax, 1e-12); scale = a/448,
 * scale_inv = 448/a, each a single fp32 division. */
void orc_scale_from_amax(float amax, float *scale, float *scale_inv)
{
    volatile float a = amax < 1e-12f ? 1e-12f : amax;  /* clamp_min(1e-12); NaN stays */
    volatile float s = a / 448.0f;
    volatile float si = 448.0f / a;
    *scale = s;
    *scale_inv = si;
}

/* ------------------------------------------------------------ quantise ---- */

/* q[i] = e4m3(fl32(x[i] * scale_inv)); returns amax of x as well. */
float orc_quantize(const uint16_t *x, int64_t n, float scale_inv, uint8_t *q)
{
    for (int64_t i = 0; i < n; i++) {
        volatile float v = orc_bf16_to_f32(x[i]) * scale_inv;
        q[i] = orc_e4m3_encode(v);
    }
    return orc_amax_bf16(x, n);
}

/* qt[c, r] = q[r, c] for a row-major [rows, cols] byte matrix. */
void orc_transpose_u8(const uint8_t *q, int64_t rows, int64_t cols, uint8_t *qt)
{
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++)
            qt[c * rows + r] = q[r * cols + c];
}

/* ------------------------------------------------------ block quantise ---- */

/* Row tiles of 1 x tile elements along the columns of a [rows, cols] bf16
 * matrix (the contraction dimension of an activation or a gradient).  For
 * each tile: amax, scale by the lag rule, quantise with that tile's scale_inv.
 * scale/scale_inv are [rows, cols/tile]. */
void orc_quantize_rowtiles(const uint16_t *x, int64_t rows, int64_t cols, int64_t tile,
                           uint8_t *q, float *scale, float *scale_inv)
{
    int64_t nt = cols / tile;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t t = 0; t < nt; t++) {
            const uint16_t *xs = x + r * cols + t * tile;
            float amax = orc_amax_bf16(xs, tile);
            float s, si;
            orc_scale_from_amax(amax, &s, &si);
            scale[r * nt + t] = s;
            scale_inv[r * nt + t] = si;
            for (int64_t k = 0; k < tile; k++) {
                volatile float v = orc_bf16_to_f32(xs[k]) * si;
                q[r * cols + t * tile + k] = orc_e4m3_encode(v);
            }
        }
}

/* Column tiles of tile x 1 elements (tile consecutive rows of one column),
 * written transposed: qt is [cols, rows] and scale/scale_inv are
 * [cols, rows/tile], so that the rows of the original become the
 * contraction dimension of qt. */
void orc_quantize_coltiles_t(const uint16_t *x, int64_t rows, int64_t cols, int64_t tile,
                             uint8_t *qt, float *scale, float *scale_inv)
{
    int64_t nt = rows / tile;
    for (int64_t c = 0; c < cols; c++)
        for (int64_t t = 0; t < nt; t++) {
            float amax = 0.0f;
            for (int64_t k = 0; k < tile; k++) {
                uint16_t h = x[(t * tile + k) * cols + c];
                float v = orc_amax_bf16(&h, 1);
                if (v > amax || isnan(v)) amax = v;
            }
            float s, si;
            orc_scale_from_amax(amax, &s, &si);
            scale[c * nt + t] = s;
            scale_inv[c * nt + t] = si;
            for (int64_t k = 0; k < tile; k++) {
                volatile float v = orc_bf16_to_f32(x[(t * tile + k) * cols + c]) * si;
                qt[c * rows + t * tile + k] = orc_e4m3_encode(v);
            }
        }
}

/* Square tiles of tile x tile elements (weights).  scale/scale_inv are
 * [rows/tile, cols/tile]. */
void orc_quantize_sqtiles(const uint16_t *x, int64_t rows, int64_t cols, int64_t tile,
                          uint8_t *q, float *scale, float *scale_inv)
{
    int64_t nr = rows / tile, nc = cols / tile;
    for (int64_t tr = 0; tr < nr; tr++)
        for (int64_t tc = 0; tc < nc; tc++) {
            float amax = 0.0f;
            for (int64_t r = 0; r < tile; r++) {
                float a = orc_amax_bf16(x + (tr * tile + r) * cols + tc * tile, tile);
                if (a > amax || isnan(a)) amax = a;
            }
            float s, si;
            orc_scale_from_amax(amax, &s, &si);
            scale[tr * nc + tc] = s;
            scale_inv[tr * nc + tc] = si;
            for (int64_t r = 0; r < tile; r++)
                for (int64_t c = 0; c < tile; c++) {
                    int64_t i = (tr * tile + r) * cols + tc * tile + c;
                    volatile float v = orc_bf16_to_f32(x[i]) * si;
                    q[i] = orc_e4m3_encode(v);
                }
        }
}

/* ---------------------------------------------------------------- GEMM ---- */

/* D[i, j] = s_a * s_b * sum_k dec(A[i, k]) * dec(B[j, k]) for the entries
 * (ii[t], jj[t]), A [M, K] and B [N, K] row-major e4m3 codes (both with the
 * contraction dimension contiguous).  Also returns the error-bound weight
 * s_a * s_b * sum_k |dec(A[i,k])| * |dec(B[j,k])| and, when bias is given,
 * adds bf16 bias[j] before rounding.  d_bf16 is D rounded to bf16. */
void orc_gemm_entries(const uint8_t *A, const uint8_t *B, int64_t K,
                      float s_a, float s_b, const uint16_t *bias,
                      const int64_t *ii, const int64_t *jj, int64_t n,
                      double *d, double *d_bf16, double *bound)
{
    double lut[256];
    for (int c = 0; c < 256; c++) lut[c] = orc_e4m3_decode((uint8_t)c);
    double s = (double)s_a * (double)s_b;
    for (int64_t t = 0; t < n; t++) {
        const uint8_t *a = A + ii[t] * K;
        const uint8_t *b = B + jj[t] * K;
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double p = lut[a[k]] * lut[b[k]];
            acc += p;
            mag += fabs(p);
        }
        double v = s * acc;
        if (bias) v += (double)orc_bf16_to_f32(bias[jj[t]]);
        d[t] = v;
        d_bf16[t] = orc_round_to_bf16(v);
        bound[t] = s * mag;
    }
}

/* Full D [M, N] (small cases). */
void orc_gemm(const uint8_t *A, const uint8_t *B, int64_t M, int64_t N, int64_t K,
              float s_a, float s_b, const uint16_t *bias,
              double *d, double *d_bf16, double *bound)
{
    double lut[256];
    for (int c = 0; c < 256; c++) lut[c] = orc_e4m3_decode((uint8_t)c);
    double s = (double)s_a * (double)s_b;
    for (int64_t i = 0; i < M; i++)
        for (int64_t j = 0; j < N; j++) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = lut[A[i * K + k]] * lut[B[j * K + k]];
                acc += p;
                mag += fabs(p);
            }
            double v = s * acc;
            if (bias) v += (double)orc_bf16_to_f32(bias[j]);
            d[i * N + j] = v;
            d_bf16[i * N + j] = orc_round_to_bf16(v);
            bound[i * N + j] = s * mag;
        }
}

/* Block-scaled GEMM entries: the contraction is split into blocks of kb
 * elements; block b of row i of A has scale sa[i, b] ([M, K/kb]); block b of
 * row j of B has scale sb[j / b_rows, b] ([N / b_rows, K/kb]; b_rows = 1 for
 * per-row B scales, 128 for 128x128 weight tiles).  Each block's exact partial
 * sum is multiplied by its two scales and the products are added in fp64. */
void orc_gemm_block_entries(const uint8_t *A, const uint8_t *B, int64_t K, int64_t kb,
                            const float *sa, const float *sb, int64_t b_rows,
                            const int64_t *ii, const int64_t *jj, int64_t n,
                            double *d, double *d_bf16, double *bound)
{
    double lut[256];
    for (int c = 0; c < 256; c++) lut[c] = orc_e4m3_decode((uint8_t)c);
    int64_t nkb = K / kb;
    for (int64_t t = 0; t < n; t++) {
        const uint8_t *a = A + ii[t] * K;
        const uint8_t *b = B + jj[t] * K;
        double acc = 0.0, mag = 0.0;
        for (int64_t blk = 0; blk < nkb; blk++) {
            double part = 0.0, pmag = 0.0;
            for (int64_t k = blk * kb; k < (blk + 1) * kb; k++) {
                double p = lut[a[k]] * lut[b[k]];
                part += p;
                pmag += fabs(p);
            }
            double s = (double)sa[ii[t] * nkb + blk] * (double)sb[(jj[t] / b_rows) * nkb + blk];
            acc += s * part;
            mag += s * pmag;
        }
        d[t] = acc;
        d_bf16[t] = orc_round_to_bf16(acc);
        bound[t] = mag;
    }
}

/* ------------------------------------------------------------- padding ---- */

/* out = x with zero rows appended up to the next multiple of `multiple`.
 * Returns the padded row count; out must hold that many rows. */
int64_t orc_pad_rows(const uint16_t *x, int64_t rows, int64_t cols, int64_t multiple,
                     uint16_t *out)
{
    int64_t padded = (rows + multiple - 1) / multiple * multiple;
    memcpy(out, x, (size_t)(rows * cols) * sizeof(uint16_t));
    memset(out + rows * cols, 0, (size_t)((padded - rows) * cols) * sizeof(uint16_t));
    return padded;
}

/* ---------------------------------------------------------- bias gradient */

/* Bias gradient of the linear y = x w^T + b: dbias[n] = sum over the rows m of
 * the upstream gradient g[m][n].  The AstrAI page's fp8_linear_backward takes
 * aten::linear_backward's output mask, whose third entry asks for this
 * gradient; the page gives no arithmetic for it, so the definition is written
 * out: each column summed in fp64 (bf16 values have 8 significant bits, so
 * the sum of up to 2^45 of them is exact), then rounded once to bf16.
 * d gets the exact sums, d_bf16 their bf16 roundings and mag the column sums
 * of |g| (the scale of a summation-error bound). */
void orc_bias_grad(const uint16_t *g, int64_t rows, int64_t cols, double *d, double *d_bf16,
                   double *mag)
{
    for (int64_t n = 0; n < cols; ++n) {
        d[n] = 0.0;
        mag[n] = 0.0;
    }
    for (int64_t m = 0; m < rows; ++m)
        for (int64_t n = 0; n < cols; ++n) {
            double v = (double)orc_bf16_to_f32(g[m * cols + n]);
            d[n] += v;
            mag[n] += fabs(v);
        }
    for (int64_t n = 0; n < cols; ++n) d_bf16[n] = orc_round_to_bf16(d[n]);
}

/* ------------------------------------------------- padding of [B, T, H] --- */

/* Per-sequence padding of a batch-major [B, T, H] bf16 tensor to [B, Tp, H]
 * (NeMo page "Add FP8 support for SALMAutomodel": TE FP8 padding for BSHD
 * inputs): every sequence keeps its T rows and gets Tp - T zero rows at its
 * end, the same zero fill the THD path appends at the end of the packed
 * batch. */
void orc_pad_bshd(const uint16_t *x, int64_t B, int64_t T, int64_t H, int64_t Tp, uint16_t *out)
{
    for (int64_t b = 0; b < B; ++b)
        for (int64_t t = 0; t < Tp; ++t)
            for (int64_t h = 0; h < H; ++h)
                out[(b * Tp + t) * H + h] = t < T ? x[(b * T + t) * H + h] : (uint16_t)0;
}

