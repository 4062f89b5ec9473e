/*
 * q4_oracle.c -- plain, slow CPU oracle for the weight-only 4-bit matmul library.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this
 * file.  It is compiled into liboracle_q4.so and used by the tests, by the smoke
 * check and by the bench's CPU-baseline leg, and by nothing else.  It shares no
 * source, header, table or helper with the CUDA library.
 *
 * Every function below writes out the definition of one operation in the order the
 * source pages state it: no blocking, no fusion, no reordering.  Floating-point
 * work that the pages fix in fp32 (the affine dequant fmaf, the codebook product)
 * is done in fp32; everything else accumulates in fp64 with k ascending.
 *
 * Build with -ffp-contract=off: the compiler must not fuse a*b+c anywhere except
 * where fmaf() is written out, or x86 and Arm hosts would disagree.
 *
 * Sources (page title, section):
 *   [P1] onnxruntime-ep-mlx 0.27.4, src/ops/quant_fastkernel.rs -- the INT4 group-32
 *        affine MatMulNBits kernel (weight unpack and dequant) and its test-module
 *        host ground truth `make_case`.
 *   [P2] onnxruntime-ep-mlx 0.31.1, src/ops/lut4.rs -- the lookup4 kernel source,
 *        the CPU decode branch of `execute`, and the test
 *        `cpu_products_keep_branch_weights_and_transposed_layouts_distinct`.
 *   [P3] mlx-native 0.9.0, src/ops/quantized_matmul_id_ggml.rs -- module doc
 *        (routed-matmul definition), `IdMmScratch` and the map0 stage of
 *        `dispatch_id_mm_for_test` (per-expert routed lists).
 *        Also `quantized_matmul_id_swiglu_q4_0` (doc comment): the fused SwiGLU
 *        routed mat-vec.
 *   The Q4_0 block layout itself (fp16 d + 16 bytes of nibbles, low nibbles are
 *   elements 0..15, high nibbles 16..31, value (q-8)*d) is not printed on [P3]; it is
 *   the GGML Q4_0 format as the problem statement gives it.  [P3] also names Q8_0 among
 *   its routed kernels without printing its block; the GGML Q8_0 block is used: fp16 d,
 *   then 32 signed bytes, value q*d.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Scalar storage conversions, written from the IEEE-754 definitions.        */
/* ------------------------------------------------------------------------- */

/* bfloat16 is the top half of an IEEE binary32. */
float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Nearest bfloat16, ties to even.  Method: scale the value by its bf16 ulp,
 * round to an integer with rint() (default rounding mode: ties to even), scale
 * back; the result is then exactly representable and its top 16 bits are it. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(f))
        return (uint16_t)((u >> 16) | 0x0040u);
    if (isinf(f) || f == 0.0f)
        return (uint16_t)(u >> 16);
    double v = (double)f;
    int e = ilogb(v);                 /* v = m * 2^e, 1 <= |m| < 2 */
    if (e < -126)
        e = -126;                     /* subnormal range: fixed ulp 2^-133 */
    double ulp = ldexp(1.0, e - 7);   /* 8 significant bits */
    double r = rint(v / ulp) * ulp;
    if (fabs(r) >= ldexp(1.0, 128))   /* rounds past the largest finite value */
        return (uint16_t)((u & 0x80000000u) >> 16 | 0x7F80u);
    float rf = (float)r;              /* exact: r has <= 8 significant bits */
    uint32_t ru;
    memcpy(&ru, &rf, sizeof ru);
    return (uint16_t)(ru >> 16);
}

/* IEEE binary16 -> value, from the field definitions. */
float oracle_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1F;
    int man = h & 0x3FF;
    double v;
    if (ex == 0)
        v = ldexp((double)man, -24);
    else if (ex == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(man | 0x400), ex - 25);
    return (float)(sign ? -v : v);
}

/* Nearest IEEE binary16, ties to even, same method as the bf16 routine. */
uint16_t oracle_f32_to_f16(float f)
{
    uint16_t sign = signbit(f) ? 0x8000u : 0u;
    if (isnan(f))
        return (uint16_t)(sign | 0x7E00u);
    if (isinf(f))
        return (uint16_t)(sign | 0x7C00u);
    double v = fabs((double)f);
    if (v == 0.0)
        return sign;
    int e = ilogb(v);
    if (e < -14)
        e = -14;                      /* subnormal range: fixed ulp 2^-24 */
    double ulp = ldexp(1.0, e - 10);  /* 11 significant bits */
    double r = rint(v / ulp) * ulp;
    if (r > 65504.0)
        return (uint16_t)(sign | 0x7C00u);
    if (r == 0.0)
        return sign;
    int re = ilogb(r);
    if (re < -14)                     /* subnormal: mantissa counts 2^-24 units */
        return (uint16_t)(sign | (uint16_t)ldexp(r, 24));
    uint16_t man = (uint16_t)(ldexp(r, 10 - re) - 1024.0);
    return (uint16_t)(sign | (uint16_t)((re + 15) << 10) | man);
}

void oracle_f32_to_bf16_n(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_bf16(in[i]);
}

void oracle_f32_to_f16_n(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_f16(in[i]);
}

void oracle_f16_to_f32_n(const uint16_t *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f16_to_f32(in[i]);
}

/* ------------------------------------------------------------------------- */
/* INT4 group-32 affine MatMulNBits  [P1]                                    */
/*   W: uint32 [N, K/8]; element k of row n is nibble (k % 8) of word k/8,   */
/*      at bits 4*(k%8) .. 4*(k%8)+3 (low nibble first);                     */
/*   scales, biases: bf16 [N, K/32]; bias = -zp * scale;                     */
/*   value = nibble * scale + bias (P1 kernel W-tile dequant; P1 make_case).  */
/* ------------------------------------------------------------------------- */

static uint32_t q4_nibble(const uint32_t *w, int64_t K, int64_t n, int64_t k)
{
    uint32_t word = w[n * (K / 8) + k / 8];
    return (word >> (4 * (k % 8))) & 0xFu;
}

/* The dequantised weight in fp32, formed with one fused multiply-add. */
static float q4_value(const uint32_t *w, const uint16_t *s, const uint16_t *b,
                      int64_t K, int64_t n, int64_t k)
{
    int64_t g = n * (K / 32) + k / 32;
    return fmaf((float)q4_nibble(w, K, n, k), oracle_bf16_to_f32(s[g]),
                oracle_bf16_to_f32(b[g]));
}

void oracle_q4_dequant(const uint32_t *w, const uint16_t *s, const uint16_t *b,
                       int64_t N, int64_t K, float *out)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            out[n * K + k] = q4_value(w, s, b, K, n, k);
}

/* How many elements whose fp32 dequant differs from the exact product-sum
 * nibble*s + b taken in fp64 (zero whenever bias is a bf16 multiple of the
 * scale's ulp, which the affine construction bias = bf16(-zp*scale) gives). */
int64_t oracle_q4_dequant_inexact(const uint32_t *w, const uint16_t *s,
                                  const uint16_t *b, int64_t N, int64_t K)
{
    int64_t bad = 0;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            int64_t g = n * (K / 32) + k / 32;
            double exact = (double)q4_nibble(w, K, n, k) * (double)oracle_bf16_to_f32(s[g]) +
                           (double)oracle_bf16_to_f32(b[g]);
            if ((double)q4_value(w, s, b, K, n, k) != exact)
                ++bad;
        }
    return bad;
}

/* y[m][n] = sum_k x[m][k] * w[n][k], fp64, k ascending. */
void oracle_q4_matmul(const uint16_t *x, const uint32_t *w, const uint16_t *s,
                      const uint16_t *b, int64_t M, int64_t N, int64_t K, double *y)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)oracle_bf16_to_f32(x[m * K + k]) *
                       (double)q4_value(w, s, b, K, n, k);
            y[m * N + n] = acc;
        }
}

/* The same sum at chosen (m, n) pairs only, for full-size spot checks. */
void oracle_q4_matmul_at(const uint16_t *x, const uint32_t *w, const uint16_t *s,
                         const uint16_t *b, int64_t K, const int64_t *mi,
                         const int64_t *ni, int64_t count, double *out)
{
    for (int64_t i = 0; i < count; ++i) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += (double)oracle_bf16_to_f32(x[mi[i] * K + k]) *
                   (double)q4_value(w, s, b, K, ni[i], k);
        out[i] = acc;
    }
}

/* Reference affine quantizer (the pages define none; used only to pin the
 * dequant by a round trip).  Per group of 32 along k: the range [lo, hi] is
 * widened to contain 0, scale = (hi - lo) / 15 stored as bf16 s,
 * zp = clamp(rint(-lo / s), 0, 15), q = clamp(rint(w / s) + zp, 0, 15),
 * bias = bf16(-zp * s).  rint() rounds ties to even. */
void oracle_q4_quantize(const float *wf, int64_t N, int64_t K, uint32_t *words,
                        uint16_t *scales, uint16_t *biases, uint8_t *zps)
{
    memset(words, 0, (size_t)(N * (K / 8)) * sizeof *words);
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < K / 32; ++g) {
            const float *v = wf + n * K + g * 32;
            double lo = 0.0, hi = 0.0;
            for (int i = 0; i < 32; ++i) {
                if (v[i] < lo) lo = v[i];
                if (v[i] > hi) hi = v[i];
            }
            double scale = (hi - lo) / 15.0;
            if (scale == 0.0)
                scale = 1.0;
            uint16_t sb = oracle_f32_to_bf16((float)scale);
            double s = (double)oracle_bf16_to_f32(sb);
            double zp = rint(-lo / s);
            if (zp < 0) zp = 0;
            if (zp > 15) zp = 15;
            scales[n * (K / 32) + g] = sb;
            biases[n * (K / 32) + g] = oracle_f32_to_bf16((float)(-zp * s));
            zps[n * (K / 32) + g] = (uint8_t)zp;
            for (int i = 0; i < 32; ++i) {
                double q = rint((double)v[i] / s) + zp;
                if (q < 0) q = 0;
                if (q > 15) q = 15;
                int64_t k = g * 32 + i;
                words[n * (K / 8) + k / 8] |= (uint32_t)q << (4 * (k % 8));
            }
        }
}

/* ------------------------------------------------------------------------- */
/* LUT4: frozen 16-entry codebook, blocked scales  [P2]                      */
/*   flat index f over the stored [rows, cols] matrix; byte f/2 holds it,    */
/*   high nibble for even f, low nibble for odd f;                           */
/*   value = fl32(book[code] * scales[f / block]).                           */
/*   transpose = 1: stored [rows=N, cols=K], f = n*K + k;                    */
/*   transpose = 0: stored [rows=K, cols=N], f = k*N + n.                    */
/* ------------------------------------------------------------------------- */

static float lut4_value_at(const uint8_t *packed, const float *scales, const float *book,
                           int64_t f, int64_t block)
{
    uint8_t byte = packed[f / 2];
    uint32_t code = (f % 2 == 0) ? (uint32_t)(byte >> 4) : (uint32_t)(byte & 15);
    float value = book[code] * scales[f / block];   /* one fp32 product */
    return value;
}

void oracle_lut4_dequant(const uint8_t *packed, const float *scales, const float *book,
                         int64_t rows, int64_t cols, int64_t block, float *out)
{
    for (int64_t f = 0; f < rows * cols; ++f)
        out[f] = lut4_value_at(packed, scales, book, f, block);
}

static int64_t lut4_flat(int64_t n, int64_t k, int64_t N, int64_t K, int transpose)
{
    return transpose ? n * K + k : k * N + n;
}

/* y[m][n] = sum_k x[m][k] * W(k, n), fp64, k ascending. */
void oracle_lut4_matmul(const uint16_t *x, const uint8_t *packed, const float *scales,
                        const float *book, int64_t M, int64_t N, int64_t K,
                        int64_t block, int transpose, double *y)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)oracle_bf16_to_f32(x[m * K + k]) *
                       (double)lut4_value_at(packed, scales, book,
                                             lut4_flat(n, k, N, K, transpose), block);
            y[m * N + n] = acc;
        }
}

void oracle_lut4_matmul_at(const uint16_t *x, const uint8_t *packed, const float *scales,
                           const float *book, int64_t N, int64_t K, int64_t block,
                           int transpose, const int64_t *mi, const int64_t *ni,
                           int64_t count, double *out)
{
    for (int64_t i = 0; i < count; ++i) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += (double)oracle_bf16_to_f32(x[mi[i] * K + k]) *
                   (double)lut4_value_at(packed, scales, book,
                                         lut4_flat(ni[i], k, N, K, transpose), block);
        out[i] = acc;
    }
}

/* The rounded-weight variant [P2, `rounded_weight` and the Cast matcher in
 * `lookup_matmul`]: when the graph casts the decoded weight to half or bfloat16
 * (and, for the adjoint, back to float), the matmul uses the decoded value rounded
 * to that type and widened again.  rounding: 0 = none (the plain matmul above),
 * 1 = IEEE binary16, 2 = bfloat16; both round to nearest, ties to even, through the
 * conversions at the top of this file. */
static double lut4_rounded_at(const uint8_t *packed, const float *scales, const float *book,
                              int64_t f, int64_t block, int rounding)
{
    float v = lut4_value_at(packed, scales, book, f, block);
    if (rounding == 1)
        v = oracle_f16_to_f32(oracle_f32_to_f16(v));
    else if (rounding == 2)
        v = oracle_bf16_to_f32(oracle_f32_to_bf16(v));
    return (double)v;
}

/* y[m][n] = sum_k x[m][k] * round(W(k, n)), fp64, k ascending. */
void oracle_lut4_matmul_rounded(const uint16_t *x, const uint8_t *packed, const float *scales,
                                const float *book, int64_t M, int64_t N, int64_t K,
                                int64_t block, int transpose, int rounding, double *y)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)oracle_bf16_to_f32(x[m * K + k]) *
                       lut4_rounded_at(packed, scales, book, lut4_flat(n, k, N, K, transpose),
                                       block, rounding);
            y[m * N + n] = acc;
        }
}

/* The same at sampled outputs (mi[i], ni[i]). */
void oracle_lut4_matmul_rounded_at(const uint16_t *x, const uint8_t *packed, const float *scales,
                                   const float *book, int64_t N, int64_t K, int64_t block,
                                   int transpose, int rounding, const int64_t *mi,
                                   const int64_t *ni, int64_t count, double *out)
{
    for (int64_t i = 0; i < count; ++i) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += (double)oracle_bf16_to_f32(x[mi[i] * K + k]) *
                   lut4_rounded_at(packed, scales, book, lut4_flat(ni[i], k, N, K, transpose),
                                   block, rounding);
        out[i] = acc;
    }
}

/* ------------------------------------------------------------------------- */
/* GGML Q4_0 expert-routed matmul  [P3 module doc]                           */
/*   row r = token*top_k + slot; expert e = ids[r]; token row t = r / top_k; */
/*   out[r][n] = sum_k x[t][k] * q4_0(W[e])[n][k].                          */
/*   Block (32 values, 18 bytes): fp16 d (little endian), then 16 bytes qs;  */
/*   element j < 16 is (qs[j] & 15) - 8, element 16 + j is (qs[j] >> 4) - 8;*/
/*   value = (q - 8) * d.                                                    */
/*   An id >= n_experts (the pages say nothing) gives an all-zero row.       */
/* ------------------------------------------------------------------------- */

static float q4_0_value(const uint8_t *row, int64_t k)
{
    const uint8_t *blk = row + (k / 32) * 18;
    float d = oracle_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
    int64_t j = k % 32;
    int q = (j < 16) ? (blk[2 + j] & 15) : (blk[2 + j - 16] >> 4);
    return (float)(q - 8) * d;       /* exact: 4-bit integer times 11-bit d */
}

void oracle_q4_0_dequant_row(const uint8_t *row, int64_t K, float *out)
{
    for (int64_t k = 0; k < K; ++k)
        out[k] = q4_0_value(row, k);
}

static void q4_0_one_row(const float *x, const uint8_t *w, uint32_t e, int64_t t,
                         int64_t N, int64_t K, int64_t n_experts, uint64_t expert_stride,
                         double *out_row)
{
    for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        if ((int64_t)e < n_experts) {
            const uint8_t *row = w + (uint64_t)e * expert_stride + (uint64_t)(n * (K / 32) * 18);
            for (int64_t k = 0; k < K; ++k)
                acc += (double)x[t * K + k] * (double)q4_0_value(row, k);
        }
        out_row[n] = acc;
    }
}

void oracle_q4_0_matmul_id(const float *x, const uint8_t *w, const uint32_t *ids,
                           int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                           int64_t n_experts, uint64_t expert_stride, double *out)
{
    for (int64_t r = 0; r < n_tokens * top_k; ++r)
        q4_0_one_row(x, w, ids[r], r / top_k, N, K, n_experts, expert_stride, out + r * N);
}

/* Only the routed rows listed in rows[] (out is [count, N]). */
void oracle_q4_0_matmul_id_rows(const float *x, const uint8_t *w, const uint32_t *ids,
                                int64_t top_k, int64_t N, int64_t K, int64_t n_experts,
                                uint64_t expert_stride, const int64_t *rows, int64_t count,
                                double *out)
{
    for (int64_t i = 0; i < count; ++i)
        q4_0_one_row(x, w, ids[rows[i]], rows[i] / top_k, N, K, n_experts, expert_stride,
                     out + i * N);
}

/* ------------------------------------------------------------------------- */
/* GGML Q8_0 expert-routed matmul  [P3 module doc; the type is one of the     */
/* routed kernels the page names]                                            */
/*   Same routing as Q4_0.  Block (32 values, 34 bytes): fp16 d (little      */
/*   endian), then 32 signed bytes qs; element j is qs[j] (two's complement) */
/*   and its value is qs[j] * d.                                             */
/* ------------------------------------------------------------------------- */

static float q8_0_value(const uint8_t *row, int64_t k)
{
    const uint8_t *blk = row + (k / 32) * 34;
    float d = oracle_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
    int q = (int)blk[2 + k % 32];
    if (q >= 128)
        q -= 256;                    /* the byte is a signed integer */
    return (float)q * d;             /* exact: 8-bit integer times 11-bit d */
}

void oracle_q8_0_dequant_row(const uint8_t *row, int64_t K, float *out)
{
    for (int64_t k = 0; k < K; ++k)
        out[k] = q8_0_value(row, k);
}

static void q8_0_one_row(const float *x, const uint8_t *w, uint32_t e, int64_t t,
                         int64_t N, int64_t K, int64_t n_experts, uint64_t expert_stride,
                         double *out_row)
{
    for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        if ((int64_t)e < n_experts) {
            const uint8_t *row = w + (uint64_t)e * expert_stride + (uint64_t)(n * (K / 32) * 34);
            for (int64_t k = 0; k < K; ++k)
                acc += (double)x[t * K + k] * (double)q8_0_value(row, k);
        }
        out_row[n] = acc;
    }
}

void oracle_q8_0_matmul_id(const float *x, const uint8_t *w, const uint32_t *ids,
                           int64_t n_tokens, int64_t top_k, int64_t N, int64_t K,
                           int64_t n_experts, uint64_t expert_stride, double *out)
{
    for (int64_t r = 0; r < n_tokens * top_k; ++r)
        q8_0_one_row(x, w, ids[r], r / top_k, N, K, n_experts, expert_stride, out + r * N);
}

/* Only the routed rows listed in rows[] (out is [count, N]). */
void oracle_q8_0_matmul_id_rows(const float *x, const uint8_t *w, const uint32_t *ids,
                                int64_t top_k, int64_t N, int64_t K, int64_t n_experts,
                                uint64_t expert_stride, const int64_t *rows, int64_t count,
                                double *out)
{
    for (int64_t i = 0; i < count; ++i)
        q8_0_one_row(x, w, ids[rows[i]], rows[i] / top_k, N, K, n_experts, expert_stride,
                     out + i * N);
}

/* ------------------------------------------------------------------------- */
/* Fused SwiGLU + routed Q4_0 mat-vec  [P3 quantized_matmul_id_swiglu_q4_0  */
/* doc]: out[r][n] = sum_k q4_0(W[ids[r]])[n][k] * (silu(gate[r][k]) *      */
/* up[r][k]).  gate and up hold one row per ROUTED row r (not per token).    */
/* silu is not spelled out on the page; its plain definition is used:       */
/* silu(z) = z * sigmoid(z) = z / (1 + exp(-z)), evaluated in fp64.          */
/* ------------------------------------------------------------------------- */

static double silu(double z)
{
    return z / (1.0 + exp(-z));
}

static void swiglu_one_row(const float *gate, const float *up, const uint8_t *w, uint32_t e,
                           int64_t r, int64_t N, int64_t K, int64_t n_experts,
                           uint64_t expert_stride, double *out_row)
{
    for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        if ((int64_t)e < n_experts) {
            const uint8_t *row = w + (uint64_t)e * expert_stride + (uint64_t)(n * (K / 32) * 18);
            for (int64_t k = 0; k < K; ++k) {
                double h = silu((double)gate[r * K + k]) * (double)up[r * K + k];
                acc += (double)q4_0_value(row, k) * h;
            }
        }
        out_row[n] = acc;
    }
}

void oracle_q4_0_matmul_id_swiglu(const float *gate, const float *up, const uint8_t *w,
                                  const uint32_t *ids, int64_t n_rows, int64_t N, int64_t K,
                                  int64_t n_experts, uint64_t expert_stride, double *out)
{
    for (int64_t r = 0; r < n_rows; ++r)
        swiglu_one_row(gate, up, w, ids[r], r, N, K, n_experts, expert_stride, out + r * N);
}

/* Only the routed rows listed in rows[] (out is [count, N]). */
void oracle_q4_0_matmul_id_swiglu_rows(const float *gate, const float *up, const uint8_t *w,
                                       const uint32_t *ids, int64_t N, int64_t K,
                                       int64_t n_experts, uint64_t expert_stride,
                                       const int64_t *rows, int64_t count, double *out)
{
    for (int64_t i = 0; i < count; ++i)
        swiglu_one_row(gate, up, w, ids[rows[i]], rows[i], N, K, n_experts, expert_stride,
                       out + i * N);
}

/* Per-expert routed lists (the map0 stage): htpe[e] = number of rows r with
 * ids[r] == e; hids holds, expert after expert (e ascending), each expert's rows
 * r in ascending order, so expert e's list starts at sum_{e' < e} htpe[e'].
 * Rows with ids[r] >= n_experts are in no list; n_invalid counts them. */
void oracle_q4_0_route(const uint32_t *ids, int64_t n_rows, int64_t n_experts,
                       uint32_t *htpe, int32_t *hids, uint32_t *n_invalid)
{
    int64_t pos = 0;
    uint32_t bad = 0;
    for (int64_t e = 0; e < n_experts; ++e) {
        uint32_t count = 0;
        for (int64_t r = 0; r < n_rows; ++r)
            if ((int64_t)ids[r] == e) {
                hids[pos++] = (int32_t)r;
                ++count;
            }
        htpe[e] = count;
    }
    for (int64_t r = 0; r < n_rows; ++r)
        if ((int64_t)ids[r] >= n_experts)
            ++bad;
    *n_invalid = bad;
}
