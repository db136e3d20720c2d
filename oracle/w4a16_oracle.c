/*
 * w4a16_oracle.c -- plain, slow CPU oracle for the W4A16 group-wise path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load it.  It shares no code, header, table or constant
 * with the CUDA kernels.
 *
 * Sources (web pages, cited by title and section):
 *   [P4] "LLM quantization from IEEE 754 to GPTQ/AWQ/GGUF" tutorial
 *        (qaqbuyan.com article 126), chapter "量化的数学基石":
 *          §1   FP16 bit layout  value = (-1)^S * 2^(E-15) * (1 + M/1024)
 *          §2   symmetric quantization  x_q = clamp(round(x/s), -8, 7),
 *               s = max|x| / 7; asymmetric quantization
 *               x_q = clamp(round(x/s) + z, 0, 15), s = (max - min) / 15,
 *               z = -round(min / s)
 *          §3   per-group granularity and the per_group_symmetric_quantize /
 *               per_group_symmetric_dequantize functions (groups along
 *               in_features, low nibble = even index, stored as q + 8,
 *               scale clamp(min=1e-8), scales stored as fp16, dequant in
 *               fp32 intermediate).
 *          "INT8 对称量化的精度实测": per-channel symmetric INT8 weights
 *               (the §2 formula with b = 8: s = max|x| / 127,
 *               x_q = clamp(round(x/s), -128, 127)), fp16 activations;
 *          GGUF section: the Q4_0 block, 32 weights in 18 bytes -- d (fp16)
 *               then 16 bytes, byte i holding element 2i in its low nibble
 *               and 2i+1 in its high nibble, decoded as (nibble - 8) * d;
 *          AWQ section "AWQ 的数学原理": activation scaling per input
 *               channel x~_j = x_j * alpha_j with W~_{:,j} = W_{:,j} / alpha_j
 *               (the alpha search needs calibration data: not restated).
 *   [P1] "W4A16 量化算子解码性能基准跑分与端侧大模型推理显存实测报告"
 *        (mhpq.cn) §一: group size 128, symmetric INT4, fp16 scales;
 *        §二/§五: y = x * W^T computed from the packed weights.
 *
 * Readings taken where the pages are silent:
 *   - all quantizer arithmetic is IEEE binary32 on the exactly-upcast fp16
 *     input; q is chosen against the fp32 scale s32, the stored scale is
 *     half_rne(s32);
 *   - round() is round-half-to-even (torch.round semantics);
 *   - the clamp(min=1e-8) is applied to s32 in binary32;
 *   - asymmetric: min and max are taken over the group and 0 (the zero
 *     point is the code of 0.0, so 0 lies in the quantized range and z is a
 *     4-bit code in [0, 15]); the nibble stores q itself and the zero point
 *     is stored as one byte per group; the same clamp(min=1e-8) guards s;
 *   - per-channel quantization is one group spanning the whole row
 *     (group = K);
 *   - W8A16: one fp16 scale per output row (per-channel), the same binary32
 *     arithmetic and clamp(min=1e-8) as the INT4 quantizer; codes are stored
 *     as q + 128 in one byte, row-major [N, K];
 *   - Q4_0 codes are the §2/§3 symmetric quantizer with groups of 32 (the
 *     pages give the block's decoder, not a separate quantizer), laid out
 *     block after block along each row, rows one after another;
 *   - AWQ's scaled activation is rounded once to fp16: x~ = fp16_rne(x * alpha),
 *     the product of two fp16 values being exact in binary32;
 *   - the GEMM reference is the exact dequantized weight (nib-8)*scale16 in
 *     binary64, summed sequentially over k in binary64, never rounded to fp16.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fno-fast-math
 *        [-fopenmp].  OpenMP only splits independent output rows; every row
 *        is the same sequential loop, so results do not depend on threads.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* FP16 <-> binary64/binary32, written from the bit layout of [P4] §1. */
/* ------------------------------------------------------------------ */

/* Exact value of an IEEE half.  E = 0 is the subnormal range
 * 2^-14 * (M/1024); E = 31 is inf/NaN. */
double orc_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);             /* 2^-14 * m / 2^10 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + (double)m, e - 25); /* 2^(e-15) * (1024+m)/2^10 */
    return sign ? -v : v;
}

/* Round a binary32 value to the nearest half, ties to even, keeping
 * subnormals and overflowing to infinity.  Works on the exact value in
 * binary64 so that every scaling step below is exact and rint() (default
 * rounding mode: to nearest, ties to even) makes the single rounding. */
uint16_t orc_float_to_half(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    double a = fabs((double)f);

    if (isnan(f))
        return (uint16_t)(sign | 0x7e00u);
    /* largest half is 65504 = (2 - 2^-10) * 2^15; half-way to the next
     * binade is 65520 and its tie goes to the even (infinite) side. */
    if (a >= 65520.0)
        return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal: value = m * 2^-24 */
        double m = rint(ldexp(a, 24));          /* m in [0, 1024] */
        return (uint16_t)(sign | (uint16_t)m);  /* m == 1024 is 2^-14 */
    }
    int ex;
    (void)frexp(a, &ex);                        /* a = fr * 2^ex, fr in [0.5,1) */
    int e = ex - 1;                             /* a in [2^e, 2^(e+1)) */
    double m = rint(ldexp(a, 10 - e)) - 1024.0; /* (a/2^e - 1) * 1024 */
    if (m >= 1024.0) {                          /* rounded up into next binade */
        m = 0.0;
        e += 1;
    }
    if (e + 15 >= 31)
        return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)m);
}

/* Vector helpers for the Python wrapper. */
void orc_half_to_double_n(const uint16_t *h, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_half_to_double(h[i]);
}

void orc_float_to_half_n(const float *f, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_float_to_half(f[i]);
}

/* ------------------------------------------------------------------ */
/* Quantizer: [P4] §2 symmetric formula + §3 per-group quantizer.       */
/* ------------------------------------------------------------------ */

/* Quantize one group of `group` fp16 weights.
 * Returns the fp16 scale bits and writes q in [-8, 7]. */
static uint16_t quantize_group(const uint16_t *w16, int64_t group, int8_t *q)
{
    /* scale = max|w| / 7 over the group (INT4 symmetric range [-8, 7]) */
    float amax = 0.0f;
    for (int64_t i = 0; i < group; ++i) {
        float a = fabsf((float)orc_half_to_double(w16[i]));
        if (a > amax)
            amax = a;
    }
    float s = amax / 7.0f;   /* IEEE binary32 division */
    if (s < 1e-8f)           /* clamp(min=1e-8): avoids dividing by zero */
        s = 1e-8f;

    /* q = clamp(round(w / s), -8, 7) with round-half-to-even */
    for (int64_t i = 0; i < group; ++i) {
        float w = (float)orc_half_to_double(w16[i]);
        float r = w / s;
        float rq = nearbyintf(r);
        if (rq < -8.0f)
            rq = -8.0f;
        if (rq > 7.0f)
            rq = 7.0f;
        q[i] = (int8_t)rq;
    }
    return orc_float_to_half(s);
}

/* W: fp16 bits [N, K] row-major (rows = out_features, K = in_features).
 * qweight: [N, K/2] bytes; byte j of a row holds k = 2j in its low nibble
 *          and k = 2j+1 in its high nibble, each stored as q + 8.
 * scales:  fp16 bits [N, K/group].
 * Returns 0, or -1 on a shape the quantizer does not accept. */
int orc_quantize(const uint16_t *W, int64_t N, int64_t K, int64_t group,
                 uint8_t *qweight, uint16_t *scales)
{
    if (N < 0 || K <= 0 || group <= 0 || group % 2 != 0 || K % group != 0 ||
        group > 32768)
        return -1;
    int64_t ngroups = K / group;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n) {
        int8_t q[32768];
        for (int64_t g = 0; g < ngroups; ++g) {
            const uint16_t *wg = W + n * K + g * group;
            scales[n * ngroups + g] = quantize_group(wg, group, q);
            for (int64_t i = 0; i < group; i += 2) {
                uint8_t lo = (uint8_t)((q[i] + 8) & 0x0f);
                uint8_t hi = (uint8_t)((q[i + 1] + 8) & 0x0f);
                qweight[n * (K / 2) + (g * group + i) / 2] = (uint8_t)((hi << 4) | lo);
            }
        }
    }
    return 0;
}

/* Quantize one group asymmetrically ([P4] §2 asymmetric formula).
 * Returns the fp16 scale bits, writes q in [0, 15] and the zero point. */
static uint16_t quantize_group_asym(const uint16_t *w16, int64_t group, uint8_t *q,
                                    uint8_t *zero)
{
    /* min and max over the group and 0 */
    float mn = 0.0f, mx = 0.0f;
    for (int64_t i = 0; i < group; ++i) {
        float v = (float)orc_half_to_double(w16[i]);
        if (v < mn)
            mn = v;
        if (v > mx)
            mx = v;
    }
    float s = (mx - mn) / 15.0f;  /* IEEE binary32 subtraction and division */
    if (s < 1e-8f)
        s = 1e-8f;
    float z = -nearbyintf(mn / s); /* z = -round(min / s), in [0, 15] */

    /* q = clamp(round(w / s) + z, 0, 15) with round-half-to-even */
    for (int64_t i = 0; i < group; ++i) {
        float w = (float)orc_half_to_double(w16[i]);
        float rq = nearbyintf(w / s) + z;
        if (rq < 0.0f)
            rq = 0.0f;
        if (rq > 15.0f)
            rq = 15.0f;
        q[i] = (uint8_t)rq;
    }
    *zero = (uint8_t)z;
    return orc_float_to_half(s);
}

/* Asymmetric variant of orc_quantize: the nibbles hold q in [0, 15]
 * (low nibble = even k), zeros: [N, K/group] bytes. */
int orc_quantize_asym(const uint16_t *W, int64_t N, int64_t K, int64_t group,
                      uint8_t *qweight, uint16_t *scales, uint8_t *zeros)
{
    if (N < 0 || K <= 0 || group <= 0 || group % 2 != 0 || K % group != 0 ||
        group > 32768)
        return -1;
    int64_t ngroups = K / group;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n) {
        uint8_t q[32768];
        for (int64_t g = 0; g < ngroups; ++g) {
            const uint16_t *wg = W + n * K + g * group;
            scales[n * ngroups + g] = quantize_group_asym(wg, group, q, &zeros[n * ngroups + g]);
            for (int64_t i = 0; i < group; i += 2)
                qweight[n * (K / 2) + (g * group + i) / 2] =
                    (uint8_t)(((q[i + 1] & 0x0f) << 4) | (q[i] & 0x0f));
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Dequantizer: [P4] §3 per_group_symmetric_dequantize, kept exact.     */
/* ------------------------------------------------------------------ */

/* Exact dequantized weight of row n: (nibble - z) * scale16 in binary64,
 * z the group's zero point (asymmetric: zrow != NULL) or 8 (symmetric: the
 * nibble holds q + 8).  An fp16 scale times an integer of magnitude <= 15
 * needs at most 15 significant bits, so binary64 holds it exactly. */
static void dequant_row(const uint8_t *qrow, const uint16_t *srow, const uint8_t *zrow,
                        int64_t K, int64_t group, double *out)
{
    for (int64_t k = 0; k < K; ++k) {
        uint8_t byte = qrow[k / 2];
        int nib = (k % 2 == 0) ? (byte & 0x0f) : ((byte >> 4) & 0x0f);
        int z = zrow ? zrow[k / group] : 8;
        out[k] = (double)(nib - z) * orc_half_to_double(srow[k / group]);
    }
}

int orc_dequantize(const uint8_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                   int64_t N, int64_t K, int64_t group, double *out)
{
    if (N < 0 || K <= 0 || group <= 0 || K % group != 0 || K % 2 != 0)
        return -1;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n)
        dequant_row(qweight + n * (K / 2), scales + n * (K / group),
                    zeros ? zeros + n * (K / group) : NULL, K, group, out + n * K);
    return 0;
}

/* The page's own fp16 dequantized weight: float(q) * float(scale) rounded
 * once to fp16 ([P4] §3 dequantize, "float32 intermediate").  Used by the
 * tests to bound the rounding a kernel adds when it stages fp16 q*scale. */
int orc_dequantize_f16(const uint8_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                       int64_t N, int64_t K, int64_t group, uint16_t *out)
{
    if (N < 0 || K <= 0 || group <= 0 || K % group != 0 || K % 2 != 0)
        return -1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = qweight[n * (K / 2) + k / 2];
            int nib = (k % 2 == 0) ? (byte & 0x0f) : ((byte >> 4) & 0x0f);
            float s = (float)orc_half_to_double(scales[n * (K / group) + k / group]);
            int z = zeros ? zeros[n * (K / group) + k / group] : 8;
            float v = (float)(nib - z) * s;
            out[n * K + k] = orc_float_to_half(v);
        }
    return 0;
}

/* ------------------------------------------------------------------ */
/* W8A16: per-channel symmetric INT8 ([P4] §2 formula with b = 8, INT8 */
/* section "per-channel, 对称").                                        */
/* ------------------------------------------------------------------ */

/* W: fp16 bits [N, K]; q8: [N, K] bytes holding q + 128; scales: fp16 bits [N]. */
int orc_quantize_w8(const uint16_t *W, int64_t N, int64_t K, uint8_t *q8, uint16_t *scales)
{
    if (N < 0 || K <= 0)
        return -1;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf((float)orc_half_to_double(W[n * K + k]));
            if (a > amax)
                amax = a;
        }
        float s = amax / 127.0f;   /* 2^(b-1) - 1 = 127 */
        if (s < 1e-8f)
            s = 1e-8f;
        for (int64_t k = 0; k < K; ++k) {
            float r = nearbyintf((float)orc_half_to_double(W[n * K + k]) / s);
            if (r < -128.0f)
                r = -128.0f;
            if (r > 127.0f)
                r = 127.0f;
            q8[n * K + k] = (uint8_t)((int)r + 128);
        }
        scales[n] = orc_float_to_half(s);
    }
    return 0;
}

/* Exact dequantized row: (code - 128) * scale16, binary64. */
static void dequant_row_w8(const uint8_t *qrow, uint16_t scale, int64_t K, double *out)
{
    double s = orc_half_to_double(scale);
    for (int64_t k = 0; k < K; ++k)
        out[k] = (double)((int)qrow[k] - 128) * s;
}

int orc_dequantize_w8(const uint8_t *q8, const uint16_t *scales, int64_t N, int64_t K,
                      double *out)
{
    for (int64_t n = 0; n < N; ++n)
        dequant_row_w8(q8 + n * K, scales[n], K, out + n * K);
    return 0;
}

/* Rows `rows` of y = x * Wd^T for W8A16 weights; y is [M, nrows] binary64. */
int orc_gemm_rows_w8(const uint16_t *x, int64_t M, int64_t K, const uint8_t *q8,
                     const uint16_t *scales, int64_t N, const int64_t *rows, int64_t nrows,
                     double *y)
{
    if (M < 0 || N < 0 || K <= 0 || K > 32768)
        return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N)
            return -1;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
        double wd[32768];
        dequant_row_w8(q8 + rows[r] * K, scales[rows[r]], K, wd);
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += orc_half_to_double(x[m * K + k]) * wd[k];
            y[m * nrows + r] = acc;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* GGUF Q4_0 blocks ([P4] GGUF section).                                */
/* ------------------------------------------------------------------ */

/* (qweight [N, K/2] canonical bytes, scales [N, K/32]) -> blocks [N * K/32][18]. */
int orc_pack_q4_0(const uint8_t *qweight, const uint16_t *scales, int64_t N, int64_t K,
                  uint8_t *blocks)
{
    if (N < 0 || K <= 0 || K % 32 != 0)
        return -1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < K / 32; ++b) {
            uint8_t *blk = blocks + (n * (K / 32) + b) * 18;
            uint16_t d = scales[n * (K / 32) + b];
            blk[0] = (uint8_t)(d & 0xff);        /* little-endian fp16 */
            blk[1] = (uint8_t)(d >> 8);
            for (int i = 0; i < 16; ++i)         /* byte i: elements 2i (low), 2i+1 (high) */
                blk[2 + i] = qweight[n * (K / 2) + b * 16 + i];
        }
    return 0;
}

/* Exact decode of Q4_0 blocks: out[n, k] = (nibble - 8) * d in binary64. */
int orc_dequantize_q4_0(const uint8_t *blocks, int64_t N, int64_t K, double *out)
{
    if (N < 0 || K <= 0 || K % 32 != 0)
        return -1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < K / 32; ++b) {
            const uint8_t *blk = blocks + (n * (K / 32) + b) * 18;
            double d = orc_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
            for (int i = 0; i < 16; ++i) {
                out[n * K + b * 32 + 2 * i] = (double)((blk[2 + i] & 0x0f) - 8) * d;
                out[n * K + b * 32 + 2 * i + 1] = (double)(((blk[2 + i] >> 4) & 0x0f) - 8) * d;
            }
        }
    return 0;
}

/* ------------------------------------------------------------------ */
/* AWQ activation scaling ([P4] AWQ section): x~[m, k] = x[m, k] * alpha[k] */
/* ------------------------------------------------------------------ */

void orc_scale_activations(const uint16_t *x, int64_t M, int64_t K, const uint16_t *alpha,
                           uint16_t *out)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            float p = (float)orc_half_to_double(x[m * K + k]) *
                      (float)orc_half_to_double(alpha[k]);   /* exact in binary32 */
            out[m * K + k] = orc_float_to_half(p);
        }
}

/* ------------------------------------------------------------------ */
/* GEMM: y[m, n] = sum_k x[m, k] * Wd[n, k]  ([P1] §二/§五, y = x W^T).  */
/* ------------------------------------------------------------------ */

/* Rows `rows[0..nrows)` of W only; y is [M, nrows] binary64, unrounded.
 * x: fp16 bits [M, K]. */
int orc_gemm_rows(const uint16_t *x, int64_t M, int64_t K, const uint8_t *qweight,
                  const uint16_t *scales, const uint8_t *zeros, int64_t N, int64_t group,
                  const int64_t *rows, int64_t nrows, double *y)
{
    if (M < 0 || N < 0 || K <= 0 || group <= 0 || K % group != 0 || K % 2 != 0 ||
        K > 32768)
        return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N)
            return -1;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t n = rows[r];
        double wd[32768];
        double xv;
        dequant_row(qweight + n * (K / 2), scales + n * (K / group),
                    zeros ? zeros + n * (K / group) : NULL, K, group, wd);
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                xv = orc_half_to_double(x[m * K + k]);
                acc += xv * wd[k];
            }
            y[m * nrows + r] = acc;
        }
    }
    return 0;
}

/* All rows: y is [M, N]. */
int orc_gemm(const uint16_t *x, int64_t M, int64_t K, const uint8_t *qweight,
             const uint16_t *scales, const uint8_t *zeros, int64_t N, int64_t group, double *y)
{
    if (M < 0 || N < 0 || K <= 0 || group <= 0 || K % group != 0 || K % 2 != 0 ||
        K > 32768)
        return -1;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n) {
        double wd[32768];
        dequant_row(qweight + n * (K / 2), scales + n * (K / group),
                    zeros ? zeros + n * (K / group) : NULL, K, group, wd);
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += orc_half_to_double(x[m * K + k]) * wd[k];
            y[m * N + n] = acc;
        }
    }
    return 0;
}

/* Threads OpenMP would use (1 without OpenMP). */
int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
