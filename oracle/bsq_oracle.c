/*
 * bsq_oracle.c -- plain, slow, CPU reference for the block-scaled
 * low-precision linear layer.  TEST INFRASTRUCTURE ONLY: nothing in the
 * library path may link, load or call this file.  It shares no code,
 * table or header with the CUDA sources.
 *
 * Sources of the rules written out here (the pages print no formulas):
 *  - "FP8 Training Infrastructure: Next-Generation Numerical Precision"
 *    (introl.com), section "O panorama da precisao numerica": E4M3 stores
 *    values up to +-448 and is used for forward activations and weights,
 *    E5M2 has the wider range and is used for gradients.
 *  - same page, section "Estrategias de escalonamento e estabilidade":
 *    block-level (microscaling) scale factors on Blackwell.
 *  - "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs"
 *    (gist.science summary of arXiv 2603.02731), section 2 "Metodologia",
 *    "Algoritmo de Conversao Direta": MXFP4 uses 32-element blocks with
 *    power-of-two scales; the FP4->FP8 conversion stays in the integer
 *    domain and preserves numerical equivalence.
 *  - Element formats E4M3 / E5M2 / E2M1 / E8M0 and the block-scale rule
 *    follow the public OCP Microscaling Formats v1.0 definitions; NVFP4's
 *    16-element block with an E4M3 block scale and an FP32 tensor scale
 *    amax/(448*6) follows the workload statement of the NVFP4 forward.
 *
 * Every floating-point value here is an exact double unless a step says
 * FP32; encodes are round-to-nearest, ties to the even code, then
 * saturation to the largest finite magnitude.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

/* element format ids used across this file's API */
enum { O_E4M3 = 0, O_E5M2 = 1, O_E2M1 = 2, O_UE4M3 = 3 };

/* ---------------------------------------------------------------------
 * Element decode, written from each format's field definition.
 * ------------------------------------------------------------------- */
double bsqo_decode(int fmt, unsigned code)
{
    int s, e, m;
    double mag;
    switch (fmt) {
    case O_E4M3:
    case O_UE4M3:
        /* sign | 4-bit exponent, bias 7 | 3-bit mantissa; S.1111.111 = NaN,
         * no infinities; exponent field 0 = subnormal m/8 * 2^(1-7). */
        code &= 0xFF;
        s = code >> 7; e = (code >> 3) & 0xF; m = code & 7;
        if (e == 15 && m == 7) return NAN;
        mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
        return s ? -mag : mag;
    case O_E5M2:
        /* sign | 5-bit exponent, bias 15 | 2-bit mantissa; IEEE-style
         * Inf (e=31, m=0) and NaN (e=31, m!=0). */
        code &= 0xFF;
        s = code >> 7; e = (code >> 2) & 0x1F; m = code & 3;
        if (e == 31) return m ? NAN : (s ? -INFINITY : INFINITY);
        mag = (e == 0) ? ldexp((double)m, -16) : ldexp(1.0 + m / 4.0, e - 15);
        return s ? -mag : mag;
    case O_E2M1:
        /* sign | 2-bit exponent, bias 1 | 1-bit mantissa; e=0 -> m * 0.5 */
        code &= 0xF;
        s = code >> 3; e = (code >> 1) & 3; m = code & 1;
        mag = (e == 0) ? 0.5 * m : ldexp(1.0 + m / 2.0, e - 1);
        return s ? -mag : mag;
    }
    return NAN;
}

/* E8M0 shared scale: 2^(b-127); 0xFF is NaN. */
double bsqo_decode_e8m0(unsigned b)
{
    b &= 0xFF;
    if (b == 0xFF) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* number of non-negative finite codes; they are 0..n-1 in increasing value */
static int n_finite(int fmt)
{
    switch (fmt) {
    case O_E4M3: case O_UE4M3: return 127; /* 0x00..0x7E, 0x7F is NaN */
    case O_E5M2: return 124;               /* 0x00..0x7B, 0x7C is Inf */
    case O_E2M1: return 8;
    }
    return 0;
}

static int sign_shift(int fmt) { return fmt == O_E2M1 ? 3 : 7; }

/* canonical NaN code of a format (E2M1 has none: 0) */
static unsigned nan_code(int fmt) { return fmt == O_E2M1 ? 0u : 0x7Fu; }

double bsqo_max_finite(int fmt) { return bsqo_decode(fmt, (unsigned)(n_finite(fmt) - 1)); }

/* Round-to-nearest, ties to the even code (mantissa LSB = code LSB), then
 * saturate |v| above the largest finite value to that value.  The sign bit
 * is kept, so negative values that round to zero give the -0 code. */
unsigned bsqo_encode(int fmt, double v)
{
    int n = n_finite(fmt), lo, hi, i;
    unsigned sign, code;
    double a, vlo, vhi;
    if (isnan(v)) return nan_code(fmt);
    sign = signbit(v) ? 1u : 0u;
    a = fabs(v);
    if (a >= bsqo_decode(fmt, (unsigned)(n - 1))) {
        code = (unsigned)(n - 1);
    } else {
        /* largest i with value(i) <= a (binary search over the code order) */
        lo = 0; hi = n - 1;
        while (hi - lo > 1) {
            int mid = (lo + hi) / 2;
            if (bsqo_decode(fmt, (unsigned)mid) <= a) lo = mid; else hi = mid;
        }
        i = lo;
        vlo = bsqo_decode(fmt, (unsigned)i);
        vhi = bsqo_decode(fmt, (unsigned)(i + 1));
        if (a - vlo < vhi - a) code = (unsigned)i;
        else if (a - vlo > vhi - a) code = (unsigned)(i + 1);
        else code = (i % 2 == 0) ? (unsigned)i : (unsigned)(i + 1);
    }
    if (fmt == O_UE4M3) return code;           /* unsigned scale: no sign */
    return (sign << sign_shift(fmt)) | code;
}

/* BF16 bit pattern -> exact double */
double bsqo_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static float bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* largest finite element exponent: floor(log2(max finite value)) */
static int emax_elem(int fmt)
{
    int ex;
    frexp(bsqo_max_finite(fmt), &ex);
    return ex - 1;            /* 8 for E4M3, 15 for E5M2, 2 for E2M1 */
}

/* ---------------------------------------------------------------------
 * One MX block: shared exponent e = floor(log2(amax)) - emax_elem, clamped
 * to the E8M0 range [-127, 127]; an all-zero block takes e = -127; a block
 * holding NaN or Inf gets the NaN scale 0xFF and NaN element codes (E2M1,
 * which has no NaN, gets zero codes).  Codes = encode(v * 2^-e).
 * ------------------------------------------------------------------- */
void bsqo_mx_block(int fmt, const double* v, int n, uint8_t* codes, uint8_t* scale)
{
    int i, ex, e;
    double amax = 0.0;
    int nonfinite = 0;
    for (i = 0; i < n; i++) {
        if (!isfinite(v[i])) nonfinite = 1;
        else if (fabs(v[i]) > amax) amax = fabs(v[i]);
    }
    if (nonfinite) {
        *scale = 0xFF;
        for (i = 0; i < n; i++) codes[i] = (uint8_t)nan_code(fmt);
        return;
    }
    if (amax == 0.0) {
        e = -127;
    } else {
        frexp(amax, &ex);     /* amax = f * 2^ex, f in [0.5, 1) */
        e = (ex - 1) - emax_elem(fmt);
        if (e < -127) e = -127;
        if (e > 127) e = 127;
    }
    *scale = (uint8_t)(e + 127);
    for (i = 0; i < n; i++) codes[i] = (uint8_t)bsqo_encode(fmt, ldexp(v[i], -e));
}

/* MX quantize of a row-major BF16 matrix [R, C], blocks of `blk` along C.
 * codes: [R, C], one code per byte (FP4 codes unpacked);
 * scales: [R, C/blk] row-major. */
void bsqo_mx_quantize_rows(int fmt, int blk, const uint16_t* x, int64_t R, int64_t C,
                           uint8_t* codes, uint8_t* scales)
{
    int64_t r;
    /* rows are independent: spread over threads, each row as written */
#pragma omp parallel for schedule(static)
    for (r = 0; r < R; r++) {
        int64_t j;
        int i;
        double v[64];
        for (j = 0; j < C / blk; j++) {
            for (i = 0; i < blk; i++) v[i] = bsqo_bf16_to_double(x[r * C + j * blk + i]);
            bsqo_mx_block(fmt, v, blk, codes + r * C + j * blk, scales + r * (C / blk) + j);
        }
    }
}

/* ---------------------------------------------------------------------
 * NVFP4, all arithmetic IEEE FP32 with round-to-nearest, in this order:
 *  amax_t = max |x| over the finite entries of the tensor
 *  s_t    = amax_t / 2688   (2688 = 448 * 6; s_t = 1 when amax_t = 0)
 *  per 16-block: q = (amax_b / 6) / s_t ; s_b = UE4M3 encode(q)
 *    s_b code 0 -> all element codes 0
 *    else d = value(s_b) * s_t ; code_i = E2M1 encode(x_i / d)
 *  a block holding NaN or Inf gets the E4M3 NaN scale 0x7F and zero codes.
 * ------------------------------------------------------------------- */
float bsqo_nvfp4_tensor_scale(const uint16_t* x, int64_t n)
{
    int64_t i;
    float amax = 0.0f, s_t;
    for (i = 0; i < n; i++) {
        float f = bf16_to_float(x[i]);
        if (isfinite(f) && fabsf(f) > amax) amax = fabsf(f);
    }
    if (amax == 0.0f) return 1.0f;
    s_t = amax / 2688.0f;
    return s_t;
}

/* Largest finite |x| of a BF16 tensor: the tensor amax of the NVFP4 recipe
 * (non-finite values are skipped, as in bsqo_nvfp4_tensor_scale). */
float bsqo_tensor_amax(const uint16_t* x, int64_t n)
{
    int64_t i;
    float amax = 0.0f;
    for (i = 0; i < n; i++) {
        float f = bf16_to_float(x[i]);
        if (isfinite(f) && fabsf(f) > amax) amax = fabsf(f);
    }
    return amax;
}

/* Delayed scaling ("FP8 Training Infrastructure", sections "Transformer
 * Engine: a fundacao de software" and "Estrategias de escalonamento e
 * estabilidade": scale factors come from the amax values observed in
 * previous iterations; history length 16, algorithm "max", margin 0).
 * For NVFP4 the tensor scale of the current step is
 *   s_t = max(history) / 2688   (FP32, round to nearest),
 * and 1 when the history holds no positive finite value (the same rule as
 * an all-zero tensor in the just-in-time recipe). */
float bsqo_nvfp4_delayed_tensor_scale(const float* hist, int64_t n)
{
    int64_t i;
    float m = 0.0f;
    for (i = 0; i < n; i++)
        if (isfinite(hist[i]) && hist[i] > m) m = hist[i];
    if (m == 0.0f) return 1.0f;
    return m / 2688.0f;
}

void bsqo_nvfp4_quantize_rows(const uint16_t* x, int64_t R, int64_t C, float s_t,
                              uint8_t* codes, uint8_t* scales)
{
    int64_t r;
    /* rows are independent: spread over threads, each row as written */
#pragma omp parallel for schedule(static)
    for (r = 0; r < R; r++) {
        int64_t j;
        int i;
        for (j = 0; j < C / 16; j++) {
            const uint16_t* xb = x + r * C + j * 16;
            uint8_t* cb = codes + r * C + j * 16;
            float amax_b = 0.0f, q, d;
            unsigned sb;
            int nonfinite = 0;
            for (i = 0; i < 16; i++) {
                float f = bf16_to_float(xb[i]);
                if (!isfinite(f)) nonfinite = 1;
                else if (fabsf(f) > amax_b) amax_b = fabsf(f);
            }
            if (nonfinite) {
                scales[r * (C / 16) + j] = 0x7F;
                for (i = 0; i < 16; i++) cb[i] = 0;
                continue;
            }
            q = amax_b / 6.0f;
            q = q / s_t;
            sb = bsqo_encode(O_UE4M3, (double)q);
            scales[r * (C / 16) + j] = (uint8_t)sb;
            if (sb == 0) {
                for (i = 0; i < 16; i++) cb[i] = 0;
                continue;
            }
            d = (float)bsqo_decode(O_UE4M3, sb) * s_t;
            for (i = 0; i < 16; i++) {
                float qi = bf16_to_float(xb[i]) / d;
                cb[i] = (uint8_t)bsqo_encode(O_E2M1, (double)qi);
            }
        }
    }
}

/* ---------------------------------------------------------------------
 * Dequantize to exact doubles.  MX: value(code) * 2^(scale-127).
 * NVFP4: value(code) * value(s_b) * s_t.
 * ------------------------------------------------------------------- */
void bsqo_mx_dequant_rows(int fmt, int blk, const uint8_t* codes, const uint8_t* scales,
                          int64_t R, int64_t C, double* out)
{
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < R; r++) {
        int64_t k;
        for (k = 0; k < C; k++)
            out[r * C + k] = bsqo_decode(fmt, codes[r * C + k]) *
                             bsqo_decode_e8m0(scales[r * (C / blk) + k / blk]);
    }
}

void bsqo_nvfp4_dequant_rows(const uint8_t* codes, const uint8_t* scales, float s_t,
                             int64_t R, int64_t C, double* out)
{
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < R; r++) {
        int64_t k;
        for (k = 0; k < C; k++)
            out[r * C + k] = bsqo_decode(O_E2M1, codes[r * C + k]) *
                             bsqo_decode(O_UE4M3, scales[r * (C / 16) + k / 16]) * (double)s_t;
    }
}

/* ---------------------------------------------------------------------
 * MXFP4 -> MXFP8 (E4M3) re-encode.  Definition used: the E4M3 MX quantize
 * of the exactly dequantized MXFP4 block (same 32-element block, same
 * rule as bsqo_mx_block).  This is the "numerically equivalent" result the
 * direct integer-domain conversion must reproduce.
 * ------------------------------------------------------------------- */
void bsqo_mxfp4_to_mxfp8_rows(const uint8_t* codes4, const uint8_t* scales4, int64_t R, int64_t C,
                              uint8_t* codes8, uint8_t* scales8)
{
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < R; r++) {
        int64_t j;
        int i;
        double v[32];
        for (j = 0; j < C / 32; j++) {
            double s = bsqo_decode_e8m0(scales4[r * (C / 32) + j]);
            for (i = 0; i < 32; i++) v[i] = bsqo_decode(O_E2M1, codes4[r * C + j * 32 + i]) * s;
            bsqo_mx_block(O_E4M3, v, 32, codes8 + r * C + j * 32, scales8 + r * (C / 32) + j);
        }
    }
}

/* ---------------------------------------------------------------------
 * GEMM reference, C[m][n] = sum_k A[m][k] * B[n][k] over exactly
 * dequantized operands (both K-major).  Inputs are dequantized doubles
 * [M][K] and [N][K].  For each requested (m, n) pair it returns
 * ref = sum_k a*b and mag = sum_k |a*b| in FP64.
 * ------------------------------------------------------------------- */
/* FP4RowToFP8Col ("Practical FP4 Training for Large-Scale MoE Models on
 * Hopper GPUs", section 2, "Kernels": dequantize, transpose and
 * re-quantize column-wise in one step, for the weight gradient).  Reading:
 * the MXFP8 E4M3 quantization, blocks of 32 along the rows, of the exactly
 * dequantized MXFP4 matrix, stored transposed.
 *   in:  codes4 [R, C] (one E2M1 code per byte), scales4 [R, C/32] (E8M0)
 *   out: codes8 [C, R] (E4M3), scales8 [C, R/32] (E8M0); R % 32 == 0. */
void bsqo_mxfp4_row_to_mxfp8_col(const uint8_t* codes4, const uint8_t* scales4, int64_t R, int64_t C,
                                 uint8_t* codes8, uint8_t* scales8)
{
    int64_t c, j;
    int i;
    double v[32];
    for (c = 0; c < C; c++)
        for (j = 0; j < R / 32; j++) {
            for (i = 0; i < 32; i++) {
                const int64_t r = j * 32 + i;
                v[i] = bsqo_decode(O_E2M1, codes4[r * C + c]) * bsqo_decode_e8m0(scales4[r * (C / 32) + c / 32]);
            }
            bsqo_mx_block(O_E4M3, v, 32, codes8 + c * R + j * 32, scales8 + c * (R / 32) + j);
        }
}

/* MXFP4 -> FP8 E4M3 with 1x128 blocks, the FP8 block of the Hopper path
 * ("Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs",
 * section 2, "Algoritmo de Conversao Direta": FP8 blocks hold 128
 * elements, the conversion takes the largest of the four FP4 block scales
 * and moves each element's exponent to it).  Readings: the 128-block scale
 * is the largest E8M0 byte among the (up to four) 32-blocks it covers, kept
 * as an E8M0 byte; each element is the E4M3 code (RNE) of its exact value
 * divided by that scale, so it is exact while its own block scale is within
 * a few binades of the largest and rounds (into E4M3's subnormals, then to
 * zero) beyond; a NaN scale byte (0xFF, the largest byte) makes the whole
 * 128-block NaN.
 *   in:  codes4 [R, C] (one E2M1 code per byte), scales4 [R, C/32] (E8M0)
 *   out: codes8 [R, C] (E4M3), scales8 [R, ceil(C/128)] (E8M0); C % 32 == 0. */
void bsqo_mxfp4_to_fp8_1x128(const uint8_t* codes4, const uint8_t* scales4, int64_t R, int64_t C,
                             uint8_t* codes8, uint8_t* scales8)
{
    const int64_t S = C / 32, G = (C + 127) / 128;
    int64_t r, g, c, j;
    for (r = 0; r < R; r++)
        for (g = 0; g < G; g++) {
            unsigned smax = 0;
            for (j = 4 * g; j < 4 * g + 4 && j < S; j++)
                if (scales4[r * S + j] > smax) smax = scales4[r * S + j];
            scales8[r * G + g] = (uint8_t)smax;
            for (c = 128 * g; c < 128 * g + 128 && c < C; c++) {
                if (smax == 0xFFu) {
                    codes8[r * C + c] = (uint8_t)nan_code(O_E4M3);
                } else {
                    const double v = bsqo_decode(O_E2M1, codes4[r * C + c]) *
                                     bsqo_decode_e8m0(scales4[r * S + c / 32]) / bsqo_decode_e8m0(smax);
                    codes8[r * C + c] = (uint8_t)bsqo_encode(O_E4M3, v);
                }
            }
        }
}

void bsqo_gemm_pairs(const double* A, const double* B, int64_t K,
                     const int64_t* ms, const int64_t* ns, int64_t npairs,
                     double* ref, double* mag)
{
    int64_t p;
#pragma omp parallel for schedule(static)
    for (p = 0; p < npairs; p++) {
        const double* a = A + ms[p] * K;
        const double* b = B + ns[p] * K;
        double s = 0.0, t = 0.0;
        int64_t k;
        for (k = 0; k < K; k++) {
            double prod = a[k] * b[k];
            s += prod;
            t += fabs(prod);
        }
        ref[p] = s;
        mag[p] = t;
    }
}

/* all M x N outputs, rows of A against rows of B */
void bsqo_gemm_full(const double* A, const double* B, int64_t M, int64_t N, int64_t K,
                    double* ref, double* mag)
{
    int64_t m;
#pragma omp parallel for schedule(static)
    for (m = 0; m < M; m++) {
        int64_t n, k;
        for (n = 0; n < N; n++) {
            double s = 0.0, t = 0.0;
            for (k = 0; k < K; k++) {
                double prod = A[m * K + k] * B[n * K + k];
                s += prod;
                t += fabs(prod);
            }
            ref[m * N + n] = s;
            mag[m * N + n] = t;
        }
    }
}
