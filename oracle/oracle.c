/*
 * oracle.c -- plain, slow, obviously correct CPU definitions of the
 * memory-bound elementwise operators.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the reference the CUDA kernels are
 * checked against.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load or call it; the product library never
 * links it, and it shares no code, header, table or helper with the CUDA path.
 *
 * Every function is single-threaded, walks the elements in index order and
 * evaluates the textbook definition of the operation.  Floating point is done
 * in binary64 and rounded once to the storage type, except where the
 * definition itself fixes the arithmetic (SAXPY is defined through a fused
 * multiply-add, see orc_saxpy_*).  Half-precision formats are decoded and
 * encoded here from their bit-field definitions (IEEE 754 binary16, and
 * bfloat16 = the top 16 bits of binary32), with round-to-nearest-even.
 *
 * Operations and the passages they follow:
 *   add     C[i] = A[i] + B[i]            "HyperAI elementwise add on RTX 5090",
 *                                          Version 1 (FP32) and Version 3 (FP16);
 *                                          "逐元素操作算子" §一.1 (each output depends
 *                                          only on the same index of the inputs)
 *   saxpy   y[i] = alpha * x[i] + y[i]    "Puzzle 31: occupancy optimisation",
 *                                          overview (minimal kernel); fused as fmaf
 *   relu    y[i] = max(x[i], 0)           CUDA-MODE lecture notes (cyqw.cn), §5.2
 *                                          example 1
 *   copy    out[i] = in[i]                CUDA-MODE lecture notes, §3.2 coalesced
 *   gather  out[i] = in[(s*i) mod n]      CUDA-MODE lecture notes, §3.2
 *                                          non-coalesced (s = 2 on the page)
 *   ceil_div(n, t) = (n + t - 1) / t      "逐元素操作算子" §二, launch configuration
 *   select  y[i] = x[i] even ? 2 x[i] : x[i] + 1 on 32-bit integers
 *                                          CUDA-MODE lecture notes, §6.1-6.2
 *                                          (control-divergence example)
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the design notes):
 *   - relu maps every x <= 0, including -0, to +0; a NaN input is passed
 *     through with its bits unchanged.
 *   - saxpy is one fused multiply-add in binary32 (C99 fmaf, which is correctly
 *     rounded); for 16-bit types x and y are widened exactly to binary32, the
 *     fmaf is taken there and the result is rounded once to the 16-bit type.
 *     alpha is a binary32 value and is never rounded to the 16-bit type.
 *   - the gather index s*i is formed without overflow (128-bit product).
 *   - select works on two's complement 32-bit integers ("x % 2 == 0" on the
 *     page); 2x and x + 1 wrap modulo 2^32 instead of overflowing.
 *
 * Build: cc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fno-fast-math
 * (see oracle/build.py).  No OpenMP, no intrinsics, no architecture flags.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------ */
/* Format definitions                                                  */
/* ------------------------------------------------------------------ */

/* Round a finite, non-negative binary64 value q (already scaled so that
 * the wanted quantum is 1) to the nearest integer, ties to even. */
static double round_half_even(double q)
{
    double r = floor(q);
    double frac = q - r; /* exact: q and r share an exponent range */
    if (frac > 0.5) {
        r += 1.0;
    } else if (frac == 0.5) {
        if (fmod(r, 2.0) != 0.0) r += 1.0;
    }
    return r;
}

/* Generic decoder for a binary interchange-style format with `mbits` stored
 * significand bits and `ebits` exponent bits (bias 2^(ebits-1)-1). */
static double decode_bits(uint32_t bits, int ebits, int mbits)
{
    uint32_t sign = (bits >> (ebits + mbits)) & 1u;
    uint32_t e = (bits >> mbits) & ((1u << ebits) - 1u);
    uint32_t m = bits & ((1u << mbits) - 1u);
    int bias = (1 << (ebits - 1)) - 1;
    double v;
    if (e == 0) {
        v = ldexp((double)m, 1 - bias - mbits); /* subnormal or zero */
    } else if (e == (1u << ebits) - 1u) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)((1u << mbits) + m), (int)e - bias - mbits);
    }
    return sign ? -v : v;
}

/* Generic encoder: round binary64 x to the format, nearest-even, with
 * gradual underflow and overflow to infinity.  A NaN maps to the quiet NaN
 * with an all-zero payload below the quiet bit and x's sign. */
static uint32_t encode_bits(double x, int ebits, int mbits)
{
    uint32_t sign = signbit(x) ? 1u : 0u;
    uint32_t sign_field = sign << (ebits + mbits);
    uint32_t emax_field = (1u << ebits) - 1u;
    int bias = (1 << (ebits - 1)) - 1;
    int emin = 1 - bias; /* exponent of the smallest normal */
    double a = fabs(x);

    if (isnan(x)) return sign_field | (emax_field << mbits) | (1u << (mbits - 1));
    if (isinf(a)) return sign_field | (emax_field << mbits);

    if (a < ldexp(1.0, emin)) {
        /* subnormal range: quantum is 2^(emin - mbits) */
        double r = round_half_even(ldexp(a, mbits - emin));
        /* r == 2^mbits is the smallest normal, whose encoding is also r */
        return sign_field | (uint32_t)r;
    }
    int ex;
    (void)frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;      /* a in [2^E, 2^(E+1)) */
    double r = round_half_even(ldexp(a, mbits - E)); /* in [2^mbits, 2^(mbits+1)] */
    if (r == ldexp(1.0, mbits + 1)) {
        r = ldexp(1.0, mbits);
        E += 1;
    }
    if (E > bias) return sign_field | (emax_field << mbits); /* overflow */
    uint32_t m = (uint32_t)(r - ldexp(1.0, mbits));
    return sign_field | ((uint32_t)(E + bias) << mbits) | m;
}

ORC_API double orc_f16_to_f64(uint16_t h) { return decode_bits(h, 5, 10); }
ORC_API uint16_t orc_f64_to_f16(double x) { return (uint16_t)encode_bits(x, 5, 10); }
ORC_API double orc_bf16_to_f64(uint16_t h) { return decode_bits(h, 8, 7); }
ORC_API uint16_t orc_f64_to_bf16(double x) { return (uint16_t)encode_bits(x, 8, 7); }
ORC_API float orc_f64_to_f32(double x) { return (float)x; }

/* ------------------------------------------------------------------ */
/* Launch geometry                                                      */
/* ------------------------------------------------------------------ */

ORC_API int64_t orc_ceil_div(int64_t n, int64_t t) { return (n + t - 1) / t; }

/* ------------------------------------------------------------------ */
/* C = A + B                                                            */
/* ------------------------------------------------------------------ */

ORC_API void orc_add_f32(const float *a, const float *b, float *c, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        double s = (double)a[i] + (double)b[i];
        c[i] = (float)s; /* one rounding, to nearest even */
    }
}

ORC_API void orc_add_f16(const uint16_t *a, const uint16_t *b, uint16_t *c, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        double s = orc_f16_to_f64(a[i]) + orc_f16_to_f64(b[i]);
        c[i] = orc_f64_to_f16(s);
    }
}

ORC_API void orc_add_bf16(const uint16_t *a, const uint16_t *b, uint16_t *c, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        double s = orc_bf16_to_f64(a[i]) + orc_bf16_to_f64(b[i]);
        c[i] = orc_f64_to_bf16(s);
    }
}

/* ------------------------------------------------------------------ */
/* y = alpha * x + y  (in place)                                        */
/* ------------------------------------------------------------------ */

ORC_API void orc_saxpy_f32(float alpha, const float *x, float *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = fmaf(alpha, x[i], y[i]);
}

ORC_API void orc_saxpy_f16(float alpha, const uint16_t *x, uint16_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        float xf = (float)orc_f16_to_f64(x[i]); /* exact widening */
        float yf = (float)orc_f16_to_f64(y[i]);
        float r = fmaf(alpha, xf, yf);
        y[i] = orc_f64_to_f16((double)r);
    }
}

ORC_API void orc_saxpy_bf16(float alpha, const uint16_t *x, uint16_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        float xf = (float)orc_bf16_to_f64(x[i]);
        float yf = (float)orc_bf16_to_f64(y[i]);
        float r = fmaf(alpha, xf, yf);
        y[i] = orc_f64_to_bf16((double)r);
    }
}

/* ------------------------------------------------------------------ */
/* y = max(x, 0)                                                        */
/* ------------------------------------------------------------------ */

ORC_API void orc_relu_f32(const float *x, float *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        double v = (double)x[i];
        if (isnan(v) || v > 0.0) {
            y[i] = x[i];
        } else {
            y[i] = 0.0f; /* +0 */
        }
    }
}

ORC_API void orc_relu_f16(const uint16_t *x, uint16_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        double v = orc_f16_to_f64(x[i]);
        y[i] = (isnan(v) || v > 0.0) ? x[i] : (uint16_t)0;
    }
}

ORC_API void orc_relu_bf16(const uint16_t *x, uint16_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        double v = orc_bf16_to_f64(x[i]);
        y[i] = (isnan(v) || v > 0.0) ? x[i] : (uint16_t)0;
    }
}

/* ------------------------------------------------------------------ */
/* copy and strided gather (raw element bits)                           */
/* ------------------------------------------------------------------ */

ORC_API void orc_copy(const void *in, void *out, int64_t n, int64_t elem_size)
{
    const unsigned char *src = (const unsigned char *)in;
    unsigned char *dst = (unsigned char *)out;
    for (int64_t i = 0; i < n; ++i)
        memcpy(dst + i * elem_size, src + i * elem_size, (size_t)elem_size);
}

ORC_API int64_t orc_gather_index(int64_t i, int64_t s, int64_t n)
{
    unsigned __int128 p = (unsigned __int128)(uint64_t)s * (uint64_t)i;
    return (int64_t)(p % (uint64_t)n);
}

ORC_API void orc_gather_stride(const void *in, void *out, int64_t n, int64_t s,
                               int64_t elem_size)
{
    const unsigned char *src = (const unsigned char *)in;
    unsigned char *dst = (unsigned char *)out;
    for (int64_t i = 0; i < n; ++i) {
        int64_t j = orc_gather_index(i, s, n);
        memcpy(dst + i * elem_size, src + j * elem_size, (size_t)elem_size);
    }
}

/* ------------------------------------------------------------------ */
/* y = x even ? 2x : x + 1  (32-bit integers, wrapping)                 */
/* ------------------------------------------------------------------ */

ORC_API void orc_select_even_odd_i32(const int32_t *x, int32_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u = (uint32_t)x[i];
        if (x[i] % 2 == 0) {
            y[i] = (int32_t)(u * 2u);
        } else {
            y[i] = (int32_t)(u + 1u);
        }
    }
}
