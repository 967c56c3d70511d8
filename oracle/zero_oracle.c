/*
 * CPU oracle for the sharded mixed-precision Adam step -- TEST INFRASTRUCTURE.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this code.  The GPU library never links it, and it shares no code,
 * header or constant table with the GPU library.
 *
 * What it computes is the *unpartitioned* step.  The ZeRO pages state that
 * partitioning optimizer state, gradients and parameters across the N_d
 * data-parallel ranks does not change the mathematics of a training step
 * (ZeRO visual reading, "ZeRO-DP" overview before the stage list), so the
 * plain definition of one step is:
 *
 *   1. all-reduce the N_d ranks' 16-bit gradients: an fp32 sum taken in rank
 *      order, rounded once to the 16-bit gradient type (ZeRO: 大模型训练的
 *      内存优化革命, glossary "Reduce-Scatter"/"All-Gather"; ZeRO visual
 *      reading, communication accounting: all-reduce = reduce-scatter +
 *      all-gather);
 *   2. check the reduced gradient for inf/NaN (loss-scale overflow);
 *   3. unscale by 1/(S*N_d) (mean over ranks, loss scale S removed);
 *   4. apply Adam to the fp32 master weights, momentum and variance and cast
 *      the new master weights back to the 16-bit type ("updates use fp32
 *      weights ... cast back to fp16": SC-2020 ZeRO notes, "Where Did All the
 *      Memory Go? / Model States").
 *
 * Adam itself is not on the pages; it is Kingma & Ba (ICLR 2015), Algorithm 1,
 * with bias correction and eps outside the square root, evaluated in fp32 in
 * the order written in oracle_adam below.  The exact gradient norm for
 * clipping and all scalar bookkeeping (bias-correction terms, loss scale)
 * live in oracle/__init__.py.
 *
 * fp32 training (the pages' fp32 SGD / SGD-with-momentum examples, b = 4 bytes
 * per parameter and gradient: ZeRO visual reading, worked examples C) is the
 * same step with the model-precision type binary32: the rank-order sum is
 * not rounded again and the "cast" of the master weights is the identity.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC (no FMA
 * contraction, so every fp32 operation below is one IEEE-754 rounding).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_FP16 0
#define ORACLE_BF16 1
#define ORACLE_FP32 2

/* ---------------------------------------------------------------------------
 * 16-bit formats, written from their definitions.
 *
 * binary16 (IEEE 754-2008): 1 sign bit, 5 exponent bits (bias 15), 10
 * fraction bits.  Normal numbers (1.f) * 2^(e-15); subnormals (0.f) * 2^-14;
 * e = 31 encodes inf (f = 0) and NaN.
 * bfloat16: the upper 16 bits of a binary32: 1 sign, 8 exponent (bias 127),
 * 7 fraction bits.
 * Rounding from binary32 is round-to-nearest, ties-to-even.  NaN results are
 * returned as a quiet NaN with the input's sign; only NaN-ness, never the
 * payload, carries meaning here.
 * ------------------------------------------------------------------------- */

float oracle_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 31) {
        mag = (f == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        mag = ldexp((double)f, -24);             /* 0.f * 2^-14 = f * 2^-24 */
    } else {
        mag = ldexp((double)(1024 + f), e - 25); /* 1.f * 2^(e-15) */
    }
    return (float)(sign ? -mag : mag);
}

float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;               /* bf16 is the top half of binary32 */
    float x;
    memcpy(&x, &u, sizeof x);
    return x;
}

/* Round a finite non-negative double `a` (which is exactly a binary32 value)
 * to a 16-bit format with `frac_bits` fraction bits, minimum normal exponent
 * `emin`, largest finite value `maxfin` and bias `bias`.  Returns the
 * magnitude bits (no sign).  The spacing of representable numbers around a
 * is 2^(floor(log2 a) - frac_bits), never finer than the subnormal spacing
 * 2^(emin - frac_bits). */
static uint16_t round_mag16(double a, int frac_bits, int emin, int bias, double tie_to_inf)
{
    if (a >= tie_to_inf) {
        /* At or above the midpoint between the largest finite value and
         * 2^(emax+1) the nearest (ties-to-even: the largest finite value has
         * an odd significand) is infinity. */
        return (uint16_t)(((1u << (15 - frac_bits)) - 1u) << frac_bits);
    }
    if (a == 0.0)
        return 0;
    int e2;
    frexp(a, &e2);                       /* a in [2^(e2-1), 2^e2) */
    int q = (e2 - 1) - frac_bits;        /* exponent of the spacing */
    if (q < emin - frac_bits)
        q = emin - frac_bits;            /* subnormal range */
    double n = ldexp(a, -q);             /* exact: a has 24 significant bits */
    double r = nearbyint(n);             /* default mode: nearest, ties to even */
    uint32_t ri = (uint32_t)r;
    uint32_t one = 1u << frac_bits;
    if (q == emin - frac_bits && ri < one)
        return (uint16_t)ri;             /* subnormal or zero */
    if (ri == 2 * one) {                 /* rounding carried into the next binade */
        ri = one;
        q += 1;
    }
    uint32_t biased = (uint32_t)(q + frac_bits + bias);
    return (uint16_t)((biased << frac_bits) | (ri - one));
}

uint16_t oracle_f32_to_f16(float x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x))
        return sign | 0x7e00;
    if (isinf(x))
        return sign | 0x7c00;
    /* largest finite 65504 = 2047 * 2^5; next binade would start at 2^16 */
    return sign | round_mag16(fabs((double)x), 10, -14, 15, 65520.0);
}

uint16_t oracle_f32_to_bf16(float x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x))
        return sign | 0x7fc0;
    if (isinf(x))
        return sign | 0x7f80;
    /* largest finite (2 - 2^-7) * 2^127; the tie with 2^128 is (2 - 2^-8) * 2^127 */
    return sign | round_mag16(fabs((double)x), 7, -126, 127, ldexp(2.0 - ldexp(1.0, -8), 127));
}

static float to_f32(uint16_t h, int dtype)
{
    return dtype == ORACLE_BF16 ? oracle_bf16_to_f32(h) : oracle_f16_to_f32(h);
}

static uint16_t to_16(float x, int dtype)
{
    return dtype == ORACLE_BF16 ? oracle_f32_to_bf16(x) : oracle_f32_to_f16(x);
}

/* Element i of an array of model-precision values (16-bit patterns, or
 * binary32 for ORACLE_FP32), widened to fp32; and the store that rounds an
 * fp32 value to the model precision (exact for ORACLE_FP32). */
static float get_val(const void* a, int64_t i, int dtype)
{
    if (dtype == ORACLE_FP32) {
        float x;
        memcpy(&x, (const char*)a + 4 * i, 4);
        return x;
    }
    return to_f32(((const uint16_t*)a)[i], dtype);
}

static void put_val(void* a, int64_t i, float x, int dtype)
{
    if (dtype == ORACLE_FP32)
        memcpy((char*)a + 4 * i, &x, 4);
    else
        ((uint16_t*)a)[i] = to_16(x, dtype);
}

/* Bulk conversions, for the tests that pin the format code against library
 * routines. */
void oracle_to_f32_array(int64_t n, const void* src, int32_t dtype, float* dst)
{
    for (int64_t i = 0; i < n; i++)
        dst[i] = get_val(src, i, dtype);
}

void oracle_from_f32_array(int64_t n, const float* src, int32_t dtype, void* dst)
{
    for (int64_t i = 0; i < n; i++)
        put_val(dst, i, src[i], dtype);
}

/* ---------------------------------------------------------------------------
 * Steps 1-2: gradient all-reduce in rank order, and the overflow check.
 *
 * h[i] = round16( (((0 + g_0[i]) + g_1[i]) + ...) + g_{N-1}[i] ), the sum in
 * fp32 (for ORACLE_FP32 the fp32 sum itself).  Returns 1 if any h[i] is inf
 * or NaN, else 0.
 * ------------------------------------------------------------------------- */
uint32_t oracle_reduce(int32_t n_ranks, int64_t n, const void* const* grads,
                       int32_t dtype, void* h)
{
    uint32_t overflow = 0;
    for (int64_t i = 0; i < n; i++) {
        float s = 0.0f;
        for (int32_t r = 0; r < n_ranks; r++)
            s = s + get_val(grads[r], i, dtype);
        put_val(h, i, s, dtype);
        if (!isfinite(get_val(h, i, dtype)))
            overflow = 1;
    }
    return overflow;
}

/* Exact sum of squares of 16-bit values, grouped by binary exponent.
 *
 * Every finite 16-bit value is h = M * 2^E with an integer significand M
 * (M < 2^11 for binary16, M < 2^8 for bfloat16), so h^2 = M^2 * 2^(2E).
 * bins[k] receives the integer sum of M^2 over the elements whose biased
 * exponent field is k (subnormals, k = 0, use the same E as k = 1).  No
 * rounding happens; inf/NaN elements are skipped.  The caller forms
 * sum_k bins[k] * 2^(2 E(k)) exactly. */
void oracle_sumsq_bins(int64_t n, const uint16_t* h, int32_t dtype, uint64_t bins[256])
{
    for (int k = 0; k < 256; k++)
        bins[k] = 0;
    for (int64_t i = 0; i < n; i++) {
        uint32_t e, f, M;
        if (dtype == ORACLE_BF16) {
            e = (h[i] >> 7) & 0xff;
            f = h[i] & 0x7f;
            if (e == 0xff)
                continue;
            M = e ? (f | 0x80) : f;
        } else {
            e = (h[i] >> 10) & 0x1f;
            f = h[i] & 0x3ff;
            if (e == 0x1f)
                continue;
            M = e ? (f | 0x400) : f;
        }
        bins[e] += (uint64_t)M * M;
    }
}

/* ---------------------------------------------------------------------------
 * Steps 3-4: unscale, optional clip, Adam on the fp32 master state, cast.
 * ------------------------------------------------------------------------- */
typedef struct {
    float inv_scale;        /* 1/(S*N_d), rounded to fp32 once */
    int32_t use_clip;       /* multiply by clip after unscaling */
    float clip;             /* clip coefficient min(1, max_norm/(norm+1e-6)) */
    float lr, beta1, beta2, eps;
    float one_minus_beta1;  /* 1 - beta1 in fp32 */
    float one_minus_beta2;  /* 1 - beta2 in fp32 */
    float bc1, bc2;         /* 1 - beta^t, formed in fp64 and rounded to fp32 once */
} oracle_hyper_t;

/* Kingma & Ba, Algorithm 1, one fp32 rounding per operation:
 *   g  = h * (1/(S N))            [* c when clipping]
 *   m' = beta1*m + (1-beta1)*g
 *   v' = beta2*v + (1-beta2)*(g*g)
 *   w' = w - lr * ( (m'/bc1) / (sqrt(v'/bc2) + eps) )
 *   p  = round16(w')
 * w, m, v are updated in place; p16 receives the cast. */
void oracle_adam(int64_t n, const void* h, int32_t dtype, const oracle_hyper_t* hp,
                 float* w, float* m, float* v, void* p16)
{
    for (int64_t i = 0; i < n; i++) {
        float g = get_val(h, i, dtype) * hp->inv_scale;
        if (hp->use_clip)
            g = g * hp->clip;
        float t1 = hp->beta1 * m[i];
        float t2 = hp->one_minus_beta1 * g;
        float m1 = t1 + t2;
        float t3 = g * g;
        float t4 = hp->one_minus_beta2 * t3;
        float t5 = hp->beta2 * v[i];
        float v1 = t5 + t4;
        float mh = m1 / hp->bc1;
        float vh = v1 / hp->bc2;
        float d = sqrtf(vh) + hp->eps;
        float u = mh / d;
        float step = hp->lr * u;
        float w1 = w[i] - step;
        w[i] = w1;
        m[i] = m1;
        v[i] = v1;
        put_val(p16, i, w1, dtype);
    }
}

/* SGD on the fp32 master weights (the other optimizers of the (2b+K)
 * accounting; PyTorch's SGD without dampening, Nesterov or weight decay):
 *   g  = h * (1/(S N))            [* c when clipping]
 *   with momentum mu (m != NULL):  m' = mu*m + g;  w' = w - lr*m'
 *   plain (m == NULL):             w' = w - lr*g
 *   p  = round16(w')
 * hp->beta1 carries mu; beta2, eps and the bias corrections are unused. */
void oracle_sgd(int64_t n, const void* h, int32_t dtype, const oracle_hyper_t* hp,
                float* w, float* m, void* p16)
{
    for (int64_t i = 0; i < n; i++) {
        float g = get_val(h, i, dtype) * hp->inv_scale;
        if (hp->use_clip)
            g = g * hp->clip;
        float d = g;
        if (m) {
            float t1 = hp->beta1 * m[i];
            float m1 = t1 + g;
            m[i] = m1;
            d = m1;
        }
        float step = hp->lr * d;
        float w1 = w[i] - step;
        w[i] = w1;
        put_val(p16, i, w1, dtype);
    }
}

/* The model-precision copy of the master weights (used to initialise the
 * parameters and, after a skipped step, as their unchanged value). */
void oracle_cast(int64_t n, const float* w, int32_t dtype, void* p16)
{
    for (int64_t i = 0; i < n; i++)
        put_val(p16, i, w[i], dtype);
}
