/*
 * dc_oracle.c -- plain, slow, obviously correct CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the CUDA library.  It shares no
 * code, header, table or helper with the GPU path.
 *
 * Build: gcc -std=c11 -O2 -fno-fast-math -ffp-contract=off -fPIC -shared.
 * No FTZ/DAZ: orc_subnormals_preserved() checks it at run time.
 *
 * Page cited by title:
 *   [PR491] "perf(cuda): vectorize the deterministic all-gather copy and
 *           right-size its single-block path".
 */
#include "dc_oracle.h"

#include <string.h>

/* [PR491] "What", copy_rank_ordered bullet: the gathered output is the
 * rank-ordered concatenation of the P payloads, byte for byte.  Written as
 * the definition: byte j of peer r lands at out[r*B + j]. */
int orc_all_gather(const uint8_t *const *peers, int P, size_t B, uint8_t *out)
{
    if (P < 1 || (B > 0 && (peers == NULL || out == NULL)))
        return -1;
    for (int r = 0; r < P; ++r) {
        if (B > 0 && peers[r] == NULL)
            return -1;
        for (size_t j = 0; j < B; ++j)
            out[(size_t)r * B + j] = peers[r][j];
    }
    return 0;
}

/* all_gather_many: each tensor t is gathered on its own into outs[t]
 * (no packing across tensors). */
int orc_all_gather_many(const uint8_t *const *peers, const size_t *bytes,
                        uint8_t *const *outs, int T, int P)
{
    if (T < 0 || P < 1 || (T > 0 && (peers == NULL || bytes == NULL || outs == NULL)))
        return -1;
    for (int t = 0; t < T; ++t) {
        int rc = orc_all_gather(peers + (size_t)t * (size_t)P, P, bytes[t], outs[t]);
        if (rc != 0)
            return rc;
    }
    return 0;
}

/* A BF16 value is the upper 16 bits of the binary32 value with the same
 * sign, exponent and leading 7 fraction bits, so widening is exact. */
float orc_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round to nearest, ties to even, from binary32 to BF16.
 *
 * Dropping the low 16 bits truncates toward zero in magnitude.  Adding
 * 0x7FFF plus the lowest kept bit before truncating rounds up exactly when
 * the dropped half is above one half-ulp, or equal to it with an odd kept
 * part: the definition of ties-to-even on the magnitude.  A carry out of
 * the fraction moves into the exponent, which is the correct next value
 * (and turns the largest finite values that round up into infinity).
 * Subnormals follow the same rule.  NaN must not be rounded (a carry could
 * turn it into infinity), so it becomes the quiet NaN with its sign. */
uint16_t orc_f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

int orc_f32_to_bf16_rne_array(const float *in, uint16_t *out, size_t n)
{
    if (n > 0 && (in == NULL || out == NULL))
        return -1;
    for (size_t i = 0; i < n; ++i)
        out[i] = orc_f32_to_bf16_rne(in[i]);
    return 0;
}

/* The fixed-order fold of one element across the P ranks: start from
 * rank 0's value itself (so an all-negative-zero column stays -0), then add
 * ranks 1..P-1 one at a time in binary32, then round once to BF16. */
static uint16_t fold_ranks(const uint16_t *const *in, int P, size_t i)
{
    float acc = orc_bf16_to_f32(in[0][i]);
    for (int q = 1; q < P; ++q) {
        float x = orc_bf16_to_f32(in[q][i]);
        acc = acc + x;
    }
    return orc_f32_to_bf16_rne(acc);
}

int orc_all_reduce_bf16(const uint16_t *const *in, uint16_t *const *out,
                        int P, size_t count)
{
    if (P < 1 || (count > 0 && (in == NULL || out == NULL)))
        return -1;
    for (int r = 0; r < P; ++r)
        if (count > 0 && (in[r] == NULL || out[r] == NULL))
            return -1;
    for (size_t i = 0; i < count; ++i) {
        uint16_t y = fold_ranks(in, P, i);
        for (int r = 0; r < P; ++r)
            out[r][i] = y;
    }
    return 0;
}

int orc_reduce_scatter_bf16(const uint16_t *const *in, uint16_t *const *out,
                            int P, size_t C)
{
    if (P < 1 || (C > 0 && (in == NULL || out == NULL)))
        return -1;
    for (int r = 0; r < P; ++r)
        if (C > 0 && (in[r] == NULL || out[r] == NULL))
            return -1;
    for (int r = 0; r < P; ++r)
        for (size_t j = 0; j < C; ++j)
            out[r][j] = fold_ranks(in, P, (size_t)r * C + j);
    return 0;
}

/* ------------------------------------------------------------------------
 * binary16.  Layout: sign (1), exponent (5, bias 15), fraction (10).  Normal
 * values are (1 + f/1024) * 2^(e-15); subnormals f * 2^-24. */
float orc_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1Fu;
    uint32_t f = h & 0x3FFu;
    uint32_t u;
    if (e == 0x1Fu) {                /* inf, or NaN (made quiet, payload kept) */
        u = sign | 0x7F800000u | (f << 13) | (f ? 0x00400000u : 0u);
    } else if (e != 0) {             /* normal: rebias the exponent */
        u = sign | ((e - 15u + 127u) << 23) | (f << 13);
    } else if (f == 0) {             /* signed zero */
        u = sign;
    } else {                         /* subnormal: f * 2^-24, exact in binary32 */
        float v = (float)f * 5.9604644775390625e-8f; /* 2^-24 */
        memcpy(&u, &v, sizeof u);
        u |= sign;
    }
    float out;
    memcpy(&out, &u, sizeof out);
    return out;
}

/* binary32 -> binary16, round to nearest, ties to even.
 * Normal range (|x| >= 2^-14): drop the low 13 fraction bits with the same
 * bias-and-truncate rule as the BF16 rounding, then move the exponent from
 * bias 127 to bias 15 (a carry out of the fraction correctly bumps the
 * exponent).  |x| >= 65520 is at or beyond the halfway point between the
 * largest binary16 value 65504 (odd significand) and 2^16, so it becomes
 * infinity.  Below 2^-14 the result is a multiple k of 2^-24: k is |x| / 2^-24
 * rounded to nearest even, computed on the integer significand. */
uint16_t orc_f32_to_f16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7FFFFFFFu;
    if (a > 0x7F800000u)
        return (uint16_t)(sign | 0x7E00u);
    if (a >= 0x477FF000u)            /* 65520 and above, infinity included */
        return (uint16_t)(sign | 0x7C00u);
    if (a >= 0x38800000u) {          /* 2^-14 and above: normal binary16 */
        uint32_t r = a + 0x0FFFu + ((a >> 13) & 1u);
        return (uint16_t)(sign | ((r >> 13) - (112u << 10)));
    }
    if (a < 0x00800000u)             /* binary32 subnormal or zero: below 2^-126 */
        return sign;
    uint32_t sig = (a & 0x007FFFFFu) | 0x00800000u;   /* 24-bit significand */
    int e = (int)(a >> 23) - 127;                      /* |x| = sig * 2^(e-23) */
    int sh = -(e + 1);                                 /* k = sig * 2^(e+1) = sig >> sh */
    if (sh >= 25)
        return sign;                 /* k < 1/2: below half of 2^-24, rounds to 0 */
    uint32_t q = sig >> sh;
    uint32_t rem = sig & ((1u << sh) - 1u);
    uint32_t half = 1u << (sh - 1);
    if (rem > half || (rem == half && (q & 1u)))
        ++q;
    return (uint16_t)(sign | q);     /* q = 1024 is the smallest normal, 0x0400 */
}

int orc_f32_to_f16_rne_array(const float *in, uint16_t *out, size_t n)
{
    if (n > 0 && (in == NULL || out == NULL))
        return -1;
    for (size_t i = 0; i < n; ++i)
        out[i] = orc_f32_to_f16_rne(in[i]);
    return 0;
}

/* Element i of input q, widened to binary32 (exact for every type). */
static float load_as_f32(const void *const *in, int q, size_t i, int dtype)
{
    if (dtype == ORC_F32)
        return ((const float *)in[q])[i];
    uint16_t h = ((const uint16_t *)in[q])[i];
    return dtype == ORC_F16 ? orc_f16_to_f32(h) : orc_bf16_to_f32(h);
}

static void store_from_f32(void *const *out, int r, size_t i, float v, int dtype)
{
    if (dtype == ORC_F32)
        ((float *)out[r])[i] = v;
    else if (dtype == ORC_F16)
        ((uint16_t *)out[r])[i] = orc_f32_to_f16_rne(v);
    else
        ((uint16_t *)out[r])[i] = orc_f32_to_bf16_rne(v);
}

/* The tree fold over x[lo..hi): split at the largest power of two below the
 * count, fold each side, add left + right. */
static float fold_tree(const float *x, int lo, int hi)
{
    int n = hi - lo;
    if (n == 1)
        return x[lo];
    int m = 1;
    while (m * 2 < n)
        m *= 2;
    float left = fold_tree(x, lo, lo + m);
    float right = fold_tree(x, lo + m, hi);
    return left + right;
}

static float fold_element(const void *const *in, int P, size_t i, int dtype, int order)
{
    float x[64] = {0.0f};
    for (int q = 0; q < P; ++q)
        x[q] = load_as_f32(in, q, i, dtype);
    if (order == ORC_ORDER_TREE)
        return fold_tree(x, 0, P);
    float acc = x[0];
    for (int q = 1; q < P; ++q)
        acc = acc + x[q];
    return acc;
}

static int check_args(const void *const *in, void *const *out, int P, size_t n, int dtype,
                      int order)
{
    if (P < 1 || P > 64 || dtype < ORC_BF16 || dtype > ORC_F32 ||
        (order != ORC_ORDER_LINEAR && order != ORC_ORDER_TREE))
        return -1;
    if (n == 0)
        return 0;
    if (in == NULL || out == NULL)
        return -1;
    for (int r = 0; r < P; ++r)
        if (in[r] == NULL || out[r] == NULL)
            return -1;
    return 0;
}

int orc_all_reduce(const void *const *in, void *const *out, int P, size_t count, int dtype,
                   int order)
{
    if (check_args(in, out, P, count, dtype, order) != 0)
        return -1;
    for (size_t i = 0; i < count; ++i) {
        float y = fold_element(in, P, i, dtype, order);
        for (int r = 0; r < P; ++r)
            store_from_f32(out, r, i, y, dtype);
    }
    return 0;
}

int orc_reduce_scatter(const void *const *in, void *const *out, int P, size_t C, int dtype,
                       int order)
{
    if (check_args(in, out, P, C, dtype, order) != 0)
        return -1;
    for (int r = 0; r < P; ++r)
        for (size_t j = 0; j < C; ++j)
            store_from_f32(out, r, j, fold_element(in, P, (size_t)r * C + j, dtype, order), dtype);
    return 0;
}

int orc_subnormals_preserved(void)
{
    /* 2^-140 is a binary32 subnormal; with FTZ/DAZ either the operand or
     * the result would read as zero. */
    volatile float tiny = 7.174648137343064e-43f; /* 2^-140 */
    volatile float one = 1.0f;
    volatile float prod = tiny * one;
    volatile float sum = tiny + tiny;
    return (prod != 0.0f && sum != 0.0f && sum == 2.0f * tiny) ? 1 : 0;
}
