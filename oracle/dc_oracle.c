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
