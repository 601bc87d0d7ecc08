/*
 * dc_oracle.h -- plain, slow CPU oracle for the deterministic collective's
 * data-parallel core (rank-ordered all-gather, fixed-order BF16 reductions).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  The CUDA library never
 * includes, links or calls it, and this file shares nothing with it.
 *
 * Page followed (by title):
 *   [PR491]  "perf(cuda): vectorize the deterministic all-gather copy and
 *            right-size its single-block path" (RL-Kernel pull request 491).
 *
 * Every routine returns 0 on success and a negative value on a bad argument.
 */
#ifndef DC_ORACLE_H
#define DC_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* All-gather: out = in_0 || in_1 || ... || in_{P-1}, B bytes each.
 * [PR491] section "What", copy_rank_ordered bullet: a pure rank-ordered copy
 * whose result is byte-identical to the concatenation in rank order. */
int orc_all_gather(const uint8_t *const *peers, int P, size_t B, uint8_t *out);

/* all_gather_many: T independent all-gathers; peers is tensor-major
 * (peers[t*P + r]), bytes[t] is tensor t's per-rank size, outs[t] its output.
 * [PR491] "Results" names all_gather_many beside all_gather; the author's
 * reply describes it as several gathers with no packing, so each tensor gets
 * its own rank-ordered output. */
int orc_all_gather_many(const uint8_t *const *peers, const size_t *bytes,
                        uint8_t *const *outs, int T, int P);

/* BF16 bit pattern -> binary32 (exact: the 16 bits become the top half). */
float orc_bf16_to_f32(uint16_t h);

/* binary32 -> BF16, round to nearest, ties to even, one rounding.  NaN maps
 * to the quiet NaN 0x7FC0 with the input's sign. */
uint16_t orc_f32_to_bf16_rne(float f);

/* orc_f32_to_bf16_rne applied to n values (for checking the rounding on
 * many inputs at once). */
int orc_f32_to_bf16_rne_array(const float *in, uint16_t *out, size_t n);

/* all_reduce: for every element i,
 *   acc = f32(in_0[i]); acc = acc + f32(in_q[i]) for q = 1..P-1 (binary32,
 *   round to nearest even, this order); y = rne_bf16(acc); out_r[i] = y for
 *   every r = 0..P-1.
 * The fold reads every in_q[i] before writing any out_r[i], so out_r may be
 * the same buffer as an input.  [PR491] "What" and "Not in this PR" name
 * the deterministic all_reduce but never print its arithmetic; this is the
 * plainest reading of "deterministic": fixed rank order, binary32
 * accumulation, one round to nearest even at the end. */
int orc_all_reduce_bf16(const uint16_t *const *in, uint16_t *const *out,
                        int P, size_t count);

/* reduce_scatter: each input holds P*C elements (input = world x output);
 * out_r[j] = rne_bf16(fold over q = 0..P-1 of f32(in_q[r*C + j])). */
int orc_reduce_scatter_bf16(const uint16_t *const *in, uint16_t *const *out,
                            int P, size_t C);

/* ------------------------------------------------------------------------
 * Other element types and summation orders.
 *
 * The element type sets how a value is widened to binary32 (exactly) and how
 * the binary32 total is rounded back (round to nearest, ties to even; binary32
 * totals are stored as they are).  The order sets the shape of the fold over
 * the P widened values of one element:
 *   ORC_ORDER_LINEAR: ((x0 + x1) + x2) + ... + x_{P-1};
 *   ORC_ORDER_TREE:   fold(x[lo..hi)) = x[lo] for one value, otherwise
 *                     fold(x[lo..lo+m)) + fold(x[lo+m..hi)) with m the largest
 *                     power of two below hi - lo (pairs of neighbouring ranks,
 *                     then pairs of pairs, the last odd group added last).
 * Every add is one binary32 add, round to nearest even.  Page:
 * [PR491], author's replies: the backend is named "cuda_ipc_fixed_tree" (a
 * fixed tree is named; its shape is not given, and the one above is the
 * reading used). */
enum { ORC_BF16 = 0, ORC_F16 = 1, ORC_F32 = 2 };
enum { ORC_ORDER_LINEAR = 0, ORC_ORDER_TREE = 1 };

/* IEEE binary16 bit pattern -> binary32, exact. */
float orc_f16_to_f32(uint16_t h);
/* binary32 -> IEEE binary16, round to nearest, ties to even; NaN -> quiet NaN
 * (0x7E00) with the input's sign. */
uint16_t orc_f32_to_f16_rne(float f);
int orc_f32_to_f16_rne_array(const float *in, uint16_t *out, size_t n);

/* all_reduce / reduce_scatter of element type `dtype` (element size 2 for
 * BF16 and F16, 4 for F32) in summation order `order`; same layouts and
 * aliasing rules as the BF16 functions above. */
int orc_all_reduce(const void *const *in, void *const *out, int P, size_t count, int dtype,
                   int order);
int orc_reduce_scatter(const void *const *in, void *const *out, int P, size_t C, int dtype,
                       int order);

/* 1 if binary32 subnormals survive arithmetic on this host (no FTZ/DAZ),
 * 0 otherwise.  The oracle is only meaningful when this returns 1. */
int orc_subnormals_preserved(void);

#ifdef __cplusplus
}
#endif
#endif /* DC_ORACLE_H */
