/*
 * bitnet_oracle.h -- scalar reference of the W2A8 ternary matmul (test infrastructure).
 *
 * TEST INFRASTRUCTURE ONLY. This header and bitnet_oracle.c form the oracle that the
 * CUDA library is checked against. Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it. It shares no code, header, table or helper
 * with the CUDA library, and the CUDA library never calls it.
 *
 * Conventions (all arrays row-major, all sizes in elements):
 *   w   : N x K   int8, ternary weights in {-1, 0, +1}
 *   wp  : N x K/4 uint8, i2_s packed codes (QK = 128 weights per 32-byte block)
 *   x   : M x K   fp32, or bf16 given as its raw 16-bit patterns
 *   xq  : M x K   int8, per-token absmax-quantised activations
 *   s   : M       fp32, per-token activation scale s = 127 / max(max|x|, 1e-5)
 *   acc : M x N   int32, ternary dot sum_k w[n][k] * xq[m][k]
 *   out : M x N   fp32, (acc / s) * w_scale
 * K must be a positive multiple of 128 for every function that touches wp.
 */
#ifndef BITNET_ORACLE_H
#define BITNET_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Pack ternary int8 weights into i2_s bytes. Returns the number of entries that
 * were not in {-1,0,+1} (they are mapped by sign), or -1 on bad arguments. */
int64_t oracle_pack_i2s(const int8_t *w, uint8_t *wp, int64_t N, int64_t K);

/* Unpack i2_s bytes into int8 weights, w = code - 1 for every 2-bit field
 * (so the unused code 3 reads as +2). Returns 0, or -1 on bad arguments. */
int oracle_unpack_i2s(const uint8_t *wp, int8_t *w, int64_t N, int64_t K);

/* bf16 bit pattern -> fp32 value (exact). */
float oracle_bf16_to_f32(uint16_t bits);

/* Per-token absmax int8 activation quantisation. Returns 0, or -1 on bad
 * arguments, or -2 if the rounding mode is not round-to-nearest-even. */
int oracle_quant_act_f32(const float *x, int64_t M, int64_t K,
                         int8_t *xq, float *s, int32_t *rowsum);
int oracle_quant_act_bf16(const uint16_t *x, int64_t M, int64_t K,
                          int8_t *xq, float *s, int32_t *rowsum);

/* The ternary matmul by its plain definition: unpack, integer dot, scale.
 * acc and out may each be NULL. nthreads <= 1 runs on the calling thread.
 * Returns 0, -1 on bad arguments, -3 if an accumulator leaves int32. */
int oracle_ternary_matmul(const int8_t *xq, const float *s, const uint8_t *wp,
                          float w_scale, float *out, int32_t *acc,
                          int64_t M, int64_t N, int64_t K, int nthreads);

/* The pages' raw code dot: sum over k of code(n,k) * xq[m][k], with the codes
 * 0/1/2 multiplied as stored (no -1). Returns 0 or -1. */
int oracle_raw_code_dot(const int8_t *xq, const uint8_t *wp, int32_t *raw,
                        int64_t M, int64_t N, int64_t K);

/* Weight ternarisation (the step before packing). mode 0, AbsMean ([DeepDive] §6-2,
 * [bitnet.rs] "Ternary Weight Quantisation"): scale = max(mean|w|, 1e-5) with the mean
 * taken through the exact integer sum of floor(|w| * 2^74) described in bitnet_oracle.c,
 * q = clip(rne(w / scale), -1, 1) in fp32. mode 1, the sign rule of quantize_i2_s
 * ([DeepDive] §4-2): q = 0 where |w| < 1e-6, else sign(w); scale = max|w|. q is N x K int8;
 * *scale one float. Returns 0, or -1 on bad arguments, -2 if the rounding mode is not
 * round-to-nearest-even, -4 if AbsMean meets |w| >= 2^12 (or NaN) or N*K > 2^40. */
int oracle_quant_weight_f32(const float *w, int64_t N, int64_t K, int mode, int8_t *q, float *scale);
int oracle_quant_weight_bf16(const uint16_t *w, int64_t N, int64_t K, int mode, int8_t *q, float *scale);

/* FFN inner activation ([bitnet.rs] "Forward Pass"): per row m of gate and up (M x F fp32),
 * h = max(g, 0)^2 * u, inner = (h * c) * gamma with c = 1 / sqrt(sum(h^2) / F + eps), the sum
 * of squares the plain ascending sum taken in double and rounded once to fp32. gamma is F fp32 (shared
 * by all rows), eps >= 0. inner is M x F fp32. Returns 0, -1 on bad arguments, -2 if the
 * rounding mode is not round-to-nearest-even. */
int oracle_ffn_inner(const float *gate, const float *up, const float *gamma, float eps, int64_t M, int64_t F,
                     float *inner);

#ifdef __cplusplus
}
#endif

#endif /* BITNET_ORACLE_H */
