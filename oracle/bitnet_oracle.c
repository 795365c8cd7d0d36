/*
 * bitnet_oracle.c -- plain scalar reference of the W2A8 ternary matmul.
 *
 * TEST INFRASTRUCTURE ONLY: the oracle the CUDA library is checked against. Only the
 * test-suite, the smoke check and the benchmark's CPU-baseline leg may load it. It shares
 * no code with the CUDA library and is deliberately slow and obvious: no blocking, no
 * SIMD, no reordering beyond what the definitions state. Portable C11 (x86-64 and
 * aarch64 alike), built with -ffp-contract=off so that every fp32 operation below is
 * exactly one IEEE-754 rounding.
 *
 * Sources, cited by page title and section:
 *   [DeepDive]  "BitNet 딥다이브 -- 작은 숫자를 빠른 연산으로 바꾸는 추론 엔진"
 *               (fiv.co.kr/repos/BitNet-deep-dive.html)
 *   [Scalar]    "[분석/검증-3] BitNet.cpp ARM 커널 재작성 : 스칼라 폴백구현을 통한 최종 검증"
 *               (uno-kim.tistory.com/459)
 *   [Report]    "[기술 분석 보고서] ARM64 모바일 환경에서의 1.58-bit 양자화 모델 추론 붕괴
 *               원인 분석 및 C++ 커널 역공학을 통한 해결" (uno-kim.tistory.com/461)
 *   [bitnet.rs] "bitnet.rs -- BitNet b1.58 Inference Engine in Rust"
 *               (shadowgraph.io/ryancinsight/bitnetrs)
 *
 * Readings taken where the pages are silent or disagree (each is also listed with its
 * reason in the design notes):
 *   - activation scale is the multiply form s = 127 / max(max|x|, 1e-5) of [DeepDive]
 *     §4-5, not the divide form x / (max|x|/127) of [bitnet.rs] "Mathematical Foundation";
 *   - "round" is round-half-to-even; the clamp is [-127, 127] ([bitnet.rs] prints
 *     [-128, 127]; with the multiply form |x*s| never exceeds 127 after rounding, so the
 *     two clamps give the same result);
 *   - bf16 input is widened to fp32 exactly before any arithmetic;
 *   - dequantisation is out = (acc / s) * w_scale with w_scale = mean|W| (the stored
 *     abs-mean of [DeepDive] §6-2), i.e. acc * alpha_W * alpha_x with alpha_x = amax/127;
 *     the extra "/127" printed in [bitnet.rs] "Quantised Forward Pass" is read as a double
 *     count;
 *   - the unused code 3 unpacks as 3 - 1 = +2 (the c - 1 rule applied literally).
 */
#include "bitnet_oracle.h"

#include <fenv.h>
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define QK 128          /* weights per i2_s block  ([Scalar] §3, [DeepDive] §4-2) */
#define BLOCK_BYTES 32  /* bytes per i2_s block: 128 weights x 2 bits / 8 */

/* Ternary value -> stored 2-bit code: -1 -> 0, 0 -> 1, +1 -> 2 ([DeepDive] §1-1 table).
 * Values outside {-1,0,+1} follow the sign rule of quantize_i2_s in [DeepDive] §4-2
 * (positive -> 2, negative -> 0, zero -> 1). */
static unsigned code_of(int8_t v) {
    if (v > 0) return 2u;
    if (v < 0) return 0u;
    return 1u;
}

/* Position of weight k inside a packed row ([DeepDive] §4-2, [Scalar] §3, [Report] §3.1):
 * the 128 weights of block i are read as 4 groups of 32; weight 32*j + g of the block
 * lives in byte i*32 + g at bit offset 6 - 2*j (group 0 in bits 7:6, group 3 in 1:0). */
static int64_t byte_of(int64_t k) { return (k / QK) * BLOCK_BYTES + (k % QK) % 32; }
static unsigned shift_of(int64_t k) { return 6u - 2u * (unsigned)((k % QK) / 32); }

int64_t oracle_pack_i2s(const int8_t *w, uint8_t *wp, int64_t N, int64_t K) {
    if (!w || !wp || N < 0 || K <= 0 || K % QK != 0) return -1;
    const int64_t row_bytes = K / 4;  /* [Scalar] §3: a row is bx/4 bytes, bx = K */
    int64_t bad = 0;
    memset(wp, 0, (size_t)(N * row_bytes));
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            int8_t v = w[n * K + k];
            if (v < -1 || v > 1) ++bad;
            wp[n * row_bytes + byte_of(k)] |= (uint8_t)(code_of(v) << shift_of(k));
        }
    }
    return bad;
}

int oracle_unpack_i2s(const uint8_t *wp, int8_t *w, int64_t N, int64_t K) {
    if (!w || !wp || N < 0 || K <= 0 || K % QK != 0) return -1;
    const int64_t row_bytes = K / 4;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            unsigned code = (wp[n * row_bytes + byte_of(k)] >> shift_of(k)) & 3u;
            /* weight = code - 1 ([DeepDive] §8 bit-packing exercise) */
            w[n * K + k] = (int8_t)((int)code - 1);
        }
    }
    return 0;
}

float oracle_bf16_to_f32(uint16_t bits) {
    /* bf16 is the upper half of an IEEE-754 binary32 pattern. */
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* One token row of the absmax quantiser ([DeepDive] §4-5 BitLinearKernel.quant_input;
 * [bitnet.rs] "8-bit Activation Quantisation (AbsMax, per-token)"). */
static void quant_row(const float *x, int64_t K, int8_t *q, float *s_out, int32_t *sum_out) {
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) amax = fmaxf(amax, fabsf(x[k]));
    const float s = 127.0f / fmaxf(amax, 1e-5f);
    int64_t sum = 0;
    for (int64_t k = 0; k < K; ++k) {
        float p = x[k] * s;          /* one fp32 multiply, rounded once */
        float r = nearbyintf(p);     /* round half to even (default rounding mode) */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[k] = (int8_t)r;
        sum += (int64_t)q[k];
    }
    *s_out = s;
    *sum_out = (int32_t)sum;  /* |sum| <= 127*K fits for every K the API admits */
}

int oracle_quant_act_f32(const float *x, int64_t M, int64_t K,
                         int8_t *xq, float *s, int32_t *rowsum) {
    if (!x || !xq || !s || !rowsum || M < 0 || K <= 0) return -1;
    if (fegetround() != FE_TONEAREST) return -2;
    for (int64_t m = 0; m < M; ++m) quant_row(x + m * K, K, xq + m * K, s + m, rowsum + m);
    return 0;
}

int oracle_quant_act_bf16(const uint16_t *x, int64_t M, int64_t K,
                          int8_t *xq, float *s, int32_t *rowsum) {
    if (!x || !xq || !s || !rowsum || M < 0 || K <= 0) return -1;
    if (fegetround() != FE_TONEAREST) return -2;
    float *row = (float *)malloc((size_t)K * sizeof(float));
    if (!row) return -1;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t k = 0; k < K; ++k) row[k] = oracle_bf16_to_f32(x[m * K + k]);
        quant_row(row, K, xq + m * K, s + m, rowsum + m);
    }
    free(row);
    return 0;
}

/* ---- ternary matmul by definition, optionally split over output rows ---- */

typedef struct {
    const int8_t *xq;
    const float *s;
    const uint8_t *wp;
    float w_scale;
    float *out;
    int32_t *acc;
    int64_t M, N, K, n_begin, n_end;
    int status;
} matmul_job;

static void *matmul_rows(void *arg) {
    matmul_job *j = (matmul_job *)arg;
    int8_t *wrow = (int8_t *)malloc((size_t)j->K);
    if (!wrow) { j->status = -1; return NULL; }
    j->status = 0;
    for (int64_t n = j->n_begin; n < j->n_end; ++n) {
        /* step 1: unpack row n to ternary values */
        oracle_unpack_i2s(j->wp + n * (j->K / 4), wrow, 1, j->K);
        for (int64_t m = 0; m < j->M; ++m) {
            /* step 2: the ternary dot, in 64-bit so that an overflow is seen */
            const int8_t *y = j->xq + m * j->K;
            int64_t a = 0;
            for (int64_t k = 0; k < j->K; ++k) a += (int64_t)wrow[k] * (int64_t)y[k];
            if (a > INT32_MAX || a < INT32_MIN) { j->status = -3; a = 0; }
            if (j->acc) j->acc[m * j->N + n] = (int32_t)a;
            /* step 3: dequantise, out = (acc / s) * alpha_W, left to right in fp32 */
            if (j->out) j->out[m * j->N + n] = ((float)a / j->s[m]) * j->w_scale;
        }
    }
    free(wrow);
    return NULL;
}

int oracle_ternary_matmul(const int8_t *xq, const float *s, const uint8_t *wp,
                          float w_scale, float *out, int32_t *acc,
                          int64_t M, int64_t N, int64_t K, int nthreads) {
    if (!xq || !wp || M < 0 || N < 0 || K <= 0 || K % QK != 0) return -1;
    if (out && !s) return -1;
    if (nthreads < 1) nthreads = 1;
    if ((int64_t)nthreads > N) nthreads = (int)(N > 0 ? N : 1);
    matmul_job *jobs = (matmul_job *)calloc((size_t)nthreads, sizeof(matmul_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) { free(jobs); free(tid); return -1; }
    for (int t = 0; t < nthreads; ++t) {
        matmul_job *j = &jobs[t];
        j->xq = xq; j->s = s; j->wp = wp; j->w_scale = w_scale; j->out = out; j->acc = acc;
        j->M = M; j->N = N; j->K = K;
        j->n_begin = N * t / nthreads;
        j->n_end = N * (t + 1) / nthreads;
    }
    int status = 0;
    if (nthreads == 1) {
        matmul_rows(&jobs[0]);
        status = jobs[0].status;
    } else {
        int started = 0;
        for (int t = 0; t < nthreads; ++t) {
            if (pthread_create(&tid[t], NULL, matmul_rows, &jobs[t]) != 0) break;
            ++started;
        }
        for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
        if (started < nthreads) status = -1;
        for (int t = 0; t < started; ++t)
            if (jobs[t].status != 0 && status == 0) status = jobs[t].status;
    }
    free(jobs);
    free(tid);
    return status;
}

/* The raw code dot as the pages describe the packed kernels computing it ([Scalar] §3,
 * [Report] §3.2 and §4): walk the packed bytes block by block, take the four 2-bit
 * fields of each byte from the high pair down, and multiply each stored code (0, 1, 2)
 * with the activation it is paired with, without subtracting 1. */
int oracle_raw_code_dot(const int8_t *xq, const uint8_t *wp, int32_t *raw,
                        int64_t M, int64_t N, int64_t K) {
    if (!xq || !wp || !raw || M < 0 || N < 0 || K <= 0 || K % QK != 0) return -1;
    const int64_t row_bytes = K / 4;
    for (int64_t m = 0; m < M; ++m) {
        const int8_t *y = xq + m * K;
        for (int64_t n = 0; n < N; ++n) {
            const uint8_t *row = wp + n * row_bytes;
            int64_t sum = 0;
            for (int64_t blk = 0; blk < K / QK; ++blk) {
                for (int64_t g = 0; g < 32; ++g) {
                    unsigned byte = row[blk * BLOCK_BYTES + g];
                    for (unsigned j = 0; j < 4; ++j) {
                        unsigned code = (byte >> (6u - 2u * j)) & 3u;
                        sum += (int64_t)code * (int64_t)y[blk * QK + 32 * j + g];
                    }
                }
            }
            raw[m * N + n] = (int32_t)sum;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------------------
 * Weight ternarisation.
 *
 * AbsMean ([DeepDive] §6-2: abs_mean = max(mean(abs(w)), 1e-5), q = clip(round(w / abs_mean),
 * -1, 1), the stored scale is abs_mean; [bitnet.rs] "Ternary Weight Quantisation" gives the
 * same without the floor). The pages compute the mean with a float library reduction in an
 * unstated order. A code decided by w / scale must come out the same on every
 * implementation, so the scale must be bit-identical; the mean is therefore defined through
 * an exact integer sum (a reading):
 *   S    = sum over all weights of floor(|w| * 2^74), an exact unsigned integer (each term is
 *          |w| to 74 fractional bits; |w| must be below 2^12, and N*K at most 2^40, so that
 *          S fits in 128 bits);
 *   mean = (float)((double)S * 2^-74 / (N * K)): the conversion of S to double, the
 *          division and the conversion to float each round to nearest (the scaling by 2^-74
 *          is exact);
 *   scale = max(mean, 1e-5f).
 * No summation order enters: any order of an exact integer sum gives S. "round" is
 * round-half-to-even as in numpy (the page's example, w = [-0.6, -0.2, 0.2, 0.6], asks which
 * rule: with it the codes are [-1, 0, 0, 1]).
 *
 * Sign rule ([DeepDive] §4-2, quantize_i2_s on float weights that are already ternary): a
 * value with |w| < 1e-6 (the comparison taken in double, as the C++ expression promotes
 * it) is 0, any other value its sign; the scale kept is the largest |w|.
 * --------------------------------------------------------------------------------------- */
static int quant_weight(const float *wf, const uint16_t *wb, int64_t N, int64_t K, int mode, int8_t *q,
                        float *scale) {
    if ((!wf && !wb) || !q || !scale || N < 1 || K < 1 || (mode != 0 && mode != 1)) return -1;
    if (fegetround() != FE_TONEAREST) return -2;
#define W_AT(i) (wf ? wf[(i)] : oracle_bf16_to_f32(wb[(i)]))
    float sc;
    if (mode == 0) {
        if ((double)N * (double)K > 1099511627776.0 /* 2^40 */) return -4;
        unsigned __int128 S = 0;
        for (int64_t i = 0; i < N * K; ++i) {
            const float a = fabsf(W_AT(i));
            if (!(a < 4096.0f)) return -4;                      /* |w| >= 2^12, or NaN */
            S += (unsigned __int128)(a * 0x1p74f);  /* a * 2^74 is exact; the conversion truncates */
        }
        const float mean = (float)((double)S * 0x1p-74 / ((double)N * (double)K));
        sc = fmaxf(mean, 1e-5f);
        for (int64_t i = 0; i < N * K; ++i) {
            float r = nearbyintf(W_AT(i) / sc);  /* one fp32 division, then round half to even */
            if (r > 1.0f) r = 1.0f;
            if (r < -1.0f) r = -1.0f;
            q[i] = (int8_t)r;
        }
    } else {
        sc = 0.0f;
        for (int64_t i = 0; i < N * K; ++i) {
            const float v = W_AT(i);
            sc = fmaxf(sc, fabsf(v));
            q[i] = ((double)fabsf(v) < 1e-6) ? 0 : (v > 0.0f ? 1 : -1);
        }
    }
#undef W_AT
    *scale = sc;
    return 0;
}

int oracle_quant_weight_f32(const float *w, int64_t N, int64_t K, int mode, int8_t *q, float *scale) {
    return w ? quant_weight(w, NULL, N, K, mode, q, scale) : -1;
}

int oracle_quant_weight_bf16(const uint16_t *w, int64_t N, int64_t K, int mode, int8_t *q, float *scale) {
    return w ? quant_weight(NULL, w, N, K, mode, q, scale) : -1;
}

/* ---------------------------------------------------------------------------------------
 * FFN inner activation ([bitnet.rs] "Forward Pass": the FFN applies squared-ReLU gating,
 * inner = ffn_sub_norm(sqrelu(gate(x)) * up(x)), and then out = down(inner)).
 *
 * The page prints the formula only. Readings:
 *   - sqrelu(g) = max(g, 0)^2: r = (g > 0 ? g : 0) (so NaN and -0 give +0), then r * r;
 *   - h = sqrelu(g) * u elementwise, in fp32: (r * r) * u, two roundings;
 *   - ffn_sub_norm is an RMSNorm (the norm the page's module list names) with a per-channel
 *     weight gamma and an epsilon eps, neither of which the page prints, so both are inputs:
 *     inner = (h * c) * gamma, c = 1 / sqrt(ss / F + eps), ss = sum of h^2, all in fp32, each
 *     operation one rounding (sqrtf and the divisions are correctly rounded);
 *   - the sum of squares is the plain sum over k = 0 .. F-1 in ascending order, taken in double
 *     (each h_k * h_k is exact in double, and F terms add at most F * 2^-53 relative error)
 *     and rounded once to fp32; that is the definition's value to within half an fp32 ulp.
 *     The page fixes no order; a parallel implementation may sum in any order, and its ss
 *     then differs from this one by its own rounding error only (the codes downstream are
 *     compared with that error in mind).
 * --------------------------------------------------------------------------------------- */
static void ffn_inner_row(const float *g, const float *u, const float *gamma, float eps, int64_t F,
                          float *inner) {
    double ss = 0.0;
    for (int64_t k = 0; k < F; ++k) {
        const float r = g[k] > 0.0f ? g[k] : 0.0f;
        const float h = (r * r) * u[k];
        inner[k] = h; /* h parked in the output until c is known */
        ss += (double)h * (double)h;
    }
    const float ssf = (float)ss;
    const float c = 1.0f / sqrtf(ssf / (float)F + eps);
    for (int64_t k = 0; k < F; ++k) inner[k] = (inner[k] * c) * gamma[k];
}

int oracle_ffn_inner(const float *gate, const float *up, const float *gamma, float eps, int64_t M, int64_t F,
                     float *inner) {
    if (!gate || !up || !gamma || !inner || M < 0 || F < 1 || F > (1 << 24) || !(eps >= 0.0f)) return -1;
    if (fegetround() != FE_TONEAREST) return -2;
    for (int64_t m = 0; m < M; ++m) ffn_inner_row(gate + m * F, up + m * F, gamma, eps, F, inner + m * F);
    return 0;
}
