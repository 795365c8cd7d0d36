/*
 * bitnet.h -- C ABI of the GB300 (sm_103a) W2A8 ternary matmul library (libbitnet_gb300.so).
 *
 * The library computes the BitNet b1.58 linear layer with ternary weights stored as 2-bit
 * codes in the i2_s layout and per-token absmax int8 activations:
 *
 *   out[m][n] = ( sum_k (code[n][k] - 1) * xq[m][k] ) / s[m] * w_scale
 *
 * where code in {0,1,2} encodes w in {-1,0,+1}. The integer sum is formed as the raw code
 * dot sum_k code*xq minus the activation row sum sum_k xq (an identity), which is how the
 * packed CPU kernels of bitnet.cpp compute it.
 *
 * Sources (by page title and section):
 *   [DeepDive]  "BitNet 딥다이브 -- 작은 숫자를 빠른 연산으로 바꾸는 추론 엔진", §1-1 (code map),
 *               §4-2 (i2_s packing, quantize_i2_s), §4-5 (GPU path, per-token quant_input)
 *   [Scalar]    "[분석/검증-3] BitNet.cpp ARM 커널 재작성 : 스칼라 폴백구현을 통한 최종 검증",
 *               §3 (scalar i2_s x int8 dot, row stride, 4x32 interleave)
 *   [Report]    "[기술 분석 보고서] ARM64 모바일 환경에서의 1.58-bit 양자화 모델 추론 붕괴 원인 분석
 *               및 C++ 커널 역공학을 통한 해결", §3.1 (interleave), §3.2 (codes multiplied as stored)
 *   [bitnet.rs] "bitnet.rs -- BitNet b1.58 Inference Engine in Rust", "Mathematical Foundation"
 *               (AbsMean weight scale, AbsMax activation quantisation, quantised forward pass)
 *
 * Common rules for every entry point:
 *   - All array pointers are DEVICE pointers owned by the caller; the library keeps no
 *     pointer after the call returns. No call allocates device memory, with two stated
 *     exceptions: bitnet_sweep_plan_create allocates the plan's device table (cudaMalloc,
 *     freed by bitnet_sweep_plan_destroy), and the library's device image holds a fixed
 *     64 MiB scratch array (used only by bitnet_i2s_matmul_noalloc) that every GPU which
 *     loads the library keeps until the process exits, used or not. Budget for both.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream). Results are valid once the stream has reached the call.
 *   - Arguments are validated on the host before anything is launched; an invalid call
 *     launches nothing and returns a negative status. No exception crosses the ABI.
 *   - Layouts are dense row-major. K (the reduction length) must be a positive multiple of
 *     128 (one i2_s block) wherever packed weights are involved.
 *   - Each call runs on the device that is current on the calling thread; that device must
 *     be an sm_103 GPU (GB300), else BITNET_EUNSUPPORTED.
 *   - Inputs must be finite; NaN/Inf activations are outside the contract.
 */
#ifndef BITNET_GB300_H
#define BITNET_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define BITNET_API __attribute__((visibility("default")))
#else
#define BITNET_API
#endif

/* ---- status codes ---- */
#define BITNET_OK 0
#define BITNET_EINVAL (-1)        /* null pointer, size <= 0 or out of range, K % 128 != 0, bad enum */
#define BITNET_EALIGN (-2)        /* a pointer is not aligned as the entry point requires        */
#define BITNET_ECUDA (-3)         /* a CUDA runtime call or kernel launch failed                  */
#define BITNET_EUNSUPPORTED (-4)  /* current device is not sm_103, or no device                 */
#define BITNET_ETIMEOUT (-5)      /* a device-side bounded wait gave up (reported by the next call
                                     to bitnet_last_device_error); the result is not valid      */
#define BITNET_ERANGE (-6)        /* an input value outside the operation's range, found on the
                                     device (reported by bitnet_last_device_error)              */

/* ---- activation dtypes (bitnet_quant_act) ---- */
#define BITNET_F32 0
#define BITNET_BF16 1

/* ---- weight ternarisation modes (bitnet_quant_weight) ---- */
#define BITNET_QW_ABSMEAN 0 /* scale = max(mean|w|, 1e-5), q = clip(rne(w / scale), -1, 1) */
#define BITNET_QW_SIGN 1    /* q = 0 where |w| < 1e-6, else sign(w); scale = max|w|       */

/* ---- matmul kernel selection (bitnet_i2s_matmul_algo) ---- */
#define BITNET_ALGO_AUTO 0   /* GEMV for a few rows (M < 5, or M < 3 when K > 10240),
                                the few-token kernel up to M = 64, the CTA-pair
                                prompt-length kernel beyond; K <= 32768                  */
#define BITNET_ALGO_GEMV 1   /* force the dp4a decode GEMV (any M)                   */
#define BITNET_ALGO_GEMM 2   /* force the tcgen05 tensor-core GEMM (any M)           */
#define BITNET_ALGO_SMALLM 3 /* force the few-token tensor-core kernel (any M)       */
#define BITNET_ALGO_PREFILL 4 /* force the prompt-length tensor-core kernel (any M)  */
#define BITNET_ALGO_PREFILL_PAIR 5 /* force its CTA-pair variant (any M)             */

/* Library ABI version (major*100 + minor). */
BITNET_API int bitnet_version(void);

/* Human-readable text for a status code. Never NULL; static storage. */
BITNET_API const char *bitnet_strerror(int status);

/*
 * bitnet_pack_i2s -- ternary int8 weights -> i2_s packed bytes.
 *   [DeepDive] §4-2 (quantize_i2_s, x86 ACT_PARALLEL branch) and §1-1 (code map).
 *
 *   w             : N x K int8, values in {-1, 0, +1}                      (device, read)
 *   wp            : N x K/4 uint8                                           (device, written)
 *                   Byte (n, 32*i + g) holds, at bit pairs 7:6, 5:4, 3:2, 1:0, the codes of
 *                   weights (n, 128*i + g), (n, 128*i + 32 + g), (n, 128*i + 64 + g),
 *                   (n, 128*i + 96 + g); code = w + 1.
 *   N, K          : N >= 1, K >= 128, K % 128 == 0, K <= 65536
 *   invalid_count : optional (may be NULL) device int32; set to the number of entries of w
 *                   outside {-1,0,+1}. Such entries are packed by sign (>0 -> 2, <0 -> 0).
 *   w and wp must be 16-byte aligned (BITNET_EALIGN otherwise).
 */
BITNET_API int bitnet_pack_i2s(const int8_t *w, uint8_t *wp, int64_t N, int64_t K,
                               int32_t *invalid_count, void *stream);

/*
 * bitnet_quant_act -- per-token absmax int8 quantisation of activation rows.
 *   [DeepDive] §4-5 (BitLinearKernel.quant_input: s = 127 / max(max|x|, 1e-5), round,
 *   clamp, int8); [bitnet.rs] "8-bit Activation Quantisation (AbsMax, per-token)".
 *
 *   x          : M x K, fp32 (dtype BITNET_F32) or bf16 (BITNET_BF16)       (device, read)
 *                bf16 is widened to fp32 exactly before any arithmetic.
 *   xq         : M x K int8, q = clamp(rne(x * s), -127, 127)              (device, written)
 *   act_scale  : M fp32, s = 127 / max(max_k |x|, 1e-5) (IEEE fp32 divide) (device, written)
 *   rowsum     : M int32, sum_k xq[m][k]                                    (device, written)
 *   M >= 1, K >= 128, K % 128 == 0, K <= 65536. x and xq must be 16-byte aligned.
 */
BITNET_API int bitnet_quant_act(const void *x, int dtype, int64_t M, int64_t K, int8_t *xq,
                                float *act_scale, int32_t *rowsum, void *stream);

/*
 * bitnet_i2s_matmul -- W2A8 ternary matmul with the -sum(y) correction and the scales.
 *   [Scalar] §3 and [Report] §3.2/§4 (raw code dot over the 4x32-interleaved bytes, codes
 *   multiplied as stored); the zero-point correction acc = raw - rowsum is exact; the
 *   dequantisation follows [bitnet.rs] "Quantised Forward Pass" read as
 *   out = acc * alpha_W * alpha_x with alpha_x = 1/s.
 *
 *   xq        : M x K int8 activations                                      (device, read)
 *   act_scale : M fp32 activation scales s                                   (device, read)
 *   rowsum    : M int32, sum_k xq[m][k] (as written by bitnet_quant_act)     (device, read)
 *   wp        : N x K/4 uint8, i2_s packed weights                           (device, read)
 *   w_scale   : per-tensor weight scale alpha_W = mean|W| of the source weights
 *   out       : M x N fp32, out[m][n] = ((float)acc[m][n] / s[m]) * w_scale  (device, written)
 *   acc_out   : optional (may be NULL) M x N int32, acc[m][n] = sum_k (code-1)*xq (written)
 *   M, N >= 1; M, N <= 2^31 - 1; K >= 128, K % 128 == 0, K <= 65536. The tensor-core kernels
 *   take K <= 32768 (BITNET_EINVAL if forced beyond); auto dispatch then uses the GEMV.
 *   xq and wp must be 16-byte aligned; out and acc_out 4-byte aligned.
 *   The 2-bit field value 3 never comes out of bitnet_pack_i2s; if present it is used
 *   arithmetically (3 - 1 = +2), the same rule as the unpacking of [DeepDive] §8.
 *   Kernel choice: for a few rows (M < 5, or M < 3 when K > 10240) a dp4a GEMV streams the
 *   packed weights. From there a few-token tcgen05 kernel decodes each weight once, as the
 *   e4m3 value code + 8, for up to 64 token rows, whose int8 values enter as three exact e4m3
 *   base-8 digits (weights as the MMA's M, K split over a thread-block cluster); more rows go
 *   in chunks of 64 when forced. Beyond 64 rows the prompt-length kernel takes over: TMA-staged
 *   packed weights and int8 tokens, expanded in the kernel to exact fp16 (the codes into tensor
 *   memory, the tokens into shared memory), with the 2-SM MMA (tcgen05.mma.cta_group::2): 256
 *   weight rows x 128 tokens (up to 128 rows) or x 256 tokens per pair of CTAs, K split over a
 *   cluster when the tiles are few. A one-CTA variant (256 weight rows x 128 tokens per CTA)
 *   is available when forced (BITNET_ALGO_PREFILL). Neither uses a workspace. A tcgen05 tile
 *   GEMM that expands the codes to fp16 in shared memory is available when forced
 *   (BITNET_ALGO_GEMM). The tensor-core paths are exact: every partial sum is an integer below
 *   2^24 accumulated in fp32. All give bit-identical results.
 */
BITNET_API int bitnet_i2s_matmul(const int8_t *xq, const float *act_scale, const int32_t *rowsum,
                                 const uint8_t *wp, float w_scale, float *out, int32_t *acc_out,
                                 int64_t M, int64_t N, int64_t K, void *stream);

/*
 * bitnet_i2s_matmul_ws -- the same result as bitnet_i2s_matmul, computed the prefill way with a
 * caller-provided device workspace: the codes are expanded once to fp16 (N x K) and the int8
 * activations converted once to fp16 (M x K) -- both exact -- and a TMA-fed tcgen05 GEMM runs
 * on them (fp32 accumulation of integers below 2^24, hence exact). "BitNet 딥다이브" §4-5: the
 * reference GPU path runs prefill with fp16 weights.
 *   workspace       : device memory, 256-byte aligned, at least
 *                     bitnet_i2s_matmul_workspace_size(M, N, K) bytes; contents overwritten.
 *   workspace_bytes : its size (BITNET_EINVAL if too small).
 *   Other arguments as bitnet_i2s_matmul; K <= 32768. Three launches on `stream`.
 */
BITNET_API int64_t bitnet_i2s_matmul_workspace_size(int64_t M, int64_t N, int64_t K);
BITNET_API int bitnet_i2s_matmul_ws(const int8_t *xq, const float *act_scale, const int32_t *rowsum,
                                    const uint8_t *wp, float w_scale, float *out, int32_t *acc_out,
                                    int64_t M, int64_t N, int64_t K, void *workspace,
                                    int64_t workspace_bytes, void *stream);

/*
 * bitnet_i2s_matmul_noalloc -- bitnet_i2s_matmul_ws for callers that cannot allocate device
 * memory (for example a plugin whose host framework owns all device memory and forbids
 * cudaMalloc, or a loop where a cudaMalloc/cudaFree would synchronise the device). No page
 * describes such an entry point; it exists for those callers only.
 *   It uses no caller workspace and allocates nothing: the workspace is a fixed 64 MiB
 *   scratch array in the library's device image, which every GPU that loads the library
 *   holds until the process exits. Problems whose workspace
 *   (bitnet_i2s_matmul_workspace_size) exceeds 64 MiB are refused with BITNET_EINVAL before
 *   any GPU work.
 *   The first call on each device (with that device current) looks up the array's device
 *   address and keeps it for the life of the process; make that first call before any stream
 *   capture. A cudaDeviceReset of that device after its first call is not supported: the kept
 *   address would then be stale.
 *   All calls share the array: calls that overlap on the GPU race on it. Each call overwrites
 *   what it uses, so nothing has to be cleared between calls.
 *   Other arguments, results and errors as bitnet_i2s_matmul_ws.
 */
BITNET_API int bitnet_i2s_matmul_noalloc(const int8_t *xq, const float *act_scale,
                                         const int32_t *rowsum, const uint8_t *wp, float w_scale,
                                         float *out, int32_t *acc_out, int64_t M, int64_t N,
                                         int64_t K, void *stream);

/* Same as bitnet_i2s_matmul with an explicit kernel choice (BITNET_ALGO_*). */
BITNET_API int bitnet_i2s_matmul_algo(const int8_t *xq, const float *act_scale,
                                      const int32_t *rowsum, const uint8_t *wp, float w_scale,
                                      float *out, int32_t *acc_out, int64_t M, int64_t N,
                                      int64_t K, int algo, void *stream);

/*
 * bitnet_quant_weight -- ternarise full-precision weights and pack them into i2_s, the step
 * before the matmul path (three kernels on `stream`, no workspace).
 *   BITNET_QW_ABSMEAN: "BitNet 딥다이브" §6-2 (abs_mean = max(mean(abs(w)), 1e-5), codes
 *   clip(round(w / abs_mean), -1, 1), stored scale abs_mean) and "bitnet.rs" "Ternary Weight
 *   Quantisation". "round" is round-half-to-even of the fp32 quotient. The mean is defined
 *   through an exact integer so that the scale, and every code it decides, is the same bit for
 *   bit whatever the summation order: S = sum over all N*K weights of floor(|w| * 2^74) (128-bit,
 *   exact), mean = fp32(fp64(S) * 2^-74 / (N*K)), each conversion and the division rounding to
 *   nearest. This needs |w| < 2^12: a weight at or above it, infinite or NaN sets
 *   BITNET_ERANGE in the device error word (read by bitnet_last_device_error); w_scale is then
 *   NaN and wp is unspecified.
 *   BITNET_QW_SIGN: quantize_i2_s of "BitNet 딥다이브" §4-2, for weights that are already
 *   ternary: |w| < 1e-6 (compared in double) codes as 0, other values by sign (NaN as -1);
 *   scale max|w| (NaN ignored).
 *
 *   w       : N x K fp32 or bf16 (dtype BITNET_F32 / BITNET_BF16), row-major (device, read)
 *   wp      : N x K/4 uint8, i2_s packed codes (device, written; also used as scratch before
 *             the codes are written). Must not overlap w.
 *   w_scale : 1 fp32, the scale above (device, written)
 *   N >= 1; K >= 128, K % 128 == 0, K <= 65536; N * K <= 2^40.
 *   w and wp 16-byte aligned, w_scale 4-byte aligned. Host-side errors as bitnet_pack_i2s.
 */
BITNET_API int bitnet_quant_weight(const void *w, int dtype, int mode, int64_t N, int64_t K,
                                   uint8_t *wp, float *w_scale, void *stream);

/*
 * bitnet_w2a8_linear_group -- per-token activation quantisation fused with the ternary
 * matmuls of up to 8 projections that consume the same activation rows (e.g. q/k/v, or
 * gate/up). Computes, for l = 0..count-1, exactly what bitnet_quant_act followed by
 * bitnet_i2s_matmul(xq, s, rowsum, wp[l], w_scale[l], out[l], acc_out[l], M, N[l], K) gives.
 *   [DeepDive] §4-5 (quant_input then the int8 x int2 linear), §4-3 (one decoded activation
 *   set reused for several weight columns); the arithmetic is that of bitnet_quant_act and
 *   bitnet_i2s_matmul.
 *
 *   x          : M x K fp32 (BITNET_F32) or bf16 (BITNET_BF16)                  (device, read)
 *   count      : 1..8 projections
 *   wp, w_scale, N, out, acc_out : HOST arrays of length count (acc_out may be NULL, and so
 *                may any entry); wp[l] N[l] x K/4 packed (device), out[l] M x N[l] fp32
 *                (device, written), acc_out[l] M x N[l] int32 (device, written)
 *   xq, act_scale, rowsum : M x K int8, M fp32, M int32 (device, written). With M == 1 and
 *                K <= 10240 the whole call is one kernel launch and these three may be NULL
 *                (each non-NULL one is written); otherwise they are required workspace and
 *                the call is one quantisation launch plus one matmul launch per projection.
 *   Same size, alignment and dtype rules as bitnet_quant_act and bitnet_i2s_matmul.
 */
BITNET_API int bitnet_w2a8_linear_group(const void *x, int dtype, int64_t M, int64_t K, int count,
                                        const uint8_t *const *wp, const float *w_scale,
                                        const int64_t *N, float *const *out, int32_t *const *acc_out,
                                        int8_t *xq, float *act_scale, int32_t *rowsum, void *stream);

/*
 * bitnet_w2a8_linear_group_ex -- bitnet_w2a8_linear_group plus an L2 prefetch hint: up to 8
 * device byte ranges (16-byte aligned starts; a partial last 16 bytes is skipped) that the
 * single-launch kernel pulls into L2 while it runs -- typically the packed weights of the
 * next group, so that the next call finds them on chip. The hint never changes a result and
 * is ignored on the two-launch path. prefetch_ptr / prefetch_bytes are HOST arrays.
 * The single-launch kernel also allows the following kernel in the stream to start early
 * (programmatic dependent launch); it reads x and writes its outputs only after the
 * preceding kernel in the stream has completed.
 */
BITNET_API int bitnet_w2a8_linear_group_ex(const void *x, int dtype, int64_t M, int64_t K, int count,
                                           const uint8_t *const *wp, const float *w_scale,
                                           const int64_t *N, float *const *out, int32_t *const *acc_out,
                                           int8_t *xq, float *act_scale, int32_t *rowsum,
                                           int prefetch_count, const void *const *prefetch_ptr,
                                           const int64_t *prefetch_bytes, void *stream);

/* bitnet_w2a8_linear -- bitnet_w2a8_linear_group with a single projection. */
BITNET_API int bitnet_w2a8_linear(const void *x, int dtype, int64_t M, int64_t K, const uint8_t *wp,
                                  float w_scale, int64_t N, float *out, int32_t *acc_out, int8_t *xq,
                                  float *act_scale, int32_t *rowsum, void *stream);

/*
 * bitnet_ffn_act_quant -- the FFN's inner activation fused with its per-token quantisation
 * ("bitnet.rs" "Forward Pass": inner = ffn_sub_norm(sqrelu(gate(x)) * up(x)), out =
 * down(inner); the quantisation is that of [DeepDive] §4-5). Per row m, in fp32 with one
 * rounding per operation:
 *   h = max(g, 0)^2 * u  (as (r * r) * u, r = g > 0 ? g : 0)
 *   inner = (h * c) * gamma,  c = 1 / sqrt(ss / F + eps)        (RMSNorm, weight gamma)
 *   xq, act_scale, rowsum = what bitnet_quant_act gives for the fp32 row inner.
 * The page fixes no order for ss, the sum of h^2. This library adds it in fp32 in a fixed
 * order, so repeated calls give the same bits: 256 partial sums, partial p accumulating by
 * fused multiply-add, in ascending k, the h_k with floor(k / 4) mod 256 == p; each run of 32
 * partials combined by the pairwise tree that adds partial p + d into p for d = 16, 8, 4, 2, 1;
 * the eight run sums combined as ((R0 + R1) + (R2 + R3)) + ((R4 + R5) + (R6 + R7)). That is
 * at most F/256 + 8 roundings per term away from the exact sum (8.1e-6 relative at
 * F = 32768), so inner is within 1e-5 relative of the exactly summed definition, and a code
 * can differ from the exactly summed one only next to a rounding boundary.
 *
 *   gate, up  : M x F fp32 (device, read), 16-byte aligned
 *   gamma     : F fp32 (device, read), 16-byte aligned, shared by all rows
 *   eps       : finite, > 0
 *   xq        : M x F int8 (device, written), 16-byte aligned
 *   act_scale, rowsum : M fp32 / M int32 (device, written)
 *   inner_out : M x F fp32 (device, written) or NULL, 16-byte aligned
 *   M >= 1; F >= 128, F % 128 == 0, F <= 32768. One kernel launch on `stream`.
 *   Values of h whose square overflows fp32 are outside the operation.
 */
BITNET_API int bitnet_ffn_act_quant(const float *gate, const float *up, const float *gamma, float eps,
                                    int64_t M, int64_t F, int8_t *xq, float *act_scale, int32_t *rowsum,
                                    float *inner_out, void *stream);

/*
 * bitnet_w2a8_ffn -- the FFN block of one decoder layer on packed ternary weights
 * ("bitnet.rs" "Forward Pass", FFN with squared-ReLU gating and sub-norm):
 *   gate = W2A8(x; wp_gate, a_gate), up = W2A8(x; wp_up, a_up)   (F outputs each, over K)
 *   xq', s', rowsum' = bitnet_ffn_act_quant(gate, up, gamma, eps)
 *   out = W2A8(xq', s', rowsum'; wp_down, a_down)                  (K outputs, over F)
 * where W2A8 is bitnet_quant_act followed by bitnet_i2s_matmul. The results are exactly those
 * of that sequence of calls.
 *
 *   x        : M x K fp32 or bf16 (dtype) (device, read), 16-byte aligned
 *   wp_gate, wp_up : F x K/4 packed (device), wp_down : K x F/4 packed (device), 16-byte aligned
 *   a_gate, a_up, a_down : the weight scales
 *   gamma, eps : as bitnet_ffn_act_quant
 *   gate_out, up_out : M x F fp32 (device, written), 16-byte aligned
 *   out      : M x K fp32 (device, written)
 *   xq       : M * max(K, F) bytes of int8 workspace (device), act_scale, rowsum : M each
 *              (device). On return the first M * F bytes of xq (a contiguous M x F array),
 *              act_scale and rowsum hold the down projection's input (the quantised inner rows). With
 *              M == 1 and K, F <= 10240 the call is two kernel launches (the gate/up group, then
 *              the down projection with the sub-norm and quantisation in its prologue) and these
 *              three may be NULL.
 *   workspace, workspace_bytes : optional (NULL, 0) device workspace, 256-byte aligned, of at
 *              least bitnet_w2a8_ffn_workspace_size(M, K, F) bytes. That size is 0 for every
 *              shape: the projections run on the workspace-free kernels of bitnet_i2s_matmul,
 *              which measured faster than the expand-once path of bitnet_i2s_matmul_ws at every
 *              M tried (up to 8192); a workspace that is passed is not used.
 *   M >= 1; K and F multiples of 128 with K <= 65536 and F <= 32768; eps finite and > 0.
 */
BITNET_API int64_t bitnet_w2a8_ffn_workspace_size(int64_t M, int64_t K, int64_t F);
BITNET_API int bitnet_w2a8_ffn(const void *x, int dtype, int64_t M, int64_t K, int64_t F,
                               const uint8_t *wp_gate, float a_gate, const uint8_t *wp_up, float a_up,
                               const uint8_t *wp_down, float a_down, const float *gamma, float eps,
                               float *gate_out, float *up_out, float *out, int8_t *xq, float *act_scale,
                               int32_t *rowsum, void *workspace, int64_t workspace_bytes, void *stream);

/*
 * Persistent sweep over independent projection groups -- one kernel launch that computes, for
 * every group g, exactly what bitnet_w2a8_linear_group(x, dtype, 1, K, count, wp, w_scale, N,
 * out, NULL, ...) computes for that group at M = 1 (per-token quantisation of x, then the
 * ternary matmuls; [DeepDive] §4-5 and §4-2, "bitnet.rs" "Quantised Forward Pass").
 *   The groups must be independent: no group's x may be written by any group's out in the
 *   same run. This is the set of projections of a decode step whose input rows are given,
 *   streamed at HBM rate. A chain of dependent layers is the per-group call, launch by launch.
 *   One CTA per SM streams a contiguous slice of all groups' packed weights through a
 *   216 KB shared-memory ring.
 * bitnet_sweep_plan_create validates the table and copies it to the current device (host,
 * synchronous; allocates the plan's device table). Pointers inside are bound to the plan.
 * bitnet_sweep_plan_run launches it on `stream` (no allocation; may be captured into a CUDA
 * graph); the current device must be the plan's.
 * bitnet_sweep_plan_destroy frees the plan (NULL is a no-op).
 */
typedef struct bitnet_linear_group {
  const void *x;            /* K activations, dtype of the plan (device), 16-byte aligned     */
  int64_t K;                /* multiple of 128, 128 <= K <= 10240                             */
  int count;                /* 1..8 projections                                               */
  const uint8_t *wp[8];     /* wp[l]: N[l] x K/4 packed codes (device), 16-byte aligned       */
  float w_scale[8];         /* alpha_W of each projection                                     */
  int64_t N[8];             /* rows of each projection, >= 1 (total over all groups < 2^31)   */
  float *out[8];            /* out[l]: N[l] fp32 (device, written), 4-byte aligned            */
} bitnet_linear_group;
typedef struct bitnet_sweep_plan_s *bitnet_sweep_plan;
BITNET_API int bitnet_sweep_plan_create(const bitnet_linear_group *groups, int n_groups, int dtype,
                                        bitnet_sweep_plan *plan);
BITNET_API int bitnet_sweep_plan_run(bitnet_sweep_plan plan, void *stream);
BITNET_API int bitnet_sweep_plan_destroy(bitnet_sweep_plan plan);

/*
 * bitnet_last_device_error -- read and clear the device-side error word of the current
 * device. Kernels that wait on an mbarrier give up after a bounded number of polls and
 * record BITNET_ETIMEOUT there instead of hanging; bitnet_quant_weight records BITNET_ERANGE
 * for weights outside its range. Synchronises the device.
 * Returns BITNET_OK, BITNET_ETIMEOUT, BITNET_ERANGE or BITNET_ECUDA.
 */
BITNET_API int bitnet_last_device_error(void);

/*
 * bitnet_selftest_wait_timeout -- a diagnostic of the failure handling above; the pages have
 * no counterpart (they describe no GPU failure path). One small kernel takes, on purpose, the
 * path that bounded waits take when they run out, without faulting or hanging the GPU: one
 * thread starts a bulk copy of `bytes` bytes from src into shared memory, while a warp waits
 * on an mbarrier that nothing ever arrives on, giving up after max_polls polls. The warp then
 * records BITNET_ETIMEOUT in the device error word, and the copying thread waits (bounded) for
 * its copy to land before the kernel returns, as every producer in the library does.
 *   src       : device, 16-byte aligned, at least `bytes` bytes (read)
 *   bytes     : 16..16384, a multiple of 16
 *   max_polls : 1..2^20 polls of the never-completing barrier
 *   report    : device, 3 uint32 (written): [0] 1 if the wait gave up, [1] 1 if the copy was
 *               seen to land, [2] the wrapping sum of the copied 32-bit words
 * After the kernel has run, bitnet_last_device_error returns BITNET_ETIMEOUT (and clears it).
 */
BITNET_API int bitnet_selftest_wait_timeout(const void *src, int64_t bytes, int32_t max_polls,
                                            uint32_t *report, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* BITNET_GB300_H */
