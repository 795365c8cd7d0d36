// ffn.cu -- the FFN's inner activation fused with its per-token quantisation, for M rows.
//
// Per row m ("bitnet.rs" "Forward Pass": inner = ffn_sub_norm(sqrelu(gate(x)) * up(x)), then
// out = down(inner); the quantisation is that of every W2A8 input, "BitNet 딥다이브" §4-5):
//   h     = max(g, 0)^2 * u
//   inner = (h * c) * gamma,       c = 1 / sqrt(sum(h^2) / F + eps)   (RMSNorm)
//   s     = 127 / max(max|inner|, 1e-5),  xq = rne(inner * s),  rowsum = sum xq
// with the fixed summation order and the fp32 rounding of each step described beside
// FfnIn; xq, s and rowsum are then exactly what the activation quantiser gives for the row
// inner, so the down projection can take them directly.
//
// One CTA of 256 threads per row, thread t taking 16-byte vectors t, t + 256, ... (which is
// the partial order of the sum of squares). Three passes over a shared-memory copy of the
// row: h and the sum of squares (gate and up are read once from HBM), then inner and its
// absolute maximum, then the codes.
#include "bitnet_dev.cuh"

namespace bitnet {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// x * s rounded to the nearest integer (ties to even) as an int; |x * s| <= 127.5 here
__device__ __forceinline__ int quant_one(float x, float s) { return __float2int_rn(__fmul_rn(x, s)); }

__global__ void __launch_bounds__(kThreads) ffn_act_quant_kernel(FfnIn ffn, int F, int8_t* __restrict__ xq,
                                                                 float* __restrict__ act_scale,
                                                                 int32_t* __restrict__ rowsum,
                                                                 float* __restrict__ inner_out) {
  extern __shared__ __align__(16) float4 row_s[];  // F / 4 vectors
  __shared__ float red_ss[kWarps];
  __shared__ uint32_t red_m[kWarps];
  __shared__ int red_i[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t m = blockIdx.x;
  const int nvec = F >> 2;
  const float4* g4 = reinterpret_cast<const float4*>(ffn.gate + m * F);
  const float4* u4 = reinterpret_cast<const float4*>(ffn.up + m * F);
  const float4* gm4 = reinterpret_cast<const float4*>(ffn.gamma);

  // pass 1: h, parked in shared memory, and this thread's partial of the sum of squares
  float ssp = 0.0f;
#pragma unroll 4
  for (int v = threadIdx.x; v < nvec; v += kThreads) {
    const float4 g = __ldcs(g4 + v), u = __ldcs(u4 + v);
    float4 h;
    h.x = ffn_h(g.x, u.x);
    h.y = ffn_h(g.y, u.y);
    h.z = ffn_h(g.z, u.z);
    h.w = ffn_h(g.w, u.w);
    ssp = __fmaf_rn(h.x, h.x, ssp);
    ssp = __fmaf_rn(h.y, h.y, ssp);
    ssp = __fmaf_rn(h.z, h.z, ssp);
    ssp = __fmaf_rn(h.w, h.w, ssp);
    row_s[v] = h;
  }
  ssp = ffn_run_sum(ssp);
  if (lane == 0) red_ss[warp] = ssp;
  __syncthreads();
  const float c = ffn_rms_factor(ffn_runs_total(red_ss), F, ffn.eps);

  // pass 2: inner = (h * c) * gamma, and its absolute maximum
  float amax = 0.0f;
  for (int v = threadIdx.x; v < nvec; v += kThreads) {
    const float4 h = row_s[v], gm = __ldg(gm4 + v);
    float4 y;
    y.x = __fmul_rn(__fmul_rn(h.x, c), gm.x);
    y.y = __fmul_rn(__fmul_rn(h.y, c), gm.y);
    y.z = __fmul_rn(__fmul_rn(h.z, c), gm.z);
    y.w = __fmul_rn(__fmul_rn(h.w, c), gm.w);
    amax = fmaxf(fmaxf(amax, fmaxf(fabsf(y.x), fabsf(y.y))), fmaxf(fabsf(y.z), fabsf(y.w)));
    row_s[v] = y;
    if (inner_out) __stcs(reinterpret_cast<float4*>(inner_out + m * F) + v, y);
  }
  // amax is a non-negative float (fmaxf drops NaN): its bits order like unsigned integers
  const uint32_t wmax = __reduce_max_sync(0xffffffffu, __float_as_uint(amax));
  if (lane == 0) red_m[warp] = wmax;
  __syncthreads();
  uint32_t bm = 0;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) bm = max(bm, red_m[i]);
  const float s = __fdiv_rn(127.0f, fmaxf(__uint_as_float(bm), 1e-5f));

  // pass 3: codes (the clamp to [-127, 127] is never active: s = fl(127 / a), a >= max|inner|)
  int sum = 0;
  uint32_t* xq_row = reinterpret_cast<uint32_t*>(xq + m * F);
  for (int v = threadIdx.x; v < nvec; v += kThreads) {
    const float4 y = row_s[v];
    const int q0 = quant_one(y.x, s), q1 = quant_one(y.y, s), q2 = quant_one(y.z, s), q3 = quant_one(y.w, s);
    sum += (q0 + q1) + (q2 + q3);
    xq_row[v] = (uint32_t)(q0 & 0xFF) | ((uint32_t)(q1 & 0xFF) << 8) | ((uint32_t)(q2 & 0xFF) << 16) |
                ((uint32_t)(q3 & 0xFF) << 24);
  }
  sum = __reduce_add_sync(0xffffffffu, sum);
  if (lane == 0) red_i[warp] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) t += red_i[i];
    act_scale[m] = s;
    rowsum[m] = t;
  }
}

}  // namespace

cudaError_t launch_ffn_act_quant(const FfnIn& ffn, int64_t M, int64_t F, int8_t* xq, float* act_scale,
                                 int32_t* rowsum, float* inner_out, cudaStream_t stream) {
  const int smem = (int)(F * 4);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(ffn_act_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kFfnMaxF * 4));
    if (e != cudaSuccess) return e;
  }
  ffn_act_quant_kernel<<<(unsigned)M, kThreads, smem, stream>>>(ffn, (int)F, xq, act_scale, rowsum, inner_out);
  return cudaGetLastError();
}

}  // namespace bitnet
