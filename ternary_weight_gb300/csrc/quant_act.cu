// quant_act.cu -- per-token absmax int8 activation quantisation (fp32 or bf16 rows).
//
// "BitNet 딥다이브" §4-5 (BitLinearKernel.quant_input): s = 127 / max(max|x|, 1e-5), round,
// clamp, int8; "bitnet.rs" "8-bit Activation Quantisation (AbsMax, per-token)". Round is
// round-half-to-even, the clamp [-127, 127]; bf16 is widened to fp32 exactly first. The
// row sum sum_k q is produced here as well: the matmul subtracts it from the raw code dot.
//
// One CTA of 256 threads per row. Each thread keeps its share of the row in registers
// (16-byte vectors: 4 fp32 or 8 bf16), so the row is read from HBM once: pass 1 finds
// max|x| (CTA reduction), pass 2 multiplies, rounds and stores int8, and sums q. Rows
// longer than the register budget take a variant that re-reads its vectors (L1/L2 hits).
#include "bitnet_dev.cuh"

#include <cuda_bf16.h>

namespace bitnet {
namespace {

constexpr int kThreads = 256;

template <bool BF16>
struct Vec;
template <>
struct Vec<false> {  // 4 x fp32
  static constexpr int kElems = 4;
  __device__ static void widen(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};
template <>
struct Vec<true> {  // 8 x bf16, widened exactly (bf16 bits are the top half of fp32)
  static constexpr int kElems = 8;
  __device__ static void widen(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int i = 1; i < kThreads / 32; ++i) r = fmaxf(r, red[i]);
  return r;
}

__device__ __forceinline__ int block_sum(int v, int* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int r = 0;
#pragma unroll
  for (int i = 0; i < kThreads / 32; ++i) r += red[i];
  return r;
}

// q = clamp(rne(x * s), -127, 127); the product is one fp32 multiply (no contraction).
__device__ __forceinline__ int quant_one(float x, float s) {
  int q = __float2int_rn(__fmul_rn(x, s));
  return max(-127, min(127, q));
}

template <int N>
__device__ __forceinline__ void store_q(int8_t* dst, const int (&q)[N]);
template <>
__device__ __forceinline__ void store_q<4>(int8_t* dst, const int (&q)[4]) {
  const uint32_t w = (uint32_t)(q[0] & 0xFF) | ((uint32_t)(q[1] & 0xFF) << 8) | ((uint32_t)(q[2] & 0xFF) << 16) |
                     ((uint32_t)(q[3] & 0xFF) << 24);
  *reinterpret_cast<uint32_t*>(dst) = w;
}
template <>
__device__ __forceinline__ void store_q<8>(int8_t* dst, const int (&q)[8]) {
  uint2 w;
  w.x = (uint32_t)(q[0] & 0xFF) | ((uint32_t)(q[1] & 0xFF) << 8) | ((uint32_t)(q[2] & 0xFF) << 16) |
        ((uint32_t)(q[3] & 0xFF) << 24);
  w.y = (uint32_t)(q[4] & 0xFF) | ((uint32_t)(q[5] & 0xFF) << 8) | ((uint32_t)(q[6] & 0xFF) << 16) |
        ((uint32_t)(q[7] & 0xFF) << 24);
  *reinterpret_cast<uint2*>(dst) = w;
}

// VPT > 0: each thread caches up to VPT vectors in registers. VPT == 0: re-read variant.
template <bool BF16, int VPT>
__global__ void __launch_bounds__(kThreads) quant_act_kernel(const void* __restrict__ x, int64_t K,
                                                             int8_t* __restrict__ xq, float* __restrict__ act_scale,
                                                             int32_t* __restrict__ rowsum) {
  using V = Vec<BF16>;
  constexpr int E = V::kElems;
  __shared__ float red_f[kThreads / 32];
  __shared__ int red_i[kThreads / 32];

  const int64_t m = blockIdx.x;
  const int64_t nvec = K / E;
  const uint4* row = reinterpret_cast<const uint4*>(static_cast<const char*>(x) + m * K * (BF16 ? 2 : 4));
  int8_t* qrow = xq + m * K;

  float amax = 0.0f;
  float cache[VPT > 0 ? VPT : 1][E];
  if constexpr (VPT > 0) {
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int64_t v = threadIdx.x + (int64_t)i * kThreads;
      if (v < nvec) {
        V::widen(__ldg(row + v), cache[i]);
#pragma unroll
        for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(cache[i][e]));
      }
    }
  } else {
    for (int64_t v = threadIdx.x; v < nvec; v += kThreads) {
      float f[E];
      V::widen(__ldg(row + v), f);
#pragma unroll
      for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(f[e]));
    }
  }
  amax = block_max(amax, red_f);
  const float s = __fdiv_rn(127.0f, fmaxf(amax, 1e-5f));

  int sum = 0;
  if constexpr (VPT > 0) {
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int64_t v = threadIdx.x + (int64_t)i * kThreads;
      if (v < nvec) {
        int q[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
          q[e] = quant_one(cache[i][e], s);
          sum += q[e];
        }
        store_q<E>(qrow + v * E, q);
      }
    }
  } else {
    for (int64_t v = threadIdx.x; v < nvec; v += kThreads) {
      float f[E];
      V::widen(__ldg(row + v), f);
      int q[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        q[e] = quant_one(f[e], s);
        sum += q[e];
      }
      store_q<E>(qrow + v * E, q);
    }
  }
  sum = block_sum(sum, red_i);
  if (threadIdx.x == 0) {
    act_scale[m] = s;
    rowsum[m] = sum;
  }
}

template <bool BF16>
cudaError_t launch_typed(const void* x, int64_t M, int64_t K, int8_t* xq, float* act_scale, int32_t* rowsum,
                         cudaStream_t stream) {
  constexpr int E = Vec<BF16>::kElems;
  const int64_t nvec = K / E;
  const int64_t per_thread = (nvec + kThreads - 1) / kThreads;
  dim3 grid((unsigned)M), block(kThreads);
  if (per_thread <= 2)
    quant_act_kernel<BF16, 2><<<grid, block, 0, stream>>>(x, K, xq, act_scale, rowsum);
  else if (per_thread <= 4)
    quant_act_kernel<BF16, 4><<<grid, block, 0, stream>>>(x, K, xq, act_scale, rowsum);
  else if (per_thread <= 8)
    quant_act_kernel<BF16, 8><<<grid, block, 0, stream>>>(x, K, xq, act_scale, rowsum);
  else
    quant_act_kernel<BF16, 0><<<grid, block, 0, stream>>>(x, K, xq, act_scale, rowsum);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_act(const void* x, int dtype, int64_t M, int64_t K, int8_t* xq, float* act_scale,
                             int32_t* rowsum, cudaStream_t stream) {
  return dtype == 1 ? launch_typed<true>(x, M, K, xq, act_scale, rowsum, stream)
                    : launch_typed<false>(x, M, K, xq, act_scale, rowsum, stream);
}

}  // namespace bitnet
