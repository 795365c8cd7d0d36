// quant_weight.cu -- weight ternarisation and i2_s packing (the step before the matmul path).
//
// What it computes (N x K weights, fp32 or bf16):
//   AbsMean ("BitNet 딥다이브" §6-2, "bitnet.rs" "Ternary Weight Quantisation"):
//     scale = max(mean|w|, 1e-5), q = clip(rne(w / scale), -1, 1)
//   sign rule (quantize_i2_s on weights that are already ternary, "BitNet 딥다이브" §4-2):
//     q = 0 where |w| < 1e-6 (compared in double), else sign(w); scale = max|w|
// then the codes q + 1 are packed in the i2_s layout ("BitNet 딥다이브" §4-2): weight 32j + g of
// 128-weight block i goes to byte 32i + g at bit offset 6 - 2j.
//
// The scale decides every code through w / scale, so it has to be reproducible bit for bit.
// The mean is therefore defined through an exact integer: S = sum over all weights of
// floor(|w| * 2^74), with |w| < 2^12 and N * K <= 2^40, so S < 2^126 fits 128 bits and no
// summation order enters. mean = fp32(fp64(S) * 2^-74 / (N * K)), each conversion and the
// division rounding to nearest. A weight outside the range (or NaN) is reported as an error.
//
// Three launches on the caller's stream, no workspace:
//   1. qw_reduce: a grid-stride pass over the whole matrix (flat, four 16-byte loads per thread in
//      flight); each CTA parks its partial (128-bit sum, or max |w|) in the first bytes of the
//      packed output, 16 bytes per CTA;
//   2. qw_finish: one CTA adds the partials and writes the scale (device float);
//   3. qw_pack: one thread per packed 32-bit word (16 weights: four 16-byte loads), overwriting the
//      parked partials. The codes are decided by comparisons against thresholds derived from the
//      scale that reproduce rne(fl(w / scale)) exactly (see code_threshold).
#include "bitnet_dev.cuh"

#include <cuda_bf16.h>

namespace bitnet {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;  // 16-byte vectors per thread per iteration
constexpr int kErrRange = -6;
constexpr uint32_t kAbsLimitBits = 0x45800000u;  // 4096.0f: |w| must stay below 2^12
constexpr uint32_t kInfBits = 0x7F800000u;

typedef unsigned __int128 u128;

// four weights as fp32 bit patterns from 16 bytes (fp32) or 8 bytes (bf16) at element i
template <bool BF16>
__device__ __forceinline__ uint4 load_bits4(const void* w, int64_t i) {
  if constexpr (BF16) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(w) + i));
    return make_uint4(u.x << 16, u.x & 0xFFFF0000u, u.y << 16, u.y & 0xFFFF0000u);
  } else {
    return __ldg(reinterpret_cast<const uint4*>(static_cast<const float*>(w) + i));
  }
}

// low 32 bits of (v * 2^32) >> c; PTX clamps shift counts above 64, so any c >= 64 gives 0
__device__ __forceinline__ uint32_t shr_low32(uint32_t v, uint32_t c) {
  uint64_t r;
  asm("shr.b64 %0, %1, %2;" : "=l"(r) : "l"((uint64_t)v << 32), "r"(c));
  return (uint32_t)r;
}
// (v * 2^32) >> c as 64 bits, same clamp
__device__ __forceinline__ uint64_t shr_64(uint32_t v, uint32_t c) {
  uint64_t r;
  asm("shr.b64 %0, %1, %2;" : "=l"(r) : "l"((uint64_t)v << 32), "r"(c));
  return r;
}

// floor(|w| * 2^74) = hi * 2^32 + lo for one weight with |w| bits m (sign cleared).
// |w| = sig * 2^(e - 150) for a normal float (sig = 24-bit significand, e = biased exponent), so
// |w| * 2^74 = sig * 2^(e - 76): lo = low 32 bits of that, hi = the rest (< 2^54 in range).
// Zero and subnormals (e = 0) give 0 through the shift clamp, which is exact: their
// |w| * 2^74 < 2^-52. Out-of-range values give bounded garbage; the caller flags them.
__device__ __forceinline__ void fixed_parts(uint32_t m, uint64_t& lo_acc, uint64_t& hi_acc) {
  const uint32_t e = m >> 23;
  const uint32_t sig = (m & 0x007FFFFFu) | 0x00800000u;
  lo_acc += shr_low32(sig, 108u - e);  // sig * 2^(e - 76) = (sig * 2^32) >> (108 - e)
  hi_acc += shr_64(sig, 140u - e);     // and >> 32 more for the part above bit 32
}

__device__ __forceinline__ u128 shfl_xor_u128(u128 v, int off) {
  const uint64_t lo = __shfl_xor_sync(0xffffffffu, (unsigned long long)(uint64_t)v, off);
  const uint64_t hi = __shfl_xor_sync(0xffffffffu, (unsigned long long)(uint64_t)(v >> 64), off);
  return ((u128)hi << 64) | lo;
}

// mode 0: per-CTA 128-bit partial of S (bit 127 set when a weight is out of range);
// mode 1: per-CTA max |w| bits (NaN ignored, as fmaxf does).
template <bool BF16>
__global__ void __launch_bounds__(kThreads) qw_reduce(const void* __restrict__ w, uint8_t* __restrict__ park,
                                                   int64_t total, int mode) {
  const int64_t nvec = total >> 2;  // 4-weight vectors
  const int64_t stride = (int64_t)gridDim.x * kThreads * kVecPerThread;
  uint64_t lo = 0;  // sum of the low parts (< 2^32 each, fewer than 2^32 of them per thread)
  u128 h = 0;       // sum of the high parts, folded in once per iteration
  uint32_t mx = 0;              // max |w| bits over in-range values (mode 0: over all, for the check)
  for (int64_t v0 = (int64_t)blockIdx.x * kThreads * kVecPerThread + threadIdx.x; v0 < nvec; v0 += stride) {
    uint4 b[kVecPerThread];
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      const int64_t v = v0 + (int64_t)u * kThreads;
      b[u] = v < nvec ? load_bits4<BF16>(w, v * 4) : make_uint4(0, 0, 0, 0);
    }
    if (mode == 0) {
      uint64_t hr = 0;  // 16 high parts < 2^56 each
#pragma unroll
      for (int u = 0; u < kVecPerThread; ++u) {
        const uint32_t m[4] = {b[u].x & 0x7FFFFFFFu, b[u].y & 0x7FFFFFFFu, b[u].z & 0x7FFFFFFFu,
                               b[u].w & 0x7FFFFFFFu};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          mx = max(mx, m[q]);
          fixed_parts(m[q], lo, hr);
        }
      }
      h += hr;
    } else {
#pragma unroll
      for (int u = 0; u < kVecPerThread; ++u) {
        const uint32_t m[4] = {b[u].x & 0x7FFFFFFFu, b[u].y & 0x7FFFFFFFu, b[u].z & 0x7FFFFFFFu,
                               b[u].w & 0x7FFFFFFFu};
#pragma unroll
        for (int q = 0; q < 4; ++q) mx = max(mx, m[q] > kInfBits ? 0u : m[q]);
      }
    }
  }
  __shared__ u128 red_s[kThreads / 32];
  __shared__ uint32_t red_m[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (mode == 0) {
    u128 s = (h << 32) + lo;  // this thread's exact sum
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s += shfl_xor_u128(s, off);
    if (lane == 0) red_s[warp] = s;
  }
  if (lane == 0) red_m[warp] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t m = 0;
    for (int i = 0; i < kThreads / 32; ++i) m = max(m, red_m[i]);
    uint64_t* out = reinterpret_cast<uint64_t*>(park + 16 * (int64_t)blockIdx.x);
    if (mode == 0) {
      u128 s = 0;
      for (int i = 0; i < kThreads / 32; ++i) s += red_s[i];
      if (m >= kAbsLimitBits) s |= (u128)1 << 127;
      out[0] = (uint64_t)s;
      out[1] = (uint64_t)(s >> 64);
    } else {
      out[0] = m;
    }
  }
}

// fp64 value of a 128-bit unsigned integer, rounded to nearest even: the top 64 significant
// bits with every lower bit folded into a sticky bit below the rounding position, then one
// correctly rounded 64 -> 53 bit conversion, then an exact power-of-two scaling.
__device__ double u128_to_double_rn(u128 s) {
  const uint64_t hi = (uint64_t)(s >> 64), lo = (uint64_t)s;
  if (hi == 0) return __ull2double_rn(lo);
  const int lz = __clzll((long long)hi);
  const u128 t = s << lz;  // top bit at 127
  const uint64_t top = (uint64_t)(t >> 64) | ((uint64_t)t != 0 ? 1ull : 0ull);
  return ldexp(__ull2double_rn(top), 64 - lz);
}

__global__ void __launch_bounds__(kThreads) qw_finish(const uint8_t* __restrict__ park, int nparts, float* __restrict__ w_scale,
                                                   int64_t total, int mode) {
  __shared__ u128 red_s[kThreads / 32];
  __shared__ uint32_t red_m[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  u128 s = 0;
  uint32_t bad = 0, mx = 0;
  for (int i = threadIdx.x; i < nparts; i += kThreads) {
    const uint64_t* p = reinterpret_cast<const uint64_t*>(park + 16 * (int64_t)i);
    if (mode == 0) {
      const uint64_t phi = p[1];
      bad |= (uint32_t)(phi >> 63);
      s += ((u128)(phi & 0x7FFFFFFFFFFFFFFFull) << 64) | p[0];
    } else {
      mx = max(mx, (uint32_t)p[0]);
    }
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  bad = __reduce_or_sync(0xffffffffu, bad);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) s += shfl_xor_u128(s, off);
  if (lane == 0) {
    red_s[warp] = s;
    red_m[warp] = mx | (bad << 31);  // max |w| bits never use bit 31
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  u128 t = 0;
  uint32_t m = 0, any_bad = 0;
  for (int i = 0; i < kThreads / 32; ++i) {
    t += red_s[i];
    m = max(m, red_m[i] & 0x7FFFFFFFu);
    any_bad |= red_m[i] >> 31;
  }
  if (mode == 0) {
    if (any_bad) {
      record_device_error(kErrRange);
      *w_scale = __uint_as_float(0x7FC00000u);  // NaN
      return;
    }
    const double mean = __ddiv_rn(u128_to_double_rn(t) * 0x1p-74, (double)total);
    *w_scale = fmaxf(__double2float_rn(mean), 1e-5f);
  } else {
    *w_scale = __uint_as_float(m);
  }
}

// Code thresholds. AbsMean: rne(r) with r = fl(w / s) clipped to [-1, 1] is +1 exactly when
// r > 0.5 (0.5 itself rounds to the even 0). fl(x) > 0.5 holds exactly when x > 0.5 + 2^-25:
// the next float above 0.5 is 0.5 + 2^-24, and the tie at their midpoint goes to 0.5, whose
// significand is even. So q = +1 iff w > s * (0.5 + 2^-25) (a product exact in fp64: 24 + 25
// significant bits), iff w > T with T that product rounded down to fp32 (no float lies
// strictly between T and the product). q = -1 iff w < -T by symmetry of the division.
// Sign rule: (double)|w| < 1e-6 iff |w| < T with T = 1e-6 rounded up to fp32 (1e-6 is not a
// binary fraction, so it lies strictly between two floats).
__device__ __forceinline__ float code_threshold(float scale, int mode) {
  if (mode == 0) return __double2float_rd((double)scale * (0.5 + 0x1p-25));
  return __double2float_ru(1e-6);
}

__device__ __forceinline__ uint32_t code_of(float v, float thr, int mode) {
  if (mode == 0) return 1u + (v > thr ? 1u : 0u) - (v < -thr ? 1u : 0u);
  if (fabsf(v) < thr) return 1u;
  return v > 0.0f ? 2u : 0u;  // NaN codes as -1, as the comparison in double would
}

// Thread t writes packed word t: row n, word c of the row (block i = c / 8, bytes g0..g0+3 with
// g0 = 4 (c % 8)); byte g0 + b holds the codes of k = 128 i + g0 + b + 32 j at bit 6 - 2j.
template <bool BF16>
__global__ void __launch_bounds__(kThreads) qw_pack(const void* __restrict__ w, const float* __restrict__ w_scale,
                                                 uint32_t* __restrict__ wp, int64_t N, int64_t K, int mode) {
  const float thr = code_threshold(*w_scale, mode);
  const int64_t words_per_row = K / 16;
  const int64_t total = N * words_per_row;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = t / words_per_row, c = t - n * words_per_row;
    const int64_t base = n * K + (c >> 3) * 128 + (c & 7) * 4;
    uint4 b[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) b[j] = load_bits4<BF16>(w, base + 32 * j);
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t sh = 6u - 2u * (uint32_t)j;
      word |= (code_of(__uint_as_float(b[j].x), thr, mode) << sh) |
              (code_of(__uint_as_float(b[j].y), thr, mode) << (sh + 8)) |
              (code_of(__uint_as_float(b[j].z), thr, mode) << (sh + 16)) |
              (code_of(__uint_as_float(b[j].w), thr, mode) << (sh + 24));
    }
    wp[t] = word;
  }
}

template <bool BF16>
cudaError_t launch_t(const void* w, int64_t N, int64_t K, int mode, uint8_t* wp, float* w_scale, int num_sms,
                     cudaStream_t stream) {
  const int64_t total = N * K;
  // one CTA per 4096 weights at most, so the 16-byte partials fit the packed output (N K / 4
  // bytes) with room to spare; four CTAs per SM keep enough loads in flight for HBM
  int64_t parts = (total + kThreads * kVecPerThread * 4 - 1) / (kThreads * kVecPerThread * 4);
  if (parts > (int64_t)num_sms * 4) parts = (int64_t)num_sms * 4;
  qw_reduce<BF16><<<(unsigned)parts, kThreads, 0, stream>>>(w, wp, total, mode);
  qw_finish<<<1, kThreads, 0, stream>>>(wp, (int)parts, w_scale, total, mode);
  const int64_t words = total / 16;
  int64_t blocks = (words + kThreads - 1) / kThreads;
  if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
  qw_pack<BF16><<<(unsigned)blocks, kThreads, 0, stream>>>(w, w_scale, reinterpret_cast<uint32_t*>(wp), N, K, mode);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_weight(const void* w, bool bf16, int64_t N, int64_t K, int mode, uint8_t* wp, float* w_scale,
                                int num_sms, cudaStream_t stream) {
  return bf16 ? launch_t<true>(w, N, K, mode, wp, w_scale, num_sms, stream)
              : launch_t<false>(w, N, K, mode, wp, w_scale, num_sms, stream);
}

cudaError_t read_clear_device_error_quant_weight(int* value) {
  *value = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

}  // namespace bitnet
