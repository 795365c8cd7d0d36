// gemm_i2s_tc.cu -- prefill GEMM (large M) of the W2A8 ternary matmul on the tcgen05 tensor core.
//
// Computes the same integers as the decode GEMV -- raw = sum_k code[n][k] * xq[m][k],
// acc = raw - rowsum[m], out = (acc / s[m]) * w_scale -- for many tokens at once.
// Sources: the raw code dot over the 4x32-interleaved i2_s bytes ("[분석/검증-3] BitNet.cpp ARM
// 커널 재작성" §3, "[기술 분석 보고서] ... 추론 붕괴 원인 분석" §3.2), the byte layout ("BitNet
// 딥다이브" §4-2) and the dequantisation ("bitnet.rs" "Quantised Forward Pass").
//
// Why fp16 MMAs: ptxas rejects tcgen05.mma .kind::i8 for sm_103a, so the integer product runs
// as kind::f16 with fp16 operands. Every operand is a small integer (codes 0..3, activations
// -127..127) that fp16 represents exactly, every product is exact, and every partial sum is
// an integer of magnitude <= 3 * 127 * K, below 2^24 for K <= 32768 (the host restricts this
// path to that K), so the fp32 accumulation in tensor memory is exact and the result equals
// the integer dot bit for bit.
//
// Structure of one CTA (one 128 x 256 output tile, tokens x weight rows):
//   warps 0-7  (256 threads): stream xq and the packed bytes from global memory, expand
//              them to fp16 in registers (int8 -> fp16 and 2-bit code -> fp16 via exact
//              0x6400 magic-number conversions), store them into a 4-stage ring of
//              128-byte-swizzled K-major tiles, and later run the epilogue;
//   warp 8     : allocates tensor memory and, from one elected lane, issues
//              tcgen05.mma.cta_group::1.kind::f16 (M=128, N=256, K=16) per 16-wide K slice,
//              releasing each stage with tcgen05.commit.
// Stage hand-off uses mbarriers; every wait is bounded (see bitnet_dev.cuh) and a timeout
// is recorded in the device error word instead of hanging.
#include "bitnet_dev.cuh"

#include <cuda_fp16.h>

#include <atomic>

namespace bitnet {
namespace {

constexpr int BM = 128;                   // tokens per tile (MMA M)
constexpr int BN = 256;                   // weight rows per tile (MMA N)
constexpr int BK = 64;                    // K per stage: one 128-byte swizzle atom of fp16
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;      // 16 KB
constexpr int B_BYTES = BN * BK * 2;      // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int CONV_WARPS = 8;
constexpr int CONV_THREADS = CONV_WARPS * 32;
constexpr int THREADS = CONV_THREADS + 32;  // + the MMA warp
constexpr uint32_t TMEM_COLS = 256;         // fp32 accumulator, 128 lanes x 256 columns
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;  // + alignment slack for 1024-B atoms
constexpr uint32_t IDESC = make_idesc_f16_f32(BM, BN);

// byte offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled K-major tile
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// 4 signed int8 (one 32-bit word) -> 4 exact fp16 in two 32-bit words. The byte y + 128 is
// placed under the exponent byte 0x64 (fp16 1024 + u for u < 1024), then 1152 is subtracted.
__device__ __forceinline__ void s8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t l = __byte_perm(u, 0x64646464u, 0x4140);
  const uint32_t h = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6480),
                                      __ushort_as_half((unsigned short)0x6480));  // 1152
  const __half2 rl = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
  const __half2 rh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
  lo = *reinterpret_cast<const uint32_t*>(&rl);
  hi = *reinterpret_cast<const uint32_t*>(&rh);
}

// 4 codes (0..3, one per byte) -> 4 exact fp16 (same magic with 1024).
__device__ __forceinline__ void u2x4_to_f16x4(uint32_t codes, uint32_t& lo, uint32_t& hi) {
  const uint32_t l = __byte_perm(codes, 0x64646464u, 0x4140);
  const uint32_t h = __byte_perm(codes, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6400),
                                      __ushort_as_half((unsigned short)0x6400));  // 1024
  const __half2 rl = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
  const __half2 rh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
  lo = *reinterpret_cast<const uint32_t*>(&rl);
  hi = *reinterpret_cast<const uint32_t*>(&rh);
}

__global__ void __launch_bounds__(THREADS, 1) gemm_i2s_tc_kernel(const int8_t* __restrict__ xq,
                                                               const float* __restrict__ act_scale,
                                                               const int32_t* __restrict__ rowsum,
                                                               const uint8_t* __restrict__ wp, float w_scale,
                                                               float* __restrict__ out, int32_t* __restrict__ acc_out,
                                                               int M, int N, int K) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t accum_bar;
  __shared__ uint32_t tmem_base_slot;

  // 1024-byte aligned stage ring (the swizzle pattern is taken from address bits)
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t ring_addr = smem_u32(ring);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * BM;
  const int ksteps = K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], CONV_THREADS);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&accum_bar, 1);
    fence_mbar_init();
  }
  if (warp == CONV_WARPS) {
    tmem_alloc(&tmem_base_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_d = tmem_base_slot;
  bool abort = false;

  if (warp < CONV_WARPS) {
    // ===================== producers: expand to fp16 into the swizzled ring =====================
    const int tid = threadIdx.x;
    for (int it = 0; it < ksteps; ++it) {
      const int s = it % STAGES;
      if (it >= STAGES && !mbar_wait(&empty_bar[s], ((it / STAGES) - 1) & 1, &abort)) break;
      uint8_t* a_tile = ring + s * STAGE_BYTES;
      uint8_t* b_tile = a_tile + A_BYTES;
      const int k0 = it * BK;

      // A: 128 rows x 64 int8 -> fp16. Thread handles two 16-byte pieces (row r, quarter q).
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int p = tid + u * CONV_THREADS;
        const int r = p >> 2, q = p & 3;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (m0 + r < M) v = __ldg(reinterpret_cast<const uint4*>(xq + (int64_t)(m0 + r) * K + k0) + q);
        uint4 c0, c1;
        s8x4_to_f16x4(v.x, c0.x, c0.y);
        s8x4_to_f16x4(v.y, c0.z, c0.w);
        s8x4_to_f16x4(v.z, c1.x, c1.y);
        s8x4_to_f16x4(v.w, c1.z, c1.w);
        *reinterpret_cast<uint4*>(a_tile + sw128_offset(r, 2 * q)) = c0;
        *reinterpret_cast<uint4*>(a_tile + sw128_offset(r, 2 * q + 1)) = c1;
      }

      // B: 256 weight rows, one per thread. The 64 K positions of this stage are the bit
      // pairs j = 2*hb and 2*hb+1 of block i's 32 bytes (k_local = 32*jj + g).
      {
        const int r = tid;
        const int i = it >> 1, hb = it & 1;
        uint4 b0 = make_uint4(0u, 0u, 0u, 0u), b1 = b0;
        if (n0 + r < N) {
          const uint4* src = reinterpret_cast<const uint4*>(wp + (int64_t)(n0 + r) * (K >> 2) + i * 32);
          b0 = __ldg(src);
          b1 = __ldg(src + 1);
        }
        const uint32_t words[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int shift = 6 - 2 * (2 * hb + jj);
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {  // bytes g = 8*g8 .. 8*g8+7 -> one 16-byte chunk
            uint4 c;
            u2x4_to_f16x4((words[2 * g8] >> shift) & 0x03030303u, c.x, c.y);
            u2x4_to_f16x4((words[2 * g8 + 1] >> shift) & 0x03030303u, c.z, c.w);
            *reinterpret_cast<uint4*>(b_tile + sw128_offset(r, 4 * jj + g8)) = c;
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&full_bar[s]);
    }

    // ===================== epilogue: TMEM -> registers -> correction, scale -> global ===========
    const bool have = mbar_wait_warp(&accum_bar, 0, &abort);
    tc_fence_after();
    if (have) {
      const int q = warp & 3;             // TMEM lane quarter this warp may access
      const int col0 = (warp >> 2) * 128; // column half
      const int m = m0 + q * 32 + lane;
      const bool mv = m < M;
      const int rs = mv ? __ldg(rowsum + m) : 0;
      const float sc = mv ? __ldg(act_scale + m) : 1.0f;
#pragma unroll 1
      for (int cb = 0; cb < 128; cb += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_d + ((uint32_t)(q * 32) << 16) + (uint32_t)(col0 + cb), v);
        tmem_ld_wait();
        if (mv) {
          const int64_t rowoff = (int64_t)m * N;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int n = n0 + col0 + cb + e;
            if (n < N) {
              const int a = __float2int_rn(__uint_as_float(v[e])) - rs;
              out[rowoff + n] = __fmul_rn(__fdiv_rn(__int2float_rn(a), sc), w_scale);
              if (acc_out) acc_out[rowoff + n] = a;
            }
          }
        }
      }
    }
  } else {
    // ===================== MMA issuer (one elected lane of warp 8) ==============================
    if (lane == 0) {
      for (int it = 0; it < ksteps; ++it) {
        const int s = it % STAGES;
        if (!mbar_wait(&full_bar[s], (it / STAGES) & 1, &abort)) break;
        tc_fence_after();
        const uint32_t a_addr = ring_addr + s * STAGE_BYTES;
        const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = make_sw128_kmajor_desc(a_addr + kk * 32);
          const uint64_t bd = make_sw128_kmajor_desc(b_addr + kk * 32);
          mma_f16_ss(tmem_d, ad, bd, IDESC, (it > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&empty_bar[s]);
      }
      // always signal the epilogue, also after an abort: the commit tracks every MMA issued
      mma_commit(&accum_bar);
    }
    __syncwarp();
  }

  // ---- teardown: the accumulator must be complete before the tensor memory is freed ----
  tc_fence_before();
  __syncthreads();
  if (warp == CONV_WARPS) {
    tc_fence_after();
    bool dummy = false;
    mbar_wait(&accum_bar, 0, &dummy);  // already complete unless the MMA issuer aborted
    tmem_dealloc(tmem_d, TMEM_COLS);
  }
}

}  // namespace

cudaError_t read_clear_device_error_gemm(int* value) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

cudaError_t launch_gemm_i2s_tc(const int8_t* xq, const float* act_scale, const int32_t* rowsum,
                               const uint8_t* wp, float w_scale, float* out, int32_t* acc_out, int64_t M,
                               int64_t N, int64_t K, int num_sms, cudaStream_t stream) {
  (void)num_sms;
  // the large dynamic shared-memory opt-in is a per-device function attribute: set it once
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(gemm_i2s_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
  gemm_i2s_tc_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(xq, act_scale, rowsum, wp, w_scale, out, acc_out,
                                                             (int)M, (int)N, (int)K);
  return cudaGetLastError();
}

}  // namespace bitnet
