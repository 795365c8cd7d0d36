// gemm_tc_ws.cu -- prefill GEMM of the W2A8 ternary matmul with a caller-provided workspace:
// expand once, then a TMA-fed tcgen05 GEMM.
//
// Computes raw[m][n] = sum_k code[n][k] * xq[m][k], acc = raw - rowsum[m],
// out = (acc / s[m]) * w_scale, exactly as the other matmul paths (same integers, same fp32
// operations in the same order). Sources: the raw code dot over the 4x32-interleaved i2_s
// bytes ("[분석/검증-3] BitNet.cpp ARM 커널 재작성" §3, "[기술 분석 보고서] ... 추론 붕괴 원인 분석"
// §3.2), the byte layout ("BitNet 딥다이브" §4-2) and the dequantisation ("bitnet.rs" "Quantised
// Forward Pass"). "BitNet 딥다이브" §4-5 notes that the reference GPU path runs its prefill model
// with fp16 weights; here the fp16 weights are produced per call from the 2-bit codes.
//
// Why expand first: on-the-fly expansion inside the GEMM repeats the work for every output
// tile that shares an operand tile (the activation tile once per N-tile, the weight tile
// once per M-tile), and the expanding warps become the bottleneck. Expanding once is two
// short HBM-bound passes; the GEMM itself is then a plain fp16 x fp16 -> fp32 contraction:
//   1. expand_codes_f16: each 2-bit code c -> fp16 c (0..3), written K-major, N x K;
//   2. convert_s8_f16:   each int8 activation -> fp16 (exact), M x K;
//   3. gemm_f16_ws_kernel: persistent CTAs over 128 x 256 output tiles (M fastest, so CTAs
//      running together share weight tiles in L2). Warp 0 issues 2-D TMA loads
//      (cp.async.bulk.tensor, 128-byte swizzle) of the fp16 tiles into a 4-stage ring; warp 1
//      allocates 512 columns of tensor memory and issues tcgen05.mma.cta_group::1.kind::f16
//      (M=128, N=256, K=16) into one of two 256-column fp32 accumulators, releasing stages
//      with tcgen05.commit; warps 2-5 drain the other accumulator (tcgen05.ld, -rowsum, /s,
//      *alpha_W) while the next tile accumulates.
// Exactness: every operand is a small integer fp16 holds exactly and every partial sum is an
// integer of magnitude <= 3 * 127 * K < 2^24 for K <= 32768, so the fp32 accumulation is exact.
// Every wait is bounded; a timeout is recorded in the device error word.
#include "bitnet_dev.cuh"

#include <cuda_fp16.h>

#include <atomic>
#include <cudaTypedefs.h>

namespace bitnet {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle row of fp16
constexpr int A_BYTES = BM * BK * 2;
constexpr int EPI_WARPS = 4;
constexpr int THREADS = (2 + EPI_WARPS) * 32;  // producer, MMA, 4 epilogue warps
constexpr uint32_t TMEM_COLS = 512;             // two accumulators of BN <= 256 fp32 columns
constexpr int kSmemBudget = 227 * 1024;
// epilogue staging: one 32 x 33 fp32 block per epilogue warp (the padding column keeps both the
// row-wise writes and the column-wise reads free of bank conflicts)
constexpr int EPI_PITCH = 33;
constexpr int EPI_SMEM = EPI_WARPS * 32 * EPI_PITCH * 4;

// Tile width BN (the MMA's N) is chosen per problem; the ring takes as many stages as fit.
template <int BN>
struct TileCfg {
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int RING_BUDGET = kSmemBudget - 1024 - 1024 - EPI_SMEM;
  static constexpr int STAGES = RING_BUDGET / STAGE_BYTES < 6 ? RING_BUDGET / STAGE_BYTES : 6;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + EPI_SMEM;
  static constexpr uint32_t IDESC = make_idesc_f16_f32(BM, BN);
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "MMA N and the 32-column epilogue steps");
  static_assert(STAGE_BYTES % 1024 == 0, "stages keep the 1024-byte alignment of the swizzle atoms");
  static_assert(STAGES >= 3, "pipeline depth");
};

// ---------------------------------------------------------------------------- expansion
__device__ __forceinline__ uint2 codes4_to_f16(uint32_t codes) {  // 4 codes (one per byte) -> 4 fp16
  const uint32_t l = __byte_perm(codes, 0x64646464u, 0x4140);
  const uint32_t h = __byte_perm(codes, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6400), __ushort_as_half((unsigned short)0x6400));
  const __half2 rl = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
  const __half2 rh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&rl), *reinterpret_cast<const uint32_t*>(&rh));
}

__device__ __forceinline__ uint2 s8x4_to_f16(uint32_t w) {  // 4 int8 -> 4 exact fp16
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t l = __byte_perm(u, 0x64646464u, 0x4140);
  const uint32_t h = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6480), __ushort_as_half((unsigned short)0x6480));
  const __half2 rl = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
  const __half2 rh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&rl), *reinterpret_cast<const uint32_t*>(&rh));
}

// One thread per packed 32-bit word (bytes g0..g0+3 of block i of row n): its 16 codes go to
// k = 128i + 32j + g0 + (0..3), j = 0..3 (bit pair j at offset 6 - 2j).
__global__ void __launch_bounds__(256) expand_codes_f16(const uint8_t* __restrict__ wp, uint16_t* __restrict__ w16,
                                                        int64_t N, int64_t K) {
  const int64_t wpr = K >> 4;  // words per packed row
  const int64_t total = N * wpr;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = t / wpr, c = t - n * wpr;
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(wp) + t);
    uint16_t* dst = w16 + n * K + (c >> 3) * 128 + (c & 7) * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint2*>(dst + 32 * j) = codes4_to_f16((w >> (6 - 2 * j)) & 0x03030303u);
  }
}

__global__ void __launch_bounds__(256) convert_s8_f16(const int8_t* __restrict__ xq, uint16_t* __restrict__ x16,
                                                      int64_t n16) {
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n16; t += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(xq) + t);
    const uint2 a = s8x4_to_f16(v.x), b = s8x4_to_f16(v.y), c = s8x4_to_f16(v.z), d = s8x4_to_f16(v.w);
    uint4* dst = reinterpret_cast<uint4*>(x16) + 2 * t;
    dst[0] = make_uint4(a.x, a.y, b.x, b.y);
    dst[1] = make_uint4(c.x, c.y, d.x, d.y);
  }
}

// ---------------------------------------------------------------------------- GEMM
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

template <int BN>
__global__ void __launch_bounds__(THREADS, 1) gemm_f16_ws_kernel(const __grid_constant__ CUtensorMap tmA,
                                                                 const __grid_constant__ CUtensorMap tmB,
                                                                 const float* __restrict__ act_scale,
                                                                 const int32_t* __restrict__ rowsum, float w_scale,
                                                                 float* __restrict__ out, int32_t* __restrict__ acc_out,
                                                                 int M, int N, int K) {
  using Cfg = TileCfg<BN>;
  constexpr int STAGES = Cfg::STAGES, STAGE_BYTES = Cfg::STAGE_BYTES;
  constexpr uint32_t IDESC = Cfg::IDESC;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t done_bar;
  __shared__ uint32_t tmem_slot;

  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);  // 1024-byte aligned atoms
  const uint32_t ring_addr = smem_u32(ring);
  float* epi_stage = reinterpret_cast<float*>(ring + STAGES * STAGE_BYTES);  // EPI_SMEM bytes
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_m = (M + BM - 1) / BM, num_n = (N + BN - 1) / BN;
  const int tiles = num_m * num_n;
  const int ksteps = K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], EPI_WARPS * 32);
    }
    mbar_init(&done_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  bool abort = false;

  if (warp == 0) {
    // ================================ TMA producer ================================
    if (lane == 0) {
      int it = 0;
      for (int tile = blockIdx.x; tile < tiles && !abort; tile += gridDim.x) {
        const int m0 = (tile % num_m) * BM, n0 = (tile / num_m) * BN;
        for (int ks = 0; ks < ksteps; ++ks, ++it) {
          const int s = it % STAGES, u = it / STAGES;
          if (u > 0 && !mbar_wait(&empty_bar[s], (u - 1) & 1, &abort)) break;
          uint8_t* a_dst = ring + s * STAGE_BYTES;
          mbar_arrive_expect_tx(&full_bar[s], STAGE_BYTES);
          tma_load_2d(a_dst, &tmA, ks * BK, m0, &full_bar[s]);
          tma_load_2d(a_dst + A_BYTES, &tmB, ks * BK, n0, &full_bar[s]);
        }
      }
      {  // every copy issued lands before the producer leaves: the MMA thread may have given up
         // on a full barrier (a bounded wait) while copies were still in flight
        bool dummy = false;
        for (int i = it - STAGES > 0 ? it - STAGES : 0; i < it; ++i) mbar_wait(&full_bar[i % STAGES], (i / STAGES) & 1, &dummy);
      }
    }
    __syncwarp();  // the warp reaches the teardown barrier as a whole
  } else if (warp == 1) {
    // ================================ MMA issuer ================================
    if (lane == 0) {
      int it = 0, lt = 0;
      for (int tile = blockIdx.x; tile < tiles && !abort; tile += gridDim.x, ++lt) {
        const int acc = lt & 1, ua = lt >> 1;
        if (ua > 0 && !mbar_wait(&tempty_bar[acc], (ua - 1) & 1, &abort)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * BN);
        for (int ks = 0; ks < ksteps; ++ks, ++it) {
          const int s = it % STAGES, u = it / STAGES;
          if (!mbar_wait(&full_bar[s], u & 1, &abort)) break;
          tc_fence_after();
          const uint32_t a_addr = ring_addr + s * STAGE_BYTES, b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_f16_ss(d, make_sw128_kmajor_desc(a_addr + kk * 32), make_sw128_kmajor_desc(b_addr + kk * 32), IDESC,
                       (ks > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&empty_bar[s]);
        }
        mma_commit(&tfull_bar[acc]);
      }
      mma_commit(&done_bar);  // tracks every MMA this thread issued
    }
    __syncwarp();  // the warp reaches the teardown barrier and the free as a whole
  } else {
    // ================================ epilogue (warps 2-5) ================================
    // Warp q reads accumulator lanes 32q..32q+31 (rows m0 + 32q + lane) 32 columns at a time,
    // finishes them in registers, and writes them through its 32 x 33 staging block so that
    // each store instruction covers 32 consecutive columns of one row (128 contiguous bytes).
    const int q = warp & 3;  // tensor-memory lane quarter this warp may read
    float* blk = epi_stage + (warp - 2) * 32 * EPI_PITCH;
    int* blk_i = reinterpret_cast<int*>(blk);
    int lt = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++lt) {
      const int acc = lt & 1, ua = lt >> 1;
      if (!mbar_wait_warp(&tfull_bar[acc], ua & 1, &abort)) break;
      tc_fence_after();
      const int m0 = (tile % num_m) * BM, n0 = (tile / num_m) * BN;
      const int mrow = m0 + q * 32 + lane;  // this lane's accumulator row
      const bool mv = mrow < M;
      const int rs = mv ? __ldg(rowsum + mrow) : 0;
      const float sc = mv ? __ldg(act_scale + mrow) : 1.0f;
#pragma unroll 1
      for (int cb = 0; cb < BN; cb += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + cb), v);
        tmem_ld_wait();
        const int n = n0 + cb + lane;  // the column this lane stores
        // pass 1: acc = raw - rowsum, staged row-wise (lane = row)
#pragma unroll
        for (int e = 0; e < 32; ++e) blk_i[lane * EPI_PITCH + e] = __float2int_rn(__uint_as_float(v[e])) - rs;
        __syncwarp();
        if (acc_out) {
#pragma unroll 4
          for (int r = 0; r < 32; ++r) {
            const int m = m0 + q * 32 + r;
            if (m < M && n < N) acc_out[(int64_t)m * N + n] = blk_i[r * EPI_PITCH + lane];
          }
        }
        __syncwarp();
        // pass 2: out = (acc / s) * w_scale, in the row's own lane, then stored column-wise
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int a = blk_i[lane * EPI_PITCH + e];
          blk[lane * EPI_PITCH + e] = __fmul_rn(__fdiv_rn(__int2float_rn(a), sc), w_scale);
        }
        __syncwarp();
#pragma unroll 4
        for (int r = 0; r < 32; ++r) {
          const int m = m0 + q * 32 + r;
          if (m < M && n < N) out[(int64_t)m * N + n] = blk[r * EPI_PITCH + lane];
        }
        __syncwarp();
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar[acc]);
    }
  }

  // ---- teardown: every MMA complete before the tensor memory is freed ----
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    bool dummy = false;
    mbar_wait(&done_bar, 0, &dummy);
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
  if (!f) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
      return nullptr;
    f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    fn.store(f, std::memory_order_release);
  }
  return f;
}

// 2-D fp16 tensor [rows][K] (K contiguous), box BK x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows) {
  return encode_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, (uint64_t)K, (uint64_t)rows, (uint64_t)K * 2, BK,
                       (uint32_t)box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

int64_t align256(int64_t v) { return (v + 255) & ~(int64_t)255; }

template <int BN>
cudaError_t launch_ws_gemm(const uint16_t* x16, const uint16_t* w16, const float* act_scale, const int32_t* rowsum,
                           float w_scale, float* out, int32_t* acc_out, int64_t M, int64_t N, int64_t K, int num_sms,
                           cudaStream_t stream) {
  using Cfg = TileCfg<BN>;
  CUtensorMap mA, mB;
  if (!make_map(&mA, x16, M, K, BM) || !make_map(&mB, w16, N, K, BN)) return cudaErrorInvalidValue;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(gemm_f16_ws_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int grid = (int)(tiles < num_sms ? tiles : num_sms);
  gemm_f16_ws_kernel<BN><<<grid, THREADS, Cfg::SMEM_BYTES, stream>>>(mA, mB, act_scale, rowsum, w_scale, out, acc_out,
                                                                     (int)M, (int)N, (int)K);
  return cudaGetLastError();
}

}  // namespace

bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner_elems,
                   uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner_elems, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t read_clear_device_error_gemm_ws(int* value) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

int64_t gemm_ws_bytes(int64_t M, int64_t N, int64_t K) { return align256(M * K * 2) + align256(N * K * 2); }

cudaError_t launch_gemm_tc_ws(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                              float w_scale, float* out, int32_t* acc_out, int64_t M, int64_t N, int64_t K,
                              void* workspace, int num_sms, cudaStream_t stream) {
  uint16_t* x16 = static_cast<uint16_t*>(workspace);
  uint16_t* w16 = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + align256(M * K * 2));
  const int64_t n16 = M * K / 16;
  convert_s8_f16<<<(unsigned)((n16 + 255) / 256 < 152 * 16 ? (n16 + 255) / 256 : 152 * 16), 256, 0, stream>>>(xq, x16,
                                                                                                               n16);
  const int64_t words = N * (K / 16);
  expand_codes_f16<<<(unsigned)((words + 255) / 256 < 152 * 16 ? (words + 255) / 256 : 152 * 16), 256, 0, stream>>>(
      wp, w16, N, K);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // Tile width: the persistent CTAs run the tiles in rounds of num_sms, and a tile's time
  // grows with BN plus a fixed part (operand A's loads and per-step overheads, taken as 32
  // columns' worth), so pick the BN with the least rounds x (BN + 32), ties to the wider.
  // For M = 4096, N = 2560: BN = 256 needs 3 rounds of 320 tiles (2.1 waves), BN = 192 needs
  // 3 rounds of 448 (2.95 waves) at about 0.78 of the time per tile.
  const int64_t num_m = (M + BM - 1) / BM;
  auto cost = [&](int bn) {
    const int64_t tiles = num_m * ((N + bn - 1) / bn);
    return ((tiles + num_sms - 1) / num_sms) * (bn + 32);
  };
  int bn = 256;
  for (int cand : {224, 192, 160, 128})
    if (cost(cand) < cost(bn)) bn = cand;
  switch (bn) {
    case 224: return launch_ws_gemm<224>(x16, w16, act_scale, rowsum, w_scale, out, acc_out, M, N, K, num_sms, stream);
    case 192: return launch_ws_gemm<192>(x16, w16, act_scale, rowsum, w_scale, out, acc_out, M, N, K, num_sms, stream);
    case 160: return launch_ws_gemm<160>(x16, w16, act_scale, rowsum, w_scale, out, acc_out, M, N, K, num_sms, stream);
    case 128: return launch_ws_gemm<128>(x16, w16, act_scale, rowsum, w_scale, out, acc_out, M, N, K, num_sms, stream);
    default: return launch_ws_gemm<256>(x16, w16, act_scale, rowsum, w_scale, out, acc_out, M, N, K, num_sms, stream);
  }
}

}  // namespace bitnet
