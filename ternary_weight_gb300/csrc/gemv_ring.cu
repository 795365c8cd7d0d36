// gemv_ring.cu -- the single-token W2A8 GEMV for large matrices: one CTA per SM streams its
// slice of the weight rows through a shared-memory ring of bulk copies.
//
// Computes, like every other path of the library, raw[n] = sum_k code[n][k] * xq[k],
// acc = raw - rowsum, out = (acc / s) * w_scale, with the same integers and the same fp32
// operations. Sources: the raw code dot over the 4x32-interleaved i2_s bytes ("[분석/검증-3]
// BitNet.cpp ARM 커널 재작성" §3), the byte layout ("BitNet 딥다이브" §4-2), the dequantisation
// ("bitnet.rs" "Quantised Forward Pass").
//
// Why a second M = 1 kernel: the register-double-buffer GEMV issues its 128-bit loads from the
// warps that also run the dp4a work, and on a 58.7 MB matrix it reaches 72% of the measured HBM
// bandwidth. Streaming by the copy engine into shared memory, as the persistent sweep kernel
// does for a whole decode step, frees the consumer warps for the arithmetic. Here:
//  * CTA b of G owns the rows [N b / G, N (b + 1) / G), cut into tiles of S steps of rpw rows
//    (at most 13.5 KB; the lane layout and S follow the sweep kernel's rule for K);
//  * warp 16, one lane, issues cp.async.bulk copies of consecutive tiles into a 16-slot ring,
//    each slot completing on its own mbarrier by transaction bytes. The weights do not depend
//    on the previous kernel, so the first 16 tiles are requested at once: with programmatic
//    dependent launch they stream while the previous kernel finishes;
//  * warps 0-15 wait for the previous kernel (griddepcontrol.wait), place the int8 row in the
//    four activation planes of the shared dp4a tile routine (gemv_tile.cuh), then take tile i
//    on warp i % 16: wait, dot products, epilogue, release.
// Every wait is bounded; a timeout is recorded in the device error word, the consumers stop and
// the producer waits (bounded) for the copies it issued before the CTA exits.
#include "gemv_tile.cuh"

#include <atomic>

namespace bitnet {
namespace {

constexpr int kRgConsumerWarps = 16;
constexpr int kRgConsumers = kRgConsumerWarps * 32;
constexpr int kRgThreads = kRgConsumers + 32;
constexpr int kRgSlots = 16;
constexpr int kRgSlotBytes = 13824;  // the sweep kernel's tile bound (SweepGroup layout rule)
constexpr int kRgRingBytes = kRgSlots * kRgSlotBytes;
constexpr int kRgMaxK = 10240;
constexpr int kRgSmem = kRgRingBytes + kRgMaxK + 64;
static_assert(kRgSlots % kRgConsumerWarps == 0, "each ring slot must belong to one consumer warp");
static_assert(kRgSmem + 512 <= 227 * 1024, "ring + planes + static shared memory");

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

template <int S>
__device__ __forceinline__ TileDot ring_tile(uint32_t tile_lane, uint32_t xq_u, int plane, int C, int T, int kl,
                                             int log2G, int rg, int rpw, int step_stride) {
  return tile_raw_dots<S>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride);
}

__global__ void __launch_bounds__(kRgThreads, 1) gemv_ring_kernel(const int8_t* __restrict__ xq,
                                                                  const float* __restrict__ act_scale,
                                                                  const int32_t* __restrict__ rowsum,
                                                                  const uint8_t* __restrict__ wp, float w_scale,
                                                                  float* __restrict__ out,
                                                                  int32_t* __restrict__ acc_out, int N, int K,
                                                                  int log2G, int S) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;                  // kRgSlots x kRgSlotBytes
  uint8_t* xq_s = smem + kRgRingBytes;   // the activation planes, K + 64 bytes
  __shared__ __align__(8) uint64_t full_bar[kRgSlots];
  __shared__ __align__(8) uint64_t empty_bar[kRgSlots];

  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int begin = (int)((int64_t)N * blockIdx.x / gridDim.x);
  const int end = (int)((int64_t)N * (blockIdx.x + 1) / gridDim.x);
  const int row_bytes = K >> 2, rpw = 32 >> log2G, TR = S * rpw;
  const int n_tiles = (end - begin + TR - 1) / TR;
  if (threadIdx.x < kRgSlots) {  // one barrier pair per thread
    mbar_init(&full_bar[threadIdx.x], 1);
    mbar_init(&empty_bar[threadIdx.x], 1);
    fence_mbar_init();
  }
  __syncthreads();
  bool abort = false;

  if (warp == kRgConsumerWarps) {
    // ================================ producer ================================
    if (lane == 0) {
      int issued = 0;
      for (; issued < n_tiles; ++issued) {
        const int slot = issued % kRgSlots, use = issued / kRgSlots;
        if (use > 0 && !mbar_wait(&empty_bar[slot], (uint32_t)(use - 1) & 1u, &abort)) break;
        const int r0 = begin + issued * TR;
        const int rows = min(TR, end - r0);
        const uint32_t bytes = (uint32_t)rows * (uint32_t)row_bytes;
        mbar_arrive_expect_tx(&full_bar[slot], bytes);
        bulk_copy_g2s(ring + slot * kRgSlotBytes, wp + (int64_t)r0 * row_bytes, bytes, &full_bar[slot]);
      }
      {  // every copy this CTA issued lands before the producer leaves: the consumers may have
         // given up on a full barrier (a bounded wait) while copies were still in flight
        bool dummy = false;
        for (int i = issued - kRgSlots > 0 ? issued - kRgSlots : 0; i < issued; ++i)
          mbar_wait(&full_bar[i % kRgSlots], (uint32_t)(i / kRgSlots) & 1u, &dummy);
      }
    }
    return;
  }

  // ================================ consumers ================================
  pdl_wait();  // the activations (and the outputs' previous readers) belong to the previous kernel
  const int C = K >> 6, plane = (C + 1) * 16;
  // activation planes: the 16 values k = 16p .. 16p + 15 go to plane j = (k % 128) / 32, chunk
  // c = 2 (k / 128) + (k % 32) / 16 (the chunk that bit pair j of weight chunk c multiplies);
  // chunk C of every plane is zero
  for (int p = threadIdx.x; p < (K >> 4); p += kRgConsumers) {
    const int k = p << 4, rem = k & 127;
    const int off = (rem >> 5) * plane + (2 * (k >> 7) + ((rem & 31) >> 4)) * 16;
    *reinterpret_cast<uint4*>(xq_s + off) = __ldg(reinterpret_cast<const uint4*>(xq) + p);
  }
  if (threadIdx.x < 4) *reinterpret_cast<uint4*>(xq_s + threadIdx.x * plane + C * 16) = make_uint4(0u, 0u, 0u, 0u);
  const float s_act = __ldg(act_scale);
  const int rs = __ldg(rowsum);
  named_bar_sync(1, kRgConsumers);  // the planes are written before any tile reads them

  const uint32_t xq_u = smem_u32(xq_s);
  const int G_lanes = 1 << log2G;
  const int kl = lane & (G_lanes - 1), rg = lane >> log2G;
  const int T = (C + G_lanes - 1) >> log2G;
  const int step_stride = rpw * row_bytes;
  for (int i = warp; i < n_tiles; i += kRgConsumerWarps) {
    const int slot = i % kRgSlots, use = i / kRgSlots;
    if (!mbar_wait_warp(&full_bar[slot], (uint32_t)use & 1u, &abort)) break;
    const int r0 = begin + i * TR;
    const int rows = min(TR, end - r0);
    const uint32_t tile_lane = smem_u32(ring + slot * kRgSlotBytes) + (uint32_t)(rg * row_bytes);
    TileDot r;
    switch (S) {
      case 1: r = ring_tile<1>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
      case 2: r = ring_tile<2>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
      case 3: r = ring_tile<3>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
      case 4: r = ring_tile<4>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
      case 5: r = ring_tile<5>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
      case 6: r = ring_tile<6>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
      case 7: r = ring_tile<7>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
      default: r = ring_tile<8>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
    }
    if (r.writer && r.row < rows) {
      const int n = r0 + r.row;
      const int a = r.sum - rs;
      out[n] = __fmul_rn(__fdiv_rn(__int2float_rn(a), s_act), w_scale);
      if (acc_out) acc_out[n] = a;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[slot]);
  }
}

}  // namespace

bool gemv_ring_supported(int64_t M, int64_t K) { return M == 1 && K <= kRgMaxK; }

cudaError_t launch_gemv_ring(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                             float w_scale, float* out, int32_t* acc_out, int64_t N, int64_t K, int num_sms,
                             cudaStream_t stream) {
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(gemv_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRgSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  SweepGroup g = {};  // the sweep kernel's layout rule: lanes per row and steps per tile from K
  g.K = (int)K;
  sweep_fill_layout(g);
  const int grid = (int)(N < num_sms ? N : num_sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kRgThreads);
  cfg.dynamicSmemBytes = kRgSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_ring_kernel, xq, act_scale, rowsum, wp, w_scale, out, acc_out, (int)N,
                            (int)K, g.log2G, g.S);
}

cudaError_t read_clear_device_error_gemv_ring(int* value) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

}  // namespace bitnet
