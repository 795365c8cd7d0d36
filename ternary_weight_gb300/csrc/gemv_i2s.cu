// gemv_i2s.cu -- decode GEMV (small M): i2_s packed ternary weights x int8 activations.
//
// What it computes (per output (m, n)):
//   raw = sum_k code[n][k] * xq[m][k]       codes 0/1/2 multiplied as stored
//   acc = raw - rowsum[m]                   = sum_k (code - 1) * xq, an identity
//   out = (acc / s[m]) * w_scale
// Sources: "[분석/검증-3] BitNet.cpp ARM 커널 재작성" §3 and "[기술 분석 보고서] ARM64 ... 추론 붕괴
// 원인 분석" §3.1-§4 (the 4x32 interleave and the raw code dot over the packed bytes);
// "BitNet 딥다이브" §4-2 (byte layout), §4-3 (_Nx1: decode the weights once and reuse them for
// several activation columns); "bitnet.rs" "Quantised Forward Pass" (dequantisation).
//
// Design (HBM-bound weight streaming):
//  * A packed row is K/4 bytes = C = K/64 chunks of 16 bytes. Chunk c is half of i2_s
//    block i = c/2 (bytes 16h..16h+15, h = c%2); its 32-bit word q holds, in bit pair j
//    (j = 0 at bits 7:6), the codes of k = 128i + 32j + 16h + 4q + (0..3).
//  * Instead of shifting, each word is masked four times (0xC0.., 0x30.., 0x0C.., 0x03..)
//    and dp4a'd (unsigned codes x signed int8) into four accumulators that are exact
//    multiples of 64, 16, 4 and 1; they are combined once at the end. 4 LOP + 4 dp4a per
//    16 weights.
//  * Activations of MT rows are staged once per CTA in shared memory, re-laid out as
//    [m][j][c][16 bytes] so that the 16 activation bytes paired with bit pair j of chunk c
//    are one conflict-free 16-byte load, shared by the R weight rows a lane handles.
//  * A warp works on a tile of (32/G)*R rows: G lanes per row group walk the row's chunks
//    (c = lane_in_group + G*t; G is the largest power of two <= 32 dividing C while that keeps
//    the walk at most 5 chunks, else 32 with a predicated ragged last chunk), each lane owning
//    R rows. Weight chunks are streamed with 128-bit
//    non-allocating loads, one chunk ahead (2*R loads in flight per lane). Partial sums
//    are reduced with xor-shuffles inside the G-lane group.
#include "bitnet_dev.cuh"

#include <atomic>

namespace bitnet {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxActSmem = 64 * 1024;  // bytes of staged activations per CTA

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int MT, int R>
__global__ void __launch_bounds__(kThreads) gemv_i2s_kernel(const int8_t* __restrict__ xq,
                                                            const float* __restrict__ act_scale,
                                                            const int32_t* __restrict__ rowsum,
                                                            const uint8_t* __restrict__ wp, float w_scale,
                                                            float* __restrict__ out, int32_t* __restrict__ acc_out,
                                                            int M, int N, int K, int log2G) {
  extern __shared__ __align__(16) uint8_t act[];  // MT x K bytes, [m][j][c][16]
  const int m0 = blockIdx.y * MT;
  const int C = K >> 6;
  const int plane = K >> 2;  // bytes per j-plane of one staged row

  // ---- stage MT activation rows (rows past M read as zero) ----
  {
    const int pieces = K >> 4;  // 16-byte pieces per row; piece p covers k = 16p..16p+15
    for (int idx = threadIdx.x; idx < MT * pieces; idx += kThreads) {
      const int m = idx / pieces, p = idx - m * pieces;
      const int i = p >> 3, j = (p >> 1) & 3, h = p & 1;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (m0 + m < M) v = __ldg(reinterpret_cast<const uint4*>(xq + (int64_t)(m0 + m) * K) + p);
      *reinterpret_cast<uint4*>(act + m * K + j * plane + (2 * i + h) * 16) = v;
    }
  }
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int G = 1 << log2G;
  const int kl = lane & (G - 1);
  const int rg = lane >> log2G;
  const int rows_per_tile = (32 >> log2G) * R;
  const int64_t tile = (int64_t)blockIdx.x * kWarps + warp;
  if (tile * rows_per_tile >= N) return;  // warp-uniform; no block barrier follows
  const int64_t nbase = tile * rows_per_tile + (int64_t)rg * R;
  const int T = (C + G - 1) >> log2G;  // chunks per lane per row (the last may be ragged)

  const uint4* wrow[R];
  bool rv[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    rv[r] = (nbase + r) < N;
    wrow[r] = reinterpret_cast<const uint4*>(wp + (rv[r] ? (nbase + r) : 0) * (int64_t)(K >> 2));
  }

  int acc[R][MT][4];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[r][m][j] = 0;

  uint4 cur[R];
#pragma unroll
  for (int r = 0; r < R; ++r) cur[r] = (rv[r] && kl < C) ? ldg_stream(wrow[r] + kl) : make_uint4(0u, 0u, 0u, 0u);

  for (int t = 0; t < T; ++t) {
    const int c = kl + (t << log2G);
    uint4 nxt[R];
    if (t + 1 < T) {
#pragma unroll
      for (int r = 0; r < R; ++r)
        nxt[r] = (rv[r] && c + G < C) ? ldg_stream(wrow[r] + c + G) : make_uint4(0u, 0u, 0u, 0u);
    }
    if (c < C) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 a = *reinterpret_cast<const uint4*>(act + m * K + j * plane + c * 16);
        const uint32_t mask = 0xC0C0C0C0u >> (2 * j);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          int s = acc[r][m][j];
          s = dp4a_us(cur[r].x & mask, a.x, s);
          s = dp4a_us(cur[r].y & mask, a.y, s);
          s = dp4a_us(cur[r].z & mask, a.z, s);
          s = dp4a_us(cur[r].w & mask, a.w, s);
          acc[r][m][j] = s;
        }
      }
    }
    }
    if (t + 1 < T) {
#pragma unroll
      for (int r = 0; r < R; ++r) cur[r] = nxt[r];
    }
  }

  // ---- combine the four bit-pair accumulators, reduce over the G lanes, epilogue ----
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      int raw = (acc[r][m][0] >> 6) + (acc[r][m][1] >> 4) + (acc[r][m][2] >> 2) + acc[r][m][3];
      for (int o = G >> 1; o > 0; o >>= 1) raw += __shfl_xor_sync(0xffffffffu, raw, o);
      if (kl == 0 && rv[r] && (m0 + m) < M) {
        const int64_t idx = (int64_t)(m0 + m) * N + (nbase + r);
        const int a = raw - __ldg(rowsum + m0 + m);
        out[idx] = __fmul_rn(__fdiv_rn(__int2float_rn(a), __ldg(act_scale + m0 + m)), w_scale);
        if (acc_out) acc_out[idx] = a;
      }
    }
  }
}

template <int MT, int R>
cudaError_t launch_cfg(const int8_t* xq, const float* s, const int32_t* rs, const uint8_t* wp, float w_scale,
                       float* out, int32_t* acc_out, int M, int N, int K, int log2G, cudaStream_t stream) {
  const int smem = MT * K;
  auto kern = gemv_i2s_kernel<MT, R>;
  if (smem > 48 * 1024) {
    // per-device opt-in to the largest staging size this instantiation can need, set once
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxActSmem);
      if (e != cudaSuccess) return e;
      configured.fetch_or(bit, std::memory_order_acq_rel);
    }
  }
  const int rows_per_tile = (32 >> log2G) * R;
  const int64_t tiles = ((int64_t)N + rows_per_tile - 1) / rows_per_tile;
  dim3 grid((unsigned)((tiles + kWarps - 1) / kWarps), (unsigned)((M + MT - 1) / MT));
  kern<<<grid, kThreads, smem, stream>>>(xq, s, rs, wp, w_scale, out, acc_out, M, N, K, log2G);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv_i2s(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                            float w_scale, float* out, int32_t* acc_out, int64_t M64, int64_t N64, int64_t K64,
                            int num_sms, cudaStream_t stream) {
  const int M = (int)M64, N = (int)N64, K = (int)K64;
  const int C = K >> 6;
  // lanes per row: the largest power of two <= 32 dividing C while that keeps at most 5 chunks
  // per lane, else 32 lanes with a ragged (predicated) last chunk
  int log2G = 5;
  while (log2G > 1 && (C & ((1 << log2G) - 1)) != 0) --log2G;  // C is even, so G >= 2 divides it
  if ((C >> log2G) > 5) log2G = 5;
  const int rpw = 32 >> log2G;

  // activation rows per CTA: next power of two >= M, at most 8, within the smem budget
  int MT = 1;
  while (MT < M && MT < 8) MT <<= 1;
  while (MT > 1 && (int64_t)MT * K > kMaxActSmem) MT >>= 1;

  // rows per lane: as many as keep >= 4 resident CTAs of work per SM
  auto ctas = [&](int R) { return (((int64_t)N + rpw * R - 1) / (rpw * R) + kWarps - 1) / kWarps; };
  const int64_t want = 4LL * num_sms;
  switch (MT) {
    case 1:
      if (ctas(4) >= want) return launch_cfg<1, 4>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, log2G, stream);
      if (ctas(2) >= want) return launch_cfg<1, 2>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, log2G, stream);
      return launch_cfg<1, 1>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, log2G, stream);
    case 2:
      if (ctas(4) >= want) return launch_cfg<2, 4>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, log2G, stream);
      if (ctas(2) >= want) return launch_cfg<2, 2>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, log2G, stream);
      return launch_cfg<2, 1>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, log2G, stream);
    case 4:
      if (ctas(2) >= want) return launch_cfg<4, 2>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, log2G, stream);
      return launch_cfg<4, 1>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, log2G, stream);
    default:
      return launch_cfg<8, 1>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, log2G, stream);
  }
}

}  // namespace bitnet
