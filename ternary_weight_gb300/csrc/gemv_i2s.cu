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
//  * Programmatic dependent launch: the kernel lets the next kernel in the stream launch as
//    soon as it starts and issues its first weight loads before it waits for the previous
//    kernel (griddepcontrol.wait), so back-to-back GEMVs keep HBM busy across the kernel
//    boundary. The activations, scales and row sums are read, and outputs written, only
//    after the wait. A previous kernel that does not trigger early (any kernel but this
//    library's GEMV and group kernels) still completes before this one starts.
#include "bitnet_dev.cuh"

#include <atomic>

namespace bitnet {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxActSmem = 64 * 1024;  // bytes of staged activations per CTA
constexpr int kMaxM1K = 10240;         // largest K of the persistent few-row kernel
// M = 1 takes the bulk-copy ring kernel for packed weights in [kRingMinBytes (kRingMinBytesLongK
// when K >= 4096), kRingMaxBytes]. Measured against the register-prefetch kernel, µs per call in
// back-to-back graphs: 2560 x 6912 (4.4 MB) 3.26 vs 3.60, 13824 x 2560 (8.8 MB) 4.03 vs 4.21,
// 10000 x 8192 (20.5 MB) 5.73 vs 6.27, 8192 x 10240 (21 MB) 5.79 vs 6.77; but 6912 x 2560 (4.4 MB)
// 3.22 vs 2.96, 2560 x 2560 3.14 vs 2.54, and 28672 x 8192 (58.7 MB) 12.73 vs 11.99: a CTA that
// turns the ring twice ends each launch with consumer work on buffered tiles and no copies in
// flight, which the register-prefetch kernel does not.
constexpr int64_t kRingMinBytes = 8LL << 20;
constexpr int64_t kRingMinBytesLongK = 4LL << 20;
constexpr int64_t kRingMaxBytes = 40LL << 20;
constexpr int kColBlock = 5;            // chunk columns a lane loads at once (the lane layout keeps
                                        // a row's walk at 5 columns when K <= 10240)

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

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
  pdl_launch_dependents();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int G = 1 << log2G;
  const int kl = lane & (G - 1);
  const int rg = lane >> log2G;
  const int rows_per_tile = (32 >> log2G) * R;
  const int64_t tile = (int64_t)blockIdx.x * kWarps + warp;
  const bool live = tile * rows_per_tile < N;  // warp-uniform
  const int64_t nbase = tile * rows_per_tile + (int64_t)rg * R;
  const int T = (C + G - 1) >> log2G;  // chunks per lane per row (the last may be ragged)

  const uint4* wrow[R];
  bool rv[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    rv[r] = live && (nbase + r) < N;
    wrow[r] = reinterpret_cast<const uint4*>(wp + (rv[r] ? (nbase + r) : 0) * (int64_t)(K >> 2));
  }
  // Weight chunks are loaded kColBlock columns x R rows at a time, all issued before any is
  // used (up to 320 bytes in flight per lane: HBM needs on the order of 100 KB in flight per
  // SM). The first block is loaded before the wait for the previous kernel in the stream:
  // the packed weights are read-only model state, the activations may be that kernel's output.
  uint4 w[kColBlock][R];
  auto load_block = [&](int t0) {
#pragma unroll
    for (int u = 0; u < kColBlock; ++u) {
      const int c = kl + ((t0 + u) << log2G);
#pragma unroll
      for (int r = 0; r < R; ++r) w[u][r] = (rv[r] && c < C) ? ldg_stream(wrow[r] + c) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  load_block(0);
  pdl_wait();

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
  if (!live) return;  // warp-uniform; no block barrier follows

  int acc[R][MT][4];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[r][m][j] = 0;

  for (int t0 = 0; t0 < T; t0 += kColBlock) {
    if (t0 > 0) load_block(t0);
#pragma unroll
    for (int u = 0; u < kColBlock; ++u) {
      if (t0 + u >= T) break;  // uniform: the walk is shorter than the block
      // a ragged last column past the row's end has zero weights (it adds nothing); its
      // activation load is clamped into the staged row
      const int c = min(kl + ((t0 + u) << log2G), C - 1);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 a = *reinterpret_cast<const uint4*>(act + m * K + j * plane + c * 16);
          const uint32_t mask = 0xC0C0C0C0u >> (2 * j);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            int s = acc[r][m][j];
            s = dp4a_us(w[u][r].x & mask, a.x, s);
            s = dp4a_us(w[u][r].y & mask, a.y, s);
            s = dp4a_us(w[u][r].z & mask, a.z, s);
            s = dp4a_us(w[u][r].w & mask, a.w, s);
            acc[r][m][j] = s;
          }
        }
      }
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


// ---------------------------------------------------------------------------------------
// M <= 8 token rows (MT, a power of two), K <= 10240: persistent kernel with a register double
// buffer. Each weight word is masked once into its bit-pair operands and applied to all MT
// rows (dp4a per row), so the streaming structure of the single-row case carries over.
// Warp w of the grid takes warp tiles w, w + W, w + 2W, ... (W = warps in the grid); a warp
// tile is rpw row groups x R rows, and each lane owns the TB chunk columns c = kl + G*u of its
// R rows (TB = the walk length, at most 5). While the lane computes one tile, the loads of its
// next tile are in flight: 4 or 5 16-byte chunks per lane, with four CTAs (32 warps) per SM
// about 64 KB per SM, which keeps HBM streaming without any shared-memory staging of the
// weights. The MT activation rows are
// staged once per CTA in shared memory (each [j][c][16] plus a zero column at c = C that the
// ragged lanes of a 32-lane layout read); rows past M are zero and never written out.
// ---------------------------------------------------------------------------------------
template <int MT, int R, int TB, int LB>
__global__ void __launch_bounds__(kThreads, LB) gemv_m1_kernel(const int8_t* __restrict__ xq,
                                                              const float* __restrict__ act_scale,
                                                              const int32_t* __restrict__ rowsum,
                                                              const uint8_t* __restrict__ wp, float w_scale,
                                                              float* __restrict__ out, int32_t* __restrict__ acc_out,
                                                              int M, int N, int K, int log2G) {
  extern __shared__ __align__(16) uint8_t act[];  // MT rows x 4 planes x (C + 1) x 16 bytes
  const int C = K >> 6;
  const int plane = (C + 1) * 16;
  const int act_row = 4 * plane;
  pdl_launch_dependents();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int G = 1 << log2G;
  const int kl = lane & (G - 1);
  const int rg = lane >> log2G;
  const int rows_per_tile = (32 >> log2G) * R;
  const int n_tiles = (N + rows_per_tile - 1) / rows_per_tile;
  const int stride = gridDim.x * kWarps;
  const int row_chunks = C;  // 16-byte chunks per packed row (K/4 bytes)
  const uint4* wbase = reinterpret_cast<const uint4*>(wp);

  // chunk (u, r) of warp tile `tile` for this lane, or zero past the matrix
  auto load_tile = [&](int tile, uint4 (&buf)[TB][R]) {
    const int n0 = tile * rows_per_tile + rg * R;
#pragma unroll
    for (int u = 0; u < TB; ++u) {
      const int c = kl + (u << log2G);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const bool ok = tile < n_tiles && n0 + r < N && c < C;
        buf[u][r] = ok ? ldg_stream(wbase + (int64_t)(n0 + r) * row_chunks + c) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };

  uint4 bufA[TB][R], bufB[TB][R];
  int tile = blockIdx.x * kWarps + warp;
  // the first tile is loaded before the wait for the previous kernel in the stream: the
  // packed weights are read-only model state, the activations may be that kernel's output
  load_tile(tile, bufA);
  pdl_wait();
  {
    const int pieces = K >> 4;  // piece p covers k = 16p..16p+15
    if constexpr (MT == 1) {
      for (int p = threadIdx.x; p < pieces; p += kThreads) {
        const int i = p >> 3, j = (p >> 1) & 3, h = p & 1;
        *reinterpret_cast<uint4*>(act + j * plane + (2 * i + h) * 16) = __ldg(reinterpret_cast<const uint4*>(xq) + p);
      }
    } else {
      for (int idx = threadIdx.x; idx < MT * pieces; idx += kThreads) {
        const int m = idx / pieces, p = idx - m * pieces;
        const int i = p >> 3, j = (p >> 1) & 3, h = p & 1;
        const uint4 v =
            m < M ? __ldg(reinterpret_cast<const uint4*>(xq + (int64_t)m * K) + p) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(act + m * act_row + j * plane + (2 * i + h) * 16) = v;
      }
    }
    if (threadIdx.x < 4 * MT)
      *reinterpret_cast<uint4*>(act + (threadIdx.x >> 2) * act_row + (threadIdx.x & 3) * plane + C * 16) =
          make_uint4(0u, 0u, 0u, 0u);
  }
  int rs[MT];
  float sx[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    rs[m] = (MT == 1 || m < M) ? __ldg(rowsum + m) : 0;
    sx[m] = (MT == 1 || m < M) ? __ldg(act_scale + m) : 1.0f;
  }
  __syncthreads();

  auto compute_store = [&](int t, const uint4 (&buf)[TB][R]) {
    int acc[MT][R][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[m][r][j] = 0;
#pragma unroll
    for (int u = 0; u < TB; ++u) {
      const int c = kl + (u << log2G);
      const int ca = c < C ? c : C;  // a ragged column reads the zero column
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t mask = 0xC0C0C0C0u >> (2 * j);
        // the masked operands of this bit pair, shared by the MT rows
        uint4 wm[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
          wm[r] = make_uint4(buf[u][r].x & mask, buf[u][r].y & mask, buf[u][r].z & mask, buf[u][r].w & mask);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const uint4 a = *reinterpret_cast<const uint4*>(act + m * act_row + j * plane + ca * 16);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            int v = acc[m][r][j];
            v = dp4a_us(wm[r].x, a.x, v);
            v = dp4a_us(wm[r].y, a.y, v);
            v = dp4a_us(wm[r].z, a.z, v);
            v = dp4a_us(wm[r].w, a.w, v);
            acc[m][r][j] = v;
          }
        }
      }
    }
    const int n0 = t * rows_per_tile + rg * R;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        int raw = (acc[m][r][0] >> 6) + (acc[m][r][1] >> 4) + (acc[m][r][2] >> 2) + acc[m][r][3];
        for (int o = G >> 1; o > 0; o >>= 1) raw += __shfl_xor_sync(0xffffffffu, raw, o);
        if (kl == 0 && n0 + r < N && (MT == 1 || m < M)) {
          const int a = raw - rs[m];
          const int64_t idx = (int64_t)m * N + n0 + r;
          out[idx] = __fmul_rn(__fdiv_rn(__int2float_rn(a), sx[m]), w_scale);
          if (acc_out) acc_out[idx] = a;
        }
      }
    }
  };

  // two tiles per trip, so the buffers swap roles without copies; tile < n_tiles is
  // warp-uniform, so the shuffles in compute_store see full warps
  for (; tile < n_tiles; tile += 2 * stride) {
    load_tile(tile + stride, bufB);
    compute_store(tile, bufA);
    if (tile + stride >= n_tiles) break;
    load_tile(tile + 2 * stride, bufA);
    compute_store(tile + stride, bufB);
  }
}

template <int MT, int R, int TB, int LB>
cudaError_t launch_m1(const int8_t* xq, const float* s, const int32_t* rs, const uint8_t* wp, float w_scale,
                      float* out, int32_t* acc_out, int M, int N, int K, int log2G, int num_sms, cudaStream_t stream) {
  auto kern = gemv_m1_kernel<MT, R, TB, LB>;
  const int smem = MT * (K + 64);
  if (smem > 48 * 1024) {
    // per-device opt-in to this instantiation's largest staging size, set once
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, MT * (kMaxM1K + 64));
      if (e != cudaSuccess) return e;
      configured.fetch_or(bit, std::memory_order_acq_rel);
    }
  }
  const int rows_per_tile = (32 >> log2G) * R;
  const int64_t tiles = ((int64_t)N + rows_per_tile - 1) / rows_per_tile;
  int64_t blocks = (tiles + kWarps - 1) / kWarps;
  if (blocks > (int64_t)LB * num_sms) blocks = (int64_t)LB * num_sms;  // persistent: LB CTAs per SM
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, xq, s, rs, wp, w_scale, out, acc_out, M, N, K, log2G);
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((tiles + kWarps - 1) / kWarps), (unsigned)((M + MT - 1) / MT));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, xq, s, rs, wp, w_scale, out, acc_out, M, N, K, log2G);
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

  // large single-token matrices: the bulk-copy ring kernel (the copy engine streams the weights,
  // every warp of the CTA is free for the dp4a work)
  const int64_t wbytes = (int64_t)N * (K / 4);
  if (M == 1 && gemv_ring_supported(M, K) && wbytes >= (K >= 4096 ? kRingMinBytesLongK : kRingMinBytes) &&
      wbytes <= kRingMaxBytes)
    return launch_gemv_ring(xq, act_scale, rowsum, wp, w_scale, out, acc_out, N, K, num_sms, stream);

  if (M == 1 && K <= 10240) {
    // walk length T <= 5 (the lane layout above). Large matrices (at least two tiles per
    // warp at four CTAs per SM): tiles of 2 to 5 chunks per lane, so the double buffer fits
    // in 64 registers and four CTAs (32 warps, about 64 KB of loads in flight) share an SM.
    // Smaller ones: two CTAs per SM and tiles of 5 to 8 chunks per lane (measured: 5 beats
    // 10 for the 8-lane K = 2560 layouts).
    const int T = (C + (1 << log2G) - 1) >> log2G;
    const int rpw1 = 32 >> log2G;
    const int64_t tiles_r1 = ((int64_t)N + rpw1 - 1) / rpw1;
    const bool large = tiles_r1 >= 2LL * 4 * kWarps * num_sms;
#define BITNET_M1(R_, TB_, LB_) \
  launch_m1<1, R_, TB_, LB_>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, 1, N, K, log2G, num_sms, stream)
    if (large) {
      switch (T) {
        case 1: return BITNET_M1(2, 1, 4);
        case 2: return BITNET_M1(2, 2, 4);
        case 3: return BITNET_M1(1, 3, 4);
        case 4: return BITNET_M1(1, 4, 4);
        default: return BITNET_M1(1, 5, 4);
      }
    }
    switch (T) {
      case 1: return BITNET_M1(8, 1, 2);
      case 2: return BITNET_M1(4, 2, 2);
      case 3: return BITNET_M1(2, 3, 2);
      case 4: return BITNET_M1(2, 4, 2);
      default: return BITNET_M1(1, 5, 2);
    }
#undef BITNET_M1
  }

  // 2 to 8 token rows, K <= 10240: the same persistent kernel with MT staged rows (M rounded up
  // to a power of two), each masked weight word applied to every row. The accumulators of MT
  // rows need more registers: two CTAs per SM for 2 and 4 rows, one for 8 (which is bound by
  // its dp4a work rather than by the loads in flight). Measured against the per-tile kernel
  // below, it wins up to 4 rows (N 6912, K 2560: 4.1 against 5.1 us at M = 2; N 2560, K 6912:
  // 8.0 against 10.5 us at M = 4), and from 5 to 8 rows only at long K (15.2 against 15.8 us
  // at M = 8, K 6912; 10.8 against 9.9 us at M = 8, K 2560).
  //
  // With walks of 4 or 5 chunks, each lane takes two weight rows: every 16-byte activation load
  // from shared memory then serves two rows, which halves the activation reads (at one row per
  // lane, N 6912, K 2560, M = 4 reads ~70 MB of shared memory, ~1.8 us of its bandwidth). The
  // occupancy that suits it follows the lane layout (us, bit-identical):
  //  * 32 lanes per row (K 6912): two CTAs per SM; M = 4 8.0 -> 7.5, M = 2 5.25 -> 5.0;
  //  * fewer lanes per row, several row groups per warp (K 2560): one CTA per SM for 3-4 rows
  //    (6.2 -> 5.8 at M = 4, 5.9 -> 5.5 at M = 3; two CTAs per SM were slower, 7.3); 2 rows keep
  //    one row per lane (4.2 against 4.8).
  if (M >= 2 && K <= kMaxM1K && (M <= 4 || (M <= 8 && K >= 4096))) {
    const int T = (C + (1 << log2G) - 1) >> log2G;
    const bool wide = log2G == 5;  // 32 lanes per row
#define BITNET_MT(MT_, R_, TB_, LB_) \
  launch_m1<MT_, R_, TB_, LB_>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, log2G, num_sms, stream)
#define BITNET_MT_T(MT_, LB_)                                       \
  switch (T) {                                                       \
    case 1: return BITNET_MT(MT_, 1, 1, LB_);                        \
    case 2: return BITNET_MT(MT_, 1, 2, LB_);                        \
    case 3: return BITNET_MT(MT_, 1, 3, LB_);                        \
    case 4: return BITNET_MT(MT_, 1, 4, LB_);                        \
    default: return BITNET_MT(MT_, 1, 5, LB_);                       \
  }
    if (M <= 4 && T >= 4 && (wide || M > 2)) {
      const int lb = wide ? 2 : 1;
      if (M <= 2) return T == 4 ? BITNET_MT(2, 2, 4, 2) : BITNET_MT(2, 2, 5, 2);
      if (lb == 2) return T == 4 ? BITNET_MT(4, 2, 4, 2) : BITNET_MT(4, 2, 5, 2);
      return T == 4 ? BITNET_MT(4, 2, 4, 1) : BITNET_MT(4, 2, 5, 1);
    }
    if (M <= 2) BITNET_MT_T(2, 2)
    if (M <= 4) BITNET_MT_T(4, 2)
    BITNET_MT_T(8, 1)
#undef BITNET_MT_T
#undef BITNET_MT
  }

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
