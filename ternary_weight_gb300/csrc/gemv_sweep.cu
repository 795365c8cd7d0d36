// gemv_sweep.cu -- many single-token projection groups, each with its own activation row, in
// one persistent launch.
//
// What it computes: for every group g (an activation row x_g of K_g values and up to 8 packed
// projections l that consume it), exactly what the single-group call computes:
//   xq = clamp(rne(x_g * s), -127, 127),  s = 127 / max(max|x_g|, 1e-5),  rowsum = sum_k xq[k]
//   out_l[n] = ((sum_k code_l[n][k] * xq[k] - rowsum) / s) * w_scale_l
// ("BitNet 딥다이브" §4-5 and §4-2; "bitnet.rs" "Quantised Forward Pass"). The groups are
// independent: no group reads what another writes in the same launch. That is the batch of
// projections of a decode sweep whose rows are given, not a chain of dependent layers.
//
// Design: the weights of all groups form one row space, which is streamed at HBM rate by one
// CTA per SM.
//  * CTA b owns a contiguous slice of the concatenated rows of every projection of every group
//    (in table order), balanced by packed bytes rather than rows (rows of different K differ
//    in size: 640 bytes at K = 2560, 1728 at 6912). The slice is cut into tiles of whole rows
//    (<= 13.5 KB, never across two projections).
//  * Warp 16 is the producer: one lane issues cp.async.bulk copies of consecutive tiles into a
//    16-slot x 13.5 KB shared-memory ring (216 KB, about 33 MB in flight over the GPU), each
//    slot completing on its own mbarrier by transaction bytes. It runs ahead across group
//    boundaries, bounded only by the ring.
//  * Warps 0-15 are consumers; tile i goes to warp i % 16 (one waiter per slot, in order).
//    They take the groups of the slice one at a time. They quantise the group's row into the
//    shared activation planes (the row was pulled into L2 at kernel start), then run the
//    shared dp4a tile routine (gemv_tile.cuh) on the group's tiles. A barrier among the
//    consumers then frees the planes for the next group.
//  * Every wait is bounded. A timeout is recorded in the device error word, and the kernel
//    leaves consistently: consumers stop at the next group boundary, and the producer waits
//    (bounded) for the copies it issued.
#include "gemv_tile.cuh"

#include <atomic>

namespace bitnet {
namespace {

constexpr int kSwConsumerWarps = 16;
constexpr int kSwConsumers = kSwConsumerWarps * 32;
constexpr int kSwThreads = kSwConsumers + 32;
constexpr int kSwSlots = 16;
// 13.5 KB slots: a tile of K = 6912 rows holds 8 steps (13.8 KB), one of K = 2560 rows 5 steps
// of 4 rows (12.8 KB); the ring and the largest activation planes just fit the 227 KB a CTA
// may use. Fewer, larger tiles cut the per-tile overhead (wait, reduce, epilogue, release):
// on the 2B-4T sweep 91 us against 102 us with 12 KB slots and at most 6 steps.
constexpr int kSwSlotBytes = 13824;
constexpr int kSwRingBytes = kSwSlots * kSwSlotBytes;
constexpr int kSwMaxK = 10240;
constexpr int kSwMaxS = 8;        // steps per tile, at most (the tile routine takes up to 8)
constexpr int kSwUnrollMaxS = 6;  // the column loop is unrolled for tiles of up to this many steps
static_assert(kSwMaxS >= 1 && kSwMaxS <= 8, "steps per tile");
constexpr int kSwMaxVec = kSwMaxK / 4 / kSwConsumers;  // fp32 16-byte vectors per thread
static_assert(kSwSlots % kSwConsumerWarps == 0, "each ring slot must belong to one consumer warp");
static_assert(kSwMaxK / 64 <= 32 * kMaxColsPerLane, "column loop bound");
// (the static shared memory, barriers and slot tables, is 640 bytes)
static_assert(kSwRingBytes + kSwMaxK + 64 + 768 <= 227 * 1024, "ring + planes + static shared memory");

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// tiles of group g inside the row slice [begin, end): whole-row runs of at most TR rows that
// never cross a projection
__device__ __forceinline__ int group_tiles(const SweepGroup& G, int begin, int end) {
  const int TR = G.S << (5 - G.log2G);
  int n = 0, off = G.row0;
  for (int j = 0; j < G.count; ++j) {
    const int lo = max(off, begin), hi = min(off + G.N[j], end);
    if (hi > lo) n += (hi - lo + TR - 1) / TR;
    off += G.N[j];
  }
  return n;
}

template <int S>
__device__ __forceinline__ TileDot sweep_tile(uint32_t tile_lane, uint32_t xq_u, int plane, int C, int T, int kl,
                                              int log2G, int rg, int rpw, int step_stride) {
  constexpr int kUnroll = S <= kSwUnrollMaxS ? kMaxColsPerLane : 1;
  return tile_raw_dots<S, kUnroll>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride);
}

template <bool BF16>
__global__ void __launch_bounds__(kSwThreads, 1) gemv_sweep_kernel(const SweepGroup* __restrict__ groups,
                                                                   const SweepSlice* __restrict__ slices,
                                                                   int n_groups) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;                   // kSwSlots x kSwSlotBytes
  uint8_t* xq_s = smem + kSwRingBytes;    // the current group's activation planes, K + 64 bytes
  __shared__ __align__(8) uint64_t full_bar[kSwSlots];
  __shared__ __align__(8) uint64_t empty_bar[kSwSlots];
  __shared__ float red_f[kSwConsumerWarps];
  __shared__ int red_i[kSwConsumerWarps];
  __shared__ int slot_rows[kSwSlots];
  __shared__ float* slot_out[kSwSlots];
  __shared__ float slot_ws[kSwSlots];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const SweepSlice slice = slices[blockIdx.x];
  const int begin = slice.begin, end = slice.end, g0 = slice.g0;
  if (threadIdx.x < kSwSlots) {  // one barrier pair per thread
    mbar_init(&full_bar[threadIdx.x], 1);
    mbar_init(&empty_bar[threadIdx.x], 1);
    fence_mbar_init();
  }
  // (an empty slice, begin == end, touches no group: every loop below stops at row0 >= end or
  // finds no tile)
  // pull the activation rows of the slice's groups into L2 while the weights start streaming
  if (warp == 0) {
    for (int g = g0 + lane; g < n_groups && groups[g].row0 < end; g += 32)
      prefetch_l2(groups[g].x, (uint32_t)groups[g].K * (BF16 ? 2u : 4u));
  }
  __syncthreads();
  bool abort = false;

  if (warp == kSwConsumerWarps) {
    // ================================ producer ================================
    if (lane == 0) {
      int issued = 0;
      for (int g = g0; g < n_groups && !abort; ++g) {
        const SweepGroup& G = groups[g];
        if (G.row0 >= end) break;
        const int row_bytes = G.K >> 2;
        const int TR = G.S << (5 - G.log2G);
        int off = G.row0;
        for (int j = 0; j < G.count && !abort; ++j) {
          int r = max(off, begin);
          const int hi = min(off + G.N[j], end);
          for (; r < hi; r += TR) {
            const int rows = min(TR, hi - r);
            const int slot = issued % kSwSlots, use = issued / kSwSlots;
            if (use > 0 && !mbar_wait(&empty_bar[slot], (use - 1) & 1, &abort)) break;
            slot_out[slot] = G.out[j] + (r - off);
            slot_ws[slot] = G.w_scale[j];
            slot_rows[slot] = rows;
            const uint32_t bytes = (uint32_t)rows * (uint32_t)row_bytes;
            mbar_arrive_expect_tx(&full_bar[slot], bytes);
            bulk_copy_g2s(ring + slot * kSwSlotBytes, G.wp[j] + (int64_t)(r - off) * row_bytes, bytes,
                          &full_bar[slot]);
            ++issued;
          }
          off += G.N[j];
        }
      }
      {  // every copy this CTA issued lands before the producer leaves: the consumers may have
         // given up on a full barrier (a bounded wait) while copies were still in flight
        bool dummy = false;
        for (int i = issued - kSwSlots > 0 ? issued - kSwSlots : 0; i < issued; ++i)
          mbar_wait(&full_bar[i % kSwSlots], (i / kSwSlots) & 1, &dummy);
      }
    }
    return;
  }

  // ================================ consumers ================================
  const uint32_t xq_u = smem_u32(xq_s);
  int tile_base = 0;
  for (int g = g0; g < n_groups; ++g) {
    const SweepGroup& G = groups[g];
    if (G.row0 >= end) break;
    const int K = G.K, C = K >> 6, log2G = G.log2G, S = G.S;
    const int plane = (C + 1) * 16;
    const int n_tiles = group_tiles(G, begin, end);

    // ---- quantise the group's row into the activation planes: element k goes to
    // [j][c][16] with c = 2*(k/128) + (k%32)/16, j = (k%128)/32; chunk C of every plane is zero
    float s_act;
    int rs_total;
    {
      constexpr int E = BF16 ? 8 : 4;
      const int nvec = K / E;
      const uint4* xv = static_cast<const uint4*>(G.x);
      uint4 xr[kSwMaxVec];
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < kSwMaxVec; ++i) {
        const int v = threadIdx.x + kSwConsumers * i;
        xr[i] = v < nvec ? __ldg(xv + v) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t w4[4] = {xr[i].x, xr[i].y, xr[i].z, xr[i].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if constexpr (BF16) {
            amax = fmaxf(amax, fabsf(__uint_as_float(w4[e] << 16)));
            amax = fmaxf(amax, fabsf(__uint_as_float(w4[e] & 0xFFFF0000u)));
          } else {
            amax = fmaxf(amax, fabsf(__uint_as_float(w4[e])));
          }
        }
      }
      // amax is a non-negative float (fmaxf drops NaN), so its bits order like unsigned ints
      const uint32_t wmax = __reduce_max_sync(0xffffffffu, __float_as_uint(amax));
      if (lane == 0) red_f[warp] = __uint_as_float(wmax);
      if (threadIdx.x < 4) *reinterpret_cast<uint4*>(xq_s + threadIdx.x * plane + C * 16) = make_uint4(0u, 0u, 0u, 0u);
      named_bar_sync(1, kSwConsumers);
      amax = 0.0f;
#pragma unroll
      for (int i = 0; i < kSwConsumerWarps; ++i) amax = fmaxf(amax, red_f[i]);
      s_act = __fdiv_rn(127.0f, fmaxf(amax, 1e-5f));
      uint32_t bsum = 0;
      int nel = 0;
#pragma unroll
      for (int i = 0; i < kSwMaxVec; ++i) {
        const int v = threadIdx.x + kSwConsumers * i;
        if (v < nvec) {
          const uint32_t w4[4] = {xr[i].x, xr[i].y, xr[i].z, xr[i].w};
          uint32_t qb[E];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if constexpr (BF16) {
              qb[2 * e] = quant_bits(__uint_as_float(w4[e] << 16), s_act);
              qb[2 * e + 1] = quant_bits(__uint_as_float(w4[e] & 0xFFFF0000u), s_act);
            } else {
              qb[e] = quant_bits(__uint_as_float(w4[e]), s_act);
            }
          }
#pragma unroll
          for (int e = 0; e < E; ++e) bsum += qb[e];
          nel += E;
          const int k = v * E;
          const int rem = k & 127;
          const int off = (rem >> 5) * plane + (2 * (k >> 7) + ((rem & 31) >> 4)) * 16 + (rem & 15);
          const uint32_t word0 =
              __byte_perm(__byte_perm(qb[0], qb[1], 0x0040), __byte_perm(qb[2], qb[3], 0x0040), 0x5410);
          if constexpr (BF16) {
            const uint32_t word1 =
                __byte_perm(__byte_perm(qb[4], qb[5], 0x0040), __byte_perm(qb[6], qb[7], 0x0040), 0x5410);
            *reinterpret_cast<uint2*>(xq_s + off) = make_uint2(word0, word1);
          } else {
            *reinterpret_cast<uint32_t*>(xq_s + off) = word0;
          }
        }
      }
      const int sum = (int)(bsum - (uint32_t)nel * kRoundMagicBits);
      const int wsum = __reduce_add_sync(0xffffffffu, sum);
      if (lane == 0) red_i[warp] = wsum;
      named_bar_sync(1, kSwConsumers);  // also orders the plane writes before the tile reads
      rs_total = 0;
#pragma unroll
      for (int i = 0; i < kSwConsumerWarps; ++i) rs_total += red_i[i];
    }

    // ---- this warp's tiles of the group: global tile indices tile_base .. tile_base + n_tiles - 1
    const int G_lanes = 1 << log2G;
    const int kl = lane & (G_lanes - 1), rg = lane >> log2G, rpw = 32 >> log2G;
    const int T = (C + G_lanes - 1) >> log2G;
    const int row_bytes = K >> 2;
    const int step_stride = rpw * row_bytes;
    const int first = tile_base + ((warp - tile_base) % kSwConsumerWarps + kSwConsumerWarps) % kSwConsumerWarps;
    for (int i = first; i < tile_base + n_tiles; i += kSwConsumerWarps) {
      const int slot = i % kSwSlots, use = i / kSwSlots;
      if (!mbar_wait_warp(&full_bar[slot], use & 1, &abort)) break;
      const int rows = slot_rows[slot];
      float* const out_row = slot_out[slot];
      const float ws = slot_ws[slot];
      const uint32_t tile_lane = smem_u32(ring + slot * kSwSlotBytes) + (uint32_t)(rg * row_bytes);
      TileDot r;
      switch (S) {
        case 1: r = sweep_tile<1>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
        case 2: r = sweep_tile<2>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
        case 3: r = sweep_tile<3>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
        case 4: r = sweep_tile<4>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
        case 5: r = sweep_tile<5>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
        case 6: r = sweep_tile<6>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
        case 7: r = sweep_tile<(kSwMaxS >= 7 ? 7 : 1)>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
        default: r = sweep_tile<(kSwMaxS >= 8 ? 8 : 1)>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride); break;
      }
      if (r.writer && r.row < rows) {
        const int a = r.sum - rs_total;
        out_row[r.row] = __fmul_rn(__fdiv_rn(__int2float_rn(a), s_act), ws);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[slot]);
    }
    tile_base += n_tiles;
    // every consumer is done with the planes before the next row, and all of them learn of a
    // timeout in any consumer warp at the same barrier, so they leave together
    if (named_bar_or(1, kSwConsumers, abort)) break;
  }
}

// lanes per row: the largest power of two <= 32 dividing C when that keeps at most 5 chunk
// columns per lane, else 32 lanes with a ragged last column (the group kernel's rule)
int sweep_log2g(int K) {
  const int C = K >> 6;
  int log2G = 5;
  while (log2G > 1 && (C & ((1 << log2G) - 1)) != 0) --log2G;
  if ((C >> log2G) > 5) log2G = 5;
  return log2G;
}

}  // namespace

bool gemv_sweep_supported(int64_t K) { return K <= kSwMaxK; }

void sweep_fill_layout(SweepGroup& g) {
  g.log2G = sweep_log2g(g.K);
  const int rpw = 32 >> g.log2G;
  const int step_bytes = (g.K >> 2) * rpw;
  int S = g.log2G >= 3 ? kSwSlotBytes / step_bytes : 1;
  if (S > kSwMaxS) S = kSwMaxS;
  if (S < 1) S = 1;
  g.S = S;
}

// The row at packed-byte position p of the concatenated row space (rounded down to a whole
// row; total_rows at the end). Adjacent CTAs are cut at the same positions, so their slices
// tile the row space exactly.
static int row_at_byte(const SweepGroup* groups, int n_groups, int total_rows, int64_t total_bytes, int64_t p,
                       int* group) {
  if (p >= total_bytes) {
    *group = n_groups - 1;
    return total_rows;
  }
  int g = 0;
  while (g + 1 < n_groups && groups[g + 1].byte0 <= p) ++g;
  const int64_t r = (p - groups[g].byte0) / (groups[g].K >> 2);
  *group = g;
  return groups[g].row0 + (int)(r < groups[g].rows ? r : groups[g].rows);
}

void sweep_slices(const SweepGroup* groups, int n_groups, int total_rows, int64_t total_bytes, int n,
                  SweepSlice* slices) {
  int g = 0;
  int row = row_at_byte(groups, n_groups, total_rows, total_bytes, 0, &g);
  for (int b = 0; b < n; ++b) {
    SweepSlice& sl = slices[b];
    sl.begin = row;
    // the first group of the slice: the last one whose first row is <= begin
    int g0 = 0;
    while (g0 + 1 < n_groups && groups[g0 + 1].row0 <= row) ++g0;
    sl.g0 = g0;
    const int64_t pe = (int64_t)((unsigned __int128)total_bytes * (unsigned)(b + 1) / (unsigned)n);
    row = row_at_byte(groups, n_groups, total_rows, total_bytes, pe, &g);
    sl.end = row;
  }
}

cudaError_t launch_gemv_sweep(const SweepGroup* groups_dev, int n_groups, const SweepSlice* slices_dev, int n_slices,
                              bool bf16, cudaStream_t stream) {
  auto kern = bf16 ? gemv_sweep_kernel<true> : gemv_sweep_kernel<false>;
  const int smem = kSwRingBytes + kSwMaxK + 64;
  static std::atomic<uint64_t> configured[2];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured[bf16].load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[bf16].fetch_or(bit, std::memory_order_acq_rel);
  }
  kern<<<n_slices, kSwThreads, smem, stream>>>(groups_dev, slices_dev, n_groups);
  return cudaGetLastError();
}

cudaError_t read_clear_device_error_sweep(int* value) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

}  // namespace bitnet
