// gemv_group.cu -- single-token (M = 1) decode step of one projection group: the per-token
// activation quantisation fused with the GEMVs of up to 8 projections that share the row.
//
// What it computes, per projection l and output row n:
//   xq = clamp(rne(x * s), -127, 127),  s = 127 / max(max|x|, 1e-5),  rowsum = sum_k xq[k]
//   raw = sum_k code_l[n][k] * xq[k]          codes 0/1/2 multiplied as stored
//   out_l[n] = ((raw - rowsum) / s) * w_scale_l
// Sources: "BitNet 딥다이브" §4-5 (per-token quant_input), §4-2 (i2_s layout), §4-3 (_Nx1: one
// decoded activation set reused across weight rows); "[분석/검증-3] BitNet.cpp ARM 커널 재작성" §3
// and "[기술 분석 보고서] ... 추론 붕괴 원인 분석" §3.1-§4 (raw code dot over the 4x32-interleaved
// bytes); "bitnet.rs" "8-bit Activation Quantisation", "Quantised Forward Pass".
//
// Design: latency first (a decode step is a chain of such groups). One CTA per SM, small
// enough (288 threads at <= 113 registers, ~106 KB of shared memory) that the CTA of the next
// group's kernel fits beside it, so with programmatic dependent launch the next kernel starts
// streaming its weights while this one finishes.
//  * The group's projections are concatenated into one row space; CTA b owns a contiguous
//    slice of it, cut into tiles of whole rows (<= 12 KB, never across two projections).
//  * Warp 8 is the producer: one lane issues cp.async.bulk copies of consecutive tiles into an
//    8-slot x 12 KB shared-memory ring, each slot completing on its own mbarrier by
//    transaction bytes; then it hands the L2 prefetch hint (the next group's weights) to
//    cp.async.bulk.prefetch.L2.
//  * Programmatic dependent launch: the kernel lets the next kernel in the stream launch as
//    soon as it starts, and streams its weights (read-only model state) before it waits for
//    the previous kernel (griddepcontrol.wait); the activations are read and every output is
//    written only after that wait. In a chain of such kernels the time per kernel is the
//    release latency plus what follows the wait, so everything that does not need the
//    activations happens before it: the kernel parameters are copied to shared memory (a
//    parameter's first read misses the constant cache), the tile count is computed, the
//    row gets an L2 prefetch and each consumer warp waits for its first tile.
//  * Warps 0-7 are consumers; tile i goes to warp i % 8 (the slot count is a multiple of 8,
//    so each slot belongs to one warp). They read the row once into registers (fp32 or bf16),
//    reduce max|x| (redux.sync on the bits of the non-negative maxima), quantise every
//    element once into shared memory laid out [j][c][16] (rounding by the fp32
//    add-1.5*2^23 identity) and reduce the row sum. Lane kl of a G-lane row group owns chunk columns c = kl + G*t; per
//    column it loads the 64 paired activation bytes (four conflict-free LDS.128) and applies
//    them to up to 8 row steps of the tile: per 16-byte weight chunk one LDS.128, then per
//    32-bit word w four masked operands (w & 0xC0.., (w<<2) & 0xC0.., w & 0x0C..,
//    (w<<2) & 0x0C..) and four dp4a (unsigned codes x signed int8) into two accumulators that
//    hold exact multiples of 64 and 4. The steps' partials
//    are reduced over the G lanes together with a transpose-reduce, so the epilogue (one IEEE
//    divide per output) runs on up to 8 lanes at once. CTA 0 also writes xq, s and the row
//    sum when asked.
//  * Every wait is bounded; a timeout is recorded in the device error word and the kernel
//    leaves after waiting (bounded) for the copies it issued.
#include "gemv_tile.cuh"

#include <atomic>

namespace bitnet {

static_assert(kMaxGroupLinears == 8, "LinearSet layout");

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + producer warp
constexpr int kSlots = 8;
constexpr int kSlotBytes = 12288;
constexpr int kRingBytes = kSlots * kSlotBytes;
constexpr int kMaxK = 10240;            // largest K this kernel takes
// the activation row passes through the consumers as 16-byte vectors, at most
// kMaxVecPerThread per thread; the first kRegVec of them stay in registers between the max
// and the quantise pass (all of them for K <= 6144 fp32 / 12288 bf16), the rest are re-read
constexpr int kMaxVecPerThread = kMaxK / 4 / (kConsumerWarps * 32);
constexpr int kRegVec = 6;
static_assert(kMaxK / 64 <= 32 * kMaxColsPerLane, "column loop bound");
// Tile i lives in slot i % kSlots and is consumed by warp i % kConsumerWarps. With the slot
// count a multiple of the consumer-warp count, every slot is only ever waited on by one
// warp, in order, so a parity wait can never see a stale phase of its slot.
static_assert(kSlots % kConsumerWarps == 0, "each ring slot must belong to one consumer warp");

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// The L2 prefetch hint: CTA b hands slice b of every range to cp.async.bulk.prefetch.L2.
__device__ __forceinline__ void issue_prefetch(const Prefetch& pf) {
  for (int p = 0; p < pf.count; ++p) {
    const int64_t n16 = pf.bytes[p] >> 4;
    int64_t lo = n16 * blockIdx.x / gridDim.x * 16, hi = n16 * (blockIdx.x + 1) / gridDim.x * 16;
    const char* base = static_cast<const char*>(pf.ptr[p]);
    while (lo < hi) {
      const int64_t len = (hi - lo) < (1 << 16) ? (hi - lo) : (1 << 16);
      prefetch_l2(base + lo, (uint32_t)len);
      lo += len;
    }
  }
}

// Number of tiles (whole-row runs of at most TR rows, never across two projections) in the
// concatenated row range [begin, end) of the group's count projections of N[j] rows.
__device__ __forceinline__ int count_tiles(const int* N, int count, int begin, int end, int TR) {
  int n = 0, off = 0;
  for (int j = 0; j < count; ++j) {
    const int lo = max(off, begin), hi = min(off + N[j], end);
    if (hi > lo) n += (hi - lo + TR - 1) / TR;
    off += N[j];
  }
  return n;
}

// Input row modes: fp32 x, bf16 x, or the FFN inner activation computed from the gate and up
// rows (FfnIn: squared-ReLU gate times up, RMS sub-norm with gamma; K is then F).
constexpr int kInF32 = 0, kInBF16 = 1, kInFfn = 2;

// IN: the input row mode.
// S: row steps per tile (1..8), a compile-time constant so the step loops carry no
// predicated dead steps.
template <int IN, int S>
__global__ void __launch_bounds__(kThreads, 2) gemv_group_kernel(const void* __restrict__ xin, LinearSet set,
                                                                 QuantOut qout, Prefetch pf, FfnIn ffn, int K,
                                                                 int log2G) {
  constexpr bool BF16 = IN == kInBF16;
  constexpr bool FFN = IN == kInFfn;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;                      // kSlots x kSlotBytes
  uint8_t* xq_s = smem + kRingBytes;         // K + 64 bytes, [j][c][16] (c = C is zero)
  __shared__ __align__(8) uint64_t full_bar[kSlots];
  __shared__ __align__(8) uint64_t empty_bar[kSlots];
  __shared__ __align__(16) float red_f[kConsumerWarps];  // read back as float4
  __shared__ __align__(16) int red_i[kConsumerWarps];    // read back as int4
  __shared__ __align__(16) float red_ss[kConsumerWarps]; // FFN: run sums of the squares
  // the tile held by each ring slot (written by the producer before its release-arrive on
  // the slot's full barrier, read by the consumer after its acquire-wait)
  __shared__ int slot_rows[kSlots];
  __shared__ float* slot_out[kSlots];    // output row of the tile's first row
  __shared__ int32_t* slot_acc[kSlots];  // same for the optional accumulators (or null)
  __shared__ float slot_ws[kSlots];      // weight scale of the tile's projection
  // The kernel parameters, copied to shared memory at the start. The first read of a
  // parameter in a launch misses the constant cache (about half a microsecond); staged here,
  // those misses are paid before the dependency wait instead of after it, where every
  // nanosecond lengthens the decode chain.
  __shared__ const uint8_t* p_wp[kMaxGroupLinears];
  __shared__ float* p_out[kMaxGroupLinears];
  __shared__ int32_t* p_acc[kMaxGroupLinears];
  __shared__ float p_ws[kMaxGroupLinears];
  __shared__ int p_N[kMaxGroupLinears];
  __shared__ int p_count;
  __shared__ const void* p_x;
  __shared__ QuantOut p_q;
  __shared__ FfnIn p_ffn;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int C = K >> 6;
  const int row_bytes = K >> 2;
  const int TR = S << (5 - log2G);  // rows per tile = steps x rows per step

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == 1 && lane < kMaxGroupLinears) {
    p_wp[lane] = set.wp[lane];
    p_out[lane] = set.out[lane];
    p_acc[lane] = set.acc[lane];
    p_ws[lane] = set.w_scale[lane];
    p_N[lane] = set.N[lane];
    if (lane == 0) {
      p_count = set.count;
      p_x = xin;
      p_q = qout;
      p_ffn = ffn;
    }
  }
  __syncthreads();
  pdl_launch_dependents();
  const int count = p_count;
  int total = 0;  // rows of the group (the host keeps this below 2^31)
  for (int j = 0; j < count; ++j) total += p_N[j];
  const int cta_begin = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int cta_end = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  bool abort = false;

  if (warp == kConsumerWarps) {
    // ================================ producer ================================
    if (lane == 0) {
      // walk this CTA's tiles in order: projection j, rows [r, hi) of it left to cover
      int issued = 0, j = -1, off = 0, r = 0, hi = 0, prev_n = 0;
      for (int i = 0;; ++i) {
        while (r >= hi) {  // next projection that intersects [cta_begin, cta_end)
          off += prev_n;
          if (++j >= count) break;
          prev_n = p_N[j];
          r = max(off, cta_begin);
          hi = min(off + prev_n, cta_end);
        }
        if (j >= count) break;
        const int rows = min(TR, hi - r);
        const int slot = i % kSlots, use = i / kSlots;
        if (use > 0 && !mbar_wait(&empty_bar[slot], (use - 1) & 1, &abort)) break;
        slot_out[slot] = p_out[j] + (r - off);
        slot_acc[slot] = p_acc[j] ? p_acc[j] + (r - off) : nullptr;
        slot_ws[slot] = p_ws[j];
        slot_rows[slot] = rows;
        const uint32_t bytes = (uint32_t)rows * (uint32_t)row_bytes;
        mbar_arrive_expect_tx(&full_bar[slot], bytes);
        bulk_copy_g2s(ring + slot * kSlotBytes, p_wp[j] + (int64_t)(r - off) * row_bytes, bytes, &full_bar[slot]);
        r += rows;
        issued = i + 1;
        if (issued == kSlots) issue_prefetch(pf);  // ring primed: now the L2 prefetch hint
      }
      if (issued < kSlots) issue_prefetch(pf);
      {  // every copy this CTA issued lands before the producer leaves: the consumers may have
         // given up on a full barrier (a bounded wait) while copies were still in flight
        bool dummy = false;
        for (int i = issued - kSlots > 0 ? issued - kSlots : 0; i < issued; ++i)
          mbar_wait(&full_bar[i % kSlots], (i / kSlots) & 1, &dummy);
      }
    }
    return;
  }

  // ================================ consumers ================================
  const int G = 1 << log2G;
  const int kl = lane & (G - 1);
  const int rg = lane >> log2G;
  const int rpw = 32 >> log2G;
  const int T = (C + G - 1) >> log2G;  // chunk columns per lane (the last may be ragged)
  // activation plane j holds the C chunk columns plus one zero column (index C) that the
  // ragged lanes of a 32-lane layout read instead of a column past the row's end
  const int plane = (C + 1) * 16;

  // everything that does not depend on the activations is done before the wait: the tile
  // count, the L2 prefetch of the row and the wait for this warp's first tile
  const int n_tiles = count_tiles(p_N, count, cta_begin, cta_end, TR);
  const QuantOut q_out = p_q;
  const uint4* xv = static_cast<const uint4*>(p_x);
  // an L2 prefetch of the row is safe before the wait: it returns no data, and a write by
  // the previous kernel lands in L2 all the same
  const FfnIn fi = p_ffn;
  if (threadIdx.x == 0) {
    if constexpr (FFN) {
      prefetch_l2(fi.gate, (uint32_t)K * 4u);
      prefetch_l2(fi.up, (uint32_t)K * 4u);
      prefetch_l2(fi.gamma, (uint32_t)K * 4u);  // model state: could be read before the wait too
    } else {
      prefetch_l2(xv, (uint32_t)K * (BF16 ? 2u : 4u));
    }
  }
  if (warp < n_tiles) mbar_wait_warp(&full_bar[warp], 0, &abort);  // tile `warp`: slot warp, use 0
  float s_act;
  int rs_total;
  pdl_wait();  // the activations may be the previous kernel's output
  {
    // the row is read once into registers: vector v = threadIdx.x + kConsumers * i
    constexpr int E = BF16 ? 8 : 4;  // elements per 16-byte vector
    const int nvec = K / E;
    uint4 xr[kRegVec];
    float amax = 0.0f;
    float c_ffn = 0.0f;
    const float4* g4 = reinterpret_cast<const float4*>(fi.gate);
    const float4* u4 = reinterpret_cast<const float4*>(fi.up);
    const float4* gm4 = reinterpret_cast<const float4*>(fi.gamma);
    if constexpr (FFN) {
      // pass 1: h = max(g, 0)^2 * u and this thread's partial of the sum of squares
      // (partial = thread, vectors in ascending order: the order FfnIn defines)
      float ssp = 0.0f;
#pragma unroll
      for (int i = 0; i < kMaxVecPerThread; ++i) {
        const int v = threadIdx.x + kConsumers * i;
        if (v < nvec) {
          const float4 g = __ldg(g4 + v), u = __ldg(u4 + v);
          const float h0 = ffn_h(g.x, u.x), h1 = ffn_h(g.y, u.y), h2 = ffn_h(g.z, u.z), h3 = ffn_h(g.w, u.w);
          ssp = __fmaf_rn(h0, h0, ssp);
          ssp = __fmaf_rn(h1, h1, ssp);
          ssp = __fmaf_rn(h2, h2, ssp);
          ssp = __fmaf_rn(h3, h3, ssp);
          if (i < kRegVec)
            xr[i] = make_uint4(__float_as_uint(h0), __float_as_uint(h1), __float_as_uint(h2), __float_as_uint(h3));
        }
      }
      ssp = ffn_run_sum(ssp);
      if (lane == 0) red_ss[warp] = ssp;
      named_bar_sync(1, kConsumers);
      {
        const float4 r0 = *reinterpret_cast<const float4*>(&red_ss[0]);
        const float4 r1 = *reinterpret_cast<const float4*>(&red_ss[4]);
        const float runs[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        c_ffn = ffn_rms_factor(ffn_runs_total(runs), K, fi.eps);
      }
      // pass 2: inner = (h * c) * gamma and its absolute maximum
#pragma unroll
      for (int i = 0; i < kMaxVecPerThread; ++i) {
        const int v = threadIdx.x + kConsumers * i;
        if (v < nvec) {
          float4 h;
          if (i < kRegVec) {
            h = make_float4(__uint_as_float(xr[i].x), __uint_as_float(xr[i].y), __uint_as_float(xr[i].z),
                            __uint_as_float(xr[i].w));
          } else {
            const float4 g = __ldg(g4 + v), u = __ldg(u4 + v);
            h = make_float4(ffn_h(g.x, u.x), ffn_h(g.y, u.y), ffn_h(g.z, u.z), ffn_h(g.w, u.w));
          }
          const float4 gm = __ldg(gm4 + v);
          const float y0 = __fmul_rn(__fmul_rn(h.x, c_ffn), gm.x), y1 = __fmul_rn(__fmul_rn(h.y, c_ffn), gm.y);
          const float y2 = __fmul_rn(__fmul_rn(h.z, c_ffn), gm.z), y3 = __fmul_rn(__fmul_rn(h.w, c_ffn), gm.w);
          amax = fmaxf(fmaxf(amax, fmaxf(fabsf(y0), fabsf(y1))), fmaxf(fabsf(y2), fabsf(y3)));
          if (i < kRegVec)
            xr[i] = make_uint4(__float_as_uint(y0), __float_as_uint(y1), __float_as_uint(y2), __float_as_uint(y3));
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < kMaxVecPerThread; ++i) {
        const int v = threadIdx.x + kConsumers * i;
        const uint4 u = v < nvec ? __ldg(xv + v) : make_uint4(0u, 0u, 0u, 0u);
        if (i < kRegVec) xr[i] = u;
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
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
    }
    // amax is a non-negative float (fmaxf drops NaN), so its bits order like unsigned ints
    const uint32_t wmax = __reduce_max_sync(0xffffffffu, __float_as_uint(amax));
    if (lane == 0) red_f[warp] = __uint_as_float(wmax);
    if (threadIdx.x < 4) *reinterpret_cast<uint4*>(xq_s + threadIdx.x * plane + C * 16) = make_uint4(0u, 0u, 0u, 0u);
    named_bar_sync(1, kConsumers);
    {
      const float4 r0 = *reinterpret_cast<const float4*>(&red_f[0]);
      const float4 r1 = *reinterpret_cast<const float4*>(&red_f[4]);
      amax = fmaxf(fmaxf(fmaxf(r0.x, r0.y), fmaxf(r0.z, r0.w)), fmaxf(fmaxf(r1.x, r1.y), fmaxf(r1.z, r1.w)));
    }
    s_act = __fdiv_rn(127.0f, fmaxf(amax, 1e-5f));
    // quantise each element once; element k goes to [j][c][16] with
    // c = 2*(k/128) + (k%32)/16, j = (k%128)/32. The row sum is accumulated on the biased
    // bits (each q + 0x4B400000) and unbiased at the end, modulo 2^32.
    uint32_t bsum = 0;
    int nel = 0;
    const bool publish = blockIdx.x == 0 && q_out.xq != nullptr;
#pragma unroll
    for (int i = 0; i < kMaxVecPerThread; ++i) {
      const int v = threadIdx.x + kConsumers * i;
      if (v < nvec) {
        uint4 u;
        if (i < kRegVec) {
          u = xr[i];
        } else if constexpr (FFN) {  // recompute inner for a vector that did not stay in registers
          const float4 g = __ldg(g4 + v), uu = __ldg(u4 + v), gm = __ldg(gm4 + v);
          u = make_uint4(__float_as_uint(__fmul_rn(__fmul_rn(ffn_h(g.x, uu.x), c_ffn), gm.x)),
                         __float_as_uint(__fmul_rn(__fmul_rn(ffn_h(g.y, uu.y), c_ffn), gm.y)),
                         __float_as_uint(__fmul_rn(__fmul_rn(ffn_h(g.z, uu.z), c_ffn), gm.z)),
                         __float_as_uint(__fmul_rn(__fmul_rn(ffn_h(g.w, uu.w), c_ffn), gm.w)));
        } else {
          u = __ldg(xv + v);
        }
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
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
        // low bytes of four words -> one word
        const uint32_t word0 = __byte_perm(__byte_perm(qb[0], qb[1], 0x0040), __byte_perm(qb[2], qb[3], 0x0040), 0x5410);
        if constexpr (BF16) {
          const uint32_t word1 =
              __byte_perm(__byte_perm(qb[4], qb[5], 0x0040), __byte_perm(qb[6], qb[7], 0x0040), 0x5410);
          *reinterpret_cast<uint2*>(xq_s + off) = make_uint2(word0, word1);
          if (publish) *reinterpret_cast<uint2*>(q_out.xq + k) = make_uint2(word0, word1);
        } else {
          *reinterpret_cast<uint32_t*>(xq_s + off) = word0;
          if (publish) *reinterpret_cast<uint32_t*>(q_out.xq + k) = word0;
        }
      }
    }
    const int sum = (int)(bsum - (uint32_t)nel * kRoundMagicBits);
    const int wsum = __reduce_add_sync(0xffffffffu, sum);
    if (lane == 0) red_i[warp] = wsum;
    named_bar_sync(1, kConsumers);  // also orders the shared activation writes before the reads
    {
      const int4 r0 = *reinterpret_cast<const int4*>(&red_i[0]);
      const int4 r1 = *reinterpret_cast<const int4*>(&red_i[4]);
      rs_total = ((r0.x + r0.y) + (r0.z + r0.w)) + ((r1.x + r1.y) + (r1.z + r1.w));
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      if (q_out.scale) *q_out.scale = s_act;
      if (q_out.rowsum) *q_out.rowsum = rs_total;
    }
  }

  // ---- consume this warp's tiles: a tile is S steps of rpw rows; step st of row group rg is
  // row st*rpw + rg. For each chunk column the lane loads the 64 paired activation bytes from
  // shared memory once and applies them to all S steps, keeping two accumulators per step.
  // The column loop is unrolled over its bound of 5 (the lane layout keeps C/G <= 5 for
  // K <= 10240) with every load unconditional, so loads of the next column overlap the
  // arithmetic of this one: a column past the row's end, or a row past the tile's end, reads
  // bytes inside the ring slot and the activation buffer and has its weight word zeroed.
  // A transpose-reduce over the G lanes (three halving levels, then plain xor levels) leaves
  // the total of step st in the lanes whose top three lane-in-group bits spell st, so the
  // epilogue (one IEEE divide per output) runs for up to 8 rows in parallel. ----
  const uint32_t xq_u = smem_u32(xq_s);
  const int step_stride = rpw * row_bytes;
  for (int i = warp; i < n_tiles; i += kConsumerWarps) {
    const int slot = i % kSlots, use = i / kSlots;
    if (i != warp) {
      if (!mbar_wait_warp(&full_bar[slot], use & 1, &abort)) break;
    } else if (abort) {
      break;
    }
    const int rows = slot_rows[slot];
    float* const out_row = slot_out[slot];
    int32_t* const acc_row = slot_acc[slot];
    const float ws = slot_ws[slot];
    // this lane's row of step 0; step st is st * step_stride bytes further
    const uint32_t tile_lane = smem_u32(ring + slot * kSlotBytes) + (uint32_t)(rg * row_bytes);
    const TileDot r = tile_raw_dots<S>(tile_lane, xq_u, plane, C, T, kl, log2G, rg, rpw, step_stride);
    if (r.writer && r.row < rows) {
      const int a = r.sum - rs_total;
      out_row[r.row] = __fmul_rn(__fdiv_rn(__int2float_rn(a), s_act), ws);
      if (acc_row) acc_row[r.row] = a;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[slot]);
  }
}

// lanes per row: the largest power of two <= 32 dividing C when that keeps at most 5 chunk
// columns per lane, else 32 lanes with a ragged last column (predicated)
int choose_log2g(int K) {
  const int C = K >> 6;
  int log2G = 5;
  while (log2G > 1 && (C & ((1 << log2G) - 1)) != 0) --log2G;
  if ((C >> log2G) > 5) log2G = 5;
  return log2G;
}

template <int IN, int S>
cudaError_t launch_s(const void* x, const LinearSet& set, const QuantOut& q, const Prefetch& pf, const FfnIn& ffn,
                     int K, int log2G, int blocks, cudaStream_t stream) {
  auto kern = gemv_group_kernel<IN, S>;
  const int smem = kRingBytes + K + 64;  // ring, activations + one zero column per plane
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes + kMaxK + 64);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
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
  return cudaLaunchKernelEx(&cfg, kern, x, set, q, pf, ffn, K, log2G);
}

template <int IN>
cudaError_t launch_t(const void* x, const LinearSet& set, const QuantOut& q, const Prefetch& pf, const FfnIn& ffn,
                     int K, int log2G, int num_sms, cudaStream_t stream) {
  int64_t total = 0;
  for (int j = 0; j < set.count; ++j) total += set.N[j];
  const int rpw = 32 >> log2G;
  const int64_t step_bytes = (int64_t)(K >> 2) * rpw;
  // steps per tile: at most 8 (one partial register each), the tile within one ring slot
  // (K <= 10240 keeps one step within 2560 bytes), 1 when fewer than 8 lanes share a row, and
  // no more than a consumer warp's share of the CTA's rows
  int blocks = num_sms;
  if (total < blocks) blocks = (int)total;
  const int64_t per_cta = (total + blocks - 1) / blocks;
  int64_t S = (log2G >= 3) ? kSlotBytes / step_bytes : 1;
  if (S > 8) S = 8;
  if (S < 1) S = 1;
  const int64_t want = ((per_cta + kConsumerWarps - 1) / kConsumerWarps + rpw - 1) / rpw;
  if (S > want) S = want < 1 ? 1 : want;
  switch (S) {
    case 1: return launch_s<IN, 1>(x, set, q, pf, ffn, K, log2G, blocks, stream);
    case 2: return launch_s<IN, 2>(x, set, q, pf, ffn, K, log2G, blocks, stream);
    case 3: return launch_s<IN, 3>(x, set, q, pf, ffn, K, log2G, blocks, stream);
    case 4: return launch_s<IN, 4>(x, set, q, pf, ffn, K, log2G, blocks, stream);
    case 5: return launch_s<IN, 5>(x, set, q, pf, ffn, K, log2G, blocks, stream);
    case 6: return launch_s<IN, 6>(x, set, q, pf, ffn, K, log2G, blocks, stream);
    case 7: return launch_s<IN, 7>(x, set, q, pf, ffn, K, log2G, blocks, stream);
    default: return launch_s<IN, 8>(x, set, q, pf, ffn, K, log2G, blocks, stream);
  }
}

}  // namespace

cudaError_t read_clear_device_error_gemv_group(int* value) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

bool gemv_group_supported(int64_t K) { return K <= kMaxK; }

cudaError_t launch_gemv_group(const void* x, bool bf16, const LinearSet& set, const QuantOut& qout,
                              const Prefetch& pf, int64_t K, int num_sms, cudaStream_t stream) {
  const int log2G = choose_log2g((int)K);
  const FfnIn none{};
  return bf16 ? launch_t<kInBF16>(x, set, qout, pf, none, (int)K, log2G, num_sms, stream)
              : launch_t<kInF32>(x, set, qout, pf, none, (int)K, log2G, num_sms, stream);
}

cudaError_t launch_gemv_group_ffn(const FfnIn& ffn, const LinearSet& set, const QuantOut& qout, const Prefetch& pf,
                                  int64_t F, int num_sms, cudaStream_t stream) {
  const int log2G = choose_log2g((int)F);
  return launch_t<kInFfn>(nullptr, set, qout, pf, ffn, (int)F, log2G, num_sms, stream);
}

}  // namespace bitnet
