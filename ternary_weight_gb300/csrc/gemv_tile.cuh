// gemv_tile.cuh -- the dp4a tile routine shared by the single-token kernels (gemv_group.cu, one
// launch per projection group, and gemv_sweep.cu, one persistent launch over many groups).
//
// Layouts ("BitNet 딥다이브" §4-2 for the weights; the activation layout is this library's):
//  * a weight row is K/4 bytes = C = K/64 chunks of 16 bytes; word q of chunk c holds, at bit
//    pair j, the codes of k = 128*(c/2) + 32*j + 16*(c%2) + 4q + (0..3);
//  * the quantised activations sit in shared memory as four planes j (one per bit pair), each
//    C + 1 chunks of 16 bytes [c][16]: plane j, chunk c holds the 16 activations that bit pair
//    j of weight chunk c multiplies; chunk C is all zero.
// The raw code dot of a row is the exact int32 sum_k code[k] * xq[k] ("[분석/검증-3] BitNet.cpp ARM
// 커널 재작성" §3: codes 0/1/2 multiplied as stored).
#pragma once

#include "bitnet_dev.cuh"

namespace bitnet {

// chunk columns per lane: the lane layouts used keep C/G <= 5, or G = 32 with C <= 160
constexpr int kMaxColsPerLane = 5;

// x * s rounded to the nearest integer, ties to even, returned as the bits of the fp32 sum
// x*s + 1.5*2^23: for |x*s| < 2^22 the sum lies in [2^23, 2^24), where fp32 steps by exactly 1,
// so the round-to-nearest-even add performs the integer rounding (1.5*2^23 is even, so ties
// go the same way), and bits - 0x4B400000 is the integer; its low byte is the int8 code.
// The clamp to [-127, 127] is never active: s = fl(127/a) with a >= max|x| gives
// |fl(x*s)| <= 127 (1 + 2^-24)^2 < 127.5, so the rounded value is at most 127 in magnitude.
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23
constexpr uint32_t kRoundMagicBits = 0x4B400000u;
__device__ __forceinline__ uint32_t quant_bits(float x, float s) {
  return __float_as_uint(__fadd_rn(__fmul_rn(x, s), kRoundMagic));
}

// Result of one tile for this lane: the raw dot `sum` of tile row `row`, valid when `writer`.
struct TileDot {
  int sum;
  int row;
  bool writer;
};

// One ring tile: S steps of rpw rows (rpw = 32 / G); step st of row group rg is row
// st * rpw + rg. Lane kl of a G-lane row group owns chunk columns c = kl + G * t (t < T). For
// each column the lane loads the 64 paired activation bytes from shared memory once and
// applies them to all S steps, keeping two accumulators per step. The column loop is unrolled
// over its bound of 5 with every load unconditional, so loads of the next column overlap the
// arithmetic of this one: a column past the row's end reads the row's last weight chunk
// against the zero activation column, and a row past the tile's end reads bytes inside the
// ring slot; neither is written. A transpose-reduce over the G lanes (three halving levels,
// then plain xor levels) leaves the total of step st in the lanes whose top three
// lane-in-group bits spell st, so the epilogue runs for up to 8 rows in parallel.
//   tile_lane : shared address of this lane's row of step 0 (step st is st * step_stride on)
//   xq_u      : shared address of activation plane 0; plane j is j * plane bytes on
// UNROLL: how many chunk columns the column loop unrolls (by default all 5 up to 6 steps;
// beyond that the registers of a second column would spill in the group kernel).
template <int S, int UNROLL = (S <= 6 ? kMaxColsPerLane : 1)>
__device__ __forceinline__ TileDot tile_raw_dots(uint32_t tile_lane, uint32_t xq_u, int plane, int C, int T, int kl,
                                                 int log2G, int rg, int rpw, int step_stride) {
  static_assert(S >= 1 && S <= 8, "one partial register per step, at most 8");
  const int G = 1 << log2G;
  // per step: hi = 64 * (sum of bit pairs 0 and 1), lo = 4 * (sum of bit pairs 2 and 3);
  // shifting the weight word left by 2 puts pair 1 under pair 0's mask and pair 3 under
  // pair 2's, so one accumulator serves two pairs at the same scale
  int acc[S][2];
#pragma unroll
  for (int st = 0; st < S; ++st) acc[st][0] = acc[st][1] = 0;
#pragma unroll UNROLL
  for (int t = 0; t < T; ++t) {
    const int c = kl + (t << log2G);
    const uint32_t w_off = (uint32_t)(min(c, C - 1) * 16);
    const uint32_t a_off = (uint32_t)((c < C ? c : C) * 16);
    // all of the column's shared-memory loads first: the S weight vectors, then the
    // activations
    uint4 wv[S];
#pragma unroll
    for (int st = 0; st < S; ++st) wv[st] = lds128(tile_lane + (uint32_t)(st * step_stride) + w_off);
    uint4 a[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) a[j] = lds128(xq_u + (uint32_t)(j * plane) + a_off);
#pragma unroll
    for (int st = 0; st < S; ++st) {
      const uint4 w = wv[st];
      const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
      const uint32_t a0[4] = {a[0].x, a[0].y, a[0].z, a[0].w};
      const uint32_t a1[4] = {a[1].x, a[1].y, a[1].z, a[1].w};
      const uint32_t a2[4] = {a[2].x, a[2].y, a[2].z, a[2].w};
      const uint32_t a3[4] = {a[3].x, a[3].y, a[3].z, a[3].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t sh = w4[q] << 2;
        acc[st][0] = dp4a_us(w4[q] & 0xC0C0C0C0u, a0[q], acc[st][0]);
        acc[st][0] = dp4a_us(sh & 0xC0C0C0C0u, a1[q], acc[st][0]);
        acc[st][1] = dp4a_us(w4[q] & 0x0C0C0C0Cu, a2[q], acc[st][1]);
        acc[st][1] = dp4a_us(sh & 0x0C0C0C0Cu, a3[q], acc[st][1]);
      }
    }
  }
  int v[8];
#pragma unroll
  for (int st = 0; st < 8; ++st) v[st] = st < S ? (acc[st < S ? st : 0][0] >> 6) + (acc[st < S ? st : 0][1] >> 2) : 0;
  int mine_step = 0;
  bool writer = kl == 0;
  if (G >= 8) {
    const int hb = log2G - 3;  // low lane bits left after the halving levels
    const bool up = (kl >> (log2G - 1)) & 1;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int send = up ? v[k] : v[k + 4], keep = up ? v[k + 4] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, G >> 1);
    }
    const bool up2 = (kl >> (log2G - 2)) & 1;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int send = up2 ? v[k] : v[k + 2], keep = up2 ? v[k + 2] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, G >> 2);
    }
    const bool up3 = (kl >> (log2G - 3)) & 1;
    {
      const int send = up3 ? v[0] : v[1], keep = up3 ? v[1] : v[0];
      v[0] = keep + __shfl_xor_sync(0xffffffffu, send, G >> 3);
    }
    for (int o = (G >> 4); o > 0; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    mine_step = (up ? 4 : 0) + (up2 ? 2 : 0) + (up3 ? 1 : 0);
    writer = (kl & ((1 << hb) - 1)) == 0;
  } else {
    for (int o = G >> 1; o > 0; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
  }
  return TileDot{v[0], mine_step * rpw + rg, writer && mine_step < S};
}

}  // namespace bitnet
