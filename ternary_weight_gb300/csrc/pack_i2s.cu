// pack_i2s.cu -- ternary int8 weights -> i2_s packed bytes.
//
// "BitNet 딥다이브" §4-2 (quantize_i2_s, x86 ACT_PARALLEL branch): a 128-weight block is
// read as 4 groups of 32; weight 32*j + g of block i goes to byte 32*i + g at bit offset
// 6 - 2*j; the code is w + 1 (§1-1 table: -1 -> 00, 0 -> 01, +1 -> 10). Entries outside
// {-1,0,+1} are packed by sign (>0 -> 2, <0 -> 0) and counted.
//
// One thread per output 32-bit word (bytes g0..g0+3 of one block of one row). It reads the
// four int8x4 words at block offsets g0, 32+g0, 64+g0, 96+g0 and assembles the word with
// byte-parallel compares. Off the timed path (weights are packed once).
#include "bitnet_dev.cuh"

namespace bitnet {
namespace {

// Per byte of a packed int8x4: code (0,1,2) in the same byte, and a count of bytes
// outside {-1,0,+1}.
__device__ __forceinline__ uint32_t codes_of(uint32_t v, int* bad) {
  // __vcmpgts4 / __vcmplts4 give 0xFF in every byte where the signed compare holds.
  const uint32_t pos = __vcmpgts4(v, 0u);            // w > 0
  const uint32_t neg = __vcmplts4(v, 0u);            // w < 0
  const uint32_t big = __vcmpgts4(v, 0x01010101u);   // w > 1
  const uint32_t sml = __vcmplts4(v, 0xFFFFFFFFu);   // w < -1
  *bad += __popc((big | sml) & 0x01010101u);
  // code = 1 + (w > 0) - (w < 0) per byte, formed without borrows: 0x01 | (pos & 0x02) -> 1/3,
  // then clear both bits where w < 0 and the low bit where w > 0.
  uint32_t c = 0x01010101u;
  c = (c & ~pos) | (pos & 0x02020202u);  // positive -> 2
  c = c & ~neg;                          // negative -> 0
  return c;
}

__global__ void __launch_bounds__(256) pack_i2s_kernel(const int8_t* __restrict__ w, uint8_t* __restrict__ wp,
                                                       int64_t N, int64_t K, int32_t* __restrict__ invalid_count) {
  const int64_t words_per_row = K / 16;  // K/4 bytes per row, 4 bytes per word
  const int64_t total = N * words_per_row;
  int bad = 0;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = t / words_per_row;
    const int64_t c = t - n * words_per_row;
    const int64_t blk = c >> 3;           // 8 words per 32-byte block
    const int64_t g0 = (c & 7) * 4;       // first byte of the word inside the block
    const int8_t* src = w + n * K + blk * 128 + g0;
    uint32_t out = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(src + 32 * j));
      out |= codes_of(v, &bad) << (6 - 2 * j);  // byte-wise: each code stays inside its byte
    }
    reinterpret_cast<uint32_t*>(wp)[t] = out;
  }
  if (invalid_count) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if ((threadIdx.x & 31) == 0 && bad) atomicAdd(invalid_count, bad);
  }
}

}  // namespace

cudaError_t launch_pack_i2s(const int8_t* w, uint8_t* wp, int64_t N, int64_t K, int32_t* invalid_count,
                            cudaStream_t stream) {
  if (invalid_count) {
    cudaError_t e = cudaMemsetAsync(invalid_count, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
  }
  const int64_t total = N * (K / 16);
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  pack_i2s_kernel<<<(unsigned)blocks, 256, 0, stream>>>(w, wp, N, K, invalid_count);
  return cudaGetLastError();
}

}  // namespace bitnet
