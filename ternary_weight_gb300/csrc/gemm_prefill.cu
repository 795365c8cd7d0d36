// gemm_prefill.cu -- the W2A8 ternary matmul for prompts (from ~100 tokens on) on the tensor cores,
// with no workspace: the packed weights and the int8 activations are staged by TMA and expanded to
// exact fp16 inside the kernel.
//
// Computes, like every other path of the library, raw[m][n] = sum_k code[n][k] * xq[m][k],
// acc = raw - rowsum[m], out = (acc / s[m]) * w_scale, with the same integers and the same fp32
// results. Sources: the raw code dot over the 4x32-interleaved i2_s bytes ("[분석/검증-3]
// BitNet.cpp ARM 커널 재작성" §3, "[기술 분석 보고서] ... 추론 붕괴 원인 분석" §3.2), the byte
// layout ("BitNet 딥다이브" §4-2), the dequantisation ("bitnet.rs" "Quantised Forward Pass").
// "BitNet 딥다이브" §4-5 runs prefill as a separate dense path; this is that path.
//
// Tile: 256 weight rows (two MMA tiles of 128: the MMA's M) x 128 tokens (the MMA's N) x a range
// of 128-k i2_s blocks. The contraction is tcgen05.mma.cta_group::1.kind::f16, M = 128, N = 128,
// K = 16, fp32 accumulation in tensor memory. Both operands are exact:
//  * A (weights): the code c in {0..3} as the fp16 subnormal c * 2^-24 (bit pattern c), written by
//    the converter threads straight into tensor memory with tcgen05.st (two shifts and two masks
//    give four codes as two fp16 pairs); the expanded weights never touch shared memory;
//  * B (tokens): the int8 value as an exact fp16 (0x6400 | (x + 128) = 1152 + x, minus 1152),
//    written into a 128-byte-swizzled K-major shared-memory tile that both weight tiles use;
//  * every product is c * x * 2^-24 and every partial sum an integer multiple of 2^-24 of
//    magnitude below 3 * 127 * K * 2^-24 < 1 for K <= 32768: the fp32 accumulators are exact, and
//    the epilogue's fma(D, 2^24, -rowsum) gives the integer acc = raw - rowsum exactly.
// K order inside a 64-k stage: the MMA only needs A and B to agree. Word q of a row's 32 staged
// bytes and bit pair j give, by (w >> (6 - 2j)) & 0x00030003 and the same shifted by 8 more, the
// codes of bytes (0, 2) and (1, 3) as fp16 pairs; so stage position p holds the stage's k =
// 4 (p / 4) + sigma(p % 4) with sigma = (0, 2, 1, 3), and the token bytes are laid out in B in the
// same order by the byte permutes that convert them.
//
// Pipeline, per 128-k block b of the CTA's range (two 64-k stages, h = 0, 1):
//  * warp 0, one lane: 2-D TMA (cp.async.bulk.tensor) of the block's packed weights (256 rows x
//    32 bytes) and int8 tokens (two boxes of 128 rows x 64 bytes, one per stage, so that the
//    converters' 16-byte reads of two neighbouring rows fall in different banks) into a staging
//    slot (4 slots); the weights of the first slots are requested before the dependency wait;
//  * warps 2-17 (16 converters) in two groups of 8 that take alternate stages (group g the stages
//    with h = g), so that each warp has two stage periods for its chain of loads, conversion,
//    tensor-memory store, fences and arrival: warp (tile, lane quarter) turns bit pairs 2h and
//    2h + 1 of its 32 rows into 32 tensor-memory columns of A, and each thread turns two 16-byte
//    pieces of token bytes into fp16 chunks of B; then fences and one arrival per warp;
//  * warp 1, one lane: per stage 2 x 4 MMAs (both weight tiles, four k16 steps), then a commit
//    that releases the stage (A columns and B tile) to the converters.
// The lanes of warps 0 and 1 that do not issue wait at a warp barrier: a lane suspended in an
// mbarrier poll would hold back the issuing lane of its warp.
//
// Epilogue. The division out = RN(RN(acc / s) * w_scale) is exact and branch-free: with the
// per-token y = RN(1/s) (the correctly rounded reciprocal), q = RN(acc * y) and two residual
// corrections r = fma(-q, s, acc) (exact), q = fma(r, y, q) give RN(acc / s) (Markstein's method;
// the first correction makes q faithful, the second rounds correctly). Tokens whose s lies outside
// [2^-100, 2^100] (quotients that could overflow) take the IEEE division instead. The finished
// values go to a token-major staging tile in the freed rings and leave by TMA bulk stores (which
// clip the ragged edges), 32 tokens per store as soon as both weight tiles have finished them, or,
// when the output rows are not 16-byte aligned or the int32 accumulators are requested too, by
// plain stores with consecutive lanes on consecutive n.
// Split K: for short prompts the blocks of one tile are spread over a thread-block cluster of up
// to 16 CTAs (as many as make every CTA resident at once). Every CTA stages its exact partials as
// int32, token-major, in its own shared memory; after a cluster barrier rank r owns the tokens
// [8 floor(16 r / cs), 8 floor(16 (r + 1) / cs)) of the tile and pulls their partials from every
// peer with 16-byte distributed-shared-memory loads (a warp reads 512 contiguous bytes of one
// token; every peer's 16 bytes are requested before any is added). r finishes its tokens in place
// and stores them; a second cluster barrier keeps every CTA alive until no peer reads its shared
// memory any more. (Bulk reduce-adds by the TMA engine into the owner's staging, tried for small
// clusters, were slower: 2B-4T FFN shapes, at 3 CTAs 20.3 against 17.1 us, at 2 CTAs 21.8
// against 21.4.)
// Every mbarrier wait is bounded; a timeout is recorded in the device error word, and the TMA
// producer always waits (bounded) for its last copies before it leaves.
#include "bitnet_dev.cuh"

#include <atomic>
#include <cstring>
#include <cudaTypedefs.h>

namespace bitnet {
namespace {

constexpr int TWR = 256;                 // weight rows per CTA (two MMA tiles)
constexpr int TT = 128;                  // tokens per CTA (the MMA's N)
constexpr int CONV_WARPS = 16;           // converters, then the epilogue
constexpr int CONV_THREADS = CONV_WARPS * 32;
constexpr int THREADS = CONV_THREADS + 64;
constexpr int NSS = 4;                   // staging slots (one 128-k block each)
constexpr int NAB = 4;                   // A/B stages (64 k each)
constexpr int STG_W = TWR * 32;          // staged packed weights of one block: 256 rows x 32 bytes
constexpr int STG_X = TT * 128;          // staged int8 tokens of one block: [half][128 rows][64 bytes]
constexpr int STG_BYTES = STG_W + STG_X;
constexpr int B_STAGE = TT * 128;        // fp16 B tile of one stage: 128 rows x 64 k x 2 bytes
constexpr int SMEM = 1024 + NAB * B_STAGE + NSS * STG_BYTES;
constexpr int OUT_STAGE = TT * TWR * 4;  // token-major fp32 tile (epilogue; reuses the rings)
constexpr uint32_t TMEM_COLS = 512;      // accumulators (2 x 128) + A stages (4 x 2 x 32)
constexpr int ACC_COLS = 2 * TT;
constexpr int A_STAGE_COLS = 64;         // both tiles: 2 x 32 columns (64 fp16 of k per lane)
constexpr int kMaxCluster = 16;
constexpr int kStoreRows = 32;           // tokens per TMA store of a whole tile (cluster size 1)
constexpr int BAR_ALL = 1;               // named barrier of the whole CTA
constexpr int BAR_HALF = 2;              // named barriers 2, 3: the converter warps of one token half
constexpr uint32_t IDESC = make_idesc_f16_f32(128, TT);
// split K: rank r of a cluster of cs finishes tokens [tok_lo(r), tok_lo(r + 1)) of the tile, in
// whole groups of 8 (every rank has at least one group for cs <= 16)
__host__ __device__ constexpr int tok_lo(int r, int cs) { return 8 * (16 * r / cs); }
static_assert(ACC_COLS + NAB * A_STAGE_COLS <= (int)TMEM_COLS, "tensor memory columns");
static_assert(SMEM <= 227 * 1024 - 4096, "shared memory (static part included)");
static_assert(OUT_STAGE <= NAB * B_STAGE + NSS * STG_BYTES, "the epilogue tile fits the reused rings");

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// shared -> global tile store by the TMA engine (elements outside the tensor are not written)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every bulk store of this thread is complete (its shared-memory source read, its writes done)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void sts32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void sts32i(uint32_t addr, int v) {
  asm volatile("st.shared.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// 16 bytes of a peer's shared memory (a shared::cluster address, 16-byte aligned)
__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t cluster_addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(cluster_addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16: A is 128 lanes (rows) x 8 columns (16 fp16
// along K, two per column, the lower position in the low half); the B descriptor is given as its
// two 32-bit halves (the low half carries the address).
__device__ __forceinline__ void mma_f16_ts2(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 bd;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "mov.b64 bd, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp writes lane (base + t).
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// four int8 -> four exact fp16 (as two fp16x2 words), in the stage's position order: bytes (0, 2)
// then bytes (1, 3)
__device__ __forceinline__ void s8x4_f16_perm(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;                      // x + 128 per byte
  const uint32_t l = __byte_perm(u, 0x64646464u, 0x4240);  // 0x64uu: 1024 + (x + 128)
  const uint32_t h = __byte_perm(u, 0x64646464u, 0x4341);
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(l), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(h), "r"(0x64806480u));
}

// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major tile
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// RN(a / s) for an integer-valued a (|a| < 2^25) and s in [2^-100, 2^100], given y = RN(1/s):
// Markstein's residual correction, twice (exact remainders by fma).
__device__ __forceinline__ float div_by_scale(float a, float s, float y) {
  float q = __fmul_rn(a, y);
  float r = __fmaf_rn(-q, s, a);
  q = __fmaf_rn(r, y, q);
  r = __fmaf_rn(-q, s, a);
  return __fmaf_rn(r, y, q);
}

// Per token of the tile, in shared memory as one float4: {act scale s, y = RN(1/s), -rowsum
// (exact), 1 if s lies in [2^-100, 2^100] else 0}.
__device__ __forceinline__ float4 token_const(const float4* tok, int t) { return tok[t]; }

// out = RN(RN((d * 2^24 - rowsum) / s) * w_scale) for any token (the IEEE division where the scale
// is extreme), and the integer acc
__device__ __forceinline__ float finish_any(float d, float4 c, float w_scale, int* acc_int) {
  const float a = __fmaf_rn(d, 16777216.0f, c.z);
  *acc_int = __float2int_rn(a);
  const float q = c.w != 0.0f ? div_by_scale(a, c.x, c.y) : __fdiv_rn(a, c.x);
  return __fmul_rn(q, w_scale);
}

// Two fp32 lanes per instruction (mul/fma .f32x2, each lane rounded exactly as the scalar
// operation): the epilogue's per-element arithmetic at half the instruction count.
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// RN(RN(a / s) * w_scale) for two values at once, as div_by_scale then __fmul_rn: ns2 = -s,
// y2 = RN(1/s) of their tokens (fma(q, -s, a) is fma(-q, s, a) exactly)
__device__ __forceinline__ uint64_t div_scale2(uint64_t a, uint64_t ns2, uint64_t y2, uint64_t ws2) {
  uint64_t q = mul2(a, y2);
  uint64_t r = fma2(q, ns2, a);
  q = fma2(r, y2, q);
  r = fma2(q, ns2, a);
  q = fma2(r, y2, q);
  return mul2(q, ws2);
}
// finish_fast for two values at once: d2 the raw accumulators, z2 = -rowsum of their tokens
__device__ __forceinline__ uint64_t finish_fast2(uint64_t d2, uint64_t ns2, uint64_t y2, uint64_t z2, uint64_t ws2) {
  return div_scale2(fma2(d2, 0x4B8000004B800000ull, z2), ns2, y2, ws2);  // 2^24 in both lanes
}

__global__ void __launch_bounds__(THREADS, 1) gemm_prefill_kernel(const __grid_constant__ CUtensorMap tmW,
                                                                  const __grid_constant__ CUtensorMap tmX,
                                                                  const __grid_constant__ CUtensorMap tmO,
                                                                  const float* __restrict__ act_scale,
                                                                  const int32_t* __restrict__ rowsum, float w_scale,
                                                                  float* __restrict__ out,
                                                                  int32_t* __restrict__ acc_out, int M, int N, int K,
                                                                  int tma_store) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_stg[NSS];   // a block's bytes have landed (TMA transaction bytes)
  __shared__ __align__(8) uint64_t empty_stg[NSS];  // the converters are done with a staging slot
  __shared__ __align__(8) uint64_t full_ab[NAB];    // a stage's A columns and B tile are written
  __shared__ __align__(8) uint64_t empty_ab[NAB];   // the MMAs reading a stage are done (one commit)
  __shared__ __align__(8) uint64_t done_bar;        // every MMA complete
  __shared__ uint32_t tmem_slot;
  __shared__ float4 tok[TT];
  __shared__ __align__(16) float tk_ns[TT], tk_y[TT], tk_z[TT];  // -s, RN(1/s), -rowsum per token

  pdl_launch_dependents();
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = raw_addr + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t bring = base;                      // NAB fp16 B tiles (1024-byte aligned)
  const uint32_t stg = base + NAB * B_STAGE;        // NSS staging slots: weights, then tokens
  const uint32_t ostage = base;                     // epilogue: [token][row] fp32 (after the MMAs)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * TWR, m0 = blockIdx.z * TT;
  const int cs = (int)gridDim.y;
  const int rank = cs > 1 ? (int)cluster_ctarank() : 0;
  const int nblk_all = K / 128;
  const int b_lo = nblk_all * rank / cs, b_hi = nblk_all * (rank + 1) / cs;
  const int nblk = b_hi - b_lo, nst = 2 * nblk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSS; ++s) {
      mbar_init(&full_stg[s], 1);
      mbar_init(&empty_stg[s], CONV_WARPS);
    }
    for (int s = 0; s < NAB; ++s) {
      mbar_init(&full_ab[s], CONV_WARPS / 2);  // one group writes a stage
      mbar_init(&empty_ab[s], 1);
    }
    mbar_init(&done_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
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
      int issued = 0;
      // weights do not depend on the previous kernel: the first slots' weights go before the wait
      const int pre = nblk < NSS ? nblk : NSS;
      for (int b = 0; b < pre; ++b) {
        mbar_arrive_expect_tx(&full_stg[b], STG_BYTES);
        tma_load_2d(stg + b * STG_BYTES, &tmW, 32 * (b_lo + b), n0, &full_stg[b]);
      }
      pdl_wait();  // the tokens may be the previous kernel's output
      for (int b = 0; b < pre; ++b) {
        tma_load_2d(stg + b * STG_BYTES + STG_W, &tmX, 128 * (b_lo + b), m0, &full_stg[b]);
        tma_load_2d(stg + b * STG_BYTES + STG_W + STG_X / 2, &tmX, 128 * (b_lo + b) + 64, m0, &full_stg[b]);
      }
      issued = pre;
      for (int b = pre; b < nblk; ++b) {
        const int slot = b % NSS, use = b / NSS;
        if (!mbar_wait(&empty_stg[slot], (uint32_t)(use - 1) & 1u, &abort)) break;
        mbar_arrive_expect_tx(&full_stg[slot], STG_BYTES);
        tma_load_2d(stg + slot * STG_BYTES, &tmW, 32 * (b_lo + b), n0, &full_stg[slot]);
        tma_load_2d(stg + slot * STG_BYTES + STG_W, &tmX, 128 * (b_lo + b), m0, &full_stg[slot]);
        tma_load_2d(stg + slot * STG_BYTES + STG_W + STG_X / 2, &tmX, 128 * (b_lo + b) + 64, m0, &full_stg[slot]);
        issued = b + 1;
      }
      {  // every copy issued lands before the producer leaves (the converters may have given up)
        bool dummy = false;
        for (int i = issued - NSS > 0 ? issued - NSS : 0; i < issued; ++i)
          mbar_wait(&full_stg[i % NSS], (uint32_t)(i / NSS) & 1u, &dummy);
      }
    }
    // The other lanes wait here, at a warp barrier, not in a polling loop of their own: a lane
    // suspended in mbarrier.try_wait holds back the whole warp, the producing lane included.
    __syncwarp();
  } else if (warp == 1) {
    // ================================ MMA issuer ================================
    // The issuing thread is on the critical path: a 128 x 128 x 16 MMA keeps the tensor pipe busy
    // for only ~45 cycles, and this warp shares its scheduler with four converter warps. So every
    // operand of the 8 MMAs of each of the NAB stage slots is formed once, before the loop, and
    // the loop, unrolled over the slots, issues nothing but the waits, the MMAs and the commits.
    if (lane == 0) {
      const uint64_t bdesc0 = make_sw128_kmajor_desc(bring);
      const uint32_t bhi = (uint32_t)(bdesc0 >> 32);  // the address field is in the low word and
      const uint32_t blo0 = (uint32_t)bdesc0;         // the offsets below never carry out of it
      const uint32_t acol0 = tmem + (uint32_t)ACC_COLS;
      const uint32_t d0 = tmem, d1 = tmem + (uint32_t)TT;
      auto stage = [&](int s, uint32_t acc_first) {
        const uint32_t a = acol0 + (uint32_t)(s * A_STAGE_COLS);
        const uint32_t bl = blo0 + (uint32_t)((s * B_STAGE) >> 4);
        mma_f16_ts2(d0, a, bl, bhi, IDESC, acc_first);
        mma_f16_ts2(d0, a + 8, bl + 2, bhi, IDESC, 1u);
        mma_f16_ts2(d0, a + 16, bl + 4, bhi, IDESC, 1u);
        mma_f16_ts2(d0, a + 24, bl + 6, bhi, IDESC, 1u);
        mma_f16_ts2(d1, a + 32, bl, bhi, IDESC, acc_first);
        mma_f16_ts2(d1, a + 40, bl + 2, bhi, IDESC, 1u);
        mma_f16_ts2(d1, a + 48, bl + 4, bhi, IDESC, 1u);
        mma_f16_ts2(d1, a + 56, bl + 6, bhi, IDESC, 1u);
        mma_commit(&empty_ab[s]);
      };
      int i = 0;
      for (uint32_t ph = 0; i < nst; ph ^= 1u) {
#pragma unroll
        for (int s = 0; s < NAB; ++s, ++i) {
          if (i >= nst || !mbar_wait(&full_ab[s], ph, &abort)) break;
          tc_fence_after();
          stage(s, i > 0 ? 1u : 0u);
        }
        if (abort) break;
      }
      mma_commit(&done_bar);  // tracks every MMA this thread issued
    }
    __syncwarp();  // as for the producer: the idle lanes must not poll beside the issuing lane
  } else {
    // ================================ converters ================================
    // Two groups of 8 warps take alternate stages (group g the stages with h = g of every block),
    // so each warp has two stage periods for its loads, conversion, tensor-memory store, fences
    // and arrival. Within a group, warp (tile, lane quarter) owns 32 weight rows.
    const int cw = warp - 2;                  // 0..15
    const int grp = cw >> 3, gw = cw & 7;
    const int quarter = warp & 3, tile = gw >> 2;
    const int row = tile * 128 + 32 * quarter + lane;  // this thread's weight row in the tile
    const int gt = gw * 32 + lane;            // 0..255: token pieces gt and gt + 256 of the stage
    const uint32_t a_lane = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(ACC_COLS + 32 * tile);
    for (int b = 0; b < nblk; ++b) {
      const int i = 2 * b + grp, slot = b % NSS, s = i % NAB;
      const uint32_t sb = stg + slot * STG_BYTES;
      if (!mbar_wait_warp(&full_stg[slot], (uint32_t)(b / NSS) & 1u, &abort)) break;
      // the row's 32 bytes, the two halves in a lane-dependent order (no bank conflicts)
      const uint32_t c0 = (uint32_t)(lane >> 2) & 1u;
      const uint4 va = lds_v4(sb + row * 32 + 16 * c0), vb = lds_v4(sb + row * 32 + 16 * (c0 ^ 1u));
      const uint4 v0 = c0 ? vb : va, v1 = c0 ? va : vb;
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      uint4 xv[2];  // 16 k of a token each: pieces p = gt + 256v (token p / 4, chunk p % 4)
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        const int p = gt + 256 * v;
        xv[v] = lds_v4(sb + STG_W + grp * (STG_X / 2) + (p >> 2) * 64 + 16 * (p & 3));
      }
      if (i >= NAB && !mbar_wait_warp(&empty_ab[s], (uint32_t)(i / NAB - 1) & 1u, &abort)) break;
      tc_fence_after();
      {  // A: bit pairs 2g, 2g + 1 of the row's 32 bytes -> 32 columns (pair jj: 16jj + 2q, + 1)
        uint32_t a[32];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int sh = 6 - 2 * (2 * grp + jj);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            a[16 * jj + 2 * q] = (w[q] >> sh) & 0x00030003u;            // bytes 0, 2: c * 2^-24
            a[16 * jj + 2 * q + 1] = (w[q] >> (sh + 8)) & 0x00030003u;  // bytes 1, 3
          }
        }
        tmem_st_32x32b_x32(a_lane + (uint32_t)(s * A_STAGE_COLS), a);
      }
      const uint32_t bt = bring + (uint32_t)(s * B_STAGE);
#pragma unroll
      for (int v = 0; v < 2; ++v) {  // B: 16 int8 -> 32 bytes of fp16 = chunks 2c, 2c + 1 of the token's row
        const int p = gt + 256 * v, t = p >> 2, c = p & 3;
        uint32_t f[8];
        s8x4_f16_perm(xv[v].x, f[0], f[1]);
        s8x4_f16_perm(xv[v].y, f[2], f[3]);
        s8x4_f16_perm(xv[v].z, f[4], f[5]);
        s8x4_f16_perm(xv[v].w, f[6], f[7]);
        sts128(bt + sw128(t, 2 * c), f[0], f[1], f[2], f[3]);
        sts128(bt + sw128(t, 2 * c + 1), f[4], f[5], f[6], f[7]);
      }
      tmem_st_wait();            // this thread's tensor-memory writes are complete
      fence_proxy_async_smem();  // its shared-memory writes -> the tensor core's reads
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&full_ab[s]);
        mbar_arrive(&empty_stg[slot]);  // this group is done with the block's staged bytes
      }
    }
    const int ct = cw * 32 + lane;
    // the tile's per-token constants (the scales and row sums are the previous kernel's output)
    pdl_wait();
    if (ct < TT) {
      const int m = m0 + ct;
      const float sc = m < M ? __ldg(act_scale + m) : 1.0f;
      const float4 c = make_float4(sc, __frcp_rn(sc), -(float)(m < M ? __ldg(rowsum + m) : 0),
                                   (sc >= 0x1p-100f && sc <= 0x1p100f) ? 1.0f : 0.0f);
      tok[ct] = c;
      tk_ns[ct] = -sc;
      tk_y[ct] = c.y;
      tk_z[ct] = c.z;
    }
  }

  // ---- every MMA done: the rings are free ----
  const bool conv = warp >= 2;
  bool have = false;
  {
    bool dummy = false;
    if (conv)
      have = mbar_wait_warp(&done_bar, 0, &abort);
    else
      mbar_wait_warp(&done_bar, 0, &dummy);
  }
  tc_fence_after();
  __syncthreads();  // tok[] written; every MMA read of the rings done

  // Epilogue roles: converter warp (tile, lane quarter, half): its tile's 32 accumulator rows
  // (the lane quarter it may read) and tokens [64 half, 64 half + 64).
  const int cw = warp - 2, quarter = warp & 3, tile = (cw >> 2) & 1, half = cw >> 3;
  const int row = tile * 128 + 32 * quarter + lane;  // the accumulator row this thread reads
  const int n = n0 + row;
  const uint32_t tacc = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(tile * TT);
  const bool plain = !tma_store;  // else: TMA stores of the staged tile

  if (cs == 1) {
    // the whole tile is this CTA's: finish straight from the accumulators, 32 tokens at a time;
    // each half's 8 warps meet at a named barrier and one thread stores the 32 finished tokens
    if (conv) {
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int cb = 64 * half + 32 * cc;
        if (have) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tacc + (uint32_t)cb, v);
          tmem_ld_wait();
          const bool fast = __all_sync(0xffffffffu, token_const(tok, cb + lane).w != 0.0f) && acc_out == nullptr;
          if (fast) {
            const uint64_t ws2 = f2pack(w_scale, w_scale);
#pragma unroll
            for (int e = 0; e < 32; e += 4) {  // four tokens' constants per 16-byte broadcast read
              const float4 ns4 = *reinterpret_cast<const float4*>(tk_ns + cb + e);
              const float4 y4 = *reinterpret_cast<const float4*>(tk_y + cb + e);
              const float4 z4 = *reinterpret_cast<const float4*>(tk_z + cb + e);
              float o[4];
              f2unpack(finish_fast2(f2pack(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), f2pack(ns4.x, ns4.y),
                                    f2pack(y4.x, y4.y), f2pack(z4.x, z4.y), ws2),
                       o[0], o[1]);
              f2unpack(finish_fast2(f2pack(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])), f2pack(ns4.z, ns4.w),
                                    f2pack(y4.z, y4.w), f2pack(z4.z, z4.w), ws2),
                       o[2], o[3]);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                if (plain) {
                  const int m = m0 + cb + e + i;
                  if (m < M && n < N) out[(int64_t)m * N + n] = o[i];
                } else {
                  sts32(ostage + (uint32_t)(((cb + e + i) * TWR + row) * 4), o[i]);
                }
              }
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              int ai;
              const float o = finish_any(__uint_as_float(v[e]), token_const(tok, cb + e), w_scale, &ai);
              if (plain) {
                const int m = m0 + cb + e;
                if (m < M && n < N) {
                  out[(int64_t)m * N + n] = o;
                  if (acc_out) acc_out[(int64_t)m * N + n] = ai;
                }
              } else {
                sts32(ostage + (uint32_t)(((cb + e) * TWR + row) * 4), o);
              }
            }
          }
        }
        if (!plain) {
          fence_proxy_async_smem();                      // the staged values -> the TMA engine
          named_bar_sync(BAR_HALF + half, CONV_THREADS / 2);  // this half's 8 warps
          if (cw == 8 * half && lane == 0 && have && m0 + cb < M) {
            tma_store_2d(&tmO, n0, m0 + cb, ostage + (uint32_t)(cb * TWR * 4));
            bulk_commit();
          }
          __syncwarp();  // the warp converges before the next collective tensor-memory load
        }
      }
      if (!plain && cw == 8 * half && lane == 0) bulk_wait_all();  // before the CTA may leave
      __syncwarp();  // and before the warp reaches the teardown barrier as a whole
    }
  } else {
    // split K: every CTA stages its exact partials as int32, token-major; after a cluster barrier
    // each owner pulls its tokens' partials from every peer, sums them, finishes them in place
    // and stores them.
    if (conv && have) {
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int cb = 64 * half + 32 * cc;
        uint32_t v[32];
        tmem_ld_32x32b_x32(tacc + (uint32_t)cb, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e)
          sts32i(ostage + (uint32_t)(((cb + e) * TWR + row) * 4), __float2int_rn(__uint_as_float(v[e]) * 16777216.0f));
      }
    }
    const int t_lo = tok_lo(rank, cs), t_hi = tok_lo(rank + 1, cs);
    const int ct = cw * 32 + lane;
    cluster_arrive_release();
    cluster_wait_acquire();  // every CTA's partials are staged
    if (conv && have) {
      // thread (row quad, token slot): 4 consecutive rows of one owned token at a time, every
      // peer's 16 bytes requested before any is added
      const int quad = ct & 63, r4 = 4 * quad;
#pragma unroll 1
      for (int t = t_lo + (ct >> 6); t < t_hi; t += 8) {
        const uint32_t off = ostage + (uint32_t)((t * TWR + r4) * 4);
        uint4 part[kMaxCluster];
#pragma unroll
        for (int p = 0; p < kMaxCluster; ++p)
          part[p] = p >= cs ? make_uint4(0u, 0u, 0u, 0u)
                            : (p == rank ? lds_v4(off) : ld_cluster_v4(map_to_rank(off, (uint32_t)p)));
        int sum[4] = {0, 0, 0, 0};
#pragma unroll
        for (int p = 0; p < kMaxCluster; ++p) {
          sum[0] += (int)part[p].x, sum[1] += (int)part[p].y, sum[2] += (int)part[p].z, sum[3] += (int)part[p].w;
        }
        const float4 c = token_const(tok, t);
        float a[4], o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = (float)(sum[i] + (int)c.z);  // raw - rowsum, exactly
        if (c.w != 0.0f) {  // warp-uniform (one token per warp)
          const uint64_t ns2 = f2pack(-c.x, -c.x), y2 = f2pack(c.y, c.y), ws2 = f2pack(w_scale, w_scale);
          f2unpack(div_scale2(f2pack(a[0], a[1]), ns2, y2, ws2), o[0], o[1]);
          f2unpack(div_scale2(f2pack(a[2], a[3]), ns2, y2, ws2), o[2], o[3]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i] = __fmul_rn(__fdiv_rn(a[i], c.x), w_scale);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (plain) {
            const int m = m0 + t, cn = n0 + r4 + i;
            if (m < M && cn < N) {
              out[(int64_t)m * N + cn] = o[i];
              if (acc_out) acc_out[(int64_t)m * N + cn] = (int)a[i];
            }
          }
        }
        // peers read only the tokens they own: this token is finished in place
        if (!plain) sts128(off, __float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]), __float_as_uint(o[3]));
      }
    }
    if (!plain) {  // the owned token rows leave by TMA bulk stores of 8 rows
      fence_proxy_async_smem();
      named_bar_sync(BAR_ALL, THREADS);
      if (threadIdx.x == 0 && !abort) {
        for (int t = t_lo; t < t_hi && m0 + t < M; t += 8) tma_store_2d(&tmO, n0, m0 + t, ostage + (uint32_t)(t * TWR * 4));
        bulk_commit();
        bulk_wait_all();
      }
      __syncwarp();
    }
  }

  if (cs > 1) {  // no CTA leaves while a peer may still read its shared memory
    cluster_arrive_release();
    cluster_wait_acquire();
  }

  // ---- teardown: every MMA completes before the tensor memory is freed ----
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// 2-D tensor [rows][inner] of 1- or 4-byte elements, box box_inner x box_rows, no swizzle.
bool make_map(CUtensorMap* map, CUtensorMapDataType dt, int esize, const void* base, int64_t rows, int64_t inner,
              int box_inner, int box_rows) {
  return encode_map_2d(map, dt, base, (uint64_t)inner, (uint64_t)rows, (uint64_t)(inner * esize),
                       (uint32_t)box_inner, (uint32_t)box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace

cudaError_t read_clear_device_error_prefill(int* value) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

bool gemm_prefill_supported(int64_t M, int64_t N, int64_t K) {
  return M >= 1 && N >= 1 && K >= 128 && K % 128 == 0 && K <= 32768 && (M + TT - 1) / TT <= 65535 &&
         (N + TWR - 1) / TWR <= 0x7fffffff;
}

cudaError_t launch_gemm_prefill(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                                float w_scale, float* out, int32_t* acc_out, int64_t M, int64_t N, int64_t K,
                                int num_sms, cudaStream_t stream) {
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(gemm_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_prefill_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  // One CTA per SM (the shared memory allows one). Tiles = weight tiles x token tiles; when they
  // leave SMs idle, the blocks of K are split over a cluster of cs CTAs, as large as lets every
  // CTA run at once (at least one block each, at most 16), checked with the occupancy query.
  const int64_t n_w = (N + TWR - 1) / TWR, n_t = (M + TT - 1) / TT, tiles = n_w * n_t;
  const int64_t nblk = K / 128;
  int64_t cs = num_sms / tiles;
  if (cs > kMaxCluster) cs = kMaxCluster;
  if (cs > nblk) cs = nblk;
  if (cs < 1) cs = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  for (; cs > 1; --cs) {
    attr[0].val.clusterDim.y = (unsigned)cs;
    cfg.gridDim = dim3((unsigned)n_w, (unsigned)cs, (unsigned)n_t);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_prefill_kernel, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();  // the query is only a hint; keep shrinking to the portable size
      if (cs <= 8) break;
      continue;
    }
    if (clusters >= tiles) break;
  }
  attr[0].val.clusterDim.y = (unsigned)cs;
  cfg.gridDim = dim3((unsigned)n_w, (unsigned)cs, (unsigned)n_t);
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;

  CUtensorMap mW, mX, mO;
  if (!make_map(&mW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, wp, N, K / 4, 32, TWR) ||
      !make_map(&mX, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, xq, M, K, 64, TT))
    return cudaErrorInvalidValue;
  // The finished tile leaves by TMA stores when the output rows are 16-byte aligned and the
  // int32 accumulators are not wanted; otherwise element by element.
  const bool tma_store = (N % 4 == 0) && (reinterpret_cast<uintptr_t>(out) & 15) == 0 && acc_out == nullptr;
  std::memset(&mO, 0, sizeof(mO));
  if (tma_store && !make_map(&mO, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, out, M, N, TWR, cs == 1 ? kStoreRows : 8))
    return cudaErrorInvalidValue;
  return cudaLaunchKernelEx(&cfg, gemm_prefill_kernel, mW, mX, mO, act_scale, rowsum, w_scale, out, acc_out, (int)M,
                            (int)N, (int)K, tma_store ? 1 : 0);
}

}  // namespace bitnet
