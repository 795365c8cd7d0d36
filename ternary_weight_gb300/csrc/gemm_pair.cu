// gemm_pair.cu -- the W2A8 ternary matmul for prompts (beyond 64 tokens) on CTA pairs: the
// prompt-length kernel's in-kernel expansion (packed weights and int8 tokens staged by TMA,
// expanded to exact fp16) with the 2-SM MMA, tcgen05.mma.cta_group::2.kind::f16, M = 256 weight
// rows over the pair, N = PT = 2 HT tokens (HT = 128, or 64 for prompts up to 128 tokens),
// K = 16. No workspace.
//
// Computes, like every other path of the library, raw[m][n] = sum_k code[n][k] * xq[m][k],
// acc = raw - rowsum[m], out = (acc / s[m]) * w_scale, with the same integers and the same fp32
// results. Sources: the raw code dot over the 4x32-interleaved i2_s bytes ("[분석/검증-3]
// BitNet.cpp ARM 커널 재작성" §3, "[기술 분석 보고서] ... 추론 붕괴 원인 분석" §3.2), the byte
// layout ("BitNet 딥다이브" §4-2), the dequantisation ("bitnet.rs" "Quantised Forward Pass").
// "BitNet 딥다이브" §4-5 runs prefill as a separate dense path; this is that path.
//
// Why pairs. In the one-CTA kernel (gemm_prefill.cu, 256 rows x 128 tokens per SM) the stage rate
// is set by the latency of the operand ring's cycle: the converter warps of a stage wait for the
// MMAs that last read its slot, and tensor memory holds only 4 slots of A next to the 2 x 128
// accumulator columns. Here the pair's M = 256 puts 128 weight rows in each SM: per 64-k stage and
// SM the converters expand half the weights (128 rows) and HT tokens, the accumulator is 128 rows
// x PT tokens (256 columns at HT = 128: the same flops per SM as the one-CTA kernel), A takes 32
// columns a stage, so 8 slots fit, and one MMA instruction covers what took four.
//
// Operands and K order are those of the one-CTA kernel:
//  * A (weights): the code c as the fp16 subnormal c * 2^-24, written with tcgen05.st into this
//    CTA's tensor memory; the MMA reads A from both CTAs' tensor memory at the same address;
//  * B (tokens): 0x6400 | (x + 128) minus 1152 = x as an exact fp16, into a 128-byte-swizzled
//    K-major tile in shared memory. The pair's B is split by N: CTA 0 of the pair holds tokens
//    0..HT-1 of the tile, CTA 1 tokens HT..PT-1, at the same shared-memory offset;
//  * every partial sum is a multiple of 2^-24 below 1 in magnitude (K <= 32768): exact in fp32.
// Stage position p holds k = 4 (p / 4) + sigma(p % 4), sigma = (0, 2, 1, 3), in A and B alike.
//
// Roles per CTA (576 threads):
//  * warp 0, one lane: 2-D TMA of this CTA's 128 weight rows x 32 bytes and HT tokens x 2 x 64
//    bytes per 128-k block into 4 staging slots (the weights of the first slots before the
//    dependency wait);
//  * warps 2-17: two groups of 8 converter warps on alternate 64-k stages; in a group, warp
//    (lane quarter q, half jj) writes bit pair 2h + jj of its 32 rows as 16 A columns, and every
//    thread converts HT / 64 16-byte token pieces into B. One arrival per warp on the stage's full
//    barrier, which lives in the pair's even CTA (the odd CTA's warps arrive remotely);
//  * warp 1 of the even CTA, one lane: waits for both CTAs' operands,
//    issues the stage's 4 MMAs and one commit multicast to both CTAs' empty barriers; a last
//    commit multicasts the completion of every MMA;
//  * epilogue: each CTA reads its 128 rows x PT tokens from its own tensor memory and finishes
//    them as the one-CTA kernel does (Markstein's division, two values per instruction, TMA
//    bulk stores of token-major staged rows).
// Split K: when the pair tiles leave SMs idle, cs k-slices run as a cluster of 2 x cs CTAs (rank =
// pair position + 2 x slice); each CTA stages its int32 partials and the slice r owner of tokens
// [8 floor((PT / 8) r / cs), 8 floor((PT / 8) (r + 1) / cs)) pulls them from the same pair
// position of every slice with 16-byte distributed-shared-memory loads. When the pair tiles fill
// whole waves and leave a partial one, the host runs the partial wave's token rows as a second,
// split-K launch.
// Every mbarrier wait is bounded; a timeout is recorded in the device error word, and the TMA
// producer waits (bounded) for its copies in flight before it leaves.
#include "bitnet_dev.cuh"
#include "gemm_pair.h"

#include <atomic>
#include <cstring>

namespace bitnet {
namespace {

constexpr int PR = 128;                  // weight rows per CTA (half of the pair's M)
constexpr int CONV_WARPS = 16;
constexpr int CONV_THREADS = CONV_WARPS * 32;
constexpr int THREADS = CONV_THREADS + 64;
constexpr int NAB = 8;                   // A/B stages (64 k each)
constexpr int STG_W = PR * 32;           // packed weights of one block: 128 rows x 32 bytes
constexpr uint32_t TMEM_COLS = 512;      // accumulator (up to 256) + 8 A stages x 32
constexpr int A_STAGE_COLS = 32;         // 128 rows x 64 k fp16
constexpr int kMaxSplit = 8;             // k-slices: a cluster of at most 16 CTAs
constexpr int kStoreRows = 32;           // tokens per TMA store (no split)
constexpr int BAR_ALL = 1;               // named barrier of the whole CTA
constexpr int BAR_TQ = 2;                // named barriers 2..5: the 4 warps of one token quarter

constexpr int NSS = 4;                   // staging slots (one 128-k block each); 6 or 8 measured no
                                         // faster with the 128-token tile, nor 6 with the 256-token one
// The token tile: HT tokens of B per CTA, PT = 2 HT per pair (the MMA's N): 256 for long prompts,
// 128 for prompts of about a hundred tokens (the 256-token tile would be half empty there).
template <int HT_>
struct PairTile {
  static constexpr int HT = HT_;
  static constexpr int PT = 2 * HT;
  static constexpr int XV = HT / 64;               // 16-byte token pieces per converter thread and stage
  static constexpr int STG_X = HT * 128;           // int8 tokens of one block: [half][HT rows][64 bytes]
  static constexpr int STG_BYTES = STG_W + STG_X;
  static constexpr int B_STAGE = HT * 128;         // fp16 B of one stage: HT tokens x 64 k x 2 bytes
  static constexpr int SMEM = 1024 + NAB * B_STAGE + NSS * STG_BYTES;
  static constexpr int OUT_STAGE = PT * PR * 4;    // token-major fp32 tile of the epilogue (reuses the rings)
  static constexpr int ACC_COLS = PT;
  static constexpr int TCH = PT / 128;             // 32-token chunks per epilogue warp
  static constexpr uint32_t IDESC = make_idesc_f16_f32(256, PT);
  // split K: slice r of cs owns tokens [tok_lo(r), tok_lo(r + 1)) of the pair tile, in groups of 8
  static __host__ __device__ constexpr int tok_lo(int r, int cs) { return 8 * ((PT / 8) * r / cs); }
  static_assert(HT == 64 || HT == 128, "token tile");
  static_assert(ACC_COLS + NAB * A_STAGE_COLS <= (int)TMEM_COLS, "tensor memory columns");
  static_assert(SMEM <= 227 * 1024 - 8192, "shared memory (static part included)");
  static_assert(OUT_STAGE <= NAB * B_STAGE + NSS * STG_BYTES, "the epilogue tile fits the reused rings");
};

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
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
__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
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

// ---- the CTA pair: tensor memory allocated for both, MMAs issued by the even CTA ----
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {  // one warp of each CTA
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D (both CTAs' tensor memory, 128 lanes each) (+)= A (both CTAs' tensor memory at a_tmem) * B^T
// (the descriptor's tile in both CTAs' shared memory: N / 2 rows each)
__device__ __forceinline__ void mma_pair_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 bd;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "mov.b64 bd, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], bd, %5, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(accumulate), "r"(idesc)
      : "memory");
}
// one arrival on the barrier at this offset in every CTA of cta_mask once the MMAs issued so far
// are complete
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "h"(cta_mask)
               : "memory");
}
// one arrival on a barrier in a peer CTA (a shared::cluster address), with the instruction's
// default semantics (release, CTA scope): a release at cluster scope measured ~1200-1500 cycles
// per arrival, which put it on the stage's critical path
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// bounded wait, acquire at cluster scope (the arrivals include a peer CTA's)
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, bool* abort) {
  if (*abort) return false;
  const uint32_t a = smem_u32(bar);
  for (uint32_t i = 0; i < kMaxPolls; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  record_device_error(kErrTimeout);
  *abort = true;
  return false;
}

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 4 int8 -> 4 exact fp16 in stage order: (bytes 0, 2) and (bytes 1, 3)
__device__ __forceinline__ void s8x4_f16_perm(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;  // x + 128 per byte
  const uint32_t l = __byte_perm(u, 0x64646464u, 0x4240);
  const uint32_t h = __byte_perm(u, 0x64646464u, 0x4341);
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(l), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(h), "r"(0x64806480u));
}

// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major tile
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// RN(a / s) for an integer-valued a (|a| < 2^25) and s in [2^-100, 2^100], given y = RN(1/s):
// Markstein's residual correction, twice (exact remainders by fma)
__device__ __forceinline__ float div_by_scale(float a, float s, float y) {
  float q = __fmul_rn(a, y);
  float r = __fmaf_rn(-q, s, a);
  q = __fmaf_rn(r, y, q);
  r = __fmaf_rn(-q, s, a);
  return __fmaf_rn(r, y, q);
}
// out = RN(RN((d * 2^24 - rowsum) / s) * w_scale) for any token (the IEEE division where the scale
// is extreme), and the integer acc
__device__ __forceinline__ float finish_any(float d, float4 c, float w_scale, int* acc_int) {
  const float a = __fmaf_rn(d, 16777216.0f, c.z);
  *acc_int = __float2int_rn(a);
  const float q = c.w != 0.0f ? div_by_scale(a, c.x, c.y) : __fdiv_rn(a, c.x);
  return __fmul_rn(q, w_scale);
}
// two fp32 lanes per instruction (each rounded as the scalar operation)
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
// RN(RN(a / s) * w_scale) for two values: ns2 = -s, y2 = RN(1/s) (fma(q, -s, a) is fma(-q, s, a))
__device__ __forceinline__ uint64_t div_scale2(uint64_t a, uint64_t ns2, uint64_t y2, uint64_t ws2) {
  uint64_t q = mul2(a, y2);
  uint64_t r = fma2(q, ns2, a);
  q = fma2(r, y2, q);
  r = fma2(q, ns2, a);
  q = fma2(r, y2, q);
  return mul2(q, ws2);
}
__device__ __forceinline__ uint64_t finish_fast2(uint64_t d2, uint64_t ns2, uint64_t y2, uint64_t z2, uint64_t ws2) {
  return div_scale2(fma2(d2, 0x4B8000004B800000ull, z2), ns2, y2, ws2);  // 2^24 in both lanes
}

template <int HT_>
__global__ void __launch_bounds__(THREADS, 1) gemm_pair_kernel(const __grid_constant__ CUtensorMap tmW,
                                                               const __grid_constant__ CUtensorMap tmX,
                                                               const __grid_constant__ CUtensorMap tmO,
                                                               const float* __restrict__ act_scale,
                                                               const int32_t* __restrict__ rowsum, float w_scale,
                                                               float* __restrict__ out, int32_t* __restrict__ acc_out,
                                                               int M, int N, int K, int tma_store) {
  using T = PairTile<HT_>;
  constexpr int HT = T::HT, PT = T::PT, XV = T::XV, STG_X = T::STG_X, STG_BYTES = T::STG_BYTES;
  constexpr int B_STAGE = T::B_STAGE, ACC_COLS = T::ACC_COLS, TCH = T::TCH;
  constexpr uint32_t IDESC = T::IDESC;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_stg[NSS];   // a block's bytes have landed (TMA transaction bytes)
  __shared__ __align__(8) uint64_t empty_stg[NSS];  // both groups are done with a staged block
  __shared__ __align__(8) uint64_t full_ab[NAB];    // (even CTA) both CTAs' operands of a stage are written
  __shared__ __align__(8) uint64_t empty_ab[NAB];   // the MMAs reading a stage are done (multicast commit)
  __shared__ __align__(8) uint64_t done_bar;        // every MMA complete (multicast commit)
  __shared__ uint32_t tmem_slot;
  __shared__ float4 tok[PT];
  __shared__ __align__(16) float tk_ns[PT], tk_y[PT], tk_z[PT];  // -s, RN(1/s), -rowsum per token

  pdl_launch_dependents();
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = raw_addr + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t bring = base;                      // NAB fp16 B tiles (1024-byte aligned)
  const uint32_t stg = base + NAB * B_STAGE;        // NSS staging slots: weights, then tokens
  const uint32_t ostage = base;                     // epilogue: [token][row] (after the MMAs)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pp = (int)(blockIdx.x & 1u);            // position in the pair
  const int n0 = (int)(blockIdx.x >> 1) * (2 * PR) + PR * pp;  // this CTA's weight rows
  const int m0 = (int)blockIdx.z * PT;              // the pair tile's tokens
  const int mb = m0 + HT * pp;                      // this CTA's B tokens
  const int cs = (int)gridDim.y;
  const int slice = (int)blockIdx.y;
  const uint32_t crank = cluster_ctarank();         // pp + 2 * slice
  const uint32_t lead = crank & ~1u;                // the pair's even CTA
  const uint16_t pair_mask = (uint16_t)(3u << lead);
  const int nblk_all = K / 128;
  const int b_lo = nblk_all * slice / cs, b_hi = nblk_all * (slice + 1) / cs;
  const int nblk = b_hi - b_lo, nst = 2 * nblk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSS; ++s) {
      mbar_init(&full_stg[s], 1);
      mbar_init(&empty_stg[s], CONV_WARPS);
    }
    for (int s = 0; s < NAB; ++s) {
      mbar_init(&full_ab[s], CONV_WARPS);  // one group of each CTA writes a stage
      mbar_init(&empty_ab[s], 1);
    }
    mbar_init(&done_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc_pair(&tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive_release();  // every CTA's barriers exist before a peer arrives on them
  cluster_wait_acquire();
  const uint32_t tmem = tmem_slot;
  bool abort = false;

  if (warp == 0) {
    // ================================ TMA producer ================================
    if (lane == 0) {
      int issued = 0;
      const int pre = nblk < NSS ? nblk : NSS;
      for (int b = 0; b < pre; ++b) {  // the weights do not depend on the previous kernel
        mbar_arrive_expect_tx(&full_stg[b], STG_BYTES);
        tma_load_2d(stg + b * STG_BYTES, &tmW, 32 * (b_lo + b), n0, &full_stg[b]);
      }
      pdl_wait();  // the tokens may be the previous kernel's output
      for (int b = 0; b < pre; ++b) {
        tma_load_2d(stg + b * STG_BYTES + STG_W, &tmX, 128 * (b_lo + b), mb, &full_stg[b]);
        tma_load_2d(stg + b * STG_BYTES + STG_W + STG_X / 2, &tmX, 128 * (b_lo + b) + 64, mb, &full_stg[b]);
      }
      issued = pre;
      for (int b = pre; b < nblk; ++b) {
        const int slot = b % NSS, use = b / NSS;
        if (!mbar_wait(&empty_stg[slot], (uint32_t)(use - 1) & 1u, &abort)) break;
        mbar_arrive_expect_tx(&full_stg[slot], STG_BYTES);
        tma_load_2d(stg + slot * STG_BYTES, &tmW, 32 * (b_lo + b), n0, &full_stg[slot]);
        tma_load_2d(stg + slot * STG_BYTES + STG_W, &tmX, 128 * (b_lo + b), mb, &full_stg[slot]);
        tma_load_2d(stg + slot * STG_BYTES + STG_W + STG_X / 2, &tmX, 128 * (b_lo + b) + 64, mb, &full_stg[slot]);
        issued = b + 1;
      }
      {  // every copy issued lands before the producer leaves (the converters may have given up)
        bool dummy = false;
        for (int i = issued - NSS > 0 ? issued - NSS : 0; i < issued; ++i)
          mbar_wait(&full_stg[i % NSS], (uint32_t)(i / NSS) & 1u, &dummy);
      }
    }
    // the other lanes wait at a warp barrier, not in a polling loop (a lane suspended in an
    // mbarrier poll holds back the producing lane of its warp)
    __syncwarp();
  } else if (warp == 1) {
    // ================================ MMA issuer (even CTA) ================================
    if (pp == 0 && lane == 0) {
      const uint64_t bdesc0 = make_sw128_kmajor_desc(bring);
      const uint32_t bhi = (uint32_t)(bdesc0 >> 32);
      const uint32_t blo0 = (uint32_t)bdesc0;
      const uint32_t acol0 = tmem + (uint32_t)ACC_COLS;
      auto stage = [&](int s, uint32_t acc_first) {
        const uint32_t a = acol0 + (uint32_t)(s * A_STAGE_COLS);
        const uint32_t bl = blo0 + (uint32_t)((s * B_STAGE) >> 4);
        mma_pair_ts(tmem, a, bl, bhi, IDESC, acc_first);
        mma_pair_ts(tmem, a + 8, bl + 2, bhi, IDESC, 1u);
        mma_pair_ts(tmem, a + 16, bl + 4, bhi, IDESC, 1u);
        mma_pair_ts(tmem, a + 24, bl + 6, bhi, IDESC, 1u);
        mma_commit_pair(&empty_ab[s], pair_mask);
      };
      int i = 0;
      for (uint32_t ph = 0; i < nst; ph ^= 1u) {
#pragma unroll
        for (int s = 0; s < NAB; ++s, ++i) {
          if (i >= nst || !mbar_wait_cluster(&full_ab[s], ph, &abort)) break;
          tc_fence_after();
          stage(s, i > 0 ? 1u : 0u);
        }
        if (abort) break;
      }
      mma_commit_pair(&done_bar, pair_mask);  // tracks every MMA this thread issued
    }
    __syncwarp();
  } else {
    // ================================ converters ================================
    const int cw = warp - 2;                     // 0..15
    const int grp = cw >> 3, gw = cw & 7;
    const int quarter = warp & 3, jj = gw >> 2;  // tensor-memory lane quarter; bit pair 2h + jj
    const int row = 32 * quarter + lane;         // this thread's weight row (of the CTA's 128)
    const int gt = gw * 32 + lane;               // token pieces gt (and gt + 256) of the stage
    const uint32_t a_lane = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(ACC_COLS + 16 * jj);
    const uint32_t full_remote = map_to_rank(smem_u32(&full_ab[0]), lead);
    for (int b = 0; b < nblk; ++b) {
      const int i = 2 * b + grp, slot = b % NSS, s = i % NAB;
      const uint32_t sb = stg + slot * STG_BYTES;
      if (!mbar_wait_warp(&full_stg[slot], (uint32_t)(b / NSS) & 1u, &abort)) break;
      const uint32_t c0 = (uint32_t)(lane >> 2) & 1u;  // the row's two 16-byte halves in a lane-dependent order
      const uint4 va = lds_v4(sb + row * 32 + 16 * c0), vb = lds_v4(sb + row * 32 + 16 * (c0 ^ 1u));
      const uint4 v0 = c0 ? vb : va, v1 = c0 ? va : vb;
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      uint4 xv[XV];
#pragma unroll
      for (int v = 0; v < XV; ++v) {
        const int p = gt + 256 * v;
        xv[v] = lds_v4(sb + STG_W + grp * (STG_X / 2) + (p >> 2) * 64 + 16 * (p & 3));
      }
      if (i >= NAB && !mbar_wait_warp(&empty_ab[s], (uint32_t)(i / NAB - 1) & 1u, &abort)) break;
      tc_fence_after();
      {  // A: bit pair 2h + jj of the row's 32 bytes -> 16 columns (16 jj + 2q, + 1)
        const int sh = 6 - 2 * (2 * grp + jj);
        uint32_t a[16];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          a[2 * q] = (w[q] >> sh) & 0x00030003u;            // bytes 0, 2: c * 2^-24
          a[2 * q + 1] = (w[q] >> (sh + 8)) & 0x00030003u;  // bytes 1, 3
        }
        tmem_st_32x32b_x16(a_lane + (uint32_t)(s * A_STAGE_COLS), a);
      }
      const uint32_t bt = bring + (uint32_t)(s * B_STAGE);
#pragma unroll
      for (int v = 0; v < XV; ++v) {  // B: 16 int8 -> 32 bytes of fp16 = chunks 2c, 2c + 1 of the token's row
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
        if (pp == 0)
          mbar_arrive(&full_ab[s]);
        else
          mbar_arrive_remote(full_remote + (uint32_t)(s * 8));
        mbar_arrive(&empty_stg[slot]);  // this group is done with the block's staged bytes
      }
    }
    const int ct = cw * 32 + lane;
    // the pair tile's per-token constants (the scales and row sums are the previous kernel's output)
    pdl_wait();
    if (ct < PT) {
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

  // Epilogue roles: converter warp (lane quarter, token quarter tq): its 32 accumulator rows and
  // tokens [PT/4 tq, PT/4 (tq + 1)) of the pair tile, in TCH chunks of 32.
  const int cw = warp - 2, quarter = warp & 3, tq = (cw >> 2) & 3;
  const int row = 32 * quarter + lane;
  const int n = n0 + row;
  const uint32_t tacc = tmem + ((uint32_t)(32 * quarter) << 16);
  const bool plain = !tma_store;

  if (cs == 1) {
    if (conv) {
#pragma unroll 1
      for (int cc = 0; cc < TCH; ++cc) {
        const int cb = (PT / 4) * tq + 32 * cc;
        if (have) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tacc + (uint32_t)cb, v);
          tmem_ld_wait();
          const bool fast = __all_sync(0xffffffffu, tok[cb + lane].w != 0.0f) && acc_out == nullptr;
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
                  sts32(ostage + (uint32_t)(((cb + e + i) * PR + row) * 4), o[i]);
                }
              }
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              int ai;
              const float o = finish_any(__uint_as_float(v[e]), tok[cb + e], w_scale, &ai);
              if (plain) {
                const int m = m0 + cb + e;
                if (m < M && n < N) {
                  out[(int64_t)m * N + n] = o;
                  if (acc_out) acc_out[(int64_t)m * N + n] = ai;
                }
              } else {
                sts32(ostage + (uint32_t)(((cb + e) * PR + row) * 4), o);
              }
            }
          }
        }
        if (!plain) {
          fence_proxy_async_smem();                 // the staged values -> the TMA engine
          named_bar_sync(BAR_TQ + tq, 128);          // this token quarter's 4 warps
          if (quarter == 0 && lane == 0 && have && m0 + cb < M) {
            tma_store_2d(&tmO, n0, m0 + cb, ostage + (uint32_t)(cb * PR * 4));
            bulk_commit();
          }
          __syncwarp();  // the warp converges before the next collective tensor-memory load
        }
      }
      if (!plain && quarter == 0 && lane == 0) bulk_wait_all();  // before the CTA may leave
      __syncwarp();  // and before the warp reaches the teardown barrier as a whole
    }
  } else {
    // split K: every CTA stages its exact partials as int32, token-major; after a cluster barrier
    // each owner pulls its tokens' partials from the same pair position of every slice, sums them,
    // finishes them in place and stores them.
    if (conv && have) {
#pragma unroll 1
      for (int cc = 0; cc < TCH; ++cc) {
        const int cb = (PT / 4) * tq + 32 * cc;
        uint32_t v[32];
        tmem_ld_32x32b_x32(tacc + (uint32_t)cb, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e)
          sts32i(ostage + (uint32_t)(((cb + e) * PR + row) * 4), __float2int_rn(__uint_as_float(v[e]) * 16777216.0f));
      }
    }
    const int t_lo = T::tok_lo(slice, cs), t_hi = T::tok_lo(slice + 1, cs);
    const int ct = cw * 32 + lane;
    cluster_arrive_release();
    cluster_wait_acquire();  // every CTA's partials are staged
    if (conv && have) {
      // thread (row quad, token slot): 4 consecutive rows of one owned token at a time (a warp
      // reads 512 contiguous bytes of one token), every slice's 16 bytes requested before any is
      // added
      const int quad = ct & 31, r4 = 4 * quad;
#pragma unroll 1
      for (int t = t_lo + (ct >> 5); t < t_hi; t += 16) {
        const uint32_t off = ostage + (uint32_t)((t * PR + r4) * 4);
        uint4 part[kMaxSplit];
#pragma unroll
        for (int p = 0; p < kMaxSplit; ++p)
          part[p] = p >= cs ? make_uint4(0u, 0u, 0u, 0u)
                            : (p == slice ? lds_v4(off) : ld_cluster_v4(map_to_rank(off, (uint32_t)(pp + 2 * p))));
        int sum[4] = {0, 0, 0, 0};
#pragma unroll
        for (int p = 0; p < kMaxSplit; ++p) {
          sum[0] += (int)part[p].x, sum[1] += (int)part[p].y, sum[2] += (int)part[p].z, sum[3] += (int)part[p].w;
        }
        const float4 c = tok[t];
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
        for (int t = t_lo; t < t_hi && m0 + t < M; t += 8) tma_store_2d(&tmO, n0, m0 + t, ostage + (uint32_t)(t * PR * 4));
        bulk_commit();
        bulk_wait_all();
      }
      __syncwarp();
    }
  }

  // ---- teardown: no CTA leaves while a peer may read its shared memory or the pair's MMAs may
  // still use its tensor memory; then both CTAs free the pair's tensor memory ----
  tc_fence_before();
  __syncthreads();
  cluster_arrive_release();
  cluster_wait_acquire();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

// 2-D tensor [rows][inner] of 1- or 4-byte elements, box box_inner x box_rows, no swizzle.
bool make_map(CUtensorMap* map, CUtensorMapDataType dt, int esize, const void* base, int64_t rows, int64_t inner,
              int box_inner, int box_rows) {
  return encode_map_2d(map, dt, base, (uint64_t)inner, (uint64_t)rows, (uint64_t)(inner * esize),
                       (uint32_t)box_inner, (uint32_t)box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace

namespace {

template <int HT>
cudaError_t launch_pair(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                        float w_scale, float* out, int32_t* acc_out, int64_t M, int64_t N, int64_t K, int num_sms,
                        cudaStream_t stream) {
  using T = PairTile<HT>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(gemm_pair_kernel<HT>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_pair_kernel<HT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  // One CTA per SM. Pair tiles = (N / 256) x (M / PT); when their CTAs leave SMs idle, the blocks
  // of K are split over cs slices (a cluster of 2 x cs CTAs, cs <= 8, at least one block each),
  // as many as let every CTA run at once (the occupancy query).
  const int64_t n_w = (N + 2 * PR - 1) / (2 * PR), n_t = (M + T::PT - 1) / T::PT, tiles = n_w * n_t;
  const int64_t nblk = K / 128;
  int64_t cs = num_sms / (2 * tiles);
  if (cs > kMaxSplit) cs = kMaxSplit;
  if (cs > nblk) cs = nblk;
  if (cs < 1) cs = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = T::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  for (; cs > 1; --cs) {
    attr[0].val.clusterDim.y = (unsigned)cs;
    cfg.gridDim = dim3((unsigned)(2 * n_w), (unsigned)cs, (unsigned)n_t);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_pair_kernel<HT>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();  // the query is only a hint; keep shrinking to the portable size
      if (2 * cs <= 8) break;
      continue;
    }
    if (clusters >= tiles) break;
  }
  attr[0].val.clusterDim.y = (unsigned)cs;
  cfg.gridDim = dim3((unsigned)(2 * n_w), (unsigned)cs, (unsigned)n_t);
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;

  CUtensorMap mW, mX, mO;
  if (!make_map(&mW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, wp, N, K / 4, 32, PR) ||
      !make_map(&mX, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, xq, M, K, 64, HT))
    return cudaErrorInvalidValue;
  const bool tma_store = (N % 4 == 0) && (reinterpret_cast<uintptr_t>(out) & 15) == 0 && acc_out == nullptr;
  std::memset(&mO, 0, sizeof(mO));
  if (tma_store && !make_map(&mO, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, out, M, N, PR, cs == 1 ? kStoreRows : 8))
    return cudaErrorInvalidValue;
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<HT>, mW, mX, mO, act_scale, rowsum, w_scale, out, acc_out, (int)M,
                            (int)N, (int)K, tma_store ? 1 : 0);
}

}  // namespace

bool gemm_pair_supported(int64_t M, int64_t N, int64_t K) {
  return M >= 1 && N >= 1 && K >= 128 && K % 128 == 0 && K <= 32768 && (M + 127) / 128 <= 65535 &&
         2 * ((N + 2 * PR - 1) / (2 * PR)) <= 0x7fffffff;
}

// The 128-token tile (64 per CTA) up to 128 rows, where the 256-token tile would be at least half
// empty; the 256-token tile beyond. When the pair tiles fill some whole waves (one pair per two
// SMs) and leave a partial one, the token rows of that last wave go to a second launch that
// splits K over up to 8 slices, so that the tail takes a fraction of a round instead of a whole
// one (M = 4096, N = 2560: 160 tiles on 76 pairs, 3 rounds for 2.1 rounds of work).
cudaError_t launch_gemm_pair(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                             float w_scale, float* out, int32_t* acc_out, int64_t M, int64_t N, int64_t K, int num_sms,
                             cudaStream_t stream) {
  if (M <= 128)
    return launch_pair<64>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, num_sms, stream);
  constexpr int64_t PT = PairTile<128>::PT;
  const int64_t n_w = (N + 2 * PR - 1) / (2 * PR), n_t = (M + PT - 1) / PT;
  const int64_t wave = num_sms / 2, rounds = n_w * n_t / (wave > 0 ? wave : 1);
  const int64_t n_t_main = rounds * wave / n_w;               // token rows filling whole waves
  const int64_t tail_tiles = (n_t - n_t_main) * n_w;
  if (rounds >= 1 && n_t_main >= 1 && n_t_main < n_t && wave / tail_tiles >= 2) {
    const int64_t m_main = n_t_main * PT;
    cudaError_t e = launch_pair<128>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, m_main, N, K, num_sms, stream);
    if (e != cudaSuccess) return e;
    return launch_pair<128>(xq + m_main * K, act_scale + m_main, rowsum + m_main, wp, w_scale, out + m_main * N,
                            acc_out ? acc_out + m_main * N : nullptr, M - m_main, N, K, num_sms, stream);
  }
  return launch_pair<128>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, num_sms, stream);
}

cudaError_t read_clear_device_error_pair(int* value) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

}  // namespace bitnet
