// gemm_smallm.cu -- the W2A8 ternary matmul for a few tokens (64 per CTA, more in chunks) on the tensor cores,
// with the weights as the MMA's M dimension.
//
// Computes, like every other path of the library, raw[m][n] = sum_k code[n][k] * xq[m][k],
// acc = raw - rowsum[m], out = (acc / s[m]) * w_scale, with the same integers and the same fp32
// operations. Sources: the raw code dot over the 4x32-interleaved i2_s bytes ("[분석/검증-3]
// BitNet.cpp ARM 커널 재작성" §3, "[기술 분석 보고서] ... 추론 붕괴 원인 분석" §3.2), the byte
// layout ("BitNet 딥다이브" §4-2), the dequantisation ("bitnet.rs" "Quantised Forward Pass").
//
// Why this shape: with a handful of tokens the work is 2-bit weight streaming, but the dp4a
// GEMV re-decodes every weight word once per token row it serves and runs out of issue slots
// from M ~ 8 on. Here each weight is decoded exactly once and the tensor core applies it to
// all tokens: D[n][j] += W'[n][k] * B[j][k] with tcgen05.mma kind::f8f6f4 (e4m3 x e4m3, fp32
// accumulate), M = 128 weight rows, K = 32.
//
// Operands (all exact in e4m3). A tiny MMA costs the tensor pipe a fixed ~45 cycles whatever
// its N, so the MMA count per weight byte is what bounds this kernel; the 8-bit kind takes
// K = 32 per MMA, half the count of fp16.
//  * weights: w' = 8 + code in {8..11}, the e4m3 byte 0x50 | code (one mask-and-or per four
//    codes); k positions past the end of K hold 0x00 (w' = 0);
//  * activations: u = x + 128 in [1, 255] is split into base-8 digits d0, d1 in [0, 7] and
//    d2 in [0, 3], each stored as the e4m3 byte 0x50 | d (= 8 + d). B has NB = 3 MP + 16 rows:
//    digit 0, 1 and 2 planes of the MP tokens, then 16 rows of 1.0 whose D column is the
//    weight-row sum W' = sum_k w'.
//  Then with D_i = sum_k w'_k (8 + d_ik): sum_k code_k x_k = D0 + 8 D1 + 64 D2 - 712 W' - 8 rowsum
//  (sum w' u = sum_i 8^i (D_i - 8 W'), and sum (w' - 8)(u - 128) over the K positions), so
//  acc = raw - rowsum = (D0 + 8 D1 + 64 D2 - 712 W') - 9 rowsum. Every D_i <= 11 * 15 * K < 2^24
//  for K <= 32768, so the fp32 accumulators hold exact integers; the combination is integer.
//
// Stages. The K range is walked in stages of 256 k: two i2_s blocks, eight K = 32 MMAs.
// Synchronisation is per stage: one wait, one fence and one barrier arrival per warp cover 256 k.
// The decoded weights (A, 128 rows x 256 k) are written straight into tensor memory with
// tcgen05.st and the MMA reads A from there; only the activation digits (B) go through shared
// memory.
//
// K order. Inside an i2_s block byte g holds the codes of k = g + 32j at bit pair j (j = 0 at
// bits 7:6), so the 16 bytes 16h..16h+15 of block b hold, for each j, the 16 consecutive
// k = 128b + 32j + 16h + e of the stage. Stage position p = 64q + 16j + e (q = 2b + h) holds
// that k: a thread's 16 bytes give 16 tensor-memory columns of 4 positions each, and a
// 16-byte piece of activations (16 consecutive k) is one 16-byte chunk of each digit row.
//
// Structure (one CTA per 128 weight rows, a range of stages and a chunk of up to 64 tokens; a
// thread-block cluster of up to 8 CTAs splits the stages; more than 64 tokens take grid.z chunks,
// each decoding its weight slice again from L2):
//  * warps 1-16 (workers): warp w owns tensor-memory lanes 32(w%4)..+31, i.e. weight rows, and
//    the 16-byte quarter q = (w-1)/4 of each row's 64 stage bytes. Each thread copies its own
//    16 weight bytes and up to two 16-byte pieces of the stage's int8 activations with
//    cp.async into a private ring of PD stages in shared memory (one commit group per stage, so
//    PD stages are in flight without tying up registers; the weights of the first stages are
//    requested before waiting for the previous kernel). Per stage it decodes its bytes into 16
//    tensor-memory columns of the stage's A slot, writes its activation digits into the
//    128-byte-swizzled K-major B tile, fences, and its warp arrives once;
//  * warp 0: allocates tensor memory; one lane issues the MMAs into NACC accumulators of NB
//    columns and commits one release of the slot per stage;
//  * epilogue: each worker warp reads 32 accumulator rows (its tensor-memory lane quarter) and
//    a quarter of the tokens, forms the integer partial D0 + 8 D1 + 64 D2 - 712 W', and either
//    keeps it (rows its CTA owns) or sends it with st.async (16-byte pieces) into the shared
//    memory of the cluster CTA that owns those rows, counted in bytes on that CTA's receive
//    barrier; each owner waits for exactly its expected bytes, adds them and writes the
//    outputs. (A cluster barrier after plain remote stores cost 0.7-1 us: its release waits
//    for every remote store to be acknowledged.)
// Every mbarrier wait is bounded; a timeout is recorded in the device error word.
#include "bitnet_dev.cuh"

#include <cuda_fp16.h>

#include <atomic>

namespace bitnet {
namespace {

constexpr int TW = 128;                    // weight rows per CTA (the MMA's M)
constexpr int SK = 256;                    // k per stage (two i2_s blocks)
constexpr int KSTEPS = SK / 32;            // K = 32 MMAs per stage
constexpr int WK_WARPS = 16;               // workers
constexpr int WK_THREADS = WK_WARPS * 32;  // four per weight row
constexpr int THREADS = 32 + WK_THREADS;
constexpr int kMaxCluster = 8;
constexpr uint32_t TMEM_COLS = 512;        // accumulators, then the A stages (one CTA per SM)
constexpr int A_COLS = SK / 4;             // tensor-memory columns of one e4m3 A stage

// rows [row_lo(r), row_lo(r + 1)) of the tile are finished by cluster rank r
__host__ __device__ constexpr int row_lo(int r, int cs) { return TW * r / cs; }

// most partial rows one CTA receives: (cs - 1) sources times its largest row share
constexpr int max_recv_rows() {
  int best = 0;
  for (int cs = 2; cs <= kMaxCluster; ++cs)
    for (int r = 0; r < cs; ++r) {
      const int v = (cs - 1) * (row_lo(r + 1, cs) - row_lo(r, cs));
      best = v > best ? v : best;
    }
  return best;
}

template <int MP>
struct SmallCfg {
  static_assert(MP % 16 == 0 && MP >= 16 && MP <= 64, "tokens per MMA: a multiple of 16, at most 64");
  static constexpr int NB = 3 * MP + 16;                          // B rows: 3 digit planes, 16 rows of ones
  static constexpr int ONES = 3 * MP;                             // the ones row
  static constexpr int NACC = 2 * NB <= 256 ? 2 : 1;              // accumulators
  static constexpr int ACOL = (NACC * NB + 63) / 64 * 64;         // first A column in tensor memory
  static constexpr int NS = MP <= 32 ? 4 : (MP <= 48 ? 3 : 2);    // A/B stages
  static constexpr int B_SUB = NB * 128;                          // e4m3 digits, 128 k x NB rows
  static constexpr int B_STAGE = 2 * B_SUB;
  static constexpr int XV = (MP * 16 + WK_THREADS - 1) / WK_THREADS;  // 16-byte activation pieces per thread
  static constexpr int PD = MP <= 16 ? 6 : (MP <= 32 ? 5 : 3);    // staged input stages in flight
  static constexpr int RAW_SLOT = WK_THREADS * 16 * (1 + XV);      // one stage's copies, 16 bytes per thread each
  static constexpr int NC = MP / 4;                                // tokens per epilogue warp
  static constexpr int PITCH = MP + 4;                             // int32 per received row (16-byte rows)
  static constexpr int RECV_ROWS = max_recv_rows();
  static constexpr int SMEM = 1024 + NS * B_STAGE + PD * RAW_SLOT + RECV_ROWS * PITCH * 4;
  static constexpr uint32_t IDESC = make_idesc_f16_f32(TW, NB);   // e4m3 x e4m3 has format code 0 like f16
  static_assert(NB % 16 == 0 && NB <= 256, "MMA N");
  static_assert(ACOL + NS * A_COLS <= (int)TMEM_COLS, "tensor memory columns");
  static_assert(B_SUB % 1024 == 0, "1024-byte aligned tiles");
  static_assert(SMEM <= 227 * 1024 - 256, "shared memory (static barriers included)");
};

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major tile
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
// 16 bytes into a peer CTA's shared memory; on arrival they count as completed transaction bytes
// on the peer's mbarrier (both addresses in the shared::cluster window of that CTA)
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, int a, int b, int c, int d, uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1,%2,%3,%4}, [%5];" ::"r"(
                   cluster_addr),
               "r"(a), "r"(b), "r"(c), "r"(d), "r"(cluster_bar)
               : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f8f6f4: A is 128 lanes (rows) x 8 columns (32
// e4m3 along K, four per column, the lowest k in the low byte).
__device__ __forceinline__ void mma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread t of the warp writes lane (base + t).
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x NC consecutive 32-bit columns (NC = 1, 4, 8, 12 or 16) into r[0..NC)
template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* r) {
  if constexpr (NC == 1) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r[0]) : "r"(taddr));
  } else if constexpr (NC == 4) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
  } else if constexpr (NC == 8) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
  } else if constexpr (NC == 12) {
    tmem_ld_cols<8>(taddr, r);
    tmem_ld_cols<4>(taddr + 8, r + 8);
  } else {
    static_assert(NC == 16, "1, 4, 8, 12 or 16 columns");
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
  }
}

template <int MP>
__global__ void __launch_bounds__(THREADS, 1) gemm_smallm_kernel(const int8_t* __restrict__ xq,
                                                                 const float* __restrict__ act_scale,
                                                                 const int32_t* __restrict__ rowsum,
                                                                 const uint8_t* __restrict__ wp, float w_scale,
                                                                 float* __restrict__ out, int32_t* __restrict__ acc_out,
                                                                 int M, int N, int K) {  // M: all tokens
  using Cfg = SmallCfg<MP>;
  constexpr int NS = Cfg::NS, XV = Cfg::XV, NC = Cfg::NC, PD = Cfg::PD, NACC = Cfg::NACC, NB = Cfg::NB;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[NS];   // a stage's operands written (one arrival per worker warp)
  __shared__ __align__(8) uint64_t empty_bar[NS];  // the MMAs reading a stage slot are done (one commit)
  __shared__ __align__(8) uint64_t done_bar;       // every MMA complete
  __shared__ __align__(8) uint64_t recv_bar;       // the partials of this CTA's rows from its peers (bytes)
  __shared__ uint32_t tmem_slot;

  pdl_launch_dependents();
  // this CTA's chunk of tokens: rows m0 .. m0 + M - 1 (M from here on counts the chunk's tokens)
  const int m0 = (int)blockIdx.z * MP;
  M = M - m0 < MP ? M - m0 : MP;
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t bring = raw_addr + ((1024u - (raw_addr & 1023u)) & 1023u);  // NS B tiles
  const uint32_t staged = bring + NS * Cfg::B_STAGE;                         // PD stages of copied inputs
  const uint32_t recv = staged + PD * Cfg::RAW_SLOT;                         // received partial rows

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * TW;
  const int cs = (int)gridDim.y;
  const int rank = (int)cluster_ctarank();
  const int nblk = K / 128;               // i2_s blocks
  const int nst_all = (nblk + 1) >> 1;    // 256-k stages (the last one half when nblk is odd)
  const int st_lo = nst_all * rank / cs, st_hi = nst_all * (rank + 1) / cs;
  const int nst = st_hi - st_lo;

  // worker roles (meaningful for warps 1..16): tensor-memory lane quarter, weight row, and the
  // 16-byte quarter q of the row's 64 stage bytes (i2_s block q/2 of the stage, half q%2)
  const int t = (int)threadIdx.x - 32;
  const int lq = warp & 3, q = (warp - 1) >> 2, qb = q >> 1;
  const int row = 32 * lq + lane;
  const bool row_ok = warp >= 1 && n0 + row < N;
  const uint8_t* wrow = wp + (int64_t)(row_ok ? n0 + row : 0) * (K / 4) + 16 * q;
  const uint32_t my_w = staged + (uint32_t)(16 * t);  // this thread's weight copy in stage slot 0
  auto issue_w = [&](int i) {
    const int gs = st_lo + i;
    const bool ok = row_ok && 2 * gs + qb < nblk;
    cp_async_16(my_w + (uint32_t)((i % PD) * Cfg::RAW_SLOT), ok ? wrow + 64 * (int64_t)gs : wp, ok ? 16u : 0u);
  };
  auto issue_x = [&](int i) {
    const int gs = st_lo + i;
#pragma unroll
    for (int v = 0; v < XV; ++v) {
      const int idx = t + WK_THREADS * v, m = idx >> 4, u = idx & 15;
      if (idx < MP * 16) {
        const bool ok = m < M && 2 * gs + (u >> 3) < nblk;
        cp_async_16(my_w + (uint32_t)((i % PD) * Cfg::RAW_SLOT + WK_THREADS * 16 * (1 + v)),
                    ok ? xq + (int64_t)(m0 + m) * K + 256 * (int64_t)gs + 16 * u : xq, ok ? 16u : 0u);
      }
    }
  };
  if (warp >= 1) {
    for (int p = 0; p < PD && p < nst; ++p) issue_w(p);  // weights do not depend on the previous kernel
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_bar[s], WK_WARPS);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&done_bar, 1);
    mbar_init(&recv_bar, 1);
    fence_mbar_init();
    if (cs > 1)  // every peer sends its partials of this CTA's rows: 4 bytes per row and token
      mbar_arrive_expect_tx(&recv_bar, (uint32_t)((cs - 1) * (row_lo(rank + 1, cs) - row_lo(rank, cs)) * MP * 4));
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (cs > 1) cluster_arrive_relaxed();  // this CTA's barriers exist (waited on before the first send)
  const uint32_t tmem = tmem_slot;
  bool abort = false;

  if (warp == 0) {
    // ================================ MMA issuer ================================
    if (lane == 0) {
      // The issuing thread's own arithmetic is on the critical path: a tiny MMA occupies the
      // tensor pipe for only ~45 cycles, so each issue here is a few integer adds to
      // descriptors built once (the address field is the low 14 bits; offsets never carry).
      const uint64_t bdesc0 = make_sw128_kmajor_desc(bring);
      const uint32_t acol0 = tmem + (uint32_t)Cfg::ACOL;
      int s = 0;
      uint32_t phase = 0;
      for (int i = 0; i < nst; ++i) {
        if (!mbar_wait(&full_bar[s], phase, &abort)) break;
        tc_fence_after();
        const uint32_t a_col = acol0 + (uint32_t)(s * A_COLS);
        const uint64_t bd = bdesc0 + (uint64_t)((s * Cfg::B_STAGE) >> 4);
        const uint32_t first = i > 0 ? 1u : 0u;  // accumulate unless this is an accumulator's first MMA
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks)
          mma_f8_ts(tmem + (uint32_t)((ks % NACC) * NB), a_col + (uint32_t)(8 * ks),
                    bd + (uint64_t)(((ks >> 2) * Cfg::B_SUB + (ks & 3) * 32) >> 4), Cfg::IDESC,
                    ks >= NACC ? 1u : first);
        mma_commit(&empty_bar[s]);
        if (++s == NS) {
          s = 0;
          phase ^= 1u;
        }
      }
      mma_commit(&done_bar);  // tracks every MMA this thread issued
    }
    __syncwarp();  // the warp converges before its collective tensor-memory loads
  } else {
    // ================================ workers ================================
    // the 16 rows of ones (e4m3 1.0 = 0x38) of every B slot; they never change, and each
    // thread's writes are fenced before its warp's first arrival like every tile write
    for (int o = 16 * t; o < NS * 2 * 16 * 128; o += 16 * WK_THREADS) {
      const int slot = o / (2 * 16 * 128), sub = (o / (16 * 128)) & 1, off = o % (16 * 128);
      sts128(bring + (uint32_t)(slot * Cfg::B_STAGE + sub * Cfg::B_SUB + Cfg::ONES * 128 + off), 0x38383838u,
             0x38383838u, 0x38383838u, 0x38383838u);
    }
    pdl_wait();  // the activations may be the previous kernel's output
#pragma unroll 1
    for (int p = 0; p < PD; ++p) {  // one commit group per stage (the first also holds the weights)
      if (p < nst) issue_x(p);
      cp_async_commit();
    }
    const uint32_t a_lane = tmem + ((uint32_t)(32 * lq) << 16) + (uint32_t)(Cfg::ACOL + 16 * q);
    for (int i = 0; i < nst; ++i) {
      const int s = i % NS, u = i / NS;
      const uint32_t slot = (uint32_t)((i % PD) * Cfg::RAW_SLOT);
      cp_async_wait_group<PD - 1>();  // this thread's copies of stage i have landed
      const uint4 wv = lds128(my_w + slot);
      uint4 xv[XV];
#pragma unroll
      for (int v = 0; v < XV; ++v) xv[v] = lds128(my_w + slot + (uint32_t)(WK_THREADS * 16 * (1 + v)));
      if (u > 0 && !mbar_wait_warp(&empty_bar[s], (uint32_t)(u - 1) & 1u, &abort)) break;
      tc_fence_after();
      {  // weights: 4 words x 4 bit pairs -> 64 e4m3 w' in 16 tensor-memory columns (pair j: 4j..4j+3)
        const bool blk_ok = 2 * (st_lo + i) + qb < nblk;  // past the end of K: w' = 0
        const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t a[16];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int wi = 0; wi < 4; ++wi)
            a[4 * j + wi] = blk_ok ? ((w[wi] >> (6 - 2 * j)) & 0x03030303u) | 0x50505050u : 0u;
        tmem_st_32x32b_x16(a_lane + (uint32_t)(s * A_COLS), a);
      }
#pragma unroll
      for (int v = 0; v < XV; ++v) {  // activations: 16 int8 (k = 16uu..) -> one chunk of each digit row
        const int idx = t + WK_THREADS * v, m = idx >> 4, uu = idx & 15;
        if (idx < MP * 16) {
          const uint32_t x4[4] = {xv[v].x ^ 0x80808080u, xv[v].y ^ 0x80808080u, xv[v].z ^ 0x80808080u,
                                  xv[v].w ^ 0x80808080u};  // u = x + 128, per byte
          uint32_t d[3][4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            d[0][e] = (x4[e] & 0x07070707u) | 0x50505050u;
            d[1][e] = ((x4[e] >> 3) & 0x07070707u) | 0x50505050u;
            d[2][e] = ((x4[e] >> 6) & 0x03030303u) | 0x50505050u;
          }
          // k = 16uu + e lies in block uu/8, half uu%2, bit pair (uu/2)%4: stage positions
          // 64(2(uu/8) + uu%2) + 16((uu/2)%4) + e, i.e. sub-tile uu/8, chunk 4(uu%2) + (uu/2)%4
          const int chunk = 4 * (uu & 1) + ((uu >> 1) & 3);
          const uint32_t bt = bring + (uint32_t)(s * Cfg::B_STAGE + (uu >> 3) * Cfg::B_SUB);
#pragma unroll
          for (int dg = 0; dg < 3; ++dg)
            sts128(bt + sw128(dg * MP + m, chunk), d[dg][0], d[dg][1], d[dg][2], d[dg][3]);
        }
      }
      if (i + PD < nst) {  // refill this copy slot with stage i + PD (its bytes are in registers)
        issue_w(i + PD);
        issue_x(i + PD);
      }
      cp_async_commit();
      tmem_st_wait();            // this thread's tensor-memory writes complete
      fence_proxy_async_smem();  // this thread's generic-proxy writes -> the tensor core's reads
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full_bar[s]);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // no copy may land after the CTA is gone
  }

  // ---- epilogue: integer partials per (row, token); push rows owned by other cluster CTAs ----
  const int quarter = warp & 3;             // tensor-memory lanes this warp may read
  const int c0 = ((warp - 1) >> 2) * NC;    // this warp's tokens
  int owner = 0;
  while (owner + 1 < cs && row_lo(owner + 1, cs) <= row) ++owner;
  const int o_lo = row_lo(owner, cs), o_rows = row_lo(owner + 1, cs) - o_lo;
  int part[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) part[c] = 0;
  bool have = false;
  if (warp >= 1 && mbar_wait_warp(&done_bar, 0, &abort)) {
    tc_fence_after();
    const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16);
    uint32_t v[NACC][3][NC], w1[NACC][1];
#pragma unroll
    for (int j = 0; j < NACC; ++j) {
#pragma unroll
      for (int dg = 0; dg < 3; ++dg) tmem_ld_cols<NC>(tbase + (uint32_t)(j * NB + dg * MP + c0), v[j][dg]);
      tmem_ld_cols<1>(tbase + (uint32_t)(j * NB + Cfg::ONES), w1[j]);
    }
    tmem_ld_wait();
    // every accumulator value is an integer below 2^24, so the fp32 sums and conversions are exact
    float wsum = 0.f;
#pragma unroll
    for (int j = 0; j < NACC; ++j) wsum += __uint_as_float(w1[j][0]);
    const int wprime = __float2int_rn(wsum);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      float dsum[3] = {0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < NACC; ++j)
#pragma unroll
        for (int dg = 0; dg < 3; ++dg) dsum[dg] += __uint_as_float(v[j][dg][c]);
      part[c] = __float2int_rn(dsum[0]) + 8 * __float2int_rn(dsum[1]) + 64 * __float2int_rn(dsum[2]) - 712 * wprime;
    }
    have = true;
  }
  if (cs > 1) {
    cluster_wait();  // every peer's receive barrier is initialised and armed
    if (have && owner != rank) {
      const int slot = rank - (rank > owner ? 1 : 0);
      const uint32_t dst = map_to_rank(recv + (uint32_t)(((slot * o_rows + (row - o_lo)) * Cfg::PITCH + c0) * 4),
                                       (uint32_t)owner);
      const uint32_t bar = map_to_rank(smem_u32(&recv_bar), (uint32_t)owner);
#pragma unroll
      for (int c = 0; c < NC; c += 4)
        st_async_v4(dst + (uint32_t)(c * 4), part[c], part[c + 1], part[c + 2], part[c + 3], bar);
    }
  }

  // ---- every tensor-memory access done; owners wait for their peers' partials and finish ----
  tc_fence_before();
  __syncthreads();
  if (have && owner == rank && !abort && (cs == 1 || mbar_wait(&recv_bar, 0, &abort))) {
    for (int slot = 0; slot < cs - 1; ++slot) {
      const uint32_t src = recv + (uint32_t)(((slot * o_rows + (row - o_lo)) * Cfg::PITCH + c0) * 4);
#pragma unroll
      for (int c = 0; c < NC; c += 4) {
        const float4 f = lds_f4(src + (uint32_t)(c * 4));
        part[c] += __float_as_int(f.x);
        part[c + 1] += __float_as_int(f.y);
        part[c + 2] += __float_as_int(f.z);
        part[c + 3] += __float_as_int(f.w);
      }
    }
    const int n = n0 + row;
    if (n < N) {
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const int m = c0 + c;
        if (m < M) {
          const int a = part[c] - 9 * __ldg(rowsum + m0 + m);  // raw = part - 8 rowsum; acc = raw - rowsum
          const int64_t o = (int64_t)(m0 + m) * N + n;
          out[o] = __fmul_rn(__fdiv_rn(__int2float_rn(a), __ldg(act_scale + m0 + m)), w_scale);
          if (acc_out) acc_out[o] = a;
        }
      }
    }
  }

  // ---- teardown: every MMA complete before the tensor memory is freed; and no peer may still be
  // sending into this CTA's shared memory when it exits (the owners waited for every byte unless a
  // wait gave up, so this bounded wait only matters on that path) ----
  if (cs > 1 && threadIdx.x == 32) {
    bool dummy = false;
    mbar_wait(&recv_bar, 0, &dummy);
  }
  if (warp == 0) {
    tc_fence_after();
    bool dummy = false;
    mbar_wait(&done_bar, 0, &dummy);
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int MP>
cudaError_t launch_mp(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                      float w_scale, float* out, int32_t* acc_out, int64_t M, int64_t N, int64_t K, int num_sms,
                      cudaStream_t stream) {
  using Cfg = SmallCfg<MP>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(gemm_smallm_kernel<MP>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  // The stages are split across a cluster so that all CTAs run at once, one per SM (the shared
  // memory allows one): at most 8 CTAs per cluster, at least one 256-k stage each. A cluster
  // that cannot be resident with the others runs as a second wave and doubles the time. A
  // cluster must fit in one GPC, so SMs / tiles overestimates the size that fits: with 20
  // tiles, 7-CTA clusters pack only two per GPC. The occupancy query decides, shrinking the
  // cluster until every one fits.
  const int64_t n_tiles = (N + TW - 1) / TW;
  const int64_t n_chunks = (M + MP - 1) / MP;  // token chunks (grid.z)
  const int64_t n_ctas1 = n_tiles * n_chunks;   // CTAs at cluster size 1
  const int64_t n_stages = (K / 128 + 1) / 2;
  int64_t cs = num_sms / n_ctas1;
  if (cs > kMaxCluster) cs = kMaxCluster;
  if (cs > n_stages) cs = n_stages;
  if (cs < 1) cs = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  for (; cs > 1; --cs) {
    attr[0].val.clusterDim.y = (unsigned)cs;
    cfg.gridDim = dim3((unsigned)n_tiles, (unsigned)cs, (unsigned)n_chunks);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_smallm_kernel<MP>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();  // the query is only a hint: keep the size from the SM count
      break;
    }
    if (clusters >= n_ctas1) break;
  }
  attr[0].val.clusterDim.y = (unsigned)cs;
  cfg.gridDim = dim3((unsigned)n_tiles, (unsigned)cs, (unsigned)n_chunks);
  // weights stream in while the previous kernel finishes (the kernel waits for it before reading
  // the activations or writing anything)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_smallm_kernel<MP>, xq, act_scale, rowsum, wp, w_scale, out, acc_out, (int)M,
                            (int)N, (int)K);
}

}  // namespace

cudaError_t read_clear_device_error_smallm(int* value) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

bool gemm_smallm_supported(int64_t M, int64_t K) { return M >= 1 && M <= 64LL * 65535 && K <= 32768; }

cudaError_t launch_gemm_smallm(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                               float w_scale, float* out, int32_t* acc_out, int64_t M, int64_t N, int64_t K,
                               int num_sms, cudaStream_t stream) {
  if (M <= 16) return launch_mp<16>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, num_sms, stream);
  if (M <= 32) return launch_mp<32>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, num_sms, stream);
  if (M <= 48) return launch_mp<48>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, num_sms, stream);
  return launch_mp<64>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, num_sms, stream);
}

}  // namespace bitnet
