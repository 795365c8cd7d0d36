// gemm_smallm.cu -- the W2A8 ternary matmul for a few tokens (2 <= M <= 64) on the tensor cores,
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
// from M ~ 8 on. Here each weight is decoded exactly once, into fp16 in shared memory, and the
// tensor core applies it to all tokens: D[n][m] += W[n][k] * X[m][k] with tcgen05.mma
// kind::f16, M = 128 weight rows, N = MP (the token count rounded up to 16), K = 16.
//
// K order. A 128-weight i2_s block is 32 bytes; byte g holds the codes of k = g + 32j at bit
// pair j (j = 0 at bits 7:6). The dot product does not care about the order of k as long as
// both operands agree, so the kernel uses the byte order: within a block, word w (bytes
// 4w..4w+3), pair j and byte b of the word sit at position p = 16w + 4j + b. The 64 positions
// of a k-block are then 16 contiguous packed bytes of a row, and the 4 codes that share (w, j)
// are one shift and one mask of a 32-bit word. The activations follow the same order: position
// 16w + 4j + b holds activation k = 4w + b + 32j, so 4-byte groups move as a whole.
//
// Structure (one CTA per 128 weight rows and a K range; a thread-block cluster of up to 8
// CTAs splits K at 64-k granularity):
//  * warps 1-2 (loaders) copy the inputs of 8 k-blocks at a time with 16-byte cp.async into a
//    staging ring: k-block kb is packed bytes 16kb..16kb+15 of every weight row, so a stage is
//    128 contiguous bytes per row (8 consecutive lanes per row), plus the 5 activation blocks
//    of 128 bytes per token row those k-blocks draw on. Contiguous lanes keep each warp's
//    copies to a few cache lines; copies of single 16-byte pieces per row left the loads
//    bound by the request rate. Completion is signalled on the stage's mbarrier by
//    cp.async.mbarrier.arrive.noinc, so the loads stay in flight while the loaders move on;
//  * warps 3-18 (expanders) turn a staged k-block into the fp16 weight tile (codes 0..3,
//    exact) and the fp16 activation tile (int8 values, exact) in the 128-byte-swizzled K-major
//    layout the MMA reads, in a ring of tile slots. They touch only shared memory: the proxy
//    fence they need before the tensor core reads a tile then has no global loads to wait for;
//  * warp 0: allocates tensor memory; one lane issues the MMAs, rotating over 8 independent
//    128 x MP fp32 accumulators (tiny MMAs into one accumulator would wait on each other);
//  * then eight expander warps read the accumulator and store each row's partial sums into the
//    shared memory of the cluster CTA that owns that row (distributed shared memory, remote
//    stores); after one cluster barrier each CTA sums its rows' partials locally and writes
//    those outputs.
// Exactness: every operand is a small integer fp16 holds exactly, and every partial and total
// sum is an integer of magnitude <= 3 * 127 * K < 2^24 for K <= 32768, so the fp32
// accumulations and the cross-CTA sums are exact.
// Every mbarrier wait is bounded; a timeout is recorded in the device error word.
#include "bitnet_dev.cuh"

#include <cuda_fp16.h>

#include <atomic>

namespace bitnet {
namespace {

constexpr int TW = 128;                  // weight rows per CTA (the MMA's M)
constexpr int KB = 64;                   // k positions per MMA k-block (one 128-byte fp16 row)
constexpr int A_TILE = TW * KB * 2;      // fp16 weight tile
constexpr int XP_WARPS = 16;             // expander warps (the first 8 also drain the accumulator)
constexpr int XP_THREADS = XP_WARPS * 32;
constexpr int LD_WARPS = 2;              // loader warps
constexpr int LD_THREADS = LD_WARPS * 32;
constexpr int THREADS = (1 + LD_WARPS + XP_WARPS) * 32;
constexpr int XP_WARP0 = 1 + LD_WARPS;   // first expander warp
constexpr int kMaxCluster = 8;
constexpr int KB_ST = 8;                 // k-blocks per staging stage
constexpr int W_PITCH = 16 * KB_ST + 16;  // staged packed bytes per weight row (padded: conflict-free reads)
constexpr int W_ST = TW * W_PITCH;
constexpr int X_BLKS = KB_ST / 2 + 1;    // 128-activation blocks a stage may draw on

template <int MP>
struct SmallCfg {
  static_assert(MP % 16 == 0 && MP >= 16 && MP <= 64, "tokens per MMA: a multiple of 16, at most 64");
  static constexpr int B_TILE = MP * KB * 2;          // fp16 activation tile
  static constexpr int AB_BYTES = A_TILE + B_TILE;
  static constexpr int AB_STAGES = 3;
  static constexpr int X_ROW = X_BLKS * 128;          // staged activation bytes per token row
  static constexpr int ST_BYTES = W_ST + MP * X_ROW;
  static constexpr int ST_STAGES = MP <= 32 ? 3 : 2;
  static constexpr int XCH = (MP * 8 + XP_THREADS - 1) / XP_THREADS;  // activation chunks per thread
  static constexpr int PITCH = MP + 1;                // fp32 partials per row (odd: conflict-free)
  static constexpr int RECV_BYTES = (TW + kMaxCluster) * PITCH * 4;
  static constexpr int SMEM = 1024 + AB_STAGES * AB_BYTES + ST_STAGES * ST_BYTES + RECV_BYTES + MP * 8;
  // NACC accumulators of MP columns each: MMA i of the CTA goes to accumulator i % NACC, so
  // consecutive MMAs are independent (with MP as small as 16 an MMA is far shorter than its
  // latency, and one shared accumulator would serialise them); the epilogue adds them up
  static constexpr int NACC = 8;
  static constexpr uint32_t TMEM_COLS = NACC * MP <= 128 ? 128 : (NACC * MP <= 256 ? 256 : 512);
  static constexpr uint32_t IDESC = make_idesc_f16_f32(TW, MP);
  static_assert(AB_BYTES % 1024 == 0, "1024-byte aligned tiles");
  static_assert(ST_BYTES % 16 == 0, "16-byte copies");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// rows [row_lo(r), row_lo(r + 1)) of the tile are finished by cluster rank r
__device__ __forceinline__ int row_lo(int r, int cs) { return TW * r / cs; }

__device__ __forceinline__ uint2 codes4_to_f16(uint32_t codes) {  // 4 codes (one per byte) -> 4 fp16
  const uint32_t l = __byte_perm(codes, 0x64646464u, 0x4140);
  const uint32_t h = __byte_perm(codes, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6400), __ushort_as_half((unsigned short)0x6400));
  const __half2 rl = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
  const __half2 rh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&rl), *reinterpret_cast<const uint32_t*>(&rh));
}

__device__ __forceinline__ uint2 s8x4_to_f16(uint32_t w) {  // 4 int8 -> 4 exact fp16
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t l = __byte_perm(u, 0x64646464u, 0x4140);
  const uint32_t h = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6480), __ushort_as_half((unsigned short)0x6480));
  const __half2 rl = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
  const __half2 rh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&rl), *reinterpret_cast<const uint32_t*>(&rh));
}

// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major tile
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

template <int MP>
__global__ void __launch_bounds__(THREADS, 1) gemm_smallm_kernel(const int8_t* __restrict__ xq,
                                                                 const float* __restrict__ act_scale,
                                                                 const int32_t* __restrict__ rowsum,
                                                                 const uint8_t* __restrict__ wp, float w_scale,
                                                                 float* __restrict__ out, int32_t* __restrict__ acc_out,
                                                                 int M, int N, int K) {
  using Cfg = SmallCfg<MP>;
  constexpr int AB_STAGES = Cfg::AB_STAGES, ST_STAGES = Cfg::ST_STAGES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t st_full[ST_STAGES];   // a k-block's inputs staged
  __shared__ __align__(8) uint64_t st_empty[ST_STAGES];  // expanders done with a staged k-block
  __shared__ __align__(8) uint64_t ab_full[AB_STAGES];   // fp16 tiles of a k-block written
  __shared__ __align__(8) uint64_t ab_empty[AB_STAGES];  // MMAs done reading a slot
  __shared__ __align__(8) uint64_t done_bar;             // every MMA complete
  __shared__ uint32_t tmem_slot;

  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* ab_ring = base;                                          // AB_STAGES x (A, B)
  uint8_t* st_ring = base + AB_STAGES * Cfg::AB_BYTES;              // ST_STAGES x (W, X)
  float* recv = reinterpret_cast<float*>(st_ring + ST_STAGES * Cfg::ST_BYTES);  // pushed partials
  int* tok_rs = reinterpret_cast<int*>(recv + (TW + kMaxCluster) * Cfg::PITCH);  // rowsum per token
  float* tok_s = reinterpret_cast<float*>(tok_rs + MP);                           // scale per token

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * TW;
  const int cs = (int)gridDim.y;
  const int rank = (int)cluster_ctarank();
  const int nkb_all = K / KB;
  const int kb_lo = nkb_all * rank / cs, kb_hi = nkb_all * (rank + 1) / cs;
  const int nkb = kb_hi - kb_lo;

  if (threadIdx.x == 0) {
    // expander barriers count warps: each warp's lanes order their own writes, __syncwarp,
    // and one lane arrives (hundreds of per-thread arrivals on one barrier word serialise)
    for (int s = 0; s < ST_STAGES; ++s) {
      mbar_init(&st_full[s], LD_THREADS);
      mbar_init(&st_empty[s], XP_WARPS);
    }
    for (int a = 0; a < AB_STAGES; ++a) {
      mbar_init(&ab_full[a], XP_WARPS);
      mbar_init(&ab_empty[a], 1);
    }
    mbar_init(&done_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x >= 64 && threadIdx.x < 64 + MP) {  // warps 2-3: the epilogue's per-token inputs
    const int m = threadIdx.x - 64;
    tok_rs[m] = m < M ? __ldg(rowsum + m) : 0;
    tok_s[m] = m < M ? __ldg(act_scale + m) : 1.0f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  bool abort = false;

  if (warp == 0) {
    // ================================ MMA issuer ================================
    if (lane == 0) {
      for (int kb = 0; kb < nkb; ++kb) {
        const int a = kb % AB_STAGES, ua = kb / AB_STAGES;
        if (!mbar_wait(&ab_full[a], ua & 1, &abort)) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(ab_ring + a * Cfg::AB_BYTES), b_addr = a_addr + A_TILE;
#pragma unroll
        for (int kk = 0; kk < KB / 16; ++kk) {
          const int i = kb * (KB / 16) + kk;  // MMA index within the CTA
          mma_f16_ss(tmem + (uint32_t)((i % Cfg::NACC) * MP), make_sw128_kmajor_desc(a_addr + kk * 32),
                     make_sw128_kmajor_desc(b_addr + kk * 32), Cfg::IDESC, i >= Cfg::NACC ? 1u : 0u);
        }
        mma_commit(&ab_empty[a]);
      }
      mma_commit(&done_bar);  // tracks every MMA this thread issued
    }
  } else if (warp < XP_WARP0) {
    // ================================ loaders ================================
    // stage s holds k-blocks kb_lo + 8s .. +7: weight row r's bytes 16 * those (8 chunks,
    // lanes 8i..8i+7 on one row), and token row m's activation blocks blk0 .. blk0 + 4,
    // blk0 = (kb_lo + 8s) / 2
    const int lt = threadIdx.x - 32;  // 0..63
    const int nst = (nkb + KB_ST - 1) / KB_ST;
    int st_i = 0;
    for (; st_i < nst; ++st_i) {
      const int s = st_i % ST_STAGES, u = st_i / ST_STAGES;
      if (u > 0 && !mbar_wait(&st_empty[s], (u - 1) & 1, &abort)) break;
      const int kb0 = kb_lo + st_i * KB_ST, blk0 = kb0 >> 1;
      const uint32_t st = smem_u32(st_ring + s * Cfg::ST_BYTES);
#pragma unroll 4
      for (int id = lt; id < TW * KB_ST; id += LD_THREADS) {
        const int r = id >> 3, c = id & 7;
        const bool ok = n0 + r < N && kb0 + c < kb_hi;
        cp_async_16(st + (uint32_t)(r * W_PITCH + c * 16),
                    wp + (int64_t)(ok ? n0 + r : 0) * (K / 4) + (ok ? (kb0 + c) * 16 : 0), ok ? 16u : 0u);
      }
      for (int id = lt; id < MP * X_BLKS * 8; id += LD_THREADS) {
        const int m = id / (X_BLKS * 8), c = id % (X_BLKS * 8);
        const bool ok = m < M && blk0 * 8 + c < nkb_all * 4;  // 16-byte pieces within K
        cp_async_16(st + (uint32_t)(W_ST + m * Cfg::X_ROW + c * 16),
                    xq + (ok ? (int64_t)m * K + blk0 * 128 + c * 16 : 0), ok ? 16u : 0u);
      }
      cp_async_arrive_noinc(&st_full[s]);
    }
    // every copy issued must land before the CTA can exit
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    // ================================ expanders ================================
    const int t = threadIdx.x - XP_WARP0 * 32;  // 0..511
    const int r = t >> 2, wq = t & 3;            // weight row and its word of each k-block
    for (int kbl = 0; kbl < nkb && !abort; ++kbl) {
      const int si = kbl / KB_ST, q = kbl % KB_ST;  // staging stage and k-block within it
      const int s = si % ST_STAGES, us = si / ST_STAGES;
      const int a = kbl % AB_STAGES, ua = kbl / AB_STAGES;
      if (q == 0 && !mbar_wait_warp(&st_full[s], us & 1, &abort)) break;
      if (ua > 0 && !mbar_wait_warp(&ab_empty[a], (ua - 1) & 1, &abort)) break;
      const uint8_t* st = st_ring + s * Cfg::ST_BYTES;
      uint8_t* at = ab_ring + a * Cfg::AB_BYTES;
      uint8_t* bt = at + A_TILE;
      const int kb = kb_lo + kbl;
      const int rb = (kb >> 1) - ((kb_lo + si * KB_ST) >> 1), half = kb & 1;
      const uint32_t word = *reinterpret_cast<const uint32_t*>(st + r * W_PITCH + q * 16 + wq * 4);
      uint32_t xw[Cfg::XCH][2];
#pragma unroll
      for (int i = 0; i < Cfg::XCH; ++i) {
        // chunk idx: token row idx>>3, chunk c = idx&7 = word c/2 of runs j0 = 2(c%2), j0+1;
        // run j of the k-block is the block's bytes 16*half + 32j .. +15
        const int idx = t + XP_THREADS * i;
        const int c = idx & 7;
        const uint32_t* xr =
            reinterpret_cast<const uint32_t*>(st + W_ST + (idx >> 3) * Cfg::X_ROW + rb * 128 + half * 16);
        const int j0 = (c & 1) * 2, xq_w = c >> 1;
        xw[i][0] = idx < MP * 8 ? xr[j0 * 8 + xq_w] : 0u;
        xw[i][1] = idx < MP * 8 ? xr[(j0 + 1) * 8 + xq_w] : 0u;
      }
      if (q == KB_ST - 1 || kbl == nkb - 1) {  // stage read to the end (values are in registers)
        __syncwarp();
        if (lane == 0) mbar_arrive(&st_empty[s]);
      }
      {  // positions 16*wq .. 16*wq+15 of the k-block: chunks 2wq (pairs 0, 1) and 2wq+1 (2, 3)
        const uint2 p0 = codes4_to_f16((word >> 6) & 0x03030303u);
        const uint2 p1 = codes4_to_f16((word >> 4) & 0x03030303u);
        const uint2 p2 = codes4_to_f16((word >> 2) & 0x03030303u);
        const uint2 p3 = codes4_to_f16(word & 0x03030303u);
        *reinterpret_cast<uint4*>(at + sw128(r, 2 * wq)) = make_uint4(p0.x, p0.y, p1.x, p1.y);
        *reinterpret_cast<uint4*>(at + sw128(r, 2 * wq + 1)) = make_uint4(p2.x, p2.y, p3.x, p3.y);
      }
#pragma unroll
      for (int i = 0; i < Cfg::XCH; ++i) {
        const int idx = t + XP_THREADS * i;
        if (idx < MP * 8) {
          const uint2 lo = s8x4_to_f16(xw[i][0]), hi = s8x4_to_f16(xw[i][1]);
          *reinterpret_cast<uint4*>(bt + sw128(idx >> 3, idx & 7)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
        }
      }
      fence_proxy_async_smem();  // this thread's generic-proxy writes -> the tensor core's reads
      __syncwarp();
      if (lane == 0) mbar_arrive(&ab_full[a]);
    }

    // ---- push this CTA's partial sums to the rows' owners in the cluster (8 warps) ----
    if (warp < XP_WARP0 + 8 && mbar_wait_warp(&done_bar, 0, &abort)) {
      tc_fence_after();
      const int e = warp - XP_WARP0;         // 0..7 (the first 8 expander warps)
      const int quarter = warp & 3;          // tensor-memory lanes this warp may read
      const int row = quarter * 32 + lane;   // accumulator row = weight row within the tile
      int owner = 0;
      while (owner + 1 < cs && row_lo(owner + 1, cs) <= row) ++owner;
      const int o_lo = row_lo(owner, cs), o_rows = row_lo(owner + 1, cs) - o_lo;
      const uint32_t dst = smem_u32(recv) + (uint32_t)(((rank * o_rows + (row - o_lo)) * Cfg::PITCH) * 4);
      const uint32_t dst_c = cs > 1 ? map_to_rank(dst, (uint32_t)owner) : dst;
      const int c_lo = (e >> 2) * (MP / 2);  // two warps share a lane quarter: half the columns each
      const int used = nkb * (KB / 16) < Cfg::NACC ? nkb * (KB / 16) : Cfg::NACC;  // accumulators written
      // per accumulator, every 8-column piece of this warp's half is loaded before one wait
      // (a wait after each piece serialised 32 round trips per warp at 64 tokens)
      constexpr int H = MP / 2, HC = H / 8;
      float sum[H];
#pragma unroll
      for (int i = 0; i < H; ++i) sum[i] = 0.f;
      for (int j = 0; j < used; ++j) {
        uint32_t v[HC][8];
#pragma unroll
        for (int cb = 0; cb < HC; ++cb)
          tmem_ld_32x32b_x8(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(j * MP + c_lo + cb * 8), v[cb]);
        tmem_ld_wait();
#pragma unroll
        for (int cb = 0; cb < HC; ++cb)
#pragma unroll
          for (int i = 0; i < 8; ++i) sum[cb * 8 + i] += __uint_as_float(v[cb][i]);  // integers < 2^24: exact
      }
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const uint32_t addr = dst_c + (uint32_t)((c_lo + i) * 4);
        if (cs > 1)
          st_cluster_u32(addr, __float_as_uint(sum[i]));
        else
          st_shared_u32(addr, __float_as_uint(sum[i]));
      }
    }
  }

  // ---- every partial pushed; each CTA finishes its own rows ----
  tc_fence_before();
  if (cs > 1)
    cluster_sync_all();
  else
    __syncthreads();
  if (warp >= XP_WARP0 && !abort) {
    const int t = threadIdx.x - XP_WARP0 * 32;
    const int lo = row_lo(rank, cs), rows = row_lo(rank + 1, cs) - lo;
    // rows <= 128: thread t takes row t % 128 of the slice (if any) for tokens t/128, +4, ...
    const int rl = t & (TW - 1);
    const int n = n0 + lo + rl;
    if (rl < rows && n < N) {
      for (int m = t >> 7; m < M; m += XP_THREADS / TW) {
        float sum = 0.0f;
        for (int src = 0; src < cs; ++src) sum += recv[(src * rows + rl) * Cfg::PITCH + m];
        const int a = __float2int_rn(sum) - tok_rs[m];
        const int64_t o = (int64_t)m * N + n;
        out[o] = __fmul_rn(__fdiv_rn(__int2float_rn(a), tok_s[m]), w_scale);
        if (acc_out) acc_out[o] = a;
      }
    }
  }

  // ---- teardown: every MMA complete before the tensor memory is freed ----
  if (warp == 0) {
    tc_fence_after();
    bool dummy = false;
    mbar_wait(&done_bar, 0, &dummy);
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
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
  // K split across a cluster so that all CTAs run at once, one per SM (the shared memory allows
  // one): at most 8 CTAs per cluster, at least four 64-k blocks each. A cluster that cannot be
  // resident with the others runs as a second wave and doubles the time. A cluster must fit in
  // one GPC, so SMs / tiles overestimates the size that fits: with 20 tiles, 7-CTA clusters pack
  // only two per GPC. The occupancy query decides, shrinking the cluster until every one fits.
  const int64_t n_tiles = (N + TW - 1) / TW;
  const int64_t nkb = K / KB;
  int64_t cs = num_sms / n_tiles;
  if (cs > kMaxCluster) cs = kMaxCluster;
  if (cs > nkb / 4) cs = nkb / 4;
  if (cs < 1) cs = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  for (; cs > 1; --cs) {
    attr[0].val.clusterDim.y = (unsigned)cs;
    cfg.gridDim = dim3((unsigned)n_tiles, (unsigned)cs);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_smallm_kernel<MP>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();  // the query is only a hint: keep the size from the SM count
      break;
    }
    if (clusters >= n_tiles) break;
  }
  attr[0].val.clusterDim.y = (unsigned)cs;
  cfg.gridDim = dim3((unsigned)n_tiles, (unsigned)cs);
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

bool gemm_smallm_supported(int64_t M, int64_t K) { return M >= 1 && M <= 64 && K <= 32768; }

cudaError_t launch_gemm_smallm(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                               float w_scale, float* out, int32_t* acc_out, int64_t M, int64_t N, int64_t K,
                               int num_sms, cudaStream_t stream) {
  if (M <= 16) return launch_mp<16>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, num_sms, stream);
  if (M <= 32) return launch_mp<32>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, num_sms, stream);
  if (M <= 48) return launch_mp<48>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, num_sms, stream);
  return launch_mp<64>(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, num_sms, stream);
}

}  // namespace bitnet
