// bitnet_dev.cuh -- device helpers shared by the kernels of libbitnet_gb300 (sm_103a only).
//
// Thin inline-PTX wrappers for the Blackwell pieces the kernels use: mbarriers with bounded
// waits, tcgen05 tensor-memory allocation / MMA / loads, and the shared-memory matrix
// descriptor of the 5th-generation tensor core. Also the launch declarations that the
// C-ABI translation unit calls.
#pragma once

#include <cstdint>
#include <cuda.h>  // CUtensorMap and its enums (the encoder itself comes from the runtime)
#include <cuda_runtime.h>

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030)
#error "libbitnet_gb300 is written for sm_103a (GB300) only"
#endif

namespace bitnet {

// ---------------------------------------------------------------------------------------
// Device-side error word: a kernel whose bounded wait runs out records a code here and
// returns instead of hanging. Internal linkage: each translation unit that waits owns one
// and exports a host reader (read_clear_device_error_*), called by bitnet_last_device_error.
// ---------------------------------------------------------------------------------------
static __device__ int g_device_error = 0;

constexpr int kErrTimeout = -5;
// mbarrier polls before a wait gives up. try_wait itself suspends for a bounded,
// hardware-chosen time, so this is on the order of seconds, far above any legal wait.
constexpr uint32_t kMaxPolls = 1u << 24;

__device__ __forceinline__ void record_device_error(int code) { atomicCAS(&g_device_error, 0, code); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete. Returns false (and records a
// timeout) if it did not complete within kMaxPolls polls; *abort is then set so that the
// caller's loop can leave early. Once *abort is set no further waiting is done.
__device__ __forceinline__ bool mbar_wait_polls(uint64_t* bar, uint32_t parity, bool* abort, uint32_t max_polls) {
  if (*abort) return false;
  const uint32_t a = smem_u32(bar);
  for (uint32_t i = 0; i < max_polls; ++i)
    if (mbar_try_wait(a, parity)) return true;
  record_device_error(kErrTimeout);
  *abort = true;
  return false;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, bool* abort) {
  return mbar_wait_polls(bar, parity, abort, kMaxPolls);
}

// mbar_wait by every lane of a warp, with the outcome made warp-uniform: a warp never splits at
// a timeout before warp-collective code (shuffles, tcgen05.ld). All 32 lanes must call it.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, bool* abort) {
  const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
  if (!ok) *abort = true;
  return ok;
}

// mbar_wait_warp with a caller-chosen poll limit (the failure-handling self-test).
__device__ __forceinline__ bool mbar_wait_warp_polls(uint64_t* bar, uint32_t parity, bool* abort, uint32_t max_polls) {
  const bool ok = __all_sync(0xffffffffu, mbar_wait_polls(bar, parity, abort, max_polls));
  if (!ok) *abort = true;
  return ok;
}

// One arrival that also announces tx_bytes of asynchronous (bulk copy) data for the phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t tx_bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(tx_bytes)
               : "memory");
}

// 1-D bulk copy global -> shared (TMA engine); completion is counted on the mbarrier in
// bytes. dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 16-byte load from shared memory by its 32-bit shared-window address (always an LDS, never a
// generic load that the compiler could not prove to be shared)
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// 16-byte asynchronous copy global -> shared (cp.async, L2 only); src_bytes 0 writes zeros
// and reads nothing. dst and src 16-byte aligned.
__device__ __forceinline__ void cp_async_16(uint32_t dst_smem, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst_smem), "l"(src), "r"(src_bytes)
               : "memory");
}
// One arrival on the mbarrier once every cp.async this thread issued so far has completed
// (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Named barrier over a subset of the CTA's warps (id 1..15; count a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// The same barrier, returning the OR of `pred` over all the participating threads.
__device__ __forceinline__ bool named_bar_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Generic-proxy shared-memory writes -> visible to the async proxy (tensor core reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (fp16/bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on an mbarrier when all previously issued tcgen05.mma of this thread finish.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives lane (base + t).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 32 lanes x 8 consecutive 32-bit columns (same lane mapping as the x32 form).
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------------------
// Thread-block clusters: rank, barrier, and loads from a peer CTA's shared memory
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives, then waits; shared-memory writes before
// the arrive are visible to the cluster's CTAs after the wait.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_u32(uint32_t smem_addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(smem_addr), "r"(v) : "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t cluster_addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
  return v;
}

// Shared-memory matrix descriptor (tcgen05 format), K-major operand with the 128-byte
// swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked along M/N.
//   bits  0-13 start address >> 4
//   bits 16-29 leading-dimension byte offset >> 4 (unused for swizzled K-major; 1)
//   bits 32-45 stride-dimension byte offset >> 4 (1024 B between 8-row groups)
//   bits 46-47 descriptor version (1 on sm_100-family)
//   bits 49-51 base offset (0: atoms are 1024-byte aligned)
//   bits 61-63 layout: 2 = 128-byte swizzle
__device__ __forceinline__ uint64_t make_sw128_kmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B fp16, both K-major, dense.
//   bits 4-5 D format (1 = f32); 7-9 A format (0 = f16); 10-12 B format (0 = f16);
//   15/16 A/B major (0 = K); 17-22 N >> 3; 24-28 M >> 4.
__host__ __device__ constexpr uint32_t make_idesc_f16_f32(uint32_t M, uint32_t N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// ---------------------------------------------------------------------------------------
// dp4a with unsigned a (packed u8 codes) and signed b (packed s8 activations)
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// ---------------------------------------------------------------------------------------
// Single-token projections sharing one activation row (kernel parameter, passed by value)
// ---------------------------------------------------------------------------------------
constexpr int kMaxGroupLinears = 8;
struct LinearSet {
  const uint8_t* wp[kMaxGroupLinears];  // N_l x K/4 packed weights
  float* out[kMaxGroupLinears];         // N_l fp32 outputs
  int32_t* acc[kMaxGroupLinears];       // optional N_l int32 accumulators
  float w_scale[kMaxGroupLinears];
  int N[kMaxGroupLinears];
  int count;
};
struct QuantOut {  // optional outputs of a fused quantisation (each may be null)
  int8_t* xq;
  float* scale;
  int32_t* rowsum;
};
// FFN inner activation ("bitnet.rs" "Forward Pass": inner = ffn_sub_norm(sqrelu(gate) * up)),
// the input row of the FFN's down projection. ffn_sub_norm is an RMSNorm with per-channel
// weight gamma and epsilon eps:
//   h = max(g, 0)^2 * u = (r * r) * u with r = (g > 0 ? g : 0)
//   inner = (h * c) * gamma,  c = 1 / sqrt(ss / F + eps)
// every operation one fp32 rounding. ss = sum of h^2 in a fixed order, so every
// implementation gets the same value: 256 partials, partial p taking the h_k with
// floor(k / 4) mod 256 == p in ascending k, each by one fma; then within each run of 32
// partials the xor butterfly with offsets 16, 8, 4, 2, 1 (the tree adding partial p + d into
// p); then the eight run sums as ((R0 + R1) + (R2 + R3)) + ((R4 + R5) + (R6 + R7)).
struct FfnIn {
  const float* gate;   // F fp32 per row
  const float* up;     // F fp32 per row
  const float* gamma;  // F fp32, shared by all rows
  float eps;
};
__device__ __forceinline__ float ffn_h(float g, float u) {
  const float r = g > 0.0f ? g : 0.0f;
  return __fmul_rn(__fmul_rn(r, r), u);
}
__device__ __forceinline__ float ffn_rms_factor(float ss, int F, float eps) {
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)F), eps)));
}
// the within-run tree of the sum of squares, on one warp's 32 partials (all lanes get it)
__device__ __forceinline__ float ffn_run_sum(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}
__device__ __forceinline__ float ffn_runs_total(const float* r) {
  return __fadd_rn(__fadd_rn(__fadd_rn(r[0], r[1]), __fadd_rn(r[2], r[3])),
                   __fadd_rn(__fadd_rn(r[4], r[5]), __fadd_rn(r[6], r[7])));
}

// One group of the persistent sweep (gemv_sweep.cu): an activation row and the projections
// that consume it. row0 / byte0 are the group's first row and first packed byte in the
// concatenated row space of all groups, rows its row count; log2G and S are the lane layout
// and the steps per tile chosen for K.
struct SweepGroup {
  const void* x;
  int64_t byte0;
  int K, log2G, S, count, row0, rows;
  const uint8_t* wp[kMaxGroupLinears];
  float* out[kMaxGroupLinears];
  float w_scale[kMaxGroupLinears];
  int N[kMaxGroupLinears];
};

constexpr int kMaxPrefetch = 8;
struct Prefetch {  // byte ranges to pull into L2 (a hint; 16-byte aligned starts)
  const void* ptr[kMaxPrefetch];
  int64_t bytes[kMaxPrefetch];
  int count;
};

// ---------------------------------------------------------------------------------------
// Launchers (defined in the kernel translation units). All return cudaError_t of the launch.
// ---------------------------------------------------------------------------------------
// Single-token group step (gemv_group.cu): quantise x (fp32, or bf16 if bf16) and run the
// GEMVs of a LinearSet in one launch; qout optionally written; pf an L2 prefetch hint.
// Launched with programmatic stream serialisation.
bool gemv_group_supported(int64_t K);
cudaError_t launch_gemv_group(const void* x, bool bf16, const LinearSet& set, const QuantOut& qout,
                              const Prefetch& pf, int64_t K, int num_sms, cudaStream_t stream);
// The same kernel with the FFN inner activation as its input row (F = K): the down
// projection of the FFN, fused with the sub-norm and the quantisation.
cudaError_t launch_gemv_group_ffn(const FfnIn& ffn, const LinearSet& set, const QuantOut& qout, const Prefetch& pf,
                                  int64_t F, int num_sms, cudaStream_t stream);
// One CTA's share of the sweep: rows [begin, end) of the concatenated row space, whose first
// row lies in group g0.
struct SweepSlice {
  int begin, end, g0;
};
// Persistent sweep over independent groups (gemv_sweep.cu). groups_dev (n_groups entries) and
// slices_dev (one per CTA, grid = n_slices) are device tables built by the host.
bool gemv_sweep_supported(int64_t K);
void sweep_fill_layout(SweepGroup& g);  // host: log2G and S from K
// host: the slices of n CTAs, balanced by packed bytes; total_rows >= n
void sweep_slices(const SweepGroup* groups, int n_groups, int total_rows, int64_t total_bytes, int n,
                  SweepSlice* slices);
cudaError_t launch_gemv_sweep(const SweepGroup* groups_dev, int n_groups, const SweepSlice* slices_dev, int n_slices,
                              bool bf16, cudaStream_t stream);
cudaError_t read_clear_device_error_sweep(int* value);
// FFN inner activation + per-token quantisation for M rows (ffn.cu); inner_out optional.
constexpr int64_t kFfnMaxF = 32768;
cudaError_t launch_ffn_act_quant(const FfnIn& ffn, int64_t M, int64_t F, int8_t* xq, float* act_scale,
                                 int32_t* rowsum, float* inner_out, cudaStream_t stream);
cudaError_t launch_pack_i2s(const int8_t* w, uint8_t* wp, int64_t N, int64_t K, int32_t* invalid_count,
                            cudaStream_t stream);
cudaError_t launch_quant_act(const void* x, int dtype, int64_t M, int64_t K, int8_t* xq, float* act_scale,
                             int32_t* rowsum, cudaStream_t stream);
cudaError_t launch_gemv_i2s(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                            float w_scale, float* out, int32_t* acc_out, int64_t M, int64_t N, int64_t K,
                            int num_sms, cudaStream_t stream);
// Weight ternarisation + i2_s packing (quant_weight.cu); mode 0 AbsMean, 1 the sign rule.
cudaError_t launch_quant_weight(const void* w, bool bf16, int64_t N, int64_t K, int mode, uint8_t* wp, float* w_scale,
                                int num_sms, cudaStream_t stream);

// Single-token GEMV over a bulk-copy ring (gemv_ring.cu): M = 1, K <= 10240; large matrices.
bool gemv_ring_supported(int64_t M, int64_t K);
cudaError_t launch_gemv_ring(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                             float w_scale, float* out, int32_t* acc_out, int64_t N, int64_t K, int num_sms,
                             cudaStream_t stream);
cudaError_t read_clear_device_error_gemv_ring(int* value);

// Prompt-length tensor-core matmul without a workspace (gemm_prefill.cu): TMA-staged packed
// weights and int8 tokens, expanded to exact fp16 in the kernel; K <= 32768.
bool gemm_prefill_supported(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_prefill(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                                float w_scale, float* out, int32_t* acc_out, int64_t M, int64_t N, int64_t K,
                                int num_sms, cudaStream_t stream);
cudaError_t read_clear_device_error_prefill(int* value);

// Few-token tensor-core matmul (gemm_smallm.cu): any M (64 tokens per CTA), K <= 32768.
bool gemm_smallm_supported(int64_t M, int64_t K);
cudaError_t launch_gemm_smallm(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                               float w_scale, float* out, int32_t* acc_out, int64_t M, int64_t N, int64_t K,
                               int num_sms, cudaStream_t stream);
cudaError_t read_clear_device_error_smallm(int* value);
cudaError_t read_clear_device_error_quant_weight(int* value);
// Read and clear the device error word of each translation unit that waits (synchronous).
cudaError_t read_clear_device_error_gemm(int* value);
cudaError_t read_clear_device_error_gemm_ws(int* value);
cudaError_t read_clear_device_error_gemv_group(int* value);
cudaError_t read_clear_device_error_selftest(int* value);
// Failure-handling self-test (selftest.cu): a bounded wait on a barrier nothing arrives on.
bool selftest_bytes_ok(int64_t bytes);
cudaError_t launch_wait_timeout_selftest(const void* src, int64_t bytes, uint32_t max_polls, uint32_t* report,
                                         cudaStream_t stream);

// Host: encode a 2-D tiled TMA tensor map over a row-major [rows][inner] array
// (gemm_tc_ws.cu). False if the driver entry point is missing or the encoder refuses.
bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner_elems,
                   uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle);

// Expand-then-GEMM path (gemm_tc_ws.cu): workspace bytes, and the launch (K <= 32768).
int64_t gemm_ws_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_tc_ws(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                              float w_scale, float* out, int32_t* acc_out, int64_t M, int64_t N, int64_t K,
                              void* workspace, int num_sms, cudaStream_t stream);
cudaError_t launch_gemm_i2s_tc(const int8_t* xq, const float* act_scale, const int32_t* rowsum,
                               const uint8_t* wp, float w_scale, float* out, int32_t* acc_out, int64_t M,
                               int64_t N, int64_t K, int num_sms, cudaStream_t stream);

}  // namespace bitnet
