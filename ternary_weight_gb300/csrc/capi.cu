// capi.cu -- the extern "C" boundary of libbitnet_gb300 (declared in include/bitnet.h).
//
// Every entry point validates its arguments on the host before anything is launched and
// returns a status code; no C++ exception crosses the ABI. Device-side state: one error word
// per kernel translation unit (written by bounded waits), the 64 MiB scratch array of
// noalloc.cu (part of the device image, resident on every GPU that loads the library), and
// the device table of each sweep plan, the one cudaMalloc the library makes (in
// bitnet_sweep_plan_create, freed by bitnet_sweep_plan_destroy).
#include "bitnet.h"
#include "bitnet_dev.cuh"
#include "gemm_pair.h"

#include <cmath>
#include <new>
#include <vector>

#include <atomic>
#include <cstdint>

namespace bitnet {
namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxK = 1 << 16;          // staged activation rows must fit shared memory
constexpr int64_t kMaxKTensorCore = 1 << 15; // exact fp32 accumulation bound of the GEMM
// auto dispatch: the few-token tensor-core kernel from this many rows on. The dp4a GEMV's cost
// grows with the rows (every weight word is decoded once per row); the tensor-core kernel's is
// flat up to 16 rows. Measured (N x K = 6912 x 2560, 2560 x 6912, 2560 x 2560, 28672 x 8192):
// the persistent few-row GEMV (K <= 10240) wins up to 4 rows (4 rows: 6.2 against 7.6 us at
// 6912 x 2560) and loses from 5 (9.2 against 7.6 us; 9 rows 16.9 against 7.6). Past K = 10240
// the plain GEMV takes over and loses from 3 rows (8192 x 28672: 48.4 against 39.5 us).
constexpr int64_t kSmallmMinM = 5;           // K <= 10240
constexpr int64_t kSmallmMinMLongK = 3;      // K > 10240
// auto dispatch: the CTA-pair prompt-length kernel beyond one 64-token chunk of the few-token
// kernel. Measured per call, us (N x K = 6912 x 2560 / 2560 x 6912; few-token chunks, one-CTA
// prompt-length kernel, CTA-pair kernel): M = 64: 11.1 / 12.0, 13.6 / 16.4, 12.7 / 13.6;
// M = 96: 14.3 / 14.9, 13.7 / 16.5, 12.7 / 13.6; M = 128: 14.5 / 15.0, 14.0 / 16.7, 12.8 / 13.7;
// M = 192: 27.9 / 18.7, 19.0 / 18.7, 15.9 / 17.2; M = 512: 43.2 / 56.3, 25.2 / 25.8, 21.1 / 21.7;
// M = 4096: 329 / 256, 151 / 164, 127 / 130. The one-CTA kernel stays available when forced.
constexpr int64_t kPairMinM = 65;

// per-device: 0 = unchecked, 1 = sm_103 ok, -1 = unsupported; and SM count
std::atomic<int> g_dev_state[kMaxDevices];
std::atomic<int> g_dev_sms[kMaxDevices];

int check_device(int* num_sms) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return BITNET_EUNSUPPORTED;
  }
  int st = g_dev_state[dev].load(std::memory_order_acquire);
  if (st == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return BITNET_EUNSUPPORTED;
    }
    st = (major == 10 && minor == 3) ? 1 : -1;
    g_dev_sms[dev].store(sms, std::memory_order_relaxed);
    g_dev_state[dev].store(st, std::memory_order_release);
  }
  if (st != 1) return BITNET_EUNSUPPORTED;
  if (num_sms) *num_sms = g_dev_sms[dev].load(std::memory_order_relaxed);
  return BITNET_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int status_of(cudaError_t e) { return e == cudaSuccess ? BITNET_OK : BITNET_ECUDA; }

bool valid_k(int64_t K) { return K >= 128 && K % 128 == 0 && K <= kMaxK; }

}  // namespace
}  // namespace bitnet

using namespace bitnet;

extern "C" {

BITNET_API int bitnet_version(void) { return 100; }

BITNET_API const char* bitnet_strerror(int status) {
  switch (status) {
    case BITNET_OK: return "ok";
    case BITNET_EINVAL: return "invalid argument (null pointer, size out of range, K not a multiple of 128, bad enum)";
    case BITNET_EALIGN: return "misaligned pointer (16-byte alignment required)";
    case BITNET_ECUDA: return "CUDA runtime error or kernel launch failure";
    case BITNET_EUNSUPPORTED: return "unsupported device (an sm_103 / GB300 GPU is required)";
    case BITNET_ETIMEOUT: return "a device-side bounded wait timed out; results are invalid";
    case BITNET_ERANGE: return "an input value outside the operation's supported range (found on the device)";
    default: return "unknown status";
  }
}

BITNET_API int bitnet_pack_i2s(const int8_t* w, uint8_t* wp, int64_t N, int64_t K, int32_t* invalid_count,
                               void* stream) {
  if (!w || !wp || N < 1 || N > INT32_MAX || !valid_k(K)) return BITNET_EINVAL;
  if (!aligned(w, 16) || !aligned(wp, 16) || (invalid_count && !aligned(invalid_count, 4))) return BITNET_EALIGN;
  int sms = 0;
  if (int st = check_device(&sms)) return st;
  return status_of(launch_pack_i2s(w, wp, N, K, invalid_count, static_cast<cudaStream_t>(stream)));
}

BITNET_API int bitnet_quant_act(const void* x, int dtype, int64_t M, int64_t K, int8_t* xq, float* act_scale,
                                int32_t* rowsum, void* stream) {
  if (!x || !xq || !act_scale || !rowsum) return BITNET_EINVAL;
  if (dtype != BITNET_F32 && dtype != BITNET_BF16) return BITNET_EINVAL;
  if (M < 1 || M > INT32_MAX || !valid_k(K)) return BITNET_EINVAL;
  if (!aligned(x, 16) || !aligned(xq, 16) || !aligned(act_scale, 4) || !aligned(rowsum, 4)) return BITNET_EALIGN;
  int sms = 0;
  if (int st = check_device(&sms)) return st;
  return status_of(launch_quant_act(x, dtype, M, K, xq, act_scale, rowsum, static_cast<cudaStream_t>(stream)));
}

BITNET_API int bitnet_quant_weight(const void* w, int dtype, int mode, int64_t N, int64_t K, uint8_t* wp,
                                   float* w_scale, void* stream) {
  if (!w || !wp || !w_scale) return BITNET_EINVAL;
  if (dtype != BITNET_F32 && dtype != BITNET_BF16) return BITNET_EINVAL;
  if (mode != BITNET_QW_ABSMEAN && mode != BITNET_QW_SIGN) return BITNET_EINVAL;
  if (N < 1 || !valid_k(K) || N > (int64_t(1) << 40) / K) return BITNET_EINVAL;
  if (!aligned(w, 16) || !aligned(wp, 16) || !aligned(w_scale, 4)) return BITNET_EALIGN;
  int sms = 0;
  if (int st = check_device(&sms)) return st;
  return status_of(launch_quant_weight(w, dtype == BITNET_BF16, N, K, mode, wp, w_scale, sms,
                                       static_cast<cudaStream_t>(stream)));
}

BITNET_API int bitnet_i2s_matmul_algo(const int8_t* xq, const float* act_scale, const int32_t* rowsum,
                                      const uint8_t* wp, float w_scale, float* out, int32_t* acc_out, int64_t M,
                                      int64_t N, int64_t K, int algo, void* stream) {
  if (!xq || !act_scale || !rowsum || !wp || !out) return BITNET_EINVAL;
  if (M < 1 || M > INT32_MAX || N < 1 || N > INT32_MAX || !valid_k(K)) return BITNET_EINVAL;
  if (algo < BITNET_ALGO_AUTO || algo > BITNET_ALGO_PREFILL_PAIR) return BITNET_EINVAL;
  if (!aligned(xq, 16) || !aligned(wp, 16) || !aligned(act_scale, 4) || !aligned(rowsum, 4) || !aligned(out, 4) ||
      (acc_out && !aligned(acc_out, 4)))
    return BITNET_EALIGN;
  if (algo == BITNET_ALGO_AUTO) {
    // dp4a GEMV for a few tokens (it decodes each weight word once per token row, cheap while
    // the rows are few); from 5 rows (3 past K = 10240) the few-token tensor-core kernel, which
    // decodes each weight once for up to 64 rows; beyond 64 rows the CTA-pair prompt-length
    // kernel (256 weight rows x 128 or 256 tokens per pair of CTAs). The one-CTA prompt-length
    // kernel and the in-kernel-expansion tile GEMM stay available when forced.
    const int64_t smallm_from = K > 10240 ? kSmallmMinMLongK : kSmallmMinM;
    if (K > kMaxKTensorCore || M < smallm_from)
      algo = BITNET_ALGO_GEMV;
    else if (M >= kPairMinM && gemm_pair_supported(M, N, K))
      algo = BITNET_ALGO_PREFILL_PAIR;
    else
      algo = BITNET_ALGO_SMALLM;
  }
  if (algo == BITNET_ALGO_GEMM && (K > kMaxKTensorCore || M > 65535LL * 128)) return BITNET_EINVAL;
  if (algo == BITNET_ALGO_GEMV && M > 65535LL * 8) return BITNET_EINVAL;
  if (algo == BITNET_ALGO_SMALLM && !gemm_smallm_supported(M, K)) return BITNET_EINVAL;
  if (algo == BITNET_ALGO_PREFILL && !gemm_prefill_supported(M, N, K)) return BITNET_EINVAL;
  if (algo == BITNET_ALGO_PREFILL_PAIR && !gemm_pair_supported(M, N, K)) return BITNET_EINVAL;
  int sms = 0;
  if (int st = check_device(&sms)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (algo) {
    case BITNET_ALGO_GEMV:
      e = launch_gemv_i2s(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, sms, s);
      break;
    case BITNET_ALGO_SMALLM:
      e = launch_gemm_smallm(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, sms, s);
      break;
    case BITNET_ALGO_PREFILL:
      e = launch_gemm_prefill(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, sms, s);
      break;
    case BITNET_ALGO_PREFILL_PAIR:
      e = launch_gemm_pair(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, sms, s);
      break;
    default:
      e = launch_gemm_i2s_tc(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, sms, s);
  }
  return status_of(e);
}

BITNET_API int64_t bitnet_i2s_matmul_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || M > INT32_MAX || N < 1 || N > INT32_MAX || !valid_k(K) || K > kMaxKTensorCore) return BITNET_EINVAL;
  return gemm_ws_bytes(M, N, K);
}

BITNET_API int bitnet_i2s_matmul_ws(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                                    float w_scale, float* out, int32_t* acc_out, int64_t M, int64_t N, int64_t K,
                                    void* workspace, int64_t workspace_bytes, void* stream) {
  if (!xq || !act_scale || !rowsum || !wp || !out || !workspace) return BITNET_EINVAL;
  if (M < 1 || M > INT32_MAX || N < 1 || N > INT32_MAX || !valid_k(K) || K > kMaxKTensorCore) return BITNET_EINVAL;
  if (workspace_bytes < gemm_ws_bytes(M, N, K)) return BITNET_EINVAL;
  if (!aligned(xq, 16) || !aligned(wp, 16) || !aligned(act_scale, 4) || !aligned(rowsum, 4) || !aligned(out, 4) ||
      (acc_out && !aligned(acc_out, 4)) || !aligned(workspace, 256))
    return BITNET_EALIGN;
  int sms = 0;
  if (int st = check_device(&sms)) return st;
  return status_of(launch_gemm_tc_ws(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, workspace, sms,
                                     static_cast<cudaStream_t>(stream)));
}

BITNET_API int bitnet_i2s_matmul(const int8_t* xq, const float* act_scale, const int32_t* rowsum,
                                 const uint8_t* wp, float w_scale, float* out, int32_t* acc_out, int64_t M,
                                 int64_t N, int64_t K, void* stream) {
  return bitnet_i2s_matmul_algo(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, BITNET_ALGO_AUTO,
                                stream);
}

BITNET_API int bitnet_w2a8_linear_group_ex(const void* x, int dtype, int64_t M, int64_t K, int count,
                                           const uint8_t* const* wp, const float* w_scale, const int64_t* N,
                                           float* const* out, int32_t* const* acc_out, int8_t* xq, float* act_scale,
                                           int32_t* rowsum, int prefetch_count, const void* const* prefetch_ptr,
                                           const int64_t* prefetch_bytes, void* stream) {
  if (!x || !wp || !w_scale || !N || !out) return BITNET_EINVAL;
  if (dtype != BITNET_F32 && dtype != BITNET_BF16) return BITNET_EINVAL;
  if (count < 1 || count > kMaxGroupLinears) return BITNET_EINVAL;
  if (M < 1 || M > INT32_MAX || !valid_k(K)) return BITNET_EINVAL;
  if (prefetch_count < 0 || prefetch_count > kMaxPrefetch) return BITNET_EINVAL;
  if (prefetch_count > 0 && (!prefetch_ptr || !prefetch_bytes)) return BITNET_EINVAL;
  if (!aligned(x, 16)) return BITNET_EALIGN;
  for (int l = 0; l < count; ++l) {
    if (!wp[l] || !out[l] || N[l] < 1 || N[l] > INT32_MAX) return BITNET_EINVAL;
    if (!aligned(wp[l], 16) || !aligned(out[l], 4) || (acc_out && acc_out[l] && !aligned(acc_out[l], 4)))
      return BITNET_EALIGN;
  }
  Prefetch pf{};
  for (int p = 0; p < prefetch_count; ++p) {
    if (!prefetch_ptr[p] || prefetch_bytes[p] < 0) return BITNET_EINVAL;
    if (!aligned(prefetch_ptr[p], 16)) return BITNET_EALIGN;
    pf.ptr[p] = prefetch_ptr[p];
    pf.bytes[p] = prefetch_bytes[p];
  }
  pf.count = prefetch_count;
  int64_t total_rows = 0;
  for (int l = 0; l < count; ++l) total_rows += N[l];
  const bool single_launch = (M == 1 && gemv_group_supported(K) && total_rows <= INT32_MAX);
  if (!single_launch && (!xq || !act_scale || !rowsum)) return BITNET_EINVAL;
  if ((xq && !aligned(xq, 16)) || (act_scale && !aligned(act_scale, 4)) || (rowsum && !aligned(rowsum, 4)))
    return BITNET_EALIGN;
  int sms = 0;
  if (int st = check_device(&sms)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (single_launch) {
    LinearSet set{};
    for (int l = 0; l < count; ++l) {
      set.wp[l] = wp[l];
      set.out[l] = out[l];
      set.acc[l] = acc_out ? acc_out[l] : nullptr;
      set.w_scale[l] = w_scale[l];
      set.N[l] = (int)N[l];
    }
    set.count = count;
    return status_of(launch_gemv_group(x, dtype == BITNET_BF16, set, QuantOut{xq, act_scale, rowsum}, pf, K, sms, s));
  }
  if (cudaError_t e = launch_quant_act(x, dtype, M, K, xq, act_scale, rowsum, s)) return status_of(e);
  for (int l = 0; l < count; ++l) {
    int st = bitnet_i2s_matmul_algo(xq, act_scale, rowsum, wp[l], w_scale[l], out[l], acc_out ? acc_out[l] : nullptr,
                                    M, N[l], K, BITNET_ALGO_AUTO, stream);
    if (st != BITNET_OK) return st;
  }
  return BITNET_OK;
}

BITNET_API int bitnet_w2a8_linear_group(const void* x, int dtype, int64_t M, int64_t K, int count,
                                        const uint8_t* const* wp, const float* w_scale, const int64_t* N,
                                        float* const* out, int32_t* const* acc_out, int8_t* xq, float* act_scale,
                                        int32_t* rowsum, void* stream) {
  return bitnet_w2a8_linear_group_ex(x, dtype, M, K, count, wp, w_scale, N, out, acc_out, xq, act_scale, rowsum, 0,
                                     nullptr, nullptr, stream);
}

BITNET_API int bitnet_w2a8_linear(const void* x, int dtype, int64_t M, int64_t K, const uint8_t* wp, float w_scale,
                                  int64_t N, float* out, int32_t* acc_out, int8_t* xq, float* act_scale,
                                  int32_t* rowsum, void* stream) {
  int32_t* accs[1] = {acc_out};
  return bitnet_w2a8_linear_group(x, dtype, M, K, 1, &wp, &w_scale, &N, &out, accs, xq, act_scale, rowsum, stream);
}

BITNET_API int bitnet_ffn_act_quant(const float* gate, const float* up, const float* gamma, float eps, int64_t M,
                                    int64_t F, int8_t* xq, float* act_scale, int32_t* rowsum, float* inner_out,
                                    void* stream) {
  if (!gate || !up || !gamma || !xq || !act_scale || !rowsum) return BITNET_EINVAL;
  if (M < 1 || M > INT32_MAX || !valid_k(F) || F > kFfnMaxF) return BITNET_EINVAL;
  if (!(eps > 0.0f) || !std::isfinite(eps)) return BITNET_EINVAL;
  if (!aligned(gate, 16) || !aligned(up, 16) || !aligned(gamma, 16) || !aligned(xq, 16) || !aligned(act_scale, 4) ||
      !aligned(rowsum, 4) || (inner_out && !aligned(inner_out, 16)))
    return BITNET_EALIGN;
  int sms = 0;
  if (int st = check_device(&sms)) return st;
  return status_of(launch_ffn_act_quant(FfnIn{gate, up, gamma, eps}, M, F, xq, act_scale, rowsum, inner_out,
                                        static_cast<cudaStream_t>(stream)));
}

namespace {
bool valid_ffn_shape(int64_t M, int64_t K, int64_t F) {
  return M >= 1 && M <= INT32_MAX && valid_k(K) && valid_k(F) && F <= kFfnMaxF;
}
// Workspace the FFN block uses: none. Its projections take the workspace-free kernels of auto
// dispatch at every M: the CTA-pair prompt-length kernel measured faster than the expand-once
// workspace path at every size tried (per projection, N x K = 6912 x 2560 / 2560 x 6912: M = 1024
// 41.7 / 44.0 against 52.6 / 58.0 us, M = 2048 63.9 / 86.0 against 82.9 / 94.5, M = 4096 127 /
// 130 against 145 / 151, M = 8192 252 / 218 against 269 / 272).
int64_t ffn_ws_bytes(int64_t, int64_t, int64_t) { return 0; }
}  // namespace

BITNET_API int64_t bitnet_w2a8_ffn_workspace_size(int64_t M, int64_t K, int64_t F) {
  if (!valid_ffn_shape(M, K, F)) return BITNET_EINVAL;
  return ffn_ws_bytes(M, K, F);
}

BITNET_API int bitnet_w2a8_ffn(const void* x, int dtype, int64_t M, int64_t K, int64_t F, const uint8_t* wp_gate,
                               float a_gate, const uint8_t* wp_up, float a_up, const uint8_t* wp_down, float a_down,
                               const float* gamma, float eps, float* gate_out, float* up_out, float* out, int8_t* xq,
                               float* act_scale, int32_t* rowsum, void* workspace, int64_t workspace_bytes,
                               void* stream) {
  if (!x || !wp_gate || !wp_up || !wp_down || !gamma || !gate_out || !up_out || !out) return BITNET_EINVAL;
  if (dtype != BITNET_F32 && dtype != BITNET_BF16) return BITNET_EINVAL;
  if (!valid_ffn_shape(M, K, F)) return BITNET_EINVAL;
  if (!(eps > 0.0f) || !std::isfinite(eps)) return BITNET_EINVAL;
  const bool single = M == 1 && gemv_group_supported(K) && gemv_group_supported(F);
  if (!single && (!xq || !act_scale || !rowsum)) return BITNET_EINVAL;
  const int64_t ws_need = ffn_ws_bytes(M, K, F);
  if (workspace && workspace_bytes < ws_need) return BITNET_EINVAL;
  if (!aligned(x, 16) || !aligned(wp_gate, 16) || !aligned(wp_up, 16) || !aligned(wp_down, 16) ||
      !aligned(gamma, 16) || !aligned(gate_out, 16) || !aligned(up_out, 16) || !aligned(out, 4))
    return BITNET_EALIGN;
  if ((xq && !aligned(xq, 16)) || (act_scale && !aligned(act_scale, 4)) || (rowsum && !aligned(rowsum, 4)) ||
      (workspace && !aligned(workspace, 256)))
    return BITNET_EALIGN;
  int sms = 0;
  if (int st = check_device(&sms)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const FfnIn ffn{gate_out, up_out, gamma, eps};
  if (single) {
    // two launches: the gate/up group (quantising x), then the down projection whose input
    // row is the sub-normed, quantised inner activation computed in its own prologue
    LinearSet gu{};
    gu.wp[0] = wp_gate, gu.wp[1] = wp_up;
    gu.out[0] = gate_out, gu.out[1] = up_out;
    gu.w_scale[0] = a_gate, gu.w_scale[1] = a_up;
    gu.N[0] = gu.N[1] = (int)F;
    gu.count = 2;
    if (cudaError_t e = launch_gemv_group(x, dtype == BITNET_BF16, gu, QuantOut{}, Prefetch{}, K, sms, s))
      return status_of(e);
    LinearSet dn{};
    dn.wp[0] = wp_down;
    dn.out[0] = out;
    dn.w_scale[0] = a_down;
    dn.N[0] = (int)K;
    dn.count = 1;
    return status_of(launch_gemv_group_ffn(ffn, dn, QuantOut{xq, act_scale, rowsum}, Prefetch{}, F, sms, s));
  }
  auto matmul = [&](const uint8_t* wp, float a, float* o, int64_t N, int64_t Kd) -> int {
    return bitnet_i2s_matmul_algo(xq, act_scale, rowsum, wp, a, o, nullptr, M, N, Kd, BITNET_ALGO_AUTO, stream);
  };
  if (cudaError_t e = launch_quant_act(x, dtype, M, K, xq, act_scale, rowsum, s)) return status_of(e);
  if (int st = matmul(wp_gate, a_gate, gate_out, F, K)) return st;
  if (int st = matmul(wp_up, a_up, up_out, F, K)) return st;
  if (cudaError_t e = launch_ffn_act_quant(ffn, M, F, xq, act_scale, rowsum, nullptr, s)) return status_of(e);
  return matmul(wp_down, a_down, out, K, F);
}

// ---- the persistent sweep: a plan owns device copies of the group table and of the per-CTA
// slices (built once on the host) ----
struct bitnet_sweep_plan_s {
  bitnet::SweepGroup* table;   // device, n_groups entries
  bitnet::SweepSlice* slices;  // device, n_slices entries (one per CTA)
  int n_groups;
  int n_slices;
  int dtype;
  int device;
};

BITNET_API int bitnet_sweep_plan_create(const bitnet_linear_group* groups, int n_groups, int dtype,
                                        bitnet_sweep_plan* plan) {
  if (!plan) return BITNET_EINVAL;
  *plan = nullptr;
  if (!groups || n_groups < 1 || n_groups > (1 << 20)) return BITNET_EINVAL;
  if (dtype != BITNET_F32 && dtype != BITNET_BF16) return BITNET_EINVAL;
  std::vector<SweepGroup> host((size_t)n_groups);
  int64_t rows = 0, bytes = 0;
  for (int g = 0; g < n_groups; ++g) {
    const bitnet_linear_group& in = groups[g];
    if (!in.x || in.count < 1 || in.count > kMaxGroupLinears) return BITNET_EINVAL;
    if (!valid_k(in.K) || !gemv_sweep_supported(in.K)) return BITNET_EINVAL;
    if (!aligned(in.x, 16)) return BITNET_EALIGN;
    SweepGroup& out = host[(size_t)g];
    out = SweepGroup{};
    out.x = in.x;
    out.K = (int)in.K;
    out.count = in.count;
    out.row0 = (int)rows;
    out.byte0 = bytes;
    for (int l = 0; l < in.count; ++l) {
      if (!in.wp[l] || !in.out[l] || in.N[l] < 1 || in.N[l] > INT32_MAX) return BITNET_EINVAL;
      if (!aligned(in.wp[l], 16) || !aligned(in.out[l], 4)) return BITNET_EALIGN;
      out.wp[l] = in.wp[l];
      out.out[l] = in.out[l];
      out.w_scale[l] = in.w_scale[l];
      out.N[l] = (int)in.N[l];
      rows += in.N[l];
      if (rows > INT32_MAX) return BITNET_EINVAL;
    }
    out.rows = (int)(rows - out.row0);
    bytes += (int64_t)out.rows * (in.K / 4);
    sweep_fill_layout(out);
  }
  int sms = 0;
  if (int st = check_device(&sms)) return st;
  // one CTA per SM (fewer if there are fewer rows), each with a byte-balanced slice
  const int n_slices = (int)(rows < sms ? rows : sms);
  std::vector<SweepSlice> slices((size_t)n_slices);
  sweep_slices(host.data(), n_groups, (int)rows, bytes, n_slices, slices.data());
  auto* p = new (std::nothrow) bitnet_sweep_plan_s{};
  if (!p) return BITNET_ECUDA;
  const size_t tb = sizeof(SweepGroup) * (size_t)n_groups, sb = sizeof(SweepSlice) * (size_t)n_slices;
  const bool ok = cudaGetDevice(&p->device) == cudaSuccess &&
                  cudaMalloc(reinterpret_cast<void**>(&p->table), tb) == cudaSuccess &&
                  cudaMalloc(reinterpret_cast<void**>(&p->slices), sb) == cudaSuccess &&
                  cudaMemcpy(p->table, host.data(), tb, cudaMemcpyHostToDevice) == cudaSuccess &&
                  cudaMemcpy(p->slices, slices.data(), sb, cudaMemcpyHostToDevice) == cudaSuccess;
  if (!ok) {
    cudaFree(p->table);
    cudaFree(p->slices);
    delete p;
    return BITNET_ECUDA;
  }
  p->n_groups = n_groups;
  p->n_slices = n_slices;
  p->dtype = dtype;
  *plan = p;
  return BITNET_OK;
}

BITNET_API int bitnet_sweep_plan_run(bitnet_sweep_plan plan, void* stream) {
  if (!plan) return BITNET_EINVAL;
  int sms = 0;
  if (int st = check_device(&sms)) return st;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return BITNET_ECUDA;
  if (dev != plan->device) return BITNET_EINVAL;
  return status_of(launch_gemv_sweep(plan->table, plan->n_groups, plan->slices, plan->n_slices,
                                     plan->dtype == BITNET_BF16, static_cast<cudaStream_t>(stream)));
}

BITNET_API int bitnet_sweep_plan_destroy(bitnet_sweep_plan plan) {
  if (!plan) return BITNET_OK;
  const cudaError_t e1 = cudaFree(plan->table);
  const cudaError_t e2 = cudaFree(plan->slices);
  delete plan;
  return e1 == cudaSuccess && e2 == cudaSuccess ? BITNET_OK : BITNET_ECUDA;
}

BITNET_API int bitnet_selftest_wait_timeout(const void* src, int64_t bytes, int32_t max_polls, uint32_t* report,
                                            void* stream) {
  if (!src || !report || !selftest_bytes_ok(bytes) || max_polls < 1 || max_polls > (1 << 20)) return BITNET_EINVAL;
  if (!aligned(src, 16) || !aligned(report, 4)) return BITNET_EALIGN;
  int sms = 0;
  if (int st = check_device(&sms)) return st;
  return status_of(launch_wait_timeout_selftest(src, bytes, (uint32_t)max_polls, report,
                                                static_cast<cudaStream_t>(stream)));
}

BITNET_API int bitnet_last_device_error(void) {
  int sms = 0;
  if (int st = check_device(&sms)) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return BITNET_ECUDA;
  int status = BITNET_OK;
  cudaError_t (*readers[])(int*) = {read_clear_device_error_gemm, read_clear_device_error_gemm_ws,
                                    read_clear_device_error_gemv_group, read_clear_device_error_smallm,
                                    read_clear_device_error_quant_weight, read_clear_device_error_sweep,
                                    read_clear_device_error_gemv_ring, read_clear_device_error_selftest,
                                    read_clear_device_error_prefill, read_clear_device_error_pair};
  for (auto rd : readers) {
    int v = 0;
    if (rd(&v) != cudaSuccess) return BITNET_ECUDA;
    if (v != 0 && status == BITNET_OK) status = v;
  }
  return status;
}

}  // extern "C"
