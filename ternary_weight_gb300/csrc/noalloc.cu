// noalloc.cu -- the prefill matmul for callers that cannot allocate device memory.
//
// bitnet_i2s_matmul_ws needs a device workspace for the fp16 copies of the weights and the
// activations. Some callers cannot provide one: a plugin inside a host framework that owns
// every byte of device memory through its own allocator and does not let plugins call
// cudaMalloc, or a latency-critical loop that must not call cudaMalloc/cudaFree because those
// calls can synchronise the whole device. bitnet_i2s_matmul_noalloc serves them: it runs the
// same kernels with the workspace taken from a fixed scratch array that is part of this
// library's device image.
//
// The array is a file-scope static __device__ object of kScratchBytes (64 MiB). Every GPU that
// loads the library holds it until the process exits, whether or not the entry point is used.
// Host code cannot use the array's name as a device address (on the host it names a host-side
// stand-in), so the first call on each device, with that device current, asks the runtime for
// the device address with cudaGetSymbolAddress and caches it; make that first call before any
// stream capture. The cache is never invalidated, so a cudaDeviceReset of a device after its
// first call is not supported (the module would be reloaded and the cached address stale). All calls share the one array: calls that overlap on the GPU (on different
// streams, or from several host threads without ordering) race on it. Nothing in it has to
// start at zero -- each call overwrites the part it uses before reading it.
#include "bitnet.h"
#include "bitnet_dev.cuh"

#include <atomic>
#include <cstdint>

namespace bitnet {
namespace {

constexpr int64_t kScratchBytes = 64ll << 20;  // stated maximum: 64 MiB per device
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDev = 64;
std::atomic<void*> g_scratch_ptr[kMaxDev];  // device address of g_scratch, per device

// Device address of the scratch array on the current device (set up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace bitnet

extern "C" BITNET_API int bitnet_i2s_matmul_noalloc(const int8_t* xq, const float* act_scale,
                                                    const int32_t* rowsum, const uint8_t* wp, float w_scale,
                                                    float* out, int32_t* acc_out, int64_t M, int64_t N, int64_t K,
                                                    void* stream) {
  using namespace bitnet;
  if (!xq || !act_scale || !rowsum || !wp || !out) return BITNET_EINVAL;
  if (M < 1 || M > INT32_MAX || N < 1 || N > INT32_MAX || K < 128 || K % 128 != 0 || K > 32768) return BITNET_EINVAL;
  // the scratch has a fixed size: problems that need more are refused before any GPU work
  if (gemm_ws_bytes(M, N, K) > kScratchBytes) return BITNET_EINVAL;
  if (!aligned_to(xq, 16) || !aligned_to(wp, 16) || !aligned_to(act_scale, 4) || !aligned_to(rowsum, 4) ||
      !aligned_to(out, 4) || (acc_out && !aligned_to(acc_out, 4)))
    return BITNET_EALIGN;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return BITNET_EUNSUPPORTED;
  }
  if (major != 10 || minor != 3) return BITNET_EUNSUPPORTED;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return BITNET_ECUDA;
  const cudaError_t e = launch_gemm_tc_ws(xq, act_scale, rowsum, wp, w_scale, out, acc_out, M, N, K, scratch, sms,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BITNET_OK : BITNET_ECUDA;
}
