// selftest.cu -- a diagnostic of the library's failure handling: a bounded wait that runs out.
//
// Every kernel that waits on an mbarrier gives up after a bounded number of polls, records
// BITNET_ETIMEOUT in its device error word, leaves its loops, lets the bulk copies it has in
// flight land, and returns; the host reads the word with bitnet_last_device_error. In a
// correct kernel that path is never taken, so this kernel takes it on purpose, safely:
//  * warp 1, one lane (the producer), issues a real cp.async.bulk copy of `bytes` bytes into
//    shared memory, completing on the mbarrier `landed`;
//  * warp 0 (the consumer) waits on the mbarrier `never`, on which nothing ever arrives, with
//    the caller's small poll limit: the wait runs out, records the timeout and sets the abort
//    flag, exactly as a product kernel's consumer would;
//  * the producer then drains as the product kernels do: a bounded wait on `landed` before it
//    leaves, so no copy can land in the shared memory of an exited CTA;
//  * report[0] = 1 if the consumer gave up, report[1] = 1 if the copy was seen to land,
//    report[2] = the sum of the copied 32-bit words (wrapping), read back from shared memory.
// No trap, no fault and no unbounded loop: the kernel always returns.
#include "bitnet_dev.cuh"

namespace bitnet {
namespace {

constexpr int kSelftestMaxBytes = 16384;

__global__ void __launch_bounds__(64, 1) wait_timeout_kernel(const uint4* __restrict__ src, uint32_t bytes,
                                                             uint32_t max_polls, uint32_t* __restrict__ report) {
  __shared__ __align__(128) uint8_t buf[kSelftestMaxBytes];
  __shared__ __align__(8) uint64_t landed;
  __shared__ __align__(8) uint64_t never;
  __shared__ uint32_t gave_up, arrived;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&landed, 1);
    mbar_init(&never, 1);
    fence_mbar_init();
    gave_up = 0;
    arrived = 0;
  }
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&landed, bytes);
      bulk_copy_g2s(buf, src, bytes, &landed);
      bool dummy = false;  // the drain every producer does before leaving
      arrived = mbar_wait(&landed, 0, &dummy) ? 1u : 0u;
    }
  } else {
    bool abort = false;
    const bool ok = mbar_wait_warp_polls(&never, 0, &abort, max_polls);
    if (lane == 0) gave_up = (!ok && abort) ? 1u : 0u;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t sum = 0;
    if (arrived)
      for (uint32_t i = 0; i < bytes / 4; ++i) sum += reinterpret_cast<const uint32_t*>(buf)[i];
    report[0] = gave_up;
    report[1] = arrived;
    report[2] = sum;
  }
}

}  // namespace

bool selftest_bytes_ok(int64_t bytes) { return bytes >= 16 && bytes <= kSelftestMaxBytes && bytes % 16 == 0; }

cudaError_t launch_wait_timeout_selftest(const void* src, int64_t bytes, uint32_t max_polls, uint32_t* report,
                                         cudaStream_t stream) {
  wait_timeout_kernel<<<1, 64, 0, stream>>>(static_cast<const uint4*>(src), (uint32_t)bytes, max_polls, report);
  return cudaGetLastError();
}

cudaError_t read_clear_device_error_selftest(int* value) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

}  // namespace bitnet
