// gemm_pair.h -- host entry points of the CTA-pair prompt-length matmul (gemm_pair.cu).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace bitnet {

// The prompt-length matmul on CTA pairs: tcgen05.mma.cta_group::2, 256 weight rows x 256 tokens
// per pair, packed weights and int8 tokens expanded to exact fp16 in the kernel; K <= 32768.
bool gemm_pair_supported(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_pair(const int8_t* xq, const float* act_scale, const int32_t* rowsum, const uint8_t* wp,
                             float w_scale, float* out, int32_t* acc_out, int64_t M, int64_t N, int64_t K, int num_sms,
                             cudaStream_t stream);
cudaError_t read_clear_device_error_pair(int* value);

}  // namespace bitnet
