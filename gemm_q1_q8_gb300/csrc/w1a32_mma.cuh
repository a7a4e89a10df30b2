// Tensor-core W1A32 prefill (prefill_mma.cu): the f32 activations split exactly into three bf16
// planes (32-block elements interleaved, the prefill MMA operand's order) in a caller's
// workspace, then the prefill MMA kernel with those planes as its activation operand.
#pragma once
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace gq {
size_t w1a32_mma_workspace_bytes(int M, int K);
// K % 64 == 0; x 4-byte aligned; workspace 16-byte aligned, w1a32_mma_workspace_bytes(M, K) bytes;
// signs 16-byte and wscale 8-byte aligned.
cudaError_t launch_w1a32_mma(const uint32_t* signs, const float* ws, const float* x, float* y, int M, int N, int K,
                             void* workspace, cudaStream_t s);
}  // namespace gq
