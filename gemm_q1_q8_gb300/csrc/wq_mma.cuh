// Tensor-core W8A32 / W4A32 group-128 matmuls (wq_mma.cu): the activation split into three bf16 planes in a caller's
// workspace, then one tcgen05 kernel.
#pragma once
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace gq {
size_t wq_mma_workspace_bytes(int T, int K);
// bits 8 or 4; K % 32 == 0, K >= 64; w, x and workspace 16-byte aligned, workspace of
// wq_mma_workspace_bytes(T, K).
cudaError_t launch_wq_mma(int bits, const uint32_t* w, const float* scale, const float* x, float* y, int T, int N,
                          int K, void* workspace, cudaStream_t s);
unsigned error_read_clear_wq_mma();
}  // namespace gq
