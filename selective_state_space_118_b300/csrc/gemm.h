// gemm.h -- the layer's projections: plain bf16 GEMMs on the tensor cores
// through cuBLASLt (the library's only non-hand-written device code).
#pragma once
#include <cuda_runtime.h>

#include <cstddef>

namespace mamba {

// Row-major C (M x N) = A (M x K, rows lda apart) * W^T (W: N x K, the
// nn.Linear weight layout, rows K apart) [+ bias (N)], bf16 in and out, fp32
// accumulation; bias (bf16) may be null.  `ws` is cuBLASLt's scratch.  Returns
// false when cuBLASLt refuses the problem or fails to launch.
bool gemm_bf16(const void* A, int lda, const void* W, const void* bias, void* C, int ldc, long M, int N, int K,
               void* ws, size_t ws_bytes, cudaStream_t stream);

// Scratch cuBLASLt may use per GEMM.
constexpr size_t kGemmWorkspace = 32u << 20;

}  // namespace mamba
