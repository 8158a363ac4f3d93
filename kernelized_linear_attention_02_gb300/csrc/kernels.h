// kernels.h -- launchers of the library's kernels (internal).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace la {

// CUDA-core recurrence (recurrent.cu): float32 path and uncovered shapes.
size_t recurrent_smem_bytes(const Problem& P);
cudaError_t recurrent_causal(const Problem& P, const void* q, const void* k, const void* v,
                             const void* decay, const float* S0, const float* Z0, void* y,
                             float* S_out, float* Z_out, cudaStream_t st);
cudaError_t recurrent_noncausal(const Problem& P, const void* q, const void* k, const void* v,
                                void* y, float* S_ws, float* Z_ws, cudaStream_t st);

// Decode step (decode.cu).
bool decode_supported(const Problem& P);
cudaError_t decode_step(const Problem& P, const void* q, const void* k, const void* v,
                        const void* decay, float* S, float* Z, void* y, cudaStream_t st);

}  // namespace la
