// kernels.h -- launchers of the library's kernels (internal).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace la {

// Devices the per-device caches of the library cover.
constexpr int kMaxDevices = 64;
// Identifier of the CUDA context current on the calling thread, unique for
// the life of the process (cuCtxGetId), or 0 when none is current.  After a
// device reset (cudaDeviceReset) the device gets a new context and so a new
// identifier: the per-device caches of addresses and kernel attributes are
// keyed by it and are rebuilt for the new context.
uint64_t current_context_id();

// CUDA-core recurrence (recurrent.cu): float32 path and uncovered shapes.
size_t recurrent_smem_bytes(const Problem& P);
// Scratch the causal recurrence uses to split a long sequence into segments
// (0: one segment); without it (ws null or too small) it runs unsplit.
size_t recurrent_workspace_bytes(const Problem& P);
cudaError_t recurrent_causal(const Problem& P, const void* q, const void* k, const void* v,
                             const void* decay, const float* S0, const float* Z0, void* y,
                             float* S_out, float* Z_out, cudaStream_t st, void* ws = nullptr,
                             size_t ws_bytes = 0);
cudaError_t recurrent_noncausal(const Problem& P, const void* q, const void* k, const void* v,
                                void* y, float* S_ws, float* Z_ws, cudaStream_t st);
// The delta rules (P.delta): one CTA per stream, token by token.
cudaError_t recurrent_delta(const Problem& P, const void* q, const void* k, const void* v, const void* decay,
                            const void* beta, int beta_per_head, const float* S0, void* y, float* S_out,
                            cudaStream_t st);

// Delta rules in chunk-parallel (WY) form on the tensor cores (delta_chunk.cu):
// bf16 inputs, Dk == Dv == 128, one log decay per kv head.
bool delta_chunk_supported(const Problem& P);
size_t delta_chunk_workspace_bytes(const Problem& P);
cudaError_t delta_chunk_causal(const Problem& P, const void* q, const void* k, const void* v, const void* decay,
                               const void* beta, int beta_per_head, const float* S0, void* y, float* S_out,
                               void* ws, cudaStream_t st);

// The gated rule with one log decay per key dimension in chunk-parallel form on
// the tensor cores (perdim_chunk.cu): bf16 inputs, Dk == Dv == 128.
bool perdim_chunk_supported(const Problem& P);
size_t perdim_chunk_workspace_bytes(const Problem& P);
cudaError_t perdim_chunk_causal(const Problem& P, const void* q, const void* k, const void* v, const void* decay,
                                const float* S0, void* y, float* S_out, void* ws, cudaStream_t st);

// Tensor-core chunk path (chunk_host.cu): bf16 inputs, Dk == Dv in {64, 128}.
bool chunk_supported(const Problem& P);
bool chunk_pointers_ok(const void* q, const void* k, const void* v, const void* y);
size_t chunk_workspace_bytes(const Problem& P, bool causal);
cudaError_t chunk_causal(const Problem& P, const void* q, const void* k, const void* v, const void* decay,
                         const float* S0, const float* Z0, void* y, float* S_out, float* Z_out, void* ws,
                         cudaStream_t st);
cudaError_t chunk_noncausal(const Problem& P, const void* q, const void* k, const void* v, void* y, void* ws,
                            cudaStream_t st);
// Reads (and optionally clears) the error word of the bounded waits; 0 = none.
unsigned chunk_device_error(bool reset);
// The current device's SM count and the device address of that error word
// (0 / nullptr if they cannot be queried).
int device_sm_count();
unsigned* device_error_word();

// Enqueues the bounded-wait self-test (selftest.cu): both wait forms give up
// after limit_us on a barrier nothing completes and set their bits in the
// device error word.
cudaError_t bounded_wait_selftest(uint32_t limit_us, cudaStream_t st);

// Gradients of the causal linear rule (backward.cu).
size_t backward_workspace_bytes(const Problem& P);
cudaError_t backward_causal(const Problem& P, const void* q, const void* k, const void* v, const float* S0,
                            const float* Z0, const void* dy, void* dq, void* dk, void* dv, float* dS0, float* dZ0,
                            void* ws, cudaStream_t st);

// The same gradients in chunk-parallel form on the tensor cores (bwd_chunk.cu):
// bf16 inputs, Dk == Dv in {64, 128}.
bool backward_chunk_supported(const Problem& P);
size_t backward_chunk_workspace_bytes(const Problem& P);
cudaError_t backward_chunk_causal(const Problem& P, const void* q, const void* k, const void* v, const float* S0,
                                  const float* Z0, const void* dy, void* dq, void* dk, void* dv, float* dS0,
                                  float* dZ0, void* ws, cudaStream_t st);

// Decode step (decode.cu).
bool decode_supported(const Problem& P);
cudaError_t decode_step(const Problem& P, const void* q, const void* k, const void* v,
                        const void* decay, float* S, float* Z, void* y, cudaStream_t st);

}  // namespace la
