// chunk_d64_causal_bf16.cu -- tensor-core chunk kernel, head size 64,
// causal pass with bf16 output.
#include "chunk_launch.cuh"

namespace la {
cudaError_t chunk_run_causal_d64_bf16(const chunk::Launch& L, cudaStream_t st) {
    return chunk::Dispatch<64, chunk::kCausal, 1>::run(L, st);
}
}  // namespace la

