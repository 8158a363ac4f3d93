// chunk_d64_causal_bf16_mask.cu -- tensor-core chunk kernel, head size 64,
// causal pass with bf16 output, for calls with a sequence-validity mask.
#include "chunk_launch.cuh"

namespace la {
cudaError_t chunk_run_causal_d64_bf16_mask(const chunk::Launch& L, cudaStream_t st) {
    return chunk::Dispatch<64, chunk::kCausal, 1, true>::run(L, st);
}
}  // namespace la
