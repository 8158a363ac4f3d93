// chunk_d64_causal_f32_mask.cu -- tensor-core chunk kernel, head size 64,
// causal pass with f32 output, for calls with a sequence-validity mask.
#include "chunk_launch.cuh"

namespace la {
cudaError_t chunk_run_causal_d64_f32_mask(const chunk::Launch& L, cudaStream_t st) {
    return chunk::Dispatch<64, chunk::kCausal, 0, true>::run(L, st);
}
}  // namespace la
