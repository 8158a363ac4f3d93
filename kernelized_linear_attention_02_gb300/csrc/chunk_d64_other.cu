// chunk_d64_other.cu -- tensor-core chunk kernel, head size 64: the state
// pass (sequence split, non-causal reduction) and the non-causal read-out.
#include "chunk_launch.cuh"

namespace la {
cudaError_t chunk_run_other_d64(const chunk::Launch& L, cudaStream_t st) {
    if (L.mode == chunk::kState) return chunk::Dispatch<64, chunk::kState, 1>::run(L, st);
    return L.out_bf16 ? chunk::Dispatch<64, chunk::kApply, 1>::run(L, st)
                      : chunk::Dispatch<64, chunk::kApply, 0>::run(L, st);
}
}  // namespace la

