// chunk_d128_other_mask.cu -- tensor-core chunk kernel, head size 128: the
// state pass and the non-causal read-out, for calls with a sequence-validity
// mask.
#include "chunk_launch.cuh"

namespace la {
cudaError_t chunk_run_other_d128_mask(const chunk::Launch& L, cudaStream_t st) {
    if (L.mode == chunk::kState) return chunk::Dispatch<128, chunk::kState, 1, true>::run(L, st);
    return L.out_bf16 ? chunk::Dispatch<128, chunk::kApply, 1, true>::run(L, st)
                      : chunk::Dispatch<128, chunk::kApply, 0, true>::run(L, st);
}
}  // namespace la
