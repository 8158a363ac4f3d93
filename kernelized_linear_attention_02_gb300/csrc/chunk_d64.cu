// chunk_d64.cu -- tensor-core chunk kernel, head size 64.
#include "chunk_launch.cuh"

namespace la {
cudaError_t chunk_run_d64(const chunk::Launch& L, cudaStream_t st) { return chunk::run_d<64>(L, st); }
}  // namespace la

#ifdef LA_TRACE
LA_TRACE_DUMP(la_trace_dump_d64)
#endif
